"""Paged grouped-query attention at head_dim 512 for GB300 (sm_103a): Python binding.

This module only marshals arguments into the C ABI of ``libpaged_attn.so`` (declared in
include/paged_attn.h); every step of the computation runs in the library's CUDA kernels.
Tensors must already live on the GPU.  If the library has not been built, the calls raise
instead of falling back to anything else.

    out, lse = paged_attn_decode(q, kv_cache, kv_indptr, kv_indices, kv_last_page_len,
                                 num_kv_heads=4, head_dim_vo=512, page_size=64,
                                 sm_scale=512 ** -0.5)
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libpaged_attn.so")

PA_KV_BF16, PA_KV_FP8_E4M3, PA_KV_NVFP4 = 0, 1, 2
PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_ALIGNMENT = 0, -1, -2, -3
PA_ERR_SMEM, PA_ERR_CUDA, PA_ERR_DEVICE, PA_ERR_SCRATCH = -4, -5, -6, -7
PA_NOALLOC_SCRATCH_BYTES = 32 << 20

# every symbol include/paged_attn.h declares
EXPORTED = ("paged_attn_decode", "paged_attn_prefill", "paged_attn_status_string",
            "paged_attn_release_workspace", "paged_attn_check_device_error",
            "paged_attn_set_decode_chunk_pages", "paged_attn_set_decode_direct", "paged_attn_last_variant",
            "paged_attn_profile_begin", "paged_attn_profile_end", "paged_attn_decode_noalloc",
            "paged_attn_set_prefill_dequant_limit", "paged_attn_set_prefill_cta_pairs",
            "paged_attn_append_kv", "paged_attn_prefill_custom_mask", "paged_attn_set_prefill_split_kv",
            "paged_attn_debug_set_error_word")

_lib = None


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {paged_attn_status_string(status)} (status {status})")


class _Scales(ctypes.Structure):
    _fields_ = [("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("sf", ctypes.c_void_p)]


def load(path: Optional[str] = None):
    """Load libpaged_attn.so (build it with ``python -m paged_gqa_attention_hd512_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing")
    lib = ctypes.CDLL(p)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.paged_attn_decode.restype = i32
    lib.paged_attn_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                      i32, ctypes.POINTER(_Scales), vp, vp, vp]
    lib.paged_attn_decode_noalloc.restype = i32
    lib.paged_attn_decode_noalloc.argtypes = list(lib.paged_attn_decode.argtypes)
    lib.paged_attn_prefill.restype = i32
    lib.paged_attn_prefill.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                       f32, i32, i32, i32, ctypes.POINTER(_Scales), vp, vp, vp]
    lib.paged_attn_append_kv.restype = i32
    lib.paged_attn_append_kv.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                         vp, vp, vp, vp]
    lib.paged_attn_prefill_custom_mask.restype = i32
    lib.paged_attn_prefill_custom_mask.argtypes = list(lib.paged_attn_prefill.argtypes[:-1]) + [vp, vp, vp]
    lib.paged_attn_status_string.restype = ctypes.c_char_p
    lib.paged_attn_status_string.argtypes = [i32]
    lib.paged_attn_release_workspace.restype = i32
    lib.paged_attn_check_device_error.restype = i32
    lib.paged_attn_check_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.paged_attn_debug_set_error_word.restype = i32
    lib.paged_attn_debug_set_error_word.argtypes = [i32, i32]
    lib.paged_attn_set_decode_chunk_pages.restype = i32
    lib.paged_attn_set_decode_chunk_pages.argtypes = [i32]
    lib.paged_attn_set_decode_direct.restype = i32
    lib.paged_attn_set_decode_direct.argtypes = [i32]
    lib.paged_attn_set_prefill_dequant_limit.restype = i32
    lib.paged_attn_set_prefill_dequant_limit.argtypes = [ctypes.c_longlong]
    lib.paged_attn_set_prefill_cta_pairs.restype = i32
    lib.paged_attn_set_prefill_cta_pairs.argtypes = [i32]
    lib.paged_attn_set_prefill_split_kv.restype = i32
    lib.paged_attn_set_prefill_split_kv.argtypes = [i32]
    lib.paged_attn_last_variant.restype = i32
    lib.paged_attn_last_variant.argtypes = [ctypes.c_char_p, i32]
    lib.paged_attn_profile_begin.restype = i32
    lib.paged_attn_profile_begin.argtypes = [i32]
    lib.paged_attn_profile_end.restype = i32
    lib.paged_attn_profile_end.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float)]
    if path is None:
        _lib = lib
    return lib


def paged_attn_status_string(status: int) -> str:
    return load().paged_attn_status_string(status).decode()


def _ptr(t: Optional[torch.Tensor]):
    """The device address of a contiguous CUDA tensor (an int; ctypes passes it as a
    pointer), None for None."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _x2(kv_dtype: int) -> int:
    return {PA_KV_BF16: 4, PA_KV_FP8_E4M3: 2, PA_KV_NVFP4: 1}[kv_dtype]


def _scales(kv_dtype, k_scale, v_scale, sf):
    sc = _Scales(None, None, None)
    if kv_dtype != PA_KV_BF16:
        sc.k_scale = _ptr(k_scale)
        sc.v_scale = _ptr(v_scale)
        sc.sf = _ptr(sf)
    return sc


def _num_pages(kv_cache, num_kv_heads, head_dim_qk, head_dim_vo, page_size, kv_dtype):
    page_bytes = num_kv_heads * page_size * (head_dim_qk + head_dim_vo) * _x2(kv_dtype) // 2
    return (kv_cache.numel() * kv_cache.element_size()) // page_bytes


def paged_attn_decode(q: torch.Tensor, kv_cache: torch.Tensor, kv_indptr: torch.Tensor,
                      kv_indices: torch.Tensor, kv_last_page_len: torch.Tensor, *,
                      num_kv_heads: int, head_dim_vo: int, page_size: int, sm_scale: float,
                      window_left: int = -1, kv_dtype: int = PA_KV_BF16,
                      k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                      sf: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, num_pages: Optional[int] = None,
                      stream=None, return_lse: bool = True) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Decode: q [batch, Hq, head_dim_qk] bf16 -> out [batch, Hq, head_dim_vo] bf16, lse [batch, Hq]."""
    batch, hq, dqk = q.shape
    if num_pages is None:
        num_pages = _num_pages(kv_cache, num_kv_heads, dqk, head_dim_vo, page_size, kv_dtype)
    if out is None:
        out = torch.empty(batch, hq, head_dim_vo, dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(batch, hq, dtype=torch.float32, device=q.device)
    sc = _scales(kv_dtype, k_scale, v_scale, sf)
    st = load().paged_attn_decode(_ptr(q), _ptr(kv_cache), _ptr(kv_indptr), _ptr(kv_indices),
                                  _ptr(kv_last_page_len), batch, num_pages, hq, num_kv_heads, dqk,
                                  head_dim_vo, page_size, float(sm_scale), window_left, kv_dtype,
                                  ctypes.byref(sc), _ptr(out), _ptr(lse), _stream(stream))
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_decode")
    return out, lse


def paged_attn_decode_noalloc(q: torch.Tensor, kv_cache: torch.Tensor, kv_indptr: torch.Tensor,
                              kv_indices: torch.Tensor, kv_last_page_len: torch.Tensor, *, out: torch.Tensor,
                              lse: Optional[torch.Tensor], num_kv_heads: int, head_dim_vo: int, page_size: int,
                              sm_scale: float, window_left: int = -1, kv_dtype: int = PA_KV_BF16,
                              k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                              sf: Optional[torch.Tensor] = None, num_pages: Optional[int] = None,
                              stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Decode for callers that cannot allocate device memory: the library uses only its
    fixed scratch array, and the caller passes ``out`` (and ``lse``) already allocated.
    Overlapping calls race on that array; serialise them."""
    batch, hq, dqk = q.shape
    if num_pages is None:
        num_pages = _num_pages(kv_cache, num_kv_heads, dqk, head_dim_vo, page_size, kv_dtype)
    sc = _scales(kv_dtype, k_scale, v_scale, sf)
    st = load().paged_attn_decode_noalloc(_ptr(q), _ptr(kv_cache), _ptr(kv_indptr), _ptr(kv_indices),
                                          _ptr(kv_last_page_len), batch, num_pages, hq, num_kv_heads, dqk,
                                          head_dim_vo, page_size, float(sm_scale), window_left, kv_dtype,
                                          ctypes.byref(sc), _ptr(out), _ptr(lse), _stream(stream))
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_decode_noalloc")
    return out, lse


def paged_attn_prefill(q: torch.Tensor, qo_indptr: torch.Tensor, kv_cache: torch.Tensor,
                       kv_indptr: torch.Tensor, kv_indices: torch.Tensor,
                       kv_last_page_len: torch.Tensor, *, num_kv_heads: int, head_dim_vo: int,
                       page_size: int, sm_scale: float, window_left: int = -1, causal: bool = True,
                       kv_dtype: int = PA_KV_BF16, k_scale: Optional[torch.Tensor] = None,
                       v_scale: Optional[torch.Tensor] = None, sf: Optional[torch.Tensor] = None,
                       out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                       num_pages: Optional[int] = None, stream=None,
                       return_lse: bool = True, custom_mask: Optional[torch.Tensor] = None,
                       mask_indptr: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Prefill: q [total_q, Hq, head_dim_qk] bf16 -> out [total_q, Hq, head_dim_vo] bf16.
    custom_mask (uint8 bits) with mask_indptr (int64 byte offsets per sequence) selects
    paged_attn_prefill_custom_mask."""
    total_q, hq, dqk = q.shape
    batch = qo_indptr.numel() - 1
    if num_pages is None:
        num_pages = _num_pages(kv_cache, num_kv_heads, dqk, head_dim_vo, page_size, kv_dtype)
    if out is None:
        out = torch.empty(total_q, hq, head_dim_vo, dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(total_q, hq, dtype=torch.float32, device=q.device)
    sc = _scales(kv_dtype, k_scale, v_scale, sf)
    args = (_ptr(q), _ptr(qo_indptr), total_q, _ptr(kv_cache), _ptr(kv_indptr), _ptr(kv_indices),
            _ptr(kv_last_page_len), batch, num_pages, hq, num_kv_heads, dqk, head_dim_vo, page_size,
            float(sm_scale), window_left, int(bool(causal)), kv_dtype, ctypes.byref(sc), _ptr(out), _ptr(lse))
    if custom_mask is not None:
        st = load().paged_attn_prefill_custom_mask(*args, _ptr(custom_mask), _ptr(mask_indptr), _stream(stream))
        what = "paged_attn_prefill_custom_mask"
    else:
        st = load().paged_attn_prefill(*args, _stream(stream))
        what = "paged_attn_prefill"
    if st != PA_OK:
        raise PagedAttnError(st, what)
    return out, lse


def paged_attn_append_kv(k_new: torch.Tensor, v_new: torch.Tensor, append_indptr: torch.Tensor,
                         kv_cache: torch.Tensor, kv_indptr: torch.Tensor, kv_indices: torch.Tensor,
                         kv_last_page_len: torch.Tensor, *, page_size: int, kv_dtype: int = PA_KV_BF16,
                         k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                         sf: Optional[torch.Tensor] = None, num_pages: Optional[int] = None,
                         stream=None) -> None:
    """Write k_new [total_new, Hkv, head_dim_qk] / v_new [total_new, Hkv, head_dim_vo] (bf16)
    as the last tokens of each sequence, converted to the cache's element type."""
    total_new, hkv, dqk = k_new.shape
    dvo = v_new.shape[2]
    batch = append_indptr.numel() - 1
    if num_pages is None:
        num_pages = _num_pages(kv_cache, hkv, dqk, dvo, page_size, kv_dtype)
    st = load().paged_attn_append_kv(_ptr(k_new), _ptr(v_new), _ptr(append_indptr), total_new, _ptr(kv_cache),
                                     _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len), batch,
                                     num_pages, hkv, dqk, dvo, page_size, kv_dtype, _ptr(k_scale),
                                     _ptr(v_scale), _ptr(sf), _stream(stream))
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_append_kv")


def paged_attn_release_workspace() -> None:
    st = load().paged_attn_release_workspace()
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_release_workspace")


def paged_attn_check_device_error() -> int:
    """Synchronise and return the device error word (0 = none); raises on a CUDA error."""
    code = ctypes.c_int(0)
    st = load().paged_attn_check_device_error(ctypes.byref(code))
    if st not in (PA_OK, PA_ERR_DEVICE):
        raise PagedAttnError(st, "paged_attn_check_device_error")
    return code.value


def paged_attn_debug_set_error_word(target: int, code: int) -> None:
    """Test hook: store ``code`` in the workspace's (0) or the no-alloc array's (1) device
    error word."""
    st = load().paged_attn_debug_set_error_word(target, code)
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_debug_set_error_word")


def paged_attn_set_decode_chunk_pages(pages: int) -> None:
    st = load().paged_attn_set_decode_chunk_pages(pages)
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_set_decode_chunk_pages")


def paged_attn_set_decode_direct(mode: int) -> None:
    """Single-launch decode: -1 where the library's rule applies (default), 0 never, 1
    whenever every (sequence, kv head) item fits one round of CTAs."""
    st = load().paged_attn_set_decode_direct(mode)
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_set_decode_direct")


def paged_attn_set_prefill_dequant_limit(nbytes: int) -> None:
    """Largest bf16 copy of FP8 / NVFP4 pages the prefill may build (0: convert inside the
    kernel; negative: the library default)."""
    st = load().paged_attn_set_prefill_dequant_limit(nbytes)
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_set_prefill_dequant_limit")


def paged_attn_set_prefill_cta_pairs(mode: int) -> None:
    """1: bf16 prefill on CTA pairs whenever two-CTA clusters fit; 0 or -1 (default): one
    CTA per query tile."""
    st = load().paged_attn_set_prefill_cta_pairs(mode)
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_set_prefill_cta_pairs")


def paged_attn_set_prefill_split_kv(mode: int) -> None:
    """-1 (default): prefills that leave SMs idle may split long KV ranges; 0: never."""
    st = load().paged_attn_set_prefill_split_kv(mode)
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_set_prefill_split_kv")


def paged_attn_last_variant() -> str:
    buf = ctypes.create_string_buffer(64)
    load().paged_attn_last_variant(buf, 64)
    return buf.value.decode()


def paged_attn_profile_begin(max_launches: int) -> None:
    st = load().paged_attn_profile_begin(max_launches)
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_profile_begin")


def paged_attn_profile_end() -> Tuple[int, float]:
    """(recorded launches, summed device milliseconds of the main kernel)."""
    n, ms = ctypes.c_int(0), ctypes.c_float(0.0)
    st = load().paged_attn_profile_end(ctypes.byref(n), ctypes.byref(ms))
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_profile_end")
    return n.value, ms.value


def case_args(case) -> dict:
    """Keyword arguments of a synth.Case (already on the GPU) for the two calls."""
    kw = dict(num_kv_heads=case.Hkv, head_dim_vo=case.d_vo, page_size=case.page_size,
              sm_scale=case.sm_scale, window_left=case.window_left, kv_dtype=case.kv_dtype,
              num_pages=case.num_pages)
    if case.kv_dtype != PA_KV_BF16:
        dev = case.q.device
        kw["k_scale"] = torch.tensor([case.k_scale], dtype=torch.float32, device=dev)
        kw["v_scale"] = torch.tensor([case.v_scale], dtype=torch.float32, device=dev)
        if case.kv_dtype == PA_KV_NVFP4:
            kw["sf"] = case.sf
    if case.phase == "prefill" and getattr(case, "mask", None) is not None:
        kw["custom_mask"] = case.mask
        kw["mask_indptr"] = case.mask_indptr
    return kw


def run_case(case, **extra):
    """Run the call that matches case.phase on a synth.Case that lives on the GPU."""
    kw = case_args(case)
    kw.update(extra)
    if case.phase == "decode":
        return paged_attn_decode(case.q, case.kv_cache, case.kv_indptr, case.kv_indices,
                                 case.kv_last_page_len, **kw)
    return paged_attn_prefill(case.q, case.qo_indptr, case.kv_cache, case.kv_indptr, case.kv_indices,
                              case.kv_last_page_len, causal=bool(case.causal), **kw)
