"""fp64 CPU oracle for paged grouped-query attention -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's cpu_baseline / reference legs
import this package.  The CUDA library never does, and this package never imports it.
The arithmetic lives in ``paged_attn_oracle.c`` (plain C, fp64); this module compiles it
with gcc and marshals numpy arrays through ctypes.

Every function follows the definition written at the top of ``paged_attn_oracle.c``
(sources: "[None][feat] Run Gemma4 head_dim 512 attention on Triton", Approach and Test
Coverage; "feat(attention): asymmetric VO-split NVFP4 paged prefill (qk=512/vo=256) for
Gemma-4 on SM120/121", Summary and NVFP4 split-KV correctness).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle (IEEE fp64: no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-o", out + ".tmp", src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or \
                os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            compile_oracle()
    return _LIB_PATH


def _bind(lib):
    lib.oracle_bf16_value.restype = ctypes.c_double
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1_value.restype = ctypes.c_double
    lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
    lib.oracle_rows.restype = ctypes.c_int
    lib.oracle_rows.argtypes = [
        _u16p, _i32p, _u8p, _i32p, _i32p, _i32p, _u8p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_int,
        ctypes.c_int, ctypes.c_int64, _i64p, _i32p, _i64p, _i64p, _u8p, _i64p, _f64p, _f64p, ctypes.c_int]
    lib.oracle_merge.restype = None
    lib.oracle_merge.argtypes = [ctypes.c_int, _f64p, _f64p, ctypes.c_int, _f64p, _f64p]
    lib.oracle_gather.restype = ctypes.c_int
    lib.oracle_gather.argtypes = [
        _u8p, _i32p, _i32p, _i32p, _u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, _f64p]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e2m1_encode.restype = ctypes.c_uint8
    lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
    lib.oracle_append_kv.restype = ctypes.c_int
    lib.oracle_append_kv.argtypes = [
        _u16p, _u16p, _i32p, _u8p, _i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float, _u8p]
    return lib


def load(path: Optional[str] = None):
    """Load the oracle library (compiling it first if needed).  ``path`` loads another
    build of it (the tests use this to load deliberately broken copies)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _np(t, dtype):
    """torch tensor or array -> contiguous numpy array of dtype (on the host)."""
    if hasattr(t, "detach"):
        import torch
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        a = t.numpy()
    else:
        a = np.asarray(t)
    want = np.dtype(dtype)
    if a.dtype != want:
        if a.dtype.kind in "iu" and want.kind in "iu" and a.dtype.itemsize == want.itemsize:
            a = a.view(want)
        else:
            a = a.astype(want)
    return np.ascontiguousarray(a)


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype)) if a is not None else None


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def rows(case, row_tok: Sequence[int], row_head: Sequence[int], key_lo=None, key_hi=None,
         threads: Optional[int] = None, lib=None):
    """fp64 attention output for the given (query token, query head) rows of ``case``
    (a synth.Case; an optional ``mask`` / ``mask_indptr`` attribute pair is the custom
    mask).  Returns (out [n, d_vo], lse [n])."""
    lib = lib or load()
    q = _np(case.q, np.uint16).reshape(-1)
    qo = _np(case.qo_indptr, np.int32)
    cache = _np(case.kv_cache, np.uint8).reshape(-1)
    ip = _np(case.kv_indptr, np.int32)
    ind = _np(case.kv_indices, np.int32)
    last = _np(case.kv_last_page_len, np.int32)
    sf = _np(case.sf, np.uint8).reshape(-1) if case.sf is not None else None
    rt = np.ascontiguousarray(np.asarray(row_tok, dtype=np.int64))
    rh = np.ascontiguousarray(np.asarray(row_head, dtype=np.int32))
    klo = np.ascontiguousarray(np.asarray(key_lo, dtype=np.int64)) if key_lo is not None else None
    khi = np.ascontiguousarray(np.asarray(key_hi, dtype=np.int64)) if key_hi is not None else None
    cm = getattr(case, "mask", None)
    mask = _np(cm, np.uint8).reshape(-1) if cm is not None else None
    mip = _np(case.mask_indptr, np.int64) if cm is not None else None
    n = rt.shape[0]
    out = np.zeros((n, case.d_vo), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.oracle_rows(
        _ptr(q, ctypes.c_uint16), _ptr(qo, ctypes.c_int32), _ptr(cache, ctypes.c_uint8),
        _ptr(ip, ctypes.c_int32), _ptr(ind, ctypes.c_int32), _ptr(last, ctypes.c_int32),
        _ptr(sf, ctypes.c_uint8), case.batch, case.Hq, case.Hkv, case.d_qk, case.d_vo,
        case.page_size, case.kv_dtype, case.k_scale, case.v_scale, case.sm_scale,
        case.window_left, case.causal, n, _ptr(rt, ctypes.c_int64), _ptr(rh, ctypes.c_int32),
        _ptr(klo, ctypes.c_int64), _ptr(khi, ctypes.c_int64), _ptr(mask, ctypes.c_uint8),
        _ptr(mip, ctypes.c_int64), _ptr(out, ctypes.c_double),
        _ptr(lse, ctypes.c_double), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_rows rejected its arguments")
    return out, lse


def full(case, threads: Optional[int] = None, lib=None):
    """Every output row of ``case``: (out [total_q, Hq, d_vo], lse [total_q, Hq])."""
    tq, hq = case.total_q, case.Hq
    tok = np.repeat(np.arange(tq, dtype=np.int64), hq)
    head = np.tile(np.arange(hq, dtype=np.int32), tq)
    out, lse = rows(case, tok, head, threads=threads, lib=lib)
    return out.reshape(tq, hq, case.d_vo), lse.reshape(tq, hq)


def merge(lse_parts, o_parts, lib=None):
    """Split-K merge of one row's partials: (o [d], lse)."""
    lib = lib or load()
    lp = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    op = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    d = op.shape[-1]
    o = np.zeros((d,), dtype=np.float64)
    lse = np.zeros((1,), dtype=np.float64)
    lib.oracle_merge(lp.shape[0], _ptr(lp, ctypes.c_double), _ptr(op, ctypes.c_double), d,
                     _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    return o, float(lse[0])


def gather(case, b: int, kvh: int, is_v: bool, lib=None):
    """Dequantised [kv_len, dim] block of one (sequence, kv head)."""
    lib = lib or load()
    cache = _np(case.kv_cache, np.uint8).reshape(-1)
    ip = _np(case.kv_indptr, np.int32)
    ind = _np(case.kv_indices, np.int32)
    last = _np(case.kv_last_page_len, np.int32)
    sf = _np(case.sf, np.uint8).reshape(-1) if case.sf is not None else None
    dim = case.d_vo if is_v else case.d_qk
    kv_len = case.kv_lens[b]
    dst = np.zeros((max(kv_len, 1), dim), dtype=np.float64)
    n = lib.oracle_gather(_ptr(cache, ctypes.c_uint8), _ptr(ip, ctypes.c_int32),
                          _ptr(ind, ctypes.c_int32), _ptr(last, ctypes.c_int32),
                          _ptr(sf, ctypes.c_uint8), case.Hkv, case.d_qk, case.d_vo,
                          case.page_size, case.kv_dtype, case.k_scale, case.v_scale, b, kvh,
                          int(is_v), _ptr(dst, ctypes.c_double))
    return dst[:n]


def bf16_value(bits: int, lib=None) -> float:
    return (lib or load()).oracle_bf16_value(bits)


def e4m3_value(code: int, lib=None) -> float:
    return (lib or load()).oracle_e4m3_value(code)


def e2m1_value(nibble: int, lib=None) -> float:
    return (lib or load()).oracle_e2m1_value(nibble)


# ------------------------------------------------------------------ append (quantise-on-write)
def e4m3_encode(x, lib=None) -> np.ndarray:
    """fp32 values -> e4m3 codes (nearest, ties to even, saturating, sign kept)."""
    lib = lib or load()
    a = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in a], dtype=np.uint8)


def e2m1_encode(x, lib=None) -> np.ndarray:
    """fp32 values -> e2m1 codes in [0, 15] (nearest, ties to even, saturating, sign kept)."""
    lib = lib or load()
    a = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.oracle_e2m1_encode(float(v)) for v in a], dtype=np.uint8)


def append_kv(k_new, v_new, append_indptr, kv_cache, kv_indptr, kv_indices, kv_last_page_len, *,
              num_kv_heads: int, head_dim_qk: int, head_dim_vo: int, page_size: int, kv_dtype: int,
              k_scale: float = 1.0, v_scale: float = 1.0, sf=None, lib=None):
    """The cache (and NVFP4 scale pool) after writing the new rows; inputs are not modified.

    Returns (cache bytes, scale-pool bytes or None, rows skipped)."""
    lib = lib or load()
    kn = _np(k_new, np.uint16).ravel()
    vn = _np(v_new, np.uint16).ravel()
    ai = _np(append_indptr, np.int32)
    cache = _np(kv_cache, np.uint8).ravel().copy()
    ip = _np(kv_indptr, np.int32)
    ix = _np(kv_indices, np.int32)
    lp = _np(kv_last_page_len, np.int32)
    sfa = _np(sf, np.uint8).ravel().copy() if sf is not None else None
    x2 = {0: 4, 1: 2, 2: 1}[kv_dtype]
    page_bytes = num_kv_heads * page_size * (head_dim_qk + head_dim_vo) * x2 // 2
    num_pages = cache.size // page_bytes
    skipped = lib.oracle_append_kv(
        _ptr(kn, ctypes.c_uint16), _ptr(vn, ctypes.c_uint16), _ptr(ai, ctypes.c_int32),
        _ptr(cache, ctypes.c_uint8), _ptr(ip, ctypes.c_int32), _ptr(ix, ctypes.c_int32),
        _ptr(lp, ctypes.c_int32), ai.size - 1, num_pages, num_kv_heads, head_dim_qk, head_dim_vo,
        page_size, kv_dtype, float(k_scale), float(v_scale), _ptr(sfa, ctypes.c_uint8))
    return cache, sfa, skipped
