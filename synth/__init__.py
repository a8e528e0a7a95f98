"""Seeded synthetic inputs for paged grouped-query attention.

This module is shared by the two sides of every parity check: the fp64 CPU oracle
(``oracle/``) and the CUDA library (``paged_gqa_attention_hd512_gb300``).  It holds no
attention arithmetic.  It holds only:

* a counter-based generator: element ``i`` of tensor ``t`` under seed ``s`` is a pure
  function of ``(s, t, i)`` built from 32-bit integer hashing (C. Wellons' "lowbias32"
  mixer).  The integer part is exact on any device; the final scaling is one IEEE fp32
  multiply and one round-to-nearest-even to bf16, so CPU and CUDA tensors built by the
  same call are bit-identical.
* encoders that turn the bf16 draws into the cache formats the pages name: per-tensor
  FP8 e4m3 and NVFP4 (e2m1 values, one e4m3 scale per 16 head-dim elements of one token,
  one fp32 global scale).  These produce the *input bytes*; both sides decode them with
  their own, separately written decoders.
* the page table (seeded random physical page order) and the workload recipes.

The "N(0,1)" draws the pages ask for are realised as the standardised sum of four
uniform 16-bit integers (an Irwin-Hall(4) variate), which is bit-reproducible across
devices without transcendental functions; its tails are bounded at about 3.46.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

M32 = 0xFFFFFFFF

KV_BF16, KV_FP8, KV_NVFP4 = 0, 1, 2
KV_DTYPE_NAMES = {KV_BF16: "bf16", KV_FP8: "fp8_e4m3", KV_NVFP4: "nvfp4"}

# tensor ids of the independent draws
TID_Q, TID_K, TID_V, TID_LEN, TID_PERM, TID_OUTLIER = 1, 2, 3, 4, 5, 6

# heavy tails: magnitude of the planted K / V outliers (in units of the draws' standard
# deviation), which the bounded Irwin-Hall(4) draws never reach (|x| <= 3.46)
OUTLIER_SIGMA = 8.0

# standard deviation of the sum of four uniform integers on [0, 65535]
_IH_SD = math.sqrt((65536.0 ** 2 - 1.0) / 3.0)
_IH_INV_SD_F32 = torch.tensor(1.0 / _IH_SD, dtype=torch.float32)


# --------------------------------------------------------------------------------------
# counter-based generator
# --------------------------------------------------------------------------------------
def _mul32(x, c: int):
    """(x * c) mod 2^32 for x in [0, 2^32) without leaving int64 range."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + ((x * hi) & 0xFFFF) * 65536) & M32


def hash32(x):
    """lowbias32 integer mixer; works on Python ints and int64 tensors alike."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _keys(seed: int, tid: int):
    k1 = hash32((seed * 0x9E3779B1 + tid * 0x85EBCA77) & M32)
    k2 = hash32(k1 ^ 0x27D4EB2F)
    k3 = hash32(k2 ^ 0x165667B1)
    return k1, k2, k3


def uniform_u32(seed: int, tid: int, idx: torch.Tensor):
    """Two independent 32-bit words per element index (int64 tensor)."""
    k1, k2, k3 = _keys(seed, tid)
    lo = idx & M32
    hi = idx >> 32
    h1 = hash32(hash32(lo ^ k1) ^ hash32(hi ^ k2))
    h2 = hash32(h1 ^ k3)
    return h1, h2


def normal_f32(seed: int, tid: int, idx: torch.Tensor) -> torch.Tensor:
    """Standardised Irwin-Hall(4) variate per element index, as fp32."""
    h1, h2 = uniform_u32(seed, tid, idx)
    s = (h1 & 0xFFFF) + (h1 >> 16) + (h2 & 0xFFFF) + (h2 >> 16) - 131070
    return s.to(torch.float32) * _IH_INV_SD_F32.to(idx.device)


def normal_bf16(seed: int, tid: int, start: int, n: int, device) -> torch.Tensor:
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    return normal_f32(seed, tid, idx).to(torch.bfloat16)


def randint(seed: int, tid: int, idx: int, lo: int, hi: int) -> int:
    """Integer in [lo, hi] (inclusive) for a scalar index."""
    k1, k2, k3 = _keys(seed, tid)
    h = hash32(hash32(idx & M32 ^ k1) ^ k2)
    return lo + h % (hi - lo + 1)


def permutation(seed: int, tid: int, n: int) -> torch.Tensor:
    """Seeded random permutation of range(n) (argsort of distinct 32-bit hashes)."""
    k1, k2, _ = _keys(seed, tid)
    idx = torch.arange(n, dtype=torch.int64)
    h = hash32(hash32(idx ^ k1) ^ k2)  # a bijection of 32-bit words -> distinct keys
    return torch.argsort(h).to(torch.int32)


# --------------------------------------------------------------------------------------
# input encoders (bf16 draw -> cache bytes)
# --------------------------------------------------------------------------------------
def e4m3_encode(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> e4m3 ("fn": bias 7, max 448, no inf) codes as uint8, RNE, saturating."""
    y = x.to(torch.float32).clamp(-448.0, 448.0)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def e4m3_to_f32(code: torch.Tensor) -> torch.Tensor:
    return code.view(torch.float8_e4m3fn).to(torch.float32)


def e2m1_encode(y: torch.Tensor) -> torch.Tensor:
    """fp32 -> e2m1 nibble codes (uint8 in [0, 15]), round-to-nearest-even, saturating to 6.

    Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 are codes 0..7; bit 3 is the sign.  Ties go to
    the even code: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4.
    """
    a = y.abs()
    code = torch.zeros_like(a, dtype=torch.uint8)
    code = torch.where(a > 0.25, 1, code)
    code = torch.where(a >= 0.75, 2, code)
    code = torch.where(a > 1.25, 3, code)
    code = torch.where(a >= 1.75, 4, code)
    code = torch.where(a > 2.5, 5, code)
    code = torch.where(a >= 3.5, 6, code)
    code = torch.where(a > 5.0, 7, code)
    code = code.to(torch.uint8)
    neg = (y < 0) & (code != 0)
    return torch.where(neg, code | 8, code).to(torch.uint8)


def pow2_ceil(v: float) -> float:
    """Smallest power of two >= v (v > 0), exactly."""
    m, e = math.frexp(v)  # v = m * 2^e, m in [0.5, 1)
    return math.ldexp(1.0, e - 1) if m == 0.5 else math.ldexp(1.0, e)


def nvfp4_global_scale(amax: float) -> float:
    """Power-of-two fp32 global scale: 2^ceil(log2(amax / (448 * 6)))."""
    if amax <= 0.0:
        return 1.0
    return pow2_ceil(amax / (448.0 * 6.0))


def nvfp4_encode_rows(x: torch.Tensor, global_scale: float):
    """x: [..., D] fp32 rows (D % 16 == 0) -> (packed uint8 [..., D/2], sf uint8 [..., D/16]).

    Block scale sf = e4m3_RNE(block_amax / 6 / global); value = e2m1_RNE(x / (sf * global)).
    Element 2i sits in the low nibble of byte i, element 2i+1 in the high nibble.
    """
    shp = x.shape
    d = shp[-1]
    xb = x.reshape(-1, d // 16, 16).to(torch.float32)
    bam = xb.abs().amax(dim=-1)
    g = torch.tensor(global_scale, dtype=torch.float32, device=x.device)
    sf = e4m3_encode(bam / 6.0 / g)
    sfv = e4m3_to_f32(sf) * g
    safe = torch.where(sfv > 0, sfv, torch.ones_like(sfv))
    q = torch.where(sfv[..., None] > 0, xb / safe[..., None], torch.zeros_like(xb))
    codes = e2m1_encode(q).reshape(-1, d)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8)
    return packed.reshape(*shp[:-1], d // 2), sf.reshape(*shp[:-1], d // 16)


# --------------------------------------------------------------------------------------
# cases
# --------------------------------------------------------------------------------------
@dataclass
class Case:
    """Every argument of one decode or prefill call, on one device.

    Layout of ``kv_cache`` (bytes): page p holds the K block [Hkv, page_size, d_qk] then
    the V block [Hkv, page_size, d_vo], elements of the KV dtype (NVFP4: two per byte).
    With d_qk == d_vo this is exactly [num_pages, 2, Hkv, page_size, head_dim].
    ``sf`` (NVFP4 only): page p holds [Hkv, page_size, d_qk/16] K scales then
    [Hkv, page_size, d_vo/16] V scales, e4m3 bytes.
    """

    phase: str
    batch: int
    num_pages: int
    Hq: int
    Hkv: int
    d_qk: int
    d_vo: int
    page_size: int
    kv_dtype: int
    sm_scale: float
    window_left: int
    causal: int
    q: torch.Tensor
    qo_indptr: torch.Tensor
    kv_cache: torch.Tensor
    kv_indptr: torch.Tensor
    kv_indices: torch.Tensor
    kv_last_page_len: torch.Tensor
    sf: Optional[torch.Tensor]
    k_scale: float
    v_scale: float
    kv_lens: List[int]
    qo_lens: List[int]
    meta: Dict = field(default_factory=dict)
    # optional prefill custom mask: per sequence b, bit (byte offset mask_indptr[b]) * 8 +
    # i * kv_len + j (little-endian within bytes) lets query row i attend key j
    mask: Optional[torch.Tensor] = None
    mask_indptr: Optional[torch.Tensor] = None

    @property
    def total_q(self) -> int:
        return int(sum(self.qo_lens))

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    def elem_bytes_x2(self) -> int:
        """Bytes per KV element times two (bf16 4, fp8 2, nvfp4 1)."""
        return {KV_BF16: 4, KV_FP8: 2, KV_NVFP4: 1}[self.kv_dtype]

    def page_bytes(self) -> int:
        return self.Hkv * self.page_size * (self.d_qk + self.d_vo) * self.elem_bytes_x2() // 2

    def to(self, device) -> "Case":
        c = Case(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("q", "qo_indptr", "kv_cache", "kv_indptr", "kv_indices", "kv_last_page_len", "sf", "mask",
                  "mask_indptr"):
            v = getattr(self, k)
            if v is not None:
                setattr(c, k, v.to(device))
        return c


def _page_table(seed: int, kv_lens: List[int], page_size: int):
    npages = [(L + page_size - 1) // page_size for L in kv_lens]
    total = sum(npages)
    perm = permutation(seed, TID_PERM, max(total, 1))[:total]
    indptr = [0]
    for n in npages:
        indptr.append(indptr[-1] + n)
    last = [(L - (n - 1) * page_size) if n > 0 else 0 for L, n in zip(kv_lens, npages)]
    return (torch.tensor(indptr, dtype=torch.int32), perm.clone(),
            torch.tensor(last, dtype=torch.int32), total)


def with_outliers(x: torch.Tensor, seed: int, tid: int, start: int, every: int) -> torch.Tensor:
    """x (bf16 draws of elements start, start + 1, ...) with element i replaced by
    +-OUTLIER_SIGMA where a seeded hash of i is 0 modulo ``every`` (one element in
    ``every`` on average, sign from another bit of the hash)."""
    idx = torch.arange(start, start + x.numel(), dtype=torch.int64, device=x.device)
    h1, _ = uniform_u32(seed, TID_OUTLIER * 16 + tid, idx)
    hit = (h1 % every) == 0
    sign = torch.where((h1 >> 31) & 1 == 1, -1.0, 1.0).to(torch.bfloat16)
    flat = torch.where(hit, sign * OUTLIER_SIGMA, x.reshape(-1))
    return flat.view(x.shape)


def _fill_kv(case_shape, seed, kv_dtype, device, chunk_pages=None, poison=True, kv_lens=None,
             indices=None, indptr=None, outlier_every=0):
    """Build cache bytes, NVFP4 scale pool and the fp32 K/V scales for a page pool.
    outlier_every > 0 plants +-OUTLIER_SIGMA values in K and V before quantisation (about
    one element in outlier_every), for heavy-tailed inputs."""
    num_pages, Hkv, ps, dqk, dvo = case_shape
    k_row = Hkv * ps * dqk
    v_row = Hkv * ps * dvo
    if chunk_pages is None:
        chunk_pages = max(1, (1 << 27) // max(1, k_row + v_row))

    def draw(tid, p0, p1, row):
        x = normal_bf16(seed, tid, p0 * row, (p1 - p0) * row, device)
        if outlier_every > 0:
            x = with_outliers(x, seed, tid, p0 * row, outlier_every)
        return x.view(p1 - p0, row)

    k_scale = v_scale = 1.0
    sf = None
    if kv_dtype == KV_BF16:
        cache = torch.empty(num_pages, k_row + v_row, dtype=torch.bfloat16, device=device)
        for p0 in range(0, num_pages, chunk_pages):
            p1 = min(num_pages, p0 + chunk_pages)
            cache[p0:p1, :k_row] = draw(TID_K, p0, p1, k_row)
            cache[p0:p1, k_row:] = draw(TID_V, p0, p1, v_row)
        cache_u8 = cache.view(torch.uint8).view(num_pages, -1)
    else:
        amax = [0.0, 0.0]
        for p0 in range(0, num_pages, chunk_pages):
            p1 = min(num_pages, p0 + chunk_pages)
            amax[0] = max(amax[0], float(draw(TID_K, p0, p1, k_row).abs().max()))
            amax[1] = max(amax[1], float(draw(TID_V, p0, p1, v_row).abs().max()))
        if kv_dtype == KV_FP8:
            k_scale = float(torch.tensor(amax[0] / 448.0, dtype=torch.float32))
            v_scale = float(torch.tensor(amax[1] / 448.0, dtype=torch.float32))
            cache_u8 = torch.empty(num_pages, k_row + v_row, dtype=torch.uint8, device=device)
            ks = torch.tensor(k_scale, dtype=torch.float32, device=device)
            vs = torch.tensor(v_scale, dtype=torch.float32, device=device)
            for p0 in range(0, num_pages, chunk_pages):
                p1 = min(num_pages, p0 + chunk_pages)
                cache_u8[p0:p1, :k_row] = e4m3_encode(draw(TID_K, p0, p1, k_row).float() / ks)
                cache_u8[p0:p1, k_row:] = e4m3_encode(draw(TID_V, p0, p1, v_row).float() / vs)
        else:
            k_scale = nvfp4_global_scale(amax[0])
            v_scale = nvfp4_global_scale(amax[1])
            cache_u8 = torch.empty(num_pages, (k_row + v_row) // 2, dtype=torch.uint8, device=device)
            sf = torch.empty(num_pages, (k_row + v_row) // 16, dtype=torch.uint8, device=device)
            for p0 in range(0, num_pages, chunk_pages):
                p1 = min(num_pages, p0 + chunk_pages)
                kp, ksf = nvfp4_encode_rows(draw(TID_K, p0, p1, k_row).float().view(-1, dqk), k_scale)
                vp, vsf = nvfp4_encode_rows(draw(TID_V, p0, p1, v_row).float().view(-1, dvo), v_scale)
                cache_u8[p0:p1, :k_row // 2] = kp.view(p1 - p0, -1)
                cache_u8[p0:p1, k_row // 2:] = vp.view(p1 - p0, -1)
                sf[p0:p1, :k_row // 16] = ksf.view(p1 - p0, -1)
                sf[p0:p1, k_row // 16:] = vsf.view(p1 - p0, -1)
    if poison and kv_lens is not None:
        _poison_tails(cache_u8, sf, kv_dtype, Hkv, ps, dqk, dvo, kv_lens, indices, indptr)
    return cache_u8.reshape(-1), (sf.reshape(-1) if sf is not None else None), k_scale, v_scale


def _poison_tails(cache_u8, sf, kv_dtype, Hkv, ps, dqk, dvo, kv_lens, indices, indptr):
    """Fill the unused slots of every last page with NaN codes (bf16 0x7FC0, e4m3 0x7F)
    and NaN block scales, so a kernel that reads them without masking shows it."""
    num_pages = cache_u8.shape[0]
    pv = cache_u8.view(num_pages, -1)
    ind = indices.tolist()
    ip = indptr.tolist()
    b2 = {KV_BF16: 2, KV_FP8: 1}.get(kv_dtype)
    for b, L in enumerate(kv_lens):
        n = ip[b + 1] - ip[b]
        if n == 0:
            continue
        used = L - (n - 1) * ps
        if used >= ps:
            continue
        p = ind[ip[b] + n - 1]
        for h in range(Hkv):
            for part, d, base in ((0, dqk, 0), (1, dvo, Hkv * ps * dqk)):
                r0 = base + (h * ps + used) * d
                r1 = base + (h * ps + ps) * d
                if kv_dtype == KV_BF16:
                    seg = pv[p, r0 * 2:r1 * 2].view(torch.int16)
                    seg.fill_(0x7FC0)
                elif kv_dtype == KV_FP8:
                    pv[p, r0:r1].fill_(0x7F)
                else:
                    pv[p, r0 // 2:r1 // 2].fill_(0x77)  # finite codes (e2m1 has no NaN)
                    sv = sf.view(num_pages, -1)
                    sv[p, r0 // 16:r1 // 16].fill_(0x7F)  # e4m3 NaN scale


def make_case(phase: str, *, batch: int, Hq: int, Hkv: int, d_qk: int, d_vo: int,
              page_size: int, kv_lens: List[int], qo_lens: Optional[List[int]] = None,
              kv_dtype: int = KV_BF16, sm_scale: Optional[float] = None, window_left: int = -1,
              causal: int = 1, seed: int = 1234, device="cpu", poison: bool = True,
              extra_pages: int = 0, outlier_every: int = 0) -> Case:
    """Build one call's inputs.  ``phase`` is "decode" (one query token per sequence) or
    "prefill" (``qo_lens`` new tokens per sequence, the last ``qo_len`` of ``kv_len``).
    ``outlier_every`` > 0 gives K and V heavy tails (see with_outliers)."""
    assert len(kv_lens) == batch
    if phase == "decode":
        qo_lens = [1] * batch
    assert qo_lens is not None and len(qo_lens) == batch
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d_qk)
    indptr, indices, last, total = _page_table(seed, kv_lens, page_size)
    num_pages = total + extra_pages
    if extra_pages:
        # unused physical pages at the end of the pool (never referenced)
        pass
    cache, sf, ks, vs = _fill_kv((num_pages, Hkv, page_size, d_qk, d_vo), seed, kv_dtype, device,
                                 poison=poison, kv_lens=kv_lens, indices=indices, indptr=indptr,
                                 outlier_every=outlier_every)
    total_q = sum(qo_lens)
    q = normal_bf16(seed, TID_Q, 0, total_q * Hq * d_qk, device).view(total_q, Hq, d_qk)
    qo_indptr = [0]
    for n in qo_lens:
        qo_indptr.append(qo_indptr[-1] + n)
    return Case(phase=phase, batch=batch, num_pages=num_pages, Hq=Hq, Hkv=Hkv, d_qk=d_qk,
                d_vo=d_vo, page_size=page_size, kv_dtype=kv_dtype, sm_scale=float(sm_scale),
                window_left=window_left, causal=causal, q=q,
                qo_indptr=torch.tensor(qo_indptr, dtype=torch.int32).to(device),
                kv_cache=cache, kv_indptr=indptr.to(device), kv_indices=indices.to(device),
                kv_last_page_len=last.to(device), sf=sf, k_scale=ks, v_scale=vs,
                kv_lens=list(kv_lens), qo_lens=list(qo_lens))


# --------------------------------------------------------------------------------------
# the workloads the pages' Gemma-4 layer shapes give (seed = 1000 + workload number)
# --------------------------------------------------------------------------------------
def _cfg2_lens(batch=64):
    return [randint(1002, TID_LEN, b, 1024, 8192) for b in range(batch)]


WORKLOADS = {
    "tiny_mqa_decode": dict(
        phase="decode", batch=2, Hq=8, Hkv=1, d_qk=512, d_vo=512, page_size=16,
        kv_lens=[37, 64], kv_dtype=KV_BF16, seed=1001),
    "gqa_decode_bf16": dict(
        phase="decode", batch=64, Hq=24, Hkv=4, d_qk=512, d_vo=512, page_size=64,
        kv_lens=None, kv_dtype=KV_BF16, seed=1002),
    # a quarter of the bf16 GQA decode workload (~0.6 GB of KV, above L2): profiling captures
    "gqa_decode_bf16_quarter": dict(
        phase="decode", batch=16, Hq=24, Hkv=4, d_qk=512, d_vo=512, page_size=64,
        kv_lens=None, kv_dtype=KV_BF16, seed=1002),
    "fp8_decode": dict(
        phase="decode", batch=128, Hq=12, Hkv=4, d_qk=512, d_vo=512, page_size=16,
        kv_lens=[32768] * 128, kv_dtype=KV_FP8, seed=1003),
    # the first 16 sequences of the FP8 decode workload (2.1 GB of KV, above L2): profiling captures
    "fp8_decode_small": dict(
        phase="decode", batch=16, Hq=12, Hkv=4, d_qk=512, d_vo=512, page_size=16,
        kv_lens=[32768] * 16, kv_dtype=KV_FP8, seed=1003),
    "causal_prefill_bf16": dict(
        phase="prefill", batch=4, Hq=24, Hkv=4, d_qk=512, d_vo=512, page_size=64,
        kv_lens=[2048, 3000, 4096, 6272], qo_lens=[2048, 3000, 4096, 6272],
        kv_dtype=KV_BF16, seed=1004),
    "nvfp4_asym_prefill": dict(
        phase="prefill", batch=8, Hq=16, Hkv=2, d_qk=512, d_vo=256, page_size=32,
        kv_lens=[1024] * 8, qo_lens=[1024] * 8, kv_dtype=KV_NVFP4, seed=1005),
    # a few new tokens per sequence over a long cached prefix ("extend")
    "prefill_extend_bf16": dict(
        phase="prefill", batch=4, Hq=24, Hkv=4, d_qk=512, d_vo=512, page_size=64,
        kv_lens=[16384] * 4, qo_lens=[32] * 4, kv_dtype=KV_BF16, seed=1006),
    # the first 32 sequences of the sliding-window decode (4.3 GB of cache, 0.54 GB of it
    # in the windows, above L2): profiling captures
    "sliding_decode_d256_small": dict(
        phase="decode", batch=32, Hq=32, Hkv=16, d_qk=256, d_vo=256, page_size=16,
        kv_lens=[8192] * 32, kv_dtype=KV_BF16, window_left=1023, seed=1005),
    "sliding_decode_d256": dict(
        phase="decode", batch=256, Hq=32, Hkv=16, d_qk=256, d_vo=256, page_size=16,
        kv_lens=[8192] * 256, kv_dtype=KV_BF16, window_left=1023, seed=1005),
}


def workload(name: str, device="cpu", poison: bool = True) -> Case:
    w = dict(WORKLOADS[name])
    if w["kv_lens"] is None:
        w["kv_lens"] = _cfg2_lens(w["batch"])
    return make_case(device=device, poison=poison, **w)


# --------------------------------------------------------------------------------------
# batch partitions across ranks (sequences are independent: no exchange between shards)
# --------------------------------------------------------------------------------------
def shard_sequences(batch: int, rank: int, world: int) -> range:
    """Global sequence ids of shard ``rank`` when a batch of ``batch`` sequences is cut
    into ``world`` contiguous shards whose sizes differ by at most one."""
    assert 0 <= rank < world
    base, extra = divmod(batch, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def workload_shard(name: str, rank: int, world: int, device="cpu", poison: bool = True) -> Case:
    """Shard ``rank`` of a global batch of ``world`` x batch sequences of workload ``name``
    (weak scaling: every shard has the workload's batch).  Sequence lengths are those of
    the global sequence ids; each shard has its own page pool and draws its values under
    its own seed (rank 0 under the workload's seed, so shard 0 of any world is the
    single-GPU workload)."""
    w = dict(WORKLOADS[name])
    ids = shard_sequences(w["batch"] * world, rank, world)
    if w["kv_lens"] is None:
        w["kv_lens"] = [randint(w["seed"], TID_LEN, b, 1024, 8192) for b in ids]
    w["seed"] = w["seed"] + 100003 * rank
    return make_case(device=device, poison=poison, **w)


def concat_cases(cases: List[Case]) -> Case:
    """One host case holding every sequence of ``cases`` in order (page pools appended,
    page ids and query rows offset); the cases must share shapes, dtype and scales."""
    c0 = cases[0]
    for c in cases[1:]:
        for k in ("phase", "Hq", "Hkv", "d_qk", "d_vo", "page_size", "kv_dtype", "sm_scale", "window_left",
                  "causal", "k_scale", "v_scale"):
            assert getattr(c, k) == getattr(c0, k), k
    ind, ip, qo, last, q, cache, sf = [], [0], [0], [], [], [], []
    page0 = 0
    for c in cases:
        c = c.to("cpu")
        ind.append(c.kv_indices + page0)
        for x in (c.kv_indptr[1:] - c.kv_indptr[:-1]).tolist():
            ip.append(ip[-1] + int(x))
        for x in (c.qo_indptr[1:] - c.qo_indptr[:-1]).tolist():
            qo.append(qo[-1] + int(x))
        last.append(c.kv_last_page_len)
        q.append(c.q)
        cache.append(c.kv_cache)
        if c.sf is not None:
            sf.append(c.sf)
        page0 += c.num_pages
    out = Case(**{k: getattr(c0, k) for k in c0.__dataclass_fields__})
    out.batch = sum(c.batch for c in cases)
    out.num_pages = page0
    out.q = torch.cat(q)
    out.qo_indptr = torch.tensor(qo, dtype=torch.int32)
    out.kv_cache = torch.cat(cache)
    out.kv_indptr = torch.tensor(ip, dtype=torch.int32)
    out.kv_indices = torch.cat(ind).to(torch.int32)
    out.kv_last_page_len = torch.cat(last)
    out.sf = torch.cat(sf) if sf else None
    out.kv_lens = [L for c in cases for L in c.kv_lens]
    out.qo_lens = [L for c in cases for L in c.qo_lens]
    return out


def workload_kv_lens(name: str) -> List[int]:
    w = WORKLOADS[name]
    return list(w["kv_lens"]) if w["kv_lens"] is not None else _cfg2_lens(w["batch"])
