"""Seeded inputs for the append (quantise-on-write) tests: a paged cache with random bytes,
a page table after the append, and new K / V rows (bf16) with the value classes the
conversion must handle (ordinary, zero and negative-zero blocks, values past the FP8 /
NVFP4 range, values near zero).  Input generation only: no conversion arithmetic."""

from types import SimpleNamespace

import numpy as np
import torch

BF16, FP8, NVFP4 = 0, 1, 2
X2 = {BF16: 4, FP8: 2, NVFP4: 1}


def make(*, kv_lens, n_new, Hkv, d_qk, d_vo, page_size, kv_dtype, seed, k_scale=1.0, v_scale=1.0,
         spare_pages=3, gain=1.0):
    """kv_lens: each sequence's length after the append; n_new: new rows per sequence."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    pages_per = [max(1, -(-L // page_size)) if L > 0 else 0 for L in kv_lens]
    num_pages = sum(pages_per) + spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    kv_indptr = np.zeros(len(kv_lens) + 1, dtype=np.int32)
    kv_indptr[1:] = np.cumsum(pages_per)
    kv_indices = perm[:kv_indptr[-1]].copy()
    last = np.array([(L - 1) % page_size + 1 if L > 0 else 0 for L in kv_lens], dtype=np.int32)
    page_bytes = Hkv * page_size * (d_qk + d_vo) * X2[kv_dtype] // 2
    cache = rng.integers(0, 256, size=num_pages * page_bytes, dtype=np.uint8)
    if kv_dtype == FP8:  # no NaN codes in the untouched bytes either (0x7F / 0xFF)
        cache[(cache & 0x7F) == 0x7F] = 0x3C
    sf = None
    if kv_dtype == NVFP4:
        sf = rng.integers(0, 0x7F, size=num_pages * Hkv * page_size * (d_qk + d_vo) // 16, dtype=np.uint8)
    append_indptr = np.zeros(len(kv_lens) + 1, dtype=np.int32)
    append_indptr[1:] = np.cumsum(n_new)
    total = int(append_indptr[-1])
    k = torch.randn(total, Hkv, d_qk, generator=gen) * gain
    v = torch.randn(total, Hkv, d_vo, generator=gen) * gain
    if total > 0:  # special blocks of 16 elements
        k[0, 0, 0:16] = 0.0
        k[0, 0, 16:32] = -0.0
        v[0, 0, 0:16] = torch.linspace(-3000.0, 3000.0, 16)  # past e4m3 / e2m1 range at unit scale
        v[0, 0, 16:32] = torch.linspace(-1e-4, 1e-4, 16)      # near zero
        k[total - 1, Hkv - 1, 32:48] = torch.tensor([6.0, -4.0, 3.0, -2.0, 1.5, -1.0, 0.5, 0.0] * 2)
    return SimpleNamespace(
        kv_lens=list(kv_lens), n_new=list(n_new), Hkv=Hkv, d_qk=d_qk, d_vo=d_vo, page_size=page_size,
        kv_dtype=kv_dtype, k_scale=float(k_scale), v_scale=float(v_scale), num_pages=num_pages,
        kv_indptr=kv_indptr, kv_indices=kv_indices, kv_last_page_len=last, kv_cache=cache, sf=sf,
        append_indptr=append_indptr, k_new=k.to(torch.bfloat16), v_new=v.to(torch.bfloat16))


def with_cache(case, cache, sf):
    """The same case with another cache / scale pool (for reading it back)."""
    c = SimpleNamespace(**vars(case))
    c.kv_cache = cache
    c.sf = sf
    return c
