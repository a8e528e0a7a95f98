"""Append (quantise-on-write) through the C ABI against the oracle, byte for byte (needs a
GPU): the whole cache and NVFP4 scale pool after the call, including every byte the call
must leave alone."""

import numpy as np
import pytest
import torch

import append_cases as ac
import oracle
import paged_gqa_attention_hd512_gb300 as pa
from parity import ensure_built

pytestmark = pytest.mark.gpu

CASES = [
    # (kv_dtype, dqk, dvo, Hkv, page_size, kv_lens, n_new, k_scale, v_scale, gain)
    (ac.BF16, 512, 512, 2, 16, [37, 64, 130, 1], [5, 64, 0, 1], 1.0, 1.0, 1.0),
    (ac.FP8, 512, 512, 4, 64, [300, 129, 64], [300, 1, 33], 0.05, 0.0125, 1.0),
    (ac.FP8, 256, 256, 2, 8, [20, 9], [20, 4], 2.0 ** -5, 1.0, 40.0),
    (ac.NVFP4, 512, 256, 2, 32, [1024, 77, 31], [1024, 40, 31], 2.0 ** -7, 2.0 ** -6, 1.0),
    (ac.NVFP4, 512, 512, 2, 16, [200, 16], [64, 16], 0.003, 0.0007, 1.0),
    (ac.NVFP4, 256, 256, 4, 8, [50, 3], [17, 3], 2.0 ** -9, 2.0 ** -3, 1e-3),
]


def _id(c):
    name = {ac.BF16: "bf16", ac.FP8: "fp8", ac.NVFP4: "nvfp4"}[c[0]]
    return f"{name}-{c[1]}x{c[2]}-h{c[3]}-ps{c[4]}-kv{'_'.join(map(str, c[5]))}-new{'_'.join(map(str, c[6]))}"


def _run_gpu(case):
    dev = "cuda"
    cache = torch.from_numpy(case.kv_cache.copy()).to(dev)
    sf = torch.from_numpy(case.sf.copy()).to(dev) if case.sf is not None else None
    ks = torch.tensor([case.k_scale], dtype=torch.float32, device=dev)
    vs = torch.tensor([case.v_scale], dtype=torch.float32, device=dev)
    pa.paged_attn_append_kv(
        case.k_new.to(dev), case.v_new.to(dev), torch.from_numpy(case.append_indptr).to(dev), cache,
        torch.from_numpy(case.kv_indptr).to(dev), torch.from_numpy(case.kv_indices).to(dev),
        torch.from_numpy(case.kv_last_page_len).to(dev), page_size=case.page_size, kv_dtype=case.kv_dtype,
        k_scale=ks, v_scale=vs, sf=sf, num_pages=case.num_pages)
    code = pa.paged_attn_check_device_error()
    return cache.cpu().numpy(), (sf.cpu().numpy() if sf is not None else None), code


def _oracle(case):
    return oracle.append_kv(case.k_new, case.v_new, case.append_indptr, case.kv_cache, case.kv_indptr,
                            case.kv_indices, case.kv_last_page_len, num_kv_heads=case.Hkv,
                            head_dim_qk=case.d_qk, head_dim_vo=case.d_vo, page_size=case.page_size,
                            kv_dtype=case.kv_dtype, k_scale=case.k_scale, v_scale=case.v_scale, sf=case.sf)


def _assert_bytes_equal(got, ref, what):
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{what}: {bad.size} bytes differ, first at {bad[:8].tolist()}: " \
                          f"gpu {got[bad[:8]].tolist()} oracle {ref[bad[:8]].tolist()}"


@pytest.mark.parametrize("c", CASES, ids=[_id(c) for c in CASES])
def test_append_matches_oracle(c):
    ensure_built()
    dt, dqk, dvo, hkv, ps, kv_lens, n_new, ks, vs, gain = c
    case = ac.make(kv_lens=kv_lens, n_new=n_new, Hkv=hkv, d_qk=dqk, d_vo=dvo, page_size=ps, kv_dtype=dt,
                   seed=900 + len(kv_lens) + dt, k_scale=ks, v_scale=vs, gain=gain)
    cache, sf, code = _run_gpu(case)
    ref_cache, ref_sf, skipped = _oracle(case)
    assert code == 0 and skipped == 0
    _assert_bytes_equal(cache, ref_cache, "cache")
    if dt == ac.NVFP4:
        _assert_bytes_equal(sf, ref_sf, "scale pool")
    assert pa.paged_attn_last_variant() == "append_kv_" + {ac.BF16: "bf16", ac.FP8: "fp8", ac.NVFP4: "nvfp4"}[dt]


def test_append_row_outside_its_sequence_sets_the_error_word():
    """Sequence 0 holds 10 tokens but is given 12 new rows: the 2 without a place are
    skipped and reported; every other row is written as the oracle writes it."""
    ensure_built()
    case = ac.make(kv_lens=[10, 20], n_new=[12, 3], Hkv=1, d_qk=256, d_vo=256, page_size=8,
                   kv_dtype=ac.FP8, seed=77, k_scale=0.1, v_scale=0.1)
    cache, _, code = _run_gpu(case)
    ref_cache, _, skipped = _oracle(case)
    assert skipped == 2 and code == 301
    _assert_bytes_equal(cache, ref_cache, "cache")


def test_appended_nvfp4_cache_feeds_the_prefill():
    """The written pages are read by the attention path: prefill over an NVFP4 cache that
    the append filled, against the oracle reading the same bytes."""
    ensure_built()
    from parity import compare
    case = ac.make(kv_lens=[160, 70], n_new=[160, 70], Hkv=2, d_qk=512, d_vo=256, page_size=32,
                   kv_dtype=ac.NVFP4, seed=31, k_scale=2.0 ** -7, v_scale=2.0 ** -7)
    cache, sf, code = _run_gpu(case)
    assert code == 0
    filled = ac.with_cache(case, cache, sf)
    hq = 16
    gen = torch.Generator().manual_seed(3)
    q = torch.randn(sum(case.kv_lens), hq, 512, generator=gen).to(torch.bfloat16)
    qo_indptr = torch.tensor([0, 160, 230], dtype=torch.int32)
    dev = "cuda"
    out, lse = pa.paged_attn_prefill(
        q.to(dev), qo_indptr.to(dev), torch.from_numpy(cache).to(dev), torch.from_numpy(case.kv_indptr).to(dev),
        torch.from_numpy(case.kv_indices).to(dev), torch.from_numpy(case.kv_last_page_len).to(dev),
        num_kv_heads=2, head_dim_vo=256, page_size=32, sm_scale=512 ** -0.5, causal=True,
        kv_dtype=pa.PA_KV_NVFP4, k_scale=torch.tensor([case.k_scale], device=dev),
        v_scale=torch.tensor([case.v_scale], device=dev), sf=torch.from_numpy(sf).to(dev),
        num_pages=case.num_pages)
    filled.q, filled.qo_indptr, filled.batch, filled.Hq, filled.total_q = q, qo_indptr, 2, hq, q.shape[0]
    filled.sm_scale, filled.window_left, filled.causal = 512 ** -0.5, -1, 1
    ref_out, ref_lse = oracle.full(filled)
    n = q.shape[0] * hq
    compare(out.reshape(n, -1), lse.reshape(n), ref_out.reshape(n, -1), ref_lse.reshape(n), "append -> prefill")


def _near(m, k):
    """The fp32 value k units in the last place away from m (m > 0, same binade)."""
    ulp = 2.0 ** (np.floor(np.log2(m)) - 23)
    return float(np.float32(m + k * ulp))


@pytest.mark.parametrize("k_off", [-3, -2, -1, 0, 1, 2, 3])
def test_append_fp8_quotients_at_rounding_midpoints(k_off):
    """x / scale within a few fp32 units of an e4m3 rounding midpoint (and on it): the
    codes follow the correctly rounded quotient, as in the oracle, wherever the kernel
    forms it."""
    ensure_built()
    rng = np.random.default_rng(5 + k_off)
    # midpoints between neighbouring e4m3 values: 1 and 1.125, 2.5 and 2.75, 13 and 14,
    # 416 and 448, and in the smallest normal binade 2^-6 (1 + 1/16)
    for j, m in enumerate([1.0625, 2.625, 13.5, 432.0, 2.0 ** -6 * 1.0625]):
        x = float(torch.tensor(rng.standard_normal() * 4.0 + 0.5).to(torch.bfloat16))
        if x == 0.0:
            x = 1.5
        scale = float(np.float32(abs(x) / _near(m, k_off)))
        case = ac.make(kv_lens=[3], n_new=[1], Hkv=1, d_qk=256, d_vo=256, page_size=8, kv_dtype=ac.FP8,
                       seed=40 + j, k_scale=scale, v_scale=scale)
        case.k_new[0, 0, 0] = x
        case.v_new[0, 0, 5] = -x
        cache, _, code = _run_gpu(case)
        ref_cache, _, skipped = _oracle(case)
        assert code == 0 and skipped == 0
        _assert_bytes_equal(cache, ref_cache, f"midpoint {m} offset {k_off}")


@pytest.mark.parametrize("k_off", [-3, -2, -1, 0, 1, 2, 3])
def test_append_nvfp4_quotients_at_rounding_midpoints(k_off):
    """Within an NVFP4 block, x / d within a few fp32 units of an e2m1 rounding midpoint
    (and on it), with the block scale 1.0 and a global scale chosen for it: codes as in the
    oracle."""
    ensure_built()
    for j, mid in enumerate([1.25, 1.75, 2.5, 3.5, 5.0]):
        target = _near(mid, k_off)
        g = float(np.float32(1.0 / target))            # d = 1.0 * g, so 1.0 / d is near the target
        amax = float(torch.tensor(5.88 * g).to(torch.bfloat16))  # (amax / 6) / g rounds to e4m3 1.0
        case = ac.make(kv_lens=[3], n_new=[1], Hkv=1, d_qk=256, d_vo=256, page_size=8, kv_dtype=ac.NVFP4,
                       seed=60 + j, k_scale=g, v_scale=g)
        for t in (case.k_new, case.v_new):
            t[0, 0, 0:16] = 0.0
            t[0, 0, 0] = amax
            t[0, 0, 1] = 1.0
            t[0, 0, 2] = -1.0
        cache, sf, code = _run_gpu(case)
        ref_cache, ref_sf, skipped = _oracle(case)
        assert code == 0 and skipped == 0
        _assert_bytes_equal(cache, ref_cache, f"midpoint {mid} offset {k_off}")
        _assert_bytes_equal(sf, ref_sf, f"scales, midpoint {mid} offset {k_off}")


@pytest.mark.parametrize("dt", [ac.FP8, ac.NVFP4])
def test_append_codes_that_round_to_zero_keep_their_sign(dt):
    """Values far below the smallest nonzero code (with the scale, or the block's largest
    value, fixed by one element): the codes are zero with the operand's sign, as the
    oracle writes them (e4m3 0x80, e2m1 0x8 for the negative ones)."""
    ensure_built()
    case = ac.make(kv_lens=[3], n_new=[1], Hkv=1, d_qk=256, d_vo=256, page_size=8, kv_dtype=dt,
                   seed=71, k_scale=1.0, v_scale=1.0)
    tiny = [2.0 ** -14, -(2.0 ** -14), 2.0 ** -20, -(2.0 ** -20), -(2.0 ** -12), 2.0 ** -12, -0.0, 0.0]
    for t in (case.k_new, case.v_new):
        t[0, 0, :] = 0.0
        t[0, 0, 0] = 4.0  # the block maximum (NVFP4) and one ordinary code
        for k, v in enumerate(tiny):
            t[0, 0, 1 + k] = v
            t[0, 0, 17 + k] = v  # a block of tiny values only (NVFP4: its scale rounds to 0)
    cache, sf, code = _run_gpu(case)
    ref_cache, ref_sf, skipped = _oracle(case)
    assert code == 0 and skipped == 0
    _assert_bytes_equal(cache, ref_cache, "codes that round to zero")
    if dt == ac.NVFP4:
        _assert_bytes_equal(sf, ref_sf, "scale pool")


@pytest.mark.parametrize("dt", [ac.FP8, ac.NVFP4])
def test_append_many_sequences(dt):
    """1100 sequences of 0-3 new tokens each: a warp finds its token's sequence in three
    rounds of its 32-way search over append_indptr."""
    import numpy as np
    ensure_built()
    rng = np.random.default_rng(77 + dt)
    n_new = [int(x) for x in rng.integers(0, 4, size=1100)]
    kv_lens = [n + int(x) for n, x in zip(n_new, rng.integers(0, 30, size=1100))]
    case = ac.make(kv_lens=kv_lens, n_new=n_new, Hkv=2, d_qk=256, d_vo=256, page_size=16, kv_dtype=dt,
                   seed=1100 + dt, k_scale=0.05, v_scale=0.02)
    cache, sf, code = _run_gpu(case)
    ref_cache, ref_sf, skipped = _oracle(case)
    assert code == 0 and skipped == 0
    _assert_bytes_equal(cache, ref_cache, "1100 sequences")
    if dt == ac.NVFP4:
        _assert_bytes_equal(sf, ref_sf, "1100 sequences, scales")


@pytest.mark.parametrize("per_sm", [72, 144])
@pytest.mark.parametrize("dt", [ac.BF16, ac.FP8, ac.NVFP4])
def test_append_several_tokens_per_warp(dt, per_sm):
    """Appends large enough that each warp writes two (72 new tokens per SM) or four (144)
    consecutive tokens, over sequences of 0 to 90 new tokens: a warp's tokens cross the
    ends of sequences, empty ones among them."""
    import numpy as np
    import torch
    ensure_built()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(300 + dt + per_sm)
    n_new = []
    while sum(n_new) < per_sm * sms:
        n_new.append(int(rng.integers(0, 91)) if rng.random() > 0.1 else 0)
    kv_lens = [n + int(x) for n, x in zip(n_new, rng.integers(0, 50, size=len(n_new)))]
    case = ac.make(kv_lens=kv_lens, n_new=n_new, Hkv=1, d_qk=256, d_vo=256, page_size=16, kv_dtype=dt,
                   seed=400 + dt + per_sm, k_scale=0.05, v_scale=0.02)
    cache, sf, code = _run_gpu(case)
    ref_cache, ref_sf, skipped = _oracle(case)
    assert code == 0 and skipped == 0
    _assert_bytes_equal(cache, ref_cache, f"{sum(n_new)} new tokens")
    if dt == ac.NVFP4:
        _assert_bytes_equal(sf, ref_sf, f"{sum(n_new)} new tokens, scales")
