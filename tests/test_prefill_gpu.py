"""Prefill parity: the tcgen05 path through the C ABI against the fp64 oracle (needs a GPU).

Cases span several 128-row query tiles and 128-key KV tiles, ragged sequence ends,
partial last pages, a cached prefix (bottom-right causal alignment), non-causal and
windowed attention, group sizes 1..16 (row packing P x g), the three head-dim shapes.
"""

import pytest

import paged_gqa_attention_hd512_gb300 as pa
import synth
from parity import check_full, ensure_built

pytestmark = pytest.mark.gpu

BF16 = synth.KV_BF16

CASES = [
    # (dqk, dvo, Hq, Hkv, page_size, kv_lens, qo_lens, causal, window)
    (512, 512, 8, 2, 16, [130, 70], [130, 70], 1, -1),
    (512, 512, 24, 4, 64, [300, 129, 1], [300, 129, 1], 1, -1),
    (512, 512, 8, 8, 16, [257], [257], 1, -1),
    (512, 512, 16, 1, 32, [200, 33], [200, 33], 1, -1),
    (512, 512, 12, 4, 8, [150, 40], [150, 40], 1, -1),
    (512, 512, 24, 4, 16, [300, 100], [50, 100], 1, -1),
    (512, 512, 24, 4, 16, [200, 77], [200, 77], 0, -1),
    (512, 512, 24, 4, 16, [400, 90], [400, 90], 1, 63),
    (512, 256, 16, 2, 32, [200, 64], [200, 64], 1, -1),
    (512, 256, 8, 1, 16, [333], [333], 1, -1),
    (256, 256, 32, 16, 16, [190, 17], [190, 17], 1, -1),
    (256, 256, 4, 2, 64, [129, 128], [129, 128], 1, 100),
    (512, 512, 8, 2, 8, [600, 300], [600, 300], 1, -1),
    (512, 256, 16, 2, 64, [700], [700], 1, 200),
    (512, 512, 24, 4, 32, [900, 513], [400, 513], 1, -1),
    # more than 64 KV tiles: the second pass recomputes S instead of reusing P
    (512, 512, 8, 2, 64, [9000, 300], [40, 300], 1, -1),
    (512, 512, 8, 1, 64, [8300], [20], 0, -1),
]


def _id(c):
    return (f"{c[0]}x{c[1]}-{c[2]}q{c[3]}kv-ps{c[4]}-kv{'_'.join(map(str, c[5]))}"
            f"-qo{'_'.join(map(str, c[6]))}-c{c[7]}-w{c[8]}")


def _variant():
    """The variant of the last call without the split-KV mark (which small cases get)."""
    return pa.paged_attn_last_variant().replace("_splitkv", "")


@pytest.fixture(params=["pairs", "single", "single_nosplit"])
def cta_mode(request):
    """bf16 prefill on one CTA per query tile (the default; small cases split long KV
    ranges), on one CTA per tile without splitting, and on CTA pairs."""
    ensure_built()
    pa.paged_attn_set_prefill_cta_pairs(1 if request.param == "pairs" else -1)
    pa.paged_attn_set_prefill_split_kv(0 if request.param == "single_nosplit" else -1)
    yield "_pair" if request.param == "pairs" else ""
    if request.param != "single":
        assert "_splitkv" not in pa.paged_attn_last_variant()
    pa.paged_attn_set_prefill_cta_pairs(-1)
    pa.paged_attn_set_prefill_split_kv(-1)


@pytest.mark.parametrize("c", CASES, ids=[_id(c) for c in CASES])
def test_prefill_parity(c, cta_mode):
    dqk, dvo, hq, hkv, ps, kv, qo, causal, win = c
    case = synth.make_case("prefill", batch=len(kv), Hq=hq, Hkv=hkv, d_qk=dqk, d_vo=dvo, page_size=ps,
                           kv_lens=kv, qo_lens=qo, causal=causal, window_left=win, seed=500 + len(kv))
    check_full(case, _id(c) + cta_mode)
    assert _variant() == f"prefill_{dqk}x{dvo}{cta_mode}_bf16"


@pytest.mark.parametrize("q_gain", [8.0, 32.0])
def test_prefill_rescale_replay(q_gain, cta_mode):
    """Large scores make the running maximum jump by more than 2^8 between KV tiles, so the
    first pass rescales O; with head_dim_vo 512 the second pass replays those rescales
    while reusing P.  q is scaled by a power of two (exact in bf16)."""
    case = synth.make_case("prefill", batch=2, Hq=8, Hkv=2, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[700, 333], qo_lens=[260, 333], seed=77)
    case.q = (case.q.float() * q_gain).to(case.q.dtype)
    check_full(case, f"q x {q_gain}{cta_mode}")


def test_prefill_cta_pairs_setter_rejects_other_modes():  # noqa: D103
    ensure_built()
    for bad in (2, -2):
        with pytest.raises(pa.PagedAttnError) as e:
            pa.paged_attn_set_prefill_cta_pairs(bad)
        assert e.value.status == pa.PA_ERR_INVALID_ARG
    for bad in (1, -2):
        with pytest.raises(pa.PagedAttnError) as e:
            pa.paged_attn_set_prefill_split_kv(bad)
        assert e.value.status == pa.PA_ERR_INVALID_ARG


def test_prefill_pairs_on_the_dequantised_copy(cta_mode, _dequant_limit):
    """NVFP4 pages through the bf16 copy, on CTA pairs and on single CTAs."""
    pa.paged_attn_set_prefill_dequant_limit(-1)
    case = synth.make_case("prefill", batch=2, Hq=16, Hkv=2, d_qk=512, d_vo=256, page_size=32,
                           kv_lens=[300, 100], qo_lens=[300, 100], kv_dtype=synth.KV_NVFP4, seed=602)
    check_full(case, "nvfp4 copy" + cta_mode)
    assert _variant() == f"prefill_512x256{cta_mode}_nvfp4_dequant"


@pytest.mark.parametrize("dvo", [512, 256])
def test_prefill_output_only_16_byte_aligned(dvo):
    """out 16 but not 32 bytes aligned: the epilogue keeps to 16-byte stores (32-byte
    stores need 32-byte addresses) and the rows land where they belong."""
    import torch
    ensure_built()
    case = synth.make_case("prefill", batch=2, Hq=8, Hkv=2, d_qk=512, d_vo=dvo, page_size=16,
                           kv_lens=[300, 70], qo_lens=[300, 70], seed=611)
    n = case.total_q * case.Hq * dvo
    buf = torch.zeros(n + 32, dtype=torch.bfloat16, device="cuda")
    off = next(k for k in range(16) if (buf.data_ptr() + 2 * k) % 32 == 16)
    out = buf[off:off + n].view(case.total_q, case.Hq, dvo)
    pa.paged_attn_set_prefill_split_kv(0)  # the kernel writes out itself
    try:
        check_full(case, f"out at 16 mod 32, d_vo {dvo}", out=out)
    finally:
        pa.paged_attn_set_prefill_split_kv(-1)
    assert not buf[:off].any() and not buf[off + n:].any(), "writes outside out"


SMALL_PAGE_CASES = [
    # (dtype, dqk, dvo, Hq, Hkv, page_size, kv_lens, qo_lens, causal, window)
    (BF16, 512, 512, 8, 2, 1, [130, 33], [130, 33], 1, -1),
    (BF16, 512, 512, 24, 4, 2, [300, 129, 1], [300, 129, 1], 1, -1),
    (BF16, 512, 256, 16, 2, 4, [260, 64], [200, 64], 1, 63),
    (BF16, 256, 256, 8, 8, 4, [190, 17], [190, 17], 0, -1),
    (BF16, 512, 512, 8, 2, 2, [700, 333], [260, 333], 1, -1),
    (synth.KV_FP8, 512, 512, 12, 4, 2, [150, 40], [150, 40], 1, -1),
    (synth.KV_NVFP4, 512, 256, 16, 2, 4, [300, 100], [300, 100], 1, -1),
    (synth.KV_NVFP4, 512, 512, 8, 1, 1, [70], [70], 1, 20),
]


def _sid(c):
    return {BF16: "bf16", synth.KV_FP8: "fp8", synth.KV_NVFP4: "nvfp4"}[c[0]] + "-" + _id(c[1:])


@pytest.mark.parametrize("split", [True, False])
@pytest.mark.parametrize("c", SMALL_PAGE_CASES, ids=[_sid(c) for c in SMALL_PAGE_CASES])
def test_prefill_small_pages(c, split):
    """Pages of 1, 2 and 4 tokens: the prefill reads a bf16 copy that pads each page to
    8 rows per kv head (the padding is masked); every KV dtype, windows, a cached prefix,
    non-causal rows, with and without split KV."""
    ensure_built()
    pa.paged_attn_set_prefill_split_kv(-1 if split else 0)
    try:
        dt, dqk, dvo, hq, hkv, ps, kv, qo, causal, win = c
        case = synth.make_case("prefill", batch=len(kv), Hq=hq, Hkv=hkv, d_qk=dqk, d_vo=dvo, page_size=ps,
                               kv_lens=kv, qo_lens=qo, kv_dtype=dt, causal=causal, window_left=win,
                               seed=640 + ps + len(kv))
        check_full(case, _sid(c))
        names = {BF16: "bf16", synth.KV_FP8: "fp8", synth.KV_NVFP4: "nvfp4"}
        assert _variant() == f"prefill_{dqk}x{dvo}_{names[dt]}_padded"
    finally:
        pa.paged_attn_set_prefill_split_kv(-1)


def test_prefill_small_pages_beyond_the_copy_limit_are_refused(_dequant_limit):  # noqa: D103
    ensure_built()
    pa.paged_attn_set_prefill_dequant_limit(0)
    case = synth.make_case("prefill", batch=1, Hq=8, Hkv=1, d_qk=512, d_vo=512, page_size=4,
                           kv_lens=[20], qo_lens=[20], seed=9).to("cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.run_case(case)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


QCASES = [
    # (dtype, dqk, dvo, Hq, Hkv, page_size, kv_lens, qo_lens, causal, window)
    (synth.KV_FP8, 512, 512, 24, 4, 16, [300, 129], [300, 129], 1, -1),
    (synth.KV_FP8, 512, 256, 8, 1, 64, [200], [150], 1, -1),
    (synth.KV_FP8, 256, 256, 6, 3, 16, [100, 31], [100, 31], 1, -1),
    (synth.KV_NVFP4, 512, 256, 16, 2, 32, [300, 100], [300, 100], 1, -1),
    (synth.KV_NVFP4, 512, 512, 8, 2, 16, [260, 64], [260, 64], 1, 40),
    (synth.KV_NVFP4, 256, 256, 12, 4, 8, [150, 33], [150, 33], 0, -1),
]


def _qid(c):
    return {synth.KV_FP8: "fp8", synth.KV_NVFP4: "nvfp4"}[c[0]] + "-" + _id(c[1:])


@pytest.fixture
def _dequant_limit():
    yield
    pa.paged_attn_set_prefill_dequant_limit(-1)


@pytest.mark.parametrize("mode", ["dequant", "in_kernel"])
@pytest.mark.parametrize("c", QCASES, ids=[_qid(c) for c in QCASES])
def test_prefill_parity_quantised(c, mode, _dequant_limit):
    """FP8 / NVFP4 pages converted once into a bf16 copy (the default) and converted inside
    the kernel on every read (the path for caches whose copy would exceed the limit)."""
    ensure_built()
    pa.paged_attn_set_prefill_dequant_limit(-1 if mode == "dequant" else 0)
    dt, dqk, dvo, hq, hkv, ps, kv, qo, causal, win = c
    case = synth.make_case("prefill", batch=len(kv), Hq=hq, Hkv=hkv, d_qk=dqk, d_vo=dvo, page_size=ps,
                           kv_lens=kv, qo_lens=qo, kv_dtype=dt, causal=causal, window_left=win, seed=600 + len(kv))
    check_full(case, _qid(c) + "-" + mode)
    names = {synth.KV_FP8: "fp8", synth.KV_NVFP4: "nvfp4"}
    suffix = "_dequant" if mode == "dequant" else ""
    assert _variant() == f"prefill_{dqk}x{dvo}_{names[dt]}{suffix}"


@pytest.mark.parametrize("dt,mode", [(BF16, "dequant"), (synth.KV_FP8, "dequant"), (synth.KV_FP8, "in_kernel"),
                                     (synth.KV_NVFP4, "dequant"), (synth.KV_NVFP4, "in_kernel")])
def test_prefill_heavy_tailed_kv(dt, mode, _dequant_limit):
    """K and V with +-8 sigma outliers (one element in 16 on average): the FP8 per-tensor
    scale and the NVFP4 global and block scales are set by the tails (FP8 / NVFP4 through
    the bf16 copy and converted inside the kernel)."""
    ensure_built()
    pa.paged_attn_set_prefill_dequant_limit(-1 if mode == "dequant" else 0)
    case = synth.make_case("prefill", batch=2, Hq=16, Hkv=2, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[300, 129], qo_lens=[300, 129], kv_dtype=dt, seed=48, outlier_every=16)
    check_full(case, f"heavy tails {mode}")


@pytest.mark.parametrize("lens", [([50, 20, 100], [50, 0, 30]), ([0, 40, 0], [0, 40, 0])],
                         ids=["no-new-tokens", "empty-sequences"])
def test_prefill_sequences_without_new_tokens(lens, cta_mode):
    """A sequence with cached tokens but no new ones, and sequences with neither, between
    ordinary ones: they get no work items and the other rows are unchanged."""
    kv, qo = lens
    case = synth.make_case("prefill", batch=3, Hq=8, Hkv=2, d_qk=512, d_vo=512, page_size=16, kv_lens=kv,
                           qo_lens=qo, seed=93)
    check_full(case, f"kv {kv} qo {qo}{cta_mode}")


def test_prefill_batch_beyond_the_planner_cache(cta_mode):
    """2100 sequences of 0-3 new tokens over 0-22 keys: more sequences than the planner
    keeps in shared memory (2048), so it reads their lengths from the index arrays."""
    import numpy as np
    rng = np.random.default_rng(95)
    qo = [int(x) for x in rng.integers(0, 4, size=2100)]
    kv = [q + int(x) for q, x in zip(qo, rng.integers(0, 20, size=2100))]
    case = synth.make_case("prefill", batch=2100, Hq=8, Hkv=2, d_qk=256, d_vo=256, page_size=16, kv_lens=kv,
                           qo_lens=qo, seed=95)
    check_full(case, "2100 sequences" + cta_mode)
