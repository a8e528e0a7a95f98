"""Decode parity: the CUDA path through the C ABI against the fp64 oracle (needs a GPU).

Small cases are compared on every output element; they span several tiles, page
boundaries, partial and exact last pages, ragged batches, empty sequences, every page
size, group sizes 1..16 (including the non-power-of-two 3, 6, 12), the three head-dim
shapes, the three KV dtypes, sliding windows and forced split-K chunkings.
"""

import pytest
import torch

import paged_gqa_attention_hd512_gb300 as pa
import synth
from parity import check_full, ensure_built, run_gpu

pytestmark = pytest.mark.gpu

BF16, FP8, NVFP4 = synth.KV_BF16, synth.KV_FP8, synth.KV_NVFP4


@pytest.fixture(autouse=True)
def _reset_split():
    ensure_built()
    pa.paged_attn_set_decode_chunk_pages(0)
    pa.paged_attn_set_decode_direct(-1)
    yield
    pa.paged_attn_set_decode_chunk_pages(0)
    pa.paged_attn_set_decode_direct(-1)


def test_tiny_mqa_decode_workload():
    """Two short sequences of one kv head: the single-launch path (no planner, no merge)."""
    c = synth.workload("tiny_mqa_decode")
    check_full(c, "tiny mqa decode")
    assert pa.paged_attn_last_variant() == "decode_512x512_hp8_bf16_direct"
    pa.paged_attn_set_decode_direct(0)
    check_full(c, "tiny mqa decode, planned")
    assert pa.paged_attn_last_variant() == "decode_512x512_hp8_bf16"


CASES = [
    # (dtype, dqk, dvo, Hq, Hkv, page_size, kv_lens, window)
    (BF16, 512, 512, 24, 4, 16, [1, 15, 16, 17, 37, 64], -1),
    (BF16, 512, 512, 24, 4, 64, [63, 64, 65, 130, 7], -1),
    (BF16, 512, 512, 8, 1, 1, [5, 33], -1),
    (BF16, 512, 512, 8, 2, 2, [9, 3], -1),
    (BF16, 512, 512, 12, 4, 4, [21, 40], -1),
    (BF16, 512, 512, 4, 4, 8, [77, 8], -1),
    (BF16, 512, 512, 16, 2, 32, [100, 31, 33], -1),
    (BF16, 512, 512, 16, 1, 16, [50, 200], -1),
    (BF16, 512, 512, 24, 2, 16, [45, 90], -1),
    (BF16, 512, 256, 16, 2, 16, [70, 13], -1),
    (BF16, 256, 256, 32, 16, 16, [100, 47], -1),
    (BF16, 256, 256, 6, 2, 8, [129, 1], -1),
    (FP8, 512, 512, 12, 4, 16, [100, 17, 64], -1),
    (FP8, 512, 512, 16, 1, 64, [150, 64], -1),
    (FP8, 512, 256, 8, 2, 16, [90, 33], -1),
    (FP8, 256, 256, 6, 3, 4, [70, 5], -1),
    (NVFP4, 512, 512, 8, 1, 32, [100, 37], -1),
    (NVFP4, 512, 256, 16, 2, 32, [96, 65], -1),
    (NVFP4, 256, 256, 12, 1, 16, [80, 16], -1),
    (NVFP4, 512, 512, 6, 2, 4, [45, 12], -1),
    (BF16, 512, 512, 24, 4, 16, [200, 64, 17], 0),
    (BF16, 512, 512, 24, 4, 16, [200, 64, 17], 15),
    (BF16, 256, 256, 32, 16, 16, [300, 1030], 1023),
    (FP8, 512, 512, 12, 4, 16, [150, 30], 40),
    (NVFP4, 512, 256, 8, 2, 32, [150, 30], 63),
]


def _id(c):
    names = {BF16: "bf16", FP8: "fp8", NVFP4: "nvfp4"}
    return f"{names[c[0]]}-{c[1]}x{c[2]}-{c[3]}q{c[4]}kv-ps{c[5]}-kv{'_'.join(map(str, c[6]))}-w{c[7]}"


@pytest.mark.parametrize("mode", ["planned", "direct"])
@pytest.mark.parametrize("c", CASES, ids=[_id(c) for c in CASES])
def test_decode_parity(c, mode):
    """Every case through the planner (split-K where it splits, and the merge) and through
    the single-launch path (one item per sequence and kv head)."""
    dt, dqk, dvo, hq, hkv, ps, lens, win = c
    pa.paged_attn_set_decode_direct(1 if mode == "direct" else 0)
    case = synth.make_case("decode", batch=len(lens), Hq=hq, Hkv=hkv, d_qk=dqk, d_vo=dvo, page_size=ps,
                           kv_lens=lens, kv_dtype=dt, window_left=win, seed=300 + len(CASES))
    check_full(case, _id(c) + " " + mode)
    assert pa.paged_attn_last_variant().endswith("_direct") == (mode == "direct")


@pytest.mark.parametrize("chunk_pages", [1, 2, 7])
@pytest.mark.parametrize("dt", [BF16, FP8, NVFP4])
def test_decode_forced_splits(chunk_pages, dt):
    case = synth.make_case("decode", batch=3, Hq=12, Hkv=4, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[1, 160, 97], kv_dtype=dt, seed=41)
    pa.paged_attn_set_decode_chunk_pages(chunk_pages)
    check_full(case, f"forced chunk {chunk_pages}")


def test_decode_split_equals_unsplit_nvfp4():
    """Page-aligned splits never cut an NVFP4 scale block (blocks run along head_dim of one
    token), so split-K and single-chunk results agree."""
    case = synth.make_case("decode", batch=2, Hq=8, Hkv=1, d_qk=512, d_vo=256, page_size=16,
                           kv_lens=[700, 333], kv_dtype=NVFP4, seed=42).to("cuda")
    pa.paged_attn_set_decode_chunk_pages(1000)
    o1, l1 = run_gpu(case)
    o1, l1 = o1.clone(), l1.clone()
    pa.paged_attn_set_decode_chunk_pages(3)
    o2, l2 = run_gpu(case)
    d = (o1.float() - o2.float()).abs()
    assert float(d.max()) <= 1e-2 + 1e-2 * float(o1.float().abs().max())
    assert float((l1 - l2).abs().max()) <= 1e-4


@pytest.mark.parametrize("direct", [0, 1])
def test_decode_empty_sequence_and_window_zero(direct):
    pa.paged_attn_set_decode_direct(direct)
    case = synth.make_case("decode", batch=3, Hq=6, Hkv=2, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[0, 40, 0], seed=43)
    check_full(case, "empty sequences")
    case = synth.make_case("decode", batch=2, Hq=6, Hkv=2, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[33, 16], window_left=0, seed=44)
    check_full(case, "window 0")


def test_decode_lse_optional_and_stream():
    case = synth.make_case("decode", batch=2, Hq=8, Hkv=1, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[37, 64], seed=45).to("cuda")
    ensure_built()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, lse = pa.run_case(case, return_lse=False)
    s.synchronize()
    assert lse is None
    ref, _ = pa.run_case(case)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_synth_cpu_and_gpu_inputs_are_identical():
    for dt in (BF16, FP8, NVFP4):
        kw = dict(batch=2, Hq=8, Hkv=2, d_qk=512, d_vo=256, page_size=16, kv_lens=[40, 17], kv_dtype=dt,
                  seed=46)
        a = synth.make_case("decode", device="cpu", **kw)
        b = synth.make_case("decode", device="cuda", **kw)
        assert torch.equal(a.kv_cache, b.kv_cache.cpu())
        assert torch.equal(a.q.view(torch.int16), b.q.cpu().view(torch.int16))
        assert a.k_scale == b.k_scale and a.v_scale == b.v_scale
        if dt == NVFP4:
            assert torch.equal(a.sf, b.sf.cpu())


@pytest.mark.parametrize("dt", [BF16, FP8, NVFP4])
def test_decode_heavy_tailed_kv(dt):
    """K and V with +-8 sigma outliers (one element in 16 on average), which the bounded
    synthetic draws never reach: the FP8 per-tensor scale and the NVFP4 global and block
    scales are set by the tails, most values sit far below them."""
    case = synth.make_case("decode", batch=4, Hq=12, Hkv=4, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[300, 17, 129, 64], kv_dtype=dt, seed=47, outlier_every=16)
    check_full(case, "heavy tails")
    pa.paged_attn_set_decode_chunk_pages(2)
    check_full(case, "heavy tails, split")


def test_decode_batch_beyond_one_planner_round():
    """1100 sequences: the planner's block (at most 1024 threads) walks the batch in two
    rounds for its page counts and its scan of chunk offsets."""
    import numpy as np
    lens = [int(x) for x in np.random.default_rng(48).integers(0, 40, size=1100)]
    case = synth.make_case("decode", batch=len(lens), Hq=8, Hkv=1, d_qk=256, d_vo=256, page_size=16,
                           kv_lens=lens, seed=48)
    check_full(case, "1100 sequences")
    assert not pa.paged_attn_last_variant().endswith("_direct")
    pa.paged_attn_set_decode_chunk_pages(1)
    check_full(case, "1100 sequences, one page per chunk")
