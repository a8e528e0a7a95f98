"""Prefill with a custom mask through the C ABI against the fp64 oracle (needs a GPU)."""

import pytest
import torch

import mask_cases
import paged_gqa_attention_hd512_gb300 as pa
import synth
from parity import check_full, ensure_built, run_gpu

pytestmark = pytest.mark.gpu

CASES = [
    # (kind, kv_dtype, dqk, dvo, Hq, Hkv, page_size, kv_lens, qo_lens, causal, window)
    ("random", synth.KV_BF16, 512, 512, 8, 2, 16, [300, 130], [300, 70], 0, -1),
    ("spans", synth.KV_BF16, 512, 512, 24, 4, 64, [400, 129], [400, 129], 1, -1),
    ("sparse_rows", synth.KV_BF16, 512, 256, 16, 2, 32, [260, 64], [200, 64], 0, -1),
    ("random", synth.KV_BF16, 512, 256, 16, 2, 16, [333], [333], 1, 100),
    ("spans", synth.KV_BF16, 256, 256, 12, 4, 8, [150, 40], [150, 40], 0, -1),
    ("random", synth.KV_FP8, 512, 512, 8, 2, 16, [200, 77], [200, 77], 0, -1),
    ("spans", synth.KV_NVFP4, 512, 256, 16, 2, 32, [256, 100], [256, 100], 1, -1),
    # pages of fewer than 8 tokens (read from the padded copy)
    ("random", synth.KV_BF16, 512, 512, 8, 2, 2, [300, 130], [300, 70], 0, -1),
    ("spans", synth.KV_NVFP4, 512, 256, 16, 2, 4, [256, 100], [256, 100], 1, -1),
    ("sparse_rows", synth.KV_BF16, 256, 256, 12, 4, 1, [150, 40], [150, 40], 0, 30),
]


def _id(c):
    return (f"{c[0]}-{ {0: 'bf16', 1: 'fp8', 2: 'nvfp4'}[c[1]] }-{c[2]}x{c[3]}-{c[4]}q{c[5]}kv-ps{c[6]}"
            f"-kv{'_'.join(map(str, c[7]))}-qo{'_'.join(map(str, c[8]))}-c{c[9]}-w{c[10]}").replace(" ", "")


def _case(c, seed):
    kind, dt, dqk, dvo, hq, hkv, ps, kv, qo, causal, win = c
    case = synth.make_case("prefill", batch=len(kv), Hq=hq, Hkv=hkv, d_qk=dqk, d_vo=dvo, page_size=ps,
                           kv_lens=kv, qo_lens=qo, kv_dtype=dt, causal=causal, window_left=win, seed=seed)
    return mask_cases.attach(case, kind, seed + 1)


@pytest.mark.parametrize("c", CASES, ids=[_id(c) for c in CASES])
def test_prefill_custom_mask_parity(c):
    ensure_built()
    check_full(_case(c, 700 + len(c[7])), _id(c))
    assert "_mask" in pa.paged_attn_last_variant()


def test_prefill_custom_mask_on_cta_pairs():
    ensure_built()
    pa.paged_attn_set_prefill_cta_pairs(1)
    try:
        c = ("spans", synth.KV_BF16, 512, 512, 8, 2, 16, [300, 130], [300, 130], 1, -1)
        check_full(_case(c, 731), "pairs " + _id(c))
        assert pa.paged_attn_last_variant() == "prefill_512x512_pair_bf16_mask"
    finally:
        pa.paged_attn_set_prefill_cta_pairs(-1)


@pytest.fixture
def _no_split():
    """Bit-identity needs the same KV chunking in both calls: no split KV."""
    pa.paged_attn_set_prefill_split_kv(0)
    yield
    pa.paged_attn_set_prefill_split_kv(-1)


def test_all_ones_mask_changes_nothing(_no_split):
    """A mask that allows every key takes the unmasked code path: bit-identical output."""
    ensure_built()
    case = synth.make_case("prefill", batch=2, Hq=8, Hkv=2, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[260, 90], qo_lens=[200, 90], causal=0, seed=741)
    ref_out, ref_lse = run_gpu(case.to("cuda"))
    mask_cases.attach(case, "all", 1)
    out, lse = run_gpu(case.to("cuda"))
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_causal_mask_equals_causal_prefill(_no_split):
    """Non-causal with a causal-shaped mask visits the tiles past the diagonal, fully
    masked: P is 0 there, so the output is the causal call's, bit for bit."""
    ensure_built()
    case = synth.make_case("prefill", batch=2, Hq=8, Hkv=2, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[260, 90], qo_lens=[260, 90], causal=1, seed=742)
    ref_out, ref_lse = run_gpu(case.to("cuda"))
    case.causal = 0
    mask_cases.attach(case, "causal", 2)
    out, lse = run_gpu(case.to("cuda"))
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_mask_arguments_are_checked():
    ensure_built()
    case = synth.make_case("prefill", batch=1, Hq=8, Hkv=1, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[40], qo_lens=[40], seed=743).to("cuda")
    kw = pa.case_args(case)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.paged_attn_prefill(case.q, case.qo_indptr, case.kv_cache, case.kv_indptr, case.kv_indices,
                              case.kv_last_page_len, custom_mask=torch.zeros(64, dtype=torch.uint8, device="cuda"),
                              mask_indptr=None, **kw)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
