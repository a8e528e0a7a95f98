"""Prefill of a few new tokens over a long cached prefix ("extend"): the planner splits
the KV ranges across CTAs and a merge kernel combines the partials.  Parity with the fp64
oracle through the C ABI (needs a GPU)."""

import pytest

import paged_gqa_attention_hd512_gb300 as pa
import synth
from parity import check_full, ensure_built

pytestmark = pytest.mark.gpu

CASES = [
    # (kv_dtype, dqk, dvo, Hq, Hkv, page_size, kv_lens, qo_lens, causal, window)
    (synth.KV_BF16, 512, 512, 8, 2, 16, [4000, 2500], [16, 40], 1, -1),
    (synth.KV_BF16, 512, 256, 16, 2, 32, [6000], [1], 1, -1),
    (synth.KV_BF16, 256, 256, 4, 2, 8, [3000, 100, 5000], [7, 100, 3], 1, 1023),
    (synth.KV_BF16, 512, 512, 24, 4, 64, [9000, 700], [5, 64], 0, -1),
    (synth.KV_BF16, 512, 512, 8, 1, 64, [12000], [30], 1, -1),
    # one token over 20000 keys: 157 KV tiles cut into 40 parts, more than a warp's lanes
    # hold at once in the merge
    (synth.KV_BF16, 512, 512, 8, 1, 64, [20000], [1], 1, -1),
    (synth.KV_FP8, 512, 512, 12, 4, 16, [3000, 1200], [9, 33], 1, -1),
    (synth.KV_NVFP4, 512, 256, 16, 2, 32, [4096, 1500], [24, 8], 1, -1),
]


def _id(c):
    dt = {0: "bf16", 1: "fp8", 2: "nvfp4"}[c[0]]
    return (f"{dt}-{c[1]}x{c[2]}-{c[3]}q{c[4]}kv-ps{c[5]}-kv{'_'.join(map(str, c[6]))}"
            f"-qo{'_'.join(map(str, c[7]))}-c{c[8]}-w{c[9]}")


@pytest.mark.parametrize("split", [True, False], ids=["split", "nosplit"])
@pytest.mark.parametrize("c", CASES, ids=[_id(c) for c in CASES])
def test_prefill_extend(c, split):
    ensure_built()
    dt, dqk, dvo, hq, hkv, ps, kv, qo, causal, win = c
    case = synth.make_case("prefill", batch=len(kv), Hq=hq, Hkv=hkv, d_qk=dqk, d_vo=dvo, page_size=ps,
                           kv_lens=kv, qo_lens=qo, kv_dtype=dt, causal=causal, window_left=win,
                           seed=800 + len(kv) + dt)
    pa.paged_attn_set_prefill_split_kv(-1 if split else 0)
    try:
        check_full(case, _id(c) + ("-split" if split else ""))
        assert ("_splitkv" in pa.paged_attn_last_variant()) == split
    finally:
        pa.paged_attn_set_prefill_split_kv(-1)
