"""Calls on two streams that overlap on the GPU (needs a GPU): each stream has its own
workspace (work lists, split-K partials, prefill plans and partial slots), so a decode on
one stream and a split-KV prefill on the other give the same bytes as alone."""

import pytest
import torch

import paged_gqa_attention_hd512_gb300 as pa
import synth
from parity import ensure_built

pytestmark = pytest.mark.gpu


def test_decode_and_prefill_on_two_streams():
    ensure_built()
    dec = synth.make_case("decode", batch=6, Hq=24, Hkv=4, d_qk=512, d_vo=512, page_size=16,
                          kv_lens=[700, 333, 64, 1, 900, 257], seed=91).to("cuda")
    pre = synth.make_case("prefill", batch=2, Hq=16, Hkv=2, d_qk=512, d_vo=512, page_size=32,
                          kv_lens=[600, 129], qo_lens=[40, 60], seed=92).to("cuda")
    ref_d = [t.clone() for t in pa.run_case(dec)]
    ref_p = [t.clone() for t in pa.run_case(pre)]
    assert "_direct" not in pa.paged_attn_last_variant()
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    results = []
    for _ in range(16):
        with torch.cuda.stream(s1):
            od = pa.run_case(dec)
        with torch.cuda.stream(s2):
            op = pa.run_case(pre)
        results.append((od, op))
    torch.cuda.synchronize()
    assert pa.paged_attn_check_device_error() == 0
    for od, op in results:
        assert torch.equal(od[0], ref_d[0]) and torch.equal(od[1], ref_d[1])
        assert torch.equal(op[0], ref_p[0]) and torch.equal(op[1], ref_p[1])
    pa.paged_attn_release_workspace()  # frees every stream's workspace
    od = pa.run_case(dec)
    torch.cuda.synchronize()
    assert torch.equal(od[0], ref_d[0])
