"""The calls inside a CUDA graph: after one eager call has grown the workspace, decode and
prefill (bf16, and FP8 / NVFP4 through the bf16 copy of the pages) allocate nothing,
synchronise nothing and take every size from device memory, so a captured call replays
correctly, also after its inputs change in place."""

import pytest
import torch

import paged_gqa_attention_hd512_gb300 as pa
import synth
from parity import ensure_built

pytestmark = pytest.mark.gpu


def _call(case, kw, out, lse):
    if case.phase == "decode":
        return pa.paged_attn_decode(case.q, case.kv_cache, case.kv_indptr, case.kv_indices, case.kv_last_page_len,
                                    out=out, lse=lse, **kw)
    return pa.paged_attn_prefill(case.q, case.qo_indptr, case.kv_cache, case.kv_indptr, case.kv_indices,
                                 case.kv_last_page_len, causal=bool(case.causal), out=out, lse=lse, **kw)


def _capture_and_check(case, seed_change):
    ensure_built()
    kw = pa.case_args(case)  # device scale tensors made once, outside the capture
    out0, lse0 = pa.run_case(case)
    torch.cuda.synchronize()
    out, lse = torch.empty_like(out0), torch.empty_like(lse0)
    _call(case, kw, out, lse)  # grows the workspace for this shape
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _call(case, kw, out, lse)
    out.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pa.paged_attn_check_device_error() == 0
    assert torch.equal(out, out0) and torch.equal(lse, lse0)
    # new query values in place: the replay reads them
    q2 = synth.make_case(case.phase, device="cuda", **seed_change).q
    case.q.copy_(q2)
    g.replay()
    ref_out, ref_lse = pa.run_case(case)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


@pytest.mark.parametrize("direct", [0, 1])
def test_decode_in_a_cuda_graph(direct):
    """The planned path (planner, split-K decode, merge) and the single-launch path."""
    kw = dict(batch=5, Hq=24, Hkv=4, d_qk=512, d_vo=512, page_size=16, kv_lens=[1, 100, 700, 64, 333])
    pa.paged_attn_set_decode_chunk_pages(0)
    pa.paged_attn_set_decode_direct(direct)
    try:
        case = synth.make_case("decode", seed=81, **kw).to("cuda")
        _capture_and_check(case, dict(kw, seed=82))
        assert pa.paged_attn_last_variant().endswith("_direct") == bool(direct)
    finally:
        pa.paged_attn_set_decode_direct(-1)


def test_capture_on_a_fresh_stream_uses_the_default_streams_workspace():
    """Warm-up on the default stream, capture on a stream that has never called the
    library: the call allocates nothing during the capture and replays correctly."""
    ensure_built()
    kw = dict(batch=3, Hq=8, Hkv=2, d_qk=512, d_vo=512, page_size=16, kv_lens=[90, 33, 300])
    case = synth.make_case("decode", seed=85, **kw).to("cuda")
    kwa = pa.case_args(case)
    out0, lse0 = pa.run_case(case)
    torch.cuda.synchronize()
    out, lse = torch.empty_like(out0), torch.empty_like(lse0)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _call(case, kwa, out, lse)
    g.replay()
    torch.cuda.synchronize()
    assert pa.paged_attn_check_device_error() == 0
    assert torch.equal(out, out0) and torch.equal(lse, lse0)


@pytest.mark.parametrize("dt", [synth.KV_BF16, synth.KV_FP8, synth.KV_NVFP4])
def test_prefill_in_a_cuda_graph(dt):
    kw = dict(batch=2, Hq=16, Hkv=2, d_qk=512, d_vo=512 if dt == synth.KV_BF16 else 256, page_size=32,
              kv_lens=[300, 129], qo_lens=[300, 60], kv_dtype=dt)
    case = synth.make_case("prefill", seed=83, **kw).to("cuda")
    _capture_and_check(case, dict(kw, seed=84))
