"""paged_attn_decode_noalloc: the decode call for callers that cannot allocate device
memory (a framework that owns every byte of device memory, a hard memory budget, code
that must not trigger cudaMalloc's implicit synchronisation mid-step).  It must give the
same result as paged_attn_decode, on consecutive calls that share its fixed scratch
array, and refuse problems whose scratch does not fit.

The file is named so that pytest collects it last.
"""

import pytest
import torch

import paged_gqa_attention_hd512_gb300 as pa
import synth
from parity import OUT_ABS, OUT_REL, LSE_ABS, ensure_built

pytestmark = pytest.mark.gpu


def _close(a, b, what):
    a, b = a.float(), b.float()
    err = (a - b).abs()
    assert bool(torch.all(err <= OUT_ABS + OUT_REL * b.abs())), f"{what}: max err {float(err.max())}"


@pytest.mark.parametrize("dt", [synth.KV_BF16, synth.KV_FP8, synth.KV_NVFP4])
def test_noalloc_matches_decode_on_two_calls(dt):
    ensure_built()
    pa.paged_attn_set_decode_chunk_pages(0)
    case = synth.make_case("decode", batch=8, Hq=24, Hkv=4, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[1, 37, 100, 255, 256, 640, 901, 64], kv_dtype=dt, seed=71).to("cuda")
    kw = pa.case_args(case)
    ref_out, ref_lse = pa.run_case(case)
    torch.cuda.synchronize()
    assert pa.paged_attn_check_device_error() == 0
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        pa.paged_attn_decode_noalloc(case.q, case.kv_cache, case.kv_indptr, case.kv_indices,
                                     case.kv_last_page_len, out=out, lse=lse, **kw)
        torch.cuda.synchronize()
        assert pa.paged_attn_last_variant().endswith("_noalloc")
        _close(out, ref_out, f"call {call} out")
        assert float((lse - ref_lse).abs().max()) <= LSE_ABS, f"call {call} lse"


def test_noalloc_rejects_scratch_overflow():
    ensure_built()
    batch, hq = 2048, 16  # >= 2048 split-K rows of 16 x 512 fp32 partials: above 32 MiB
    q = torch.zeros(batch, hq, 512, dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros(batch * 16 * 1024 * 2, dtype=torch.uint8, device="cuda")
    indptr = torch.arange(batch + 1, dtype=torch.int32, device="cuda")
    indices = torch.arange(batch, dtype=torch.int32, device="cuda")
    last = torch.ones(batch, dtype=torch.int32, device="cuda")
    out = torch.empty(batch, hq, 512, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.paged_attn_decode_noalloc(q, cache, indptr, indices, last, out=out, lse=None, num_kv_heads=1,
                                     head_dim_vo=512, page_size=16, sm_scale=0.04)
    assert e.value.status == pa.PA_ERR_SCRATCH
