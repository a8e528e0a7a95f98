"""paged_attn_decode_noalloc: the decode call for callers that cannot allocate device
memory (a framework that owns every byte of device memory, a hard memory budget, code
that must not trigger cudaMalloc's implicit synchronisation mid-step).  It must give the
same result as paged_attn_decode and as the oracle, on consecutive calls of different
shapes that share its fixed scratch array, including problems whose split-K partials
make it use fewer KV splits than paged_attn_decode would; it must not allocate device
memory; and it must refuse problems whose scratch does not fit.

The file is named so that pytest collects it last.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_attention_hd512_gb300 as pa
import synth
from parity import OUT_ABS, OUT_REL, LSE_ABS, compare, ensure_built

pytestmark = pytest.mark.gpu

SCRATCH = pa.PA_NOALLOC_SCRATCH_BYTES


def _close(a, b, what):
    a, b = a.float(), b.float()
    err = (a - b).abs()
    assert bool(torch.all(err <= OUT_ABS + OUT_REL * b.abs())), f"{what}: max err {float(err.max())}"


def _noalloc(case):
    """One paged_attn_decode_noalloc call on a device case, into NaN-filled outputs."""
    out = torch.full((case.batch, case.Hq, case.d_vo), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((case.batch, case.Hq), float("nan"), dtype=torch.float32, device="cuda")
    pa.paged_attn_decode_noalloc(case.q, case.kv_cache, case.kv_indptr, case.kv_indices, case.kv_last_page_len,
                                 out=out, lse=lse, **pa.case_args(case))
    torch.cuda.synchronize()
    assert pa.paged_attn_last_variant().endswith("_noalloc")
    return out, lse


def _against_oracle(host, out, lse, what):
    ref_out, ref_lse = oracle.full(host)
    n = host.batch * host.Hq
    compare(out.reshape(n, -1), lse.reshape(n), ref_out.reshape(n, -1), ref_lse.reshape(n), what)


def _split_rows(batch, hq, hkv, dvo, sms):
    """The no-alloc call's bound on split-K chunks (its fixed-array arithmetic) and the
    bound paged_attn_decode uses."""
    def up(v):
        return (v + 255) // 256 * 256
    per_chunk = 16 + hq * 8 + hq * dvo * 4
    fixed = 256 + 256 + up(batch * 8) + up(batch * hkv * 4) + 4 * 256
    fit = (SCRATCH - fixed) // per_chunk - batch
    usual = (16 * sms + hkv - 1) // hkv
    return fit, usual


@pytest.mark.parametrize("dt", [synth.KV_BF16, synth.KV_FP8, synth.KV_NVFP4])
def test_noalloc_matches_decode_on_two_calls(dt):
    """Call 1 and call 2 have different shapes (fewer sequences and chunks in call 2), so
    a work list or partial left in the shared array by call 1 cannot pass for call 2's."""
    ensure_built()
    pa.paged_attn_set_decode_chunk_pages(0)
    big = synth.make_case("decode", batch=8, Hq=24, Hkv=4, d_qk=512, d_vo=512, page_size=16,
                          kv_lens=[1, 37, 100, 255, 256, 640, 901, 64], kv_dtype=dt, seed=71).to("cuda")
    small = synth.make_case("decode", batch=3, Hq=24, Hkv=4, d_qk=512, d_vo=512, page_size=16,
                            kv_lens=[300, 17, 129], kv_dtype=dt, seed=72).to("cuda")
    for call, case in enumerate((big, small)):
        ref_out, ref_lse = pa.run_case(case)
        torch.cuda.synchronize()
        assert pa.paged_attn_check_device_error() == 0
        ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
        out, lse = _noalloc(case)
        _close(out, ref_out, f"call {call} out")
        assert float((lse - ref_lse).abs().max()) <= LSE_ABS, f"call {call} lse"
    assert pa.paged_attn_check_device_error() == 0


def test_noalloc_fewer_splits_than_usual_matches_oracle():
    """A batch whose split-K partials (batch x 16 heads x 512 fp32 per chunk) do not fit
    the fixed array at paged_attn_decode's chunk count: the call cuts fewer, longer
    chunks.  Checked against the oracle, then a second, smaller call on the same array."""
    ensure_built()
    pa.paged_attn_set_decode_chunk_pages(0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    batch, hq, hkv = 256, 16, 1
    fit, usual = _split_rows(batch, hq, hkv, 512, sms)
    assert 1 <= fit < usual, (fit, usual)  # the case reaches the reduced-split branch
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 700, batch)]
    lens[0], lens[1] = 1, 699
    host = synth.make_case("decode", batch=batch, Hq=hq, Hkv=hkv, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=lens, seed=73)
    out, lse = _noalloc(host.to("cuda"))
    assert pa.paged_attn_check_device_error() == 0
    _against_oracle(host, out, lse, "reduced splits")

    host2 = synth.make_case("decode", batch=5, Hq=8, Hkv=2, d_qk=512, d_vo=256, page_size=8,
                            kv_lens=[5, 80, 1000, 33, 64], kv_dtype=synth.KV_FP8, seed=74)
    out2, lse2 = _noalloc(host2.to("cuda"))
    assert pa.paged_attn_check_device_error() == 0
    _against_oracle(host2, out2, lse2, "second call")


def test_noalloc_allocates_no_device_memory():
    """With the library's workspace released, no-alloc calls leave free device memory
    unchanged (a call that grew the workspace would take at least its 1 MiB granule)."""
    ensure_built()
    pa.paged_attn_set_decode_chunk_pages(0)
    case = synth.make_case("decode", batch=64, Hq=16, Hkv=2, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[200 + 37 * b for b in range(64)], seed=75).to("cuda")
    kw = pa.case_args(case)
    out = torch.empty(case.batch, case.Hq, case.d_vo, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(case.batch, case.Hq, dtype=torch.float32, device="cuda")

    def call():  # creates no tensor: torch's allocator stays out of the measured window
        pa.paged_attn_decode_noalloc(case.q, case.kv_cache, case.kv_indptr, case.kv_indices,
                                     case.kv_last_page_len, out=out, lse=lse, **kw)

    call()  # the first call on the device resolves the array
    torch.cuda.synchronize()
    assert pa.load().paged_attn_release_workspace() == pa.PA_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 > free0 - (1 << 20), (free0, free1)
    assert pa.paged_attn_check_device_error() == 0


def test_noalloc_error_word_is_reported_and_cleared():
    """A wait site recorded in the fixed array's error word is reported by
    paged_attn_check_device_error and cleared by it (as is the workspace's)."""
    ensure_built()
    case = synth.make_case("decode", batch=2, Hq=8, Hkv=1, d_qk=512, d_vo=512, page_size=16,
                           kv_lens=[37, 64], seed=76).to("cuda")
    _noalloc(case)
    assert pa.paged_attn_check_device_error() == 0
    pa.paged_attn_debug_set_error_word(1, 4242)
    assert pa.paged_attn_check_device_error() == 4242
    assert pa.paged_attn_check_device_error() == 0
    pa.paged_attn_debug_set_error_word(0, 17)
    assert pa.paged_attn_check_device_error() == 17
    assert pa.paged_attn_check_device_error() == 0


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
