"""Append codes over every bf16 input value (needs a GPU): each FP8 and NVFP4 code is a
rounding of the quotient x / scale (or x / d, d the NVFP4 block's decoded scale) that the
kernel forms from a reciprocal and two exact residual corrections where the operands are in
range, and by IEEE division elsewhere.  Both must give the correctly rounded quotient's
code, which the oracle forms by fp32 division: compared byte for byte, for every finite
bf16 value (and the infinities), against divisors of either kind."""

import numpy as np
import pytest
import torch

import append_cases as ac
from parity import ensure_built
from test_append_gpu import _assert_bytes_equal, _oracle, _run_gpu

pytestmark = pytest.mark.gpu


def _bf16_values(with_inf=True):
    """Every bf16 bit pattern that is not a NaN, as int16 bits."""
    bits = np.arange(65536, dtype=np.uint32)
    exp, man = (bits >> 7) & 0xFF, bits & 0x7F
    keep = ~((exp == 0xFF) & ((man != 0) | (not with_inf)))
    return bits[keep].astype(np.uint16)


def _to_bf16(bits_u16):
    return torch.from_numpy(bits_u16.astype(np.int16)).view(torch.bfloat16)


def _f32(v):
    return float(np.float32(v))


FP8_SCALES = [1.0, 0.0125, 1.0 / 3.0, 7.1, 3.3e4, 1.37 * 2.0 ** -20, np.nextafter(np.float32(2.0), np.float32(0)),
              np.nextafter(np.float32(1.0), np.float32(2.0)), 5e-37, 2.0 ** 110]


@pytest.mark.parametrize("scale", [_f32(s) for s in FP8_SCALES])
def test_append_fp8_every_bf16_value(scale):
    """All 65282 non-NaN bf16 values, shuffled over the K and V rows of 64 new tokens, at
    one per-tensor scale (among them scales whose quotients overflow fp32 for large x, and
    one beyond the reciprocal form's range)."""
    ensure_built()
    vals = _bf16_values()
    rng = np.random.default_rng(11)
    vals = vals[rng.permutation(vals.size)]
    tokens, hkv, d = 64, 2, 256
    slots = tokens * hkv * d * 2
    buf = np.zeros(slots, dtype=np.uint16)
    buf[:vals.size] = vals
    case = ac.make(kv_lens=[tokens], n_new=[tokens], Hkv=hkv, d_qk=d, d_vo=d, page_size=16, kv_dtype=ac.FP8,
                   seed=12, k_scale=scale, v_scale=_f32(scale * 1.5))
    half = slots // 2
    case.k_new = _to_bf16(buf[:half]).view(tokens, hkv, d).clone()
    case.v_new = _to_bf16(buf[half:]).view(tokens, hkv, d).clone()
    cache, _, code = _run_gpu(case)
    ref_cache, _, skipped = _oracle(case)
    assert code == 0 and skipped == 0
    _assert_bytes_equal(cache, ref_cache, f"every bf16 value, scale {scale}")


@pytest.mark.parametrize("g", [_f32(0.7314), _f32(3.1e-3), 2.0 ** -7, _f32(2.9e4)])
def test_append_nvfp4_every_bf16_value(g):
    """Every finite bf16 value, sorted by magnitude and cut into runs of 15; each run forms
    five blocks with a sixteenth element that sets the block maximum at 1, 1.5, 2.7, 5.3
    or 12 times the run's largest magnitude, so the quotients x / d spread over the e2m1
    range (and below it), at one global scale."""
    ensure_built()
    vals = _bf16_values(with_inf=False)
    f = _to_bf16(vals).float().numpy()
    order = np.argsort(np.abs(f), kind="stable")
    vals, f = vals[order], f[order]
    n_runs = vals.size // 15
    blocks = []
    for m in (1.0, 1.5, 2.7, 5.3, 12.0):
        for r in range(n_runs):
            run = vals[15 * r:15 * r + 15]
            top = float(np.abs(f[15 * r:15 * r + 15]).max())
            anchor = torch.tensor([top * m]).to(torch.bfloat16)
            if not torch.isfinite(anchor).all():
                anchor = torch.tensor([top]).to(torch.bfloat16)
            a_bits = anchor.view(torch.int16).numpy().astype(np.uint16)
            blocks.append(np.concatenate([a_bits, run]))
    data = np.concatenate(blocks)
    hkv, d = 2, 512
    per_token = hkv * d * 2
    tokens = -(-data.size // per_token)
    buf = np.zeros(tokens * per_token, dtype=np.uint16)
    buf[:data.size] = data
    case = ac.make(kv_lens=[tokens], n_new=[tokens], Hkv=hkv, d_qk=d, d_vo=d, page_size=16, kv_dtype=ac.NVFP4,
                   seed=13, k_scale=g, v_scale=g)
    half = buf.size // 2
    case.k_new = _to_bf16(buf[:half]).view(tokens, hkv, d).clone()
    case.v_new = _to_bf16(buf[half:]).view(tokens, hkv, d).clone()
    cache, sf, code = _run_gpu(case)
    ref_cache, ref_sf, skipped = _oracle(case)
    assert code == 0 and skipped == 0
    _assert_bytes_equal(cache, ref_cache, f"every bf16 value, global scale {g}")
    _assert_bytes_equal(sf, ref_sf, f"scales, global scale {g}")


def test_append_nvfp4_saturated_block_scale():
    """A block maximum so large against the global scale that the block scale saturates
    at the e4m3 maximum: x / d then reaches past fp32's range for the largest values (the
    kernel takes the IEEE division there), and the codes saturate at 6 as in the oracle."""
    ensure_built()
    g = _f32(1e-3)
    case = ac.make(kv_lens=[2], n_new=[2], Hkv=1, d_qk=256, d_vo=256, page_size=8, kv_dtype=ac.NVFP4,
                   seed=14, k_scale=g, v_scale=g)
    big = [3.0e38, -3.0e38, 1.0e38, 2.5e36, -7.0, 1.0, 1.0e30, -1.0e-30]
    for t in (case.k_new, case.v_new):
        t[0, 0, 0:8] = torch.tensor(big)
        t[1, 0, 16:24] = torch.tensor(big[::-1])
    cache, sf, code = _run_gpu(case)
    ref_cache, ref_sf, skipped = _oracle(case)
    assert code == 0 and skipped == 0
    _assert_bytes_equal(cache, ref_cache, "saturated block scale")
    _assert_bytes_equal(sf, ref_sf, "saturated block scale, scales")
