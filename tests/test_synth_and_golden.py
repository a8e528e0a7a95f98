"""Seeded generator, input encoders and the stored oracle fixture (CPU only)."""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_mqa_decode.txt")


def test_generator_is_deterministic_and_standardised():
    a = synth.normal_bf16(5, synth.TID_K, 1000, 200000, "cpu")
    b = synth.normal_bf16(5, synth.TID_K, 1000, 200000, "cpu")
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c = synth.normal_bf16(5, synth.TID_V, 1000, 200000, "cpu")
    assert not torch.equal(a, c)
    x = a.double()
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
    assert float(x.abs().max()) <= math.sqrt(3.0 * 4.0) + 1e-2  # Irwin-Hall(4) bound


def test_generator_window_consistency():
    """An element's value does not depend on which window of indices generated it."""
    whole = synth.normal_bf16(9, synth.TID_Q, 0, 4096, "cpu")
    part = synth.normal_bf16(9, synth.TID_Q, 1000, 96, "cpu")
    assert torch.equal(whole[1000:1096].view(torch.int16), part.view(torch.int16))
    big = torch.tensor([2 ** 33 + 5, 2 ** 34 + 7], dtype=torch.int64)
    v = synth.normal_f32(9, synth.TID_Q, big)
    assert torch.isfinite(v).all()


def test_e2m1_encoder_round_to_nearest_even():
    y = torch.tensor([0.0, 0.2, 0.25, 0.26, 0.75, 1.25, 1.3, 1.75, 2.5, 2.6, 3.5, 5.0, 5.1, 9.0,
                      -0.75, -6.0])
    want = [0, 0, 0, 1, 2, 2, 3, 4, 4, 5, 6, 6, 7, 7, 8 | 2, 8 | 7]
    assert synth.e2m1_encode(y).tolist() == want


def test_nvfp4_encoder_error_bound():
    x = synth.normal_bf16(3, synth.TID_K, 0, 64 * 512, "cpu").float().view(64, 512)
    g = synth.nvfp4_global_scale(float(x.abs().max()))
    assert g == 2.0 ** round(math.log2(g))
    packed, sf = synth.nvfp4_encode_rows(x, g)
    lib = oracle.load()
    nib = torch.stack([packed & 15, packed >> 4], dim=-1).view(64, 512)
    vals = torch.tensor([lib.oracle_e2m1_value(i) for i in range(16)], dtype=torch.float64)
    sfv = torch.tensor([lib.oracle_e4m3_value(int(s)) for s in sf.view(-1).tolist()],
                       dtype=torch.float64).view(64, 32)
    deq = vals[nib.long()] * sfv.repeat_interleave(16, dim=1) * g
    # e2m1 steps are at most 2 (between 4 and 6) in units of the block scale
    bound = sfv.repeat_interleave(16, dim=1) * g * 1.0 + 1e-12
    assert torch.all((deq - x.double()).abs() <= bound)


def test_fp8_encoder_matches_definition():
    x = torch.linspace(-448.0, 448.0, 4001)
    codes = synth.e4m3_encode(x)
    lib = oracle.load()
    dec = torch.tensor([lib.oracle_e4m3_value(int(c)) for c in codes.tolist()])
    # round to nearest: no representable value is closer than the chosen one
    allv = torch.tensor([lib.oracle_e4m3_value(c) for c in range(256) if c not in (0x7F, 0xFF)])
    best = (allv[None, :] - x[:, None].double()).abs().min(dim=1).values
    assert torch.allclose((dec - x.double()).abs(), best, atol=0, rtol=0)


def test_page_table_is_a_permutation():
    c = synth.make_case("decode", batch=3, Hq=2, Hkv=1, d_qk=32, d_vo=32, page_size=4,
                        kv_lens=[5, 8, 13], seed=3)
    ind = c.kv_indices.tolist()
    assert sorted(ind) == list(range(c.num_pages))
    assert c.kv_indptr.tolist() == [0, 2, 4, 8]
    assert c.kv_last_page_len.tolist() == [1, 4, 1]


def test_workload_lengths():
    lens = synth.workload_kv_lens("gqa_decode_bf16")
    assert len(lens) == 64 and min(lens) >= 1024 and max(lens) <= 8192


def test_golden_tiny_decode():
    c = synth.workload("tiny_mqa_decode")
    out, lse = oracle.full(c, threads=1)
    rows = [l.split() for l in open(GOLDEN) if not l.startswith("#")]
    assert len(rows) == 16
    for r in rows:
        b, h = int(r[0]), int(r[1])
        vals = np.array([float(x) for x in r[2:]])
        got = np.concatenate([[lse[b, h], out[b, h].sum()], out[b, h, :8]])
        assert np.allclose(got, vals, rtol=1e-12, atol=1e-12)
