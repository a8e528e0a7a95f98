"""The append (quantise-on-write) part of the oracle against its pins (CPU only).

The encoders are pinned to torch's float8_e4m3fn cast (a library routine) and to the
e2m1 rounding table written out from the format's definition; the append itself is pinned
through the attention oracle's own page walk (``oracle.gather``): new rows must come back
as the last tokens of their sequence, every other token unchanged, FP8 values within half
an e4m3 step, and NVFP4 blocks built on the e2m1 grid exactly.
"""

import math
import os

import numpy as np
import pytest
import torch

import append_cases as ac
import oracle


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def pin_e4m3_encoder_matches_torch_cast(lib):
    mags = np.array([lib.oracle_e4m3_value(c) for c in range(127)], dtype=np.float64)
    mids = (mags[:-1] + mags[1:]) / 2  # exact in fp32 (at most 5 significant bits)
    vals = np.concatenate([mags, mids, np.nextafter(_f32(mids), np.float32(np.inf)),
                           np.nextafter(_f32(mids), np.float32(0))]).astype(np.float32)
    rng = np.random.default_rng(7)
    vals = np.concatenate([vals, _f32(2.0 ** rng.uniform(-12, math.log2(448), 4000))])
    vals = np.concatenate([vals, -vals, _f32([0.0, -0.0, 448.0, 460.0, -460.0])])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(vals, lib)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:5]]


def pin_e4m3_encoder_saturates(lib):
    got = oracle.e4m3_encode([465.0, 1e6, 3.0e38, -465.0, -1e9], lib)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


# value -> e2m1 code: the grid {0, 0.5, 1, 1.5, 2, 3, 4, 6} is codes 0..7, a tie goes to the
# even code, the sign is bit 3, magnitudes above 6 saturate
E2M1_CASES = [
    (0.0, 0), (-0.0, 8), (0.5, 1), (1.0, 2), (1.5, 3), (2.0, 4), (3.0, 5), (4.0, 6), (6.0, 7),
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
    (0.2499, 0), (0.2501, 1), (0.7499, 1), (1.2501, 3), (2.5001, 5), (4.9999, 6), (5.0001, 7),
    (6.5, 7), (1e9, 7), (-0.1, 8), (-0.75, 10), (-5.0, 14), (-7.0, 15), (-2.5, 12),
]


def pin_e2m1_encoder_table(lib):
    got = oracle.e2m1_encode([v for v, _ in E2M1_CASES], lib)
    assert [int(c) for c in got] == [c for _, c in E2M1_CASES]


def _gather_all(case):
    """Dequantised K and V of every (sequence, kv head), from the unmodified attention
    oracle (the read-back side stays fixed while the append side is mutated)."""
    out = {}
    for b, L in enumerate(case.kv_lens):
        if L == 0:
            continue
        for h in range(case.Hkv):
            out[(b, h, 0)] = oracle.gather(case, b, h, False)
            out[(b, h, 1)] = oracle.gather(case, b, h, True)
    return out


def _new_rows(case, b, h, is_v):
    lo, hi = case.append_indptr[b], case.append_indptr[b + 1]
    t = case.v_new if is_v else case.k_new
    return t[lo:hi, h].float().numpy().astype(np.float64)


SHAPES = [(512, 512, 2, 16), (512, 256, 2, 32), (256, 256, 4, 8)]


def pin_append_bf16_places_rows(lib):
    for shape in SHAPES:
        _bf16_places_rows(shape, lib)


def _bf16_places_rows(shape, lib):
    dqk, dvo, hkv, ps = shape
    case = ac.make(kv_lens=[37, 64, 130, 5], n_new=[5, 64, 0, 5], Hkv=hkv, d_qk=dqk, d_vo=dvo,
                   page_size=ps, kv_dtype=ac.BF16, seed=11)
    before = _gather_all(case)
    cache, sf, skipped = oracle.append_kv(
        case.k_new, case.v_new, case.append_indptr, case.kv_cache, case.kv_indptr, case.kv_indices,
        case.kv_last_page_len, num_kv_heads=hkv, head_dim_qk=dqk, head_dim_vo=dvo, page_size=ps,
        kv_dtype=ac.BF16, lib=lib)
    assert skipped == 0
    after = _gather_all(ac.with_cache(case, cache, sf))
    changed = 0
    for (b, h, is_v), old in before.items():
        n = case.n_new[b]
        new = after[(b, h, is_v)]
        L = case.kv_lens[b]
        np.testing.assert_array_equal(new[:L - n], old[:L - n])
        np.testing.assert_array_equal(new[L - n:], _new_rows(case, b, h, is_v))
        changed += n * (dvo if is_v else dqk) * 2
    # nothing outside the new rows was written (unused slots of last pages, spare pages)
    assert int(np.count_nonzero(cache != case.kv_cache)) <= changed


def pin_append_fp8_within_half_step(lib):
    case = ac.make(kv_lens=[40, 17], n_new=[24, 17], Hkv=2, d_qk=512, d_vo=256, page_size=16,
                   kv_dtype=ac.FP8, seed=12, k_scale=0.05, v_scale=0.0125)
    cache, sf, skipped = oracle.append_kv(
        case.k_new, case.v_new, case.append_indptr, case.kv_cache, case.kv_indptr, case.kv_indices,
        case.kv_last_page_len, num_kv_heads=2, head_dim_qk=512, head_dim_vo=256, page_size=16,
        kv_dtype=ac.FP8, k_scale=case.k_scale, v_scale=case.v_scale, lib=lib)
    assert skipped == 0
    after = _gather_all(ac.with_cache(case, cache, sf))
    for (b, h, is_v), got in after.items():
        n, L = case.n_new[b], case.kv_lens[b]
        x = _new_rows(case, b, h, is_v)
        s = case.v_scale if is_v else case.k_scale
        y = np.abs(x / s)
        # half an e4m3 step at |x / s| (3 mantissa bits, subnormal step 2^-9), saturation at 448
        e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
        half = np.where(y > 448, y - 448, 2.0 ** (e - 4)) * s
        err = np.abs(got[L - n:] - x)
        assert np.all(err <= half * (1 + 1e-6) + 1e-30), float(np.max(err - half))


def pin_append_nvfp4_grid_blocks_round_trip(lib):
    """Blocks built as e2m1 grid values times d = value(sf) * G, with 6 * d present (so the
    block scale is chosen exactly), come back unchanged; distinct values per element catch
    a swapped nibble or a misplaced scale."""
    case = ac.make(kv_lens=[48, 20], n_new=[16, 20], Hkv=2, d_qk=512, d_vo=256, page_size=32,
                   kv_dtype=ac.NVFP4, seed=13, k_scale=2.0 ** -6, v_scale=2.0 ** -4)
    rng = np.random.default_rng(5)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    e4m3 = np.array([oracle.load().oracle_e4m3_value(c) for c in range(1, 127)])  # read side: unmodified
    for t, G in ((case.k_new, case.k_scale), (case.v_new, case.v_scale)):
        shape = t.shape
        vals = rng.choice(grid, size=shape) * rng.choice([-1.0, 1.0], size=shape)
        vals = vals.reshape(shape[0], shape[1], -1, 16)
        vals[..., 0] = 6.0
        sfv = rng.choice(e4m3[(e4m3 >= 2.0 ** -4) & (e4m3 <= 64)], size=vals.shape[:3])
        x = vals * (sfv * G)[..., None]
        t.copy_(torch.from_numpy(x.reshape(shape)).to(torch.bfloat16))
        assert torch.equal(t.double(), torch.from_numpy(x.reshape(shape)))  # exact in bf16
    cache, sf, skipped = oracle.append_kv(
        case.k_new, case.v_new, case.append_indptr, case.kv_cache, case.kv_indptr, case.kv_indices,
        case.kv_last_page_len, num_kv_heads=2, head_dim_qk=512, head_dim_vo=256, page_size=32,
        kv_dtype=ac.NVFP4, k_scale=case.k_scale, v_scale=case.v_scale, sf=case.sf, lib=lib)
    assert skipped == 0
    after = _gather_all(ac.with_cache(case, cache, sf))
    for (b, h, is_v), got in after.items():
        n, L = case.n_new[b], case.kv_lens[b]
        np.testing.assert_array_equal(got[L - n:], _new_rows(case, b, h, is_v))


def pin_append_skips_rows_outside_the_sequence(lib):
    case = ac.make(kv_lens=[10, 20], n_new=[12, 3], Hkv=1, d_qk=256, d_vo=256, page_size=8,
                   kv_dtype=ac.BF16, seed=14)
    cache, _, skipped = oracle.append_kv(
        case.k_new, case.v_new, case.append_indptr, case.kv_cache, case.kv_indptr, case.kv_indices,
        case.kv_last_page_len, num_kv_heads=1, head_dim_qk=256, head_dim_vo=256, page_size=8,
        kv_dtype=ac.BF16, lib=lib)
    assert skipped == 2  # sequence 0 holds 10 tokens: its first 2 of 12 new rows have no place


APPEND_PINS = [pin_e4m3_encoder_matches_torch_cast, pin_e4m3_encoder_saturates, pin_e2m1_encoder_table,
               pin_append_bf16_places_rows, pin_append_fp8_within_half_step,
               pin_append_nvfp4_grid_blocks_round_trip, pin_append_skips_rows_outside_the_sequence]


@pytest.mark.parametrize("pin", APPEND_PINS, ids=[p.__name__ for p in APPEND_PINS])
def test_append_pin(pin):
    pin(oracle.load())


# Plausible mistakes planted in copies of the oracle's append code: each must fail a pin.
APPEND_MUTANTS = {
    "scale_multiplies": ("oracle_e4m3_encode(bf16_float(src[d]) / s)", "oracle_e4m3_encode(bf16_float(src[d]) * s)"),
    "nibbles_swapped": ("(uint8_t)(lo | (hi << 4))", "(uint8_t)(hi | (lo << 4))"),
    "block_scale_divisor": ("(amax / 6.0f) / s", "(amax / 4.0f) / s"),
    "ties_to_odd": ("(dd == bd && (c & 1) == 0)", "(dd == bd && (c & 1) == 1)"),
    "position_off_by_one": ("int64_t t = kv_len - n + j;", "int64_t t = kv_len - n + j - 1;"),
    "v_into_k_block": ("(is_v ? rows * k_row + row * v_row : row * k_row)", "(is_v ? row * v_row : row * k_row)"),
    "v_scales_into_k_scales": ("(is_v ? rows * (d_qk / 16) + row * (d_vo / 16) : row * (d_qk / 16))",
                               "(is_v ? row * (d_vo / 16) : row * (d_qk / 16))"),
    "e4m3_sign_dropped": ("return (uint8_t)(code | (signbit(v) ? 0x80 : 0));", "return (uint8_t)code;"),
    "k_scale_for_v": ("float s = is_v ? v_scale : k_scale;", "float s = k_scale;"),
    "global_scale_dropped": ("float dd = (float)oracle_e4m3_value(sfc) * s;",
                             "float dd = (float)oracle_e4m3_value(sfc);"),
    "head_stride_dropped": ("int64_t row = (int64_t)h * page_size + slot;", "int64_t row = slot;"),
}


@pytest.mark.parametrize("name", sorted(APPEND_MUTANTS))
def test_append_mutant_is_caught(name, tmp_path):
    old, new = APPEND_MUTANTS[name]
    src_path = os.path.join(os.path.dirname(oracle.__file__), "paged_attn_oracle.c")
    src = open(src_path).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique / missing"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.compile_oracle(str(path), str(tmp_path / "libmutant.so")))
    failed = []
    for pin in APPEND_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
