"""Pins of the fp64 oracle to things other than itself.

Each ``pin_*`` function takes a loaded oracle library (``oracle.load()`` or a deliberately
broken copy) and raises AssertionError when the oracle disagrees with:
  * the number-format definitions (torch's float8 decoder, the e2m1 value table),
  * an independent contiguous-layout attention built from library routines
    (tests/dense_reference.py: torch reshapes + scipy softmax / logsumexp),
  * invariants and closed forms the mathematics fixes (page-order invariance, a single
    key returns its value, identical keys return the mean, split-K merge = unsplit,
    prefill row i = decode over i+1 keys, window limits, GQA = per-head MHA, empty rows).
"""

import math

import numpy as np
import torch

import oracle
import synth
from dense_reference import E2M1_TABLE, attention_row, seq_kv
from mask_cases import attach as attach_mask

REL = 1e-12


def _close(a, b, rel=REL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), what
    assert np.array_equal(a[~fin], b[~fin]), what
    scale = max(1e-300, float(np.abs(b[fin]).max()) if fin.any() else 1.0)
    err = float(np.abs(a[fin] - b[fin]).max()) if fin.any() else 0.0
    assert err <= rel * scale, f"{what}: max err {err:.3e} vs scale {scale:.3e}"


def _all_rows(case):
    tok = np.repeat(np.arange(case.total_q), case.Hq)
    head = np.tile(np.arange(case.Hq), case.total_q)
    return tok, head


def _check_dense(case, lib, what):
    tok, head = _all_rows(case)
    out, lse = oracle.rows(case, tok, head, lib=lib, threads=2)
    for r, (t, h) in enumerate(zip(tok, head)):
        o_ref, l_ref = attention_row(case, int(t), int(h))
        _close(out[r], o_ref, what=f"{what} out row {t},{h}")
        _close([lse[r]], [l_ref], what=f"{what} lse row {t},{h}")


# ------------------------------------------------------------------------------ formats
def pin_formats_e4m3(lib):
    codes = torch.arange(256, dtype=torch.int64).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([lib.oracle_e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    # spot values from the format definition: max normal, min normal, min subnormal
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9


def pin_formats_e2m1(lib):
    got = np.array([lib.oracle_e2m1_value(c) for c in range(16)])
    ref = np.concatenate([E2M1_TABLE, -E2M1_TABLE])
    assert np.array_equal(got, ref)


def pin_formats_bf16(lib):
    g = torch.Generator().manual_seed(7)
    bits = torch.randint(0, 65536, (2000,), generator=g, dtype=torch.int64)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # finite patterns only
    ref = bits.to(torch.int16).view(torch.bfloat16).double().numpy()
    got = np.array([lib.oracle_bf16_value(int(b)) for b in bits.tolist()])
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------------------ dense
def pin_dense_tiny_mqa_decode(lib):
    _check_dense(synth.workload("tiny_mqa_decode"), lib, "tiny mqa decode")


def pin_dense_gqa_window_decode(lib):
    c = synth.make_case("decode", batch=3, Hq=6, Hkv=2, d_qk=64, d_vo=64, page_size=4,
                        kv_lens=[1, 9, 12], window_left=5, seed=11)
    _check_dense(c, lib, "gqa window decode")


def pin_dense_prefill_with_prefix(lib):
    c = synth.make_case("prefill", batch=2, Hq=4, Hkv=2, d_qk=32, d_vo=32, page_size=8,
                        kv_lens=[20, 7], qo_lens=[5, 7], seed=12)
    _check_dense(c, lib, "causal prefill with prefix")


def pin_dense_prefill_noncausal_window(lib):
    c = synth.make_case("prefill", batch=2, Hq=2, Hkv=1, d_qk=32, d_vo=32, page_size=4,
                        kv_lens=[10, 6], qo_lens=[4, 6], causal=0, window_left=3, seed=13)
    _check_dense(c, lib, "non-causal windowed prefill")


def pin_dense_fp8_decode(lib):
    c = synth.make_case("decode", batch=2, Hq=4, Hkv=2, d_qk=64, d_vo=64, page_size=8,
                        kv_lens=[13, 16], kv_dtype=synth.KV_FP8, seed=14)
    # the scales are caller inputs: make K's and V's differ so neither can stand in for
    # the other
    c.v_scale = c.v_scale * 3.0
    _check_dense(c, lib, "fp8 decode")


def pin_dense_nvfp4_asym_prefill(lib):
    c = synth.make_case("prefill", batch=2, Hq=4, Hkv=1, d_qk=64, d_vo=32, page_size=4,
                        kv_lens=[9, 6], qo_lens=[9, 6], kv_dtype=synth.KV_NVFP4, seed=15)
    _check_dense(c, lib, "nvfp4 asymmetric prefill")


# ------------------------------------------------------------------------------ invariants
def pin_page_permutation(lib):
    c = synth.make_case("decode", batch=2, Hq=4, Hkv=2, d_qk=32, d_vo=32, page_size=4,
                        kv_lens=[11, 16], seed=21)
    tok, head = _all_rows(c)
    out0, lse0 = oracle.rows(c, tok, head, lib=lib, threads=1)
    perm = torch.from_numpy(np.random.default_rng(5).permutation(c.num_pages)).long()
    pages = c.kv_cache.view(c.num_pages, -1)
    moved = torch.empty_like(pages)
    moved[perm] = pages
    c2 = c.to("cpu")
    c2.kv_cache = moved.reshape(-1)
    c2.kv_indices = perm[c.kv_indices.long()].to(torch.int32)
    out1, lse1 = oracle.rows(c2, tok, head, lib=lib, threads=1)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_single_token(lib):
    c = synth.make_case("decode", batch=1, Hq=2, Hkv=1, d_qk=64, d_vo=64, page_size=16,
                        kv_lens=[1], seed=22)
    out, lse = oracle.rows(c, [0, 0], [0, 1], lib=lib, threads=1)
    K, V = seq_kv(c, 0, 0)
    for r in range(2):
        assert np.array_equal(out[r], V[0])
        s0 = float(c.q[0, r].double().numpy() @ K[0]) * c.sm_scale
        _close([lse[r]], [s0], what="single-token lse")


def pin_identical_keys(lib):
    c = synth.make_case("decode", batch=1, Hq=1, Hkv=1, d_qk=32, d_vo=32, page_size=4,
                        kv_lens=[10], seed=23)
    H, ps, dq, dv = c.Hkv, c.page_size, c.d_qk, c.d_vo
    pages = c.kv_cache.view(torch.bfloat16).view(c.num_pages, -1)
    krow = pages[c.kv_indices[0].item(), :dq].clone()
    pages[:, :H * ps * dq] = krow.repeat(H * ps)
    out, lse = oracle.rows(c, [0], [0], lib=lib, threads=1)
    K, V = seq_kv(c, 0, 0)
    _close(out[0], V.mean(axis=0), what="identical keys mean")
    s = float(c.q[0, 0].double().numpy() @ K[0]) * c.sm_scale
    _close([lse[0]], [s + math.log(10)], what="identical keys lse")


def pin_split_merge(lib):
    c = synth.make_case("decode", batch=2, Hq=3, Hkv=1, d_qk=32, d_vo=32, page_size=4,
                        kv_lens=[23, 17], seed=24)
    rng = np.random.default_rng(3)
    for b in range(2):
        L = c.kv_lens[b]
        npg = (L + 3) // 4
        cuts = sorted(set(rng.choice(np.arange(1, npg), size=min(3, npg - 1), replace=False)))
        bounds = [0] + [4 * x for x in cuts] + [L]
        for h in range(3):
            whole, lse_w = oracle.rows(c, [b], [h], lib=lib, threads=1)
            n = len(bounds) - 1
            parts, lses = oracle.rows(c, [b] * n, [h] * n, key_lo=bounds[:-1], key_hi=bounds[1:],
                                      lib=lib, threads=1)
            o, l = oracle.merge(lses, parts, lib=lib)
            _close(o, whole[0], what="split-K merge out")
            _close([l], [lse_w[0]], what="split-K merge lse")
            # and the partial itself against the dense reference on its key range
            o_ref, l_ref = attention_row(c, b, h, key_range=(bounds[0], bounds[1]))
            _close(parts[0], o_ref, what="partial out")
            _close([lses[0]], [l_ref], what="partial lse")


def _truncated_decode(c, b, n_keys, q_rows):
    """Decode case over the first n_keys keys of sequence b of case c."""
    ps = c.page_size
    ip = c.kv_indptr.tolist()
    npg = (n_keys + ps - 1) // ps
    d = c.to("cpu")
    d.phase, d.batch, d.causal = "decode", 1, 1
    d.kv_indptr = torch.tensor([0, npg], dtype=torch.int32)
    d.kv_indices = c.kv_indices[ip[b]:ip[b] + npg].clone()
    d.kv_last_page_len = torch.tensor([n_keys - (npg - 1) * ps], dtype=torch.int32)
    d.q = q_rows.reshape(1, c.Hq, c.d_qk).clone()
    d.qo_indptr = torch.tensor([0, 1], dtype=torch.int32)
    d.kv_lens, d.qo_lens = [n_keys], [1]
    return d


def pin_prefill_row_is_decode(lib):
    c = synth.make_case("prefill", batch=1, Hq=4, Hkv=2, d_qk=32, d_vo=32, page_size=4,
                        kv_lens=[13], qo_lens=[13], seed=25)
    out, lse = oracle.rows(c, *_all_rows(c), lib=lib, threads=1)
    out = out.reshape(13, 4, -1)
    lse = lse.reshape(13, 4)
    for i in (0, 3, 4, 12):
        d = _truncated_decode(c, 0, i + 1, c.q[i])
        o2, l2 = oracle.rows(d, [0] * 4, list(range(4)), lib=lib, threads=1)
        assert np.array_equal(out[i], o2) and np.array_equal(lse[i], l2), i


def pin_window_limits(lib):
    c = synth.make_case("decode", batch=2, Hq=2, Hkv=1, d_qk=32, d_vo=32, page_size=4,
                        kv_lens=[9, 14], seed=26)
    tok, head = _all_rows(c)
    base, lb = oracle.rows(c, tok, head, lib=lib, threads=1)
    wide = c.to("cpu")
    wide.window_left = 13  # >= kv_len - 1 for every sequence
    o1, l1 = oracle.rows(wide, tok, head, lib=lib, threads=1)
    assert np.array_equal(base, o1) and np.array_equal(lb, l1)
    zero = c.to("cpu")
    zero.window_left = 0
    o0, _ = oracle.rows(zero, tok, head, lib=lib, threads=1)
    for r, t in enumerate(tok):
        _, V = seq_kv(c, int(t), 0)
        assert np.array_equal(o0[r], V[c.kv_lens[int(t)] - 1])


def _single_head(c, h):
    kvh = h // c.group
    H, ps, dq, dv, P = c.Hkv, c.page_size, c.d_qk, c.d_vo, c.num_pages
    pages = c.kv_cache.view(torch.bfloat16).view(P, -1)
    K = pages[:, :H * ps * dq].reshape(P, H, ps * dq)[:, kvh]
    V = pages[:, H * ps * dq:].reshape(P, H, ps * dv)[:, kvh]
    s = c.to("cpu")
    s.Hq, s.Hkv = 1, 1
    s.kv_cache = torch.cat([K, V], dim=1).contiguous().view(torch.uint8).reshape(-1)
    s.q = c.q[:, h:h + 1].contiguous()
    return s


def pin_gqa_per_head(lib):
    c = synth.make_case("prefill", batch=2, Hq=6, Hkv=2, d_qk=32, d_vo=32, page_size=4,
                        kv_lens=[7, 10], qo_lens=[3, 10], seed=27)
    tok, head = _all_rows(c)
    out, lse = oracle.rows(c, tok, head, lib=lib, threads=1)
    for h in range(6):
        s = _single_head(c, h)
        t = np.arange(c.total_q)
        o2, l2 = oracle.rows(s, t, np.zeros_like(t), lib=lib, threads=1)
        sel = head == h
        assert np.array_equal(out[sel], o2) and np.array_equal(lse[sel], l2), h


def pin_empty_sequence(lib):
    c = synth.make_case("decode", batch=2, Hq=2, Hkv=1, d_qk=32, d_vo=32, page_size=4,
                        kv_lens=[0, 5], seed=28)
    out, lse = oracle.rows(c, [0, 0, 1], [0, 1, 0], lib=lib, threads=1)
    assert np.all(out[:2] == 0.0) and np.all(np.isneginf(lse[:2]))
    o_ref, l_ref = attention_row(c, 1, 0)
    _close(out[2], o_ref, what="row after empty sequence")


# ------------------------------------------------------------------------- custom masks
def pin_dense_custom_mask(lib):
    """Random, span and sparse masks against the dense reference (numpy's bit unpacking)."""
    for n, (kind, causal) in enumerate((("random", 0), ("spans", 1), ("sparse_rows", 0), ("random", 1))):
        c = synth.make_case("prefill", batch=2, Hq=4, Hkv=2, d_qk=32, d_vo=32, page_size=8,
                            kv_lens=[21, 9], qo_lens=[6, 9], causal=causal, seed=40 + n)
        attach_mask(c, kind, 70 + n)
        _check_dense(c, lib, f"custom mask {kind} causal={causal}")


def pin_mask_all_ones_changes_nothing(lib):
    c = synth.make_case("prefill", batch=2, Hq=2, Hkv=1, d_qk=32, d_vo=16, page_size=4,
                        kv_lens=[13, 6], qo_lens=[5, 6], causal=0, window_left=4, seed=45)
    tok, head = _all_rows(c)
    ref_o, ref_l = oracle.rows(c, tok, head, lib=lib, threads=1)
    attach_mask(c, "all", 1)
    o, l = oracle.rows(c, tok, head, lib=lib, threads=1)
    assert np.array_equal(o, ref_o) and np.array_equal(l, ref_l)


def pin_causal_mask_equals_causal(lib):
    c = synth.make_case("prefill", batch=2, Hq=2, Hkv=1, d_qk=32, d_vo=32, page_size=8,
                        kv_lens=[19, 8], qo_lens=[7, 8], causal=1, seed=46)
    tok, head = _all_rows(c)
    ref_o, ref_l = oracle.rows(c, tok, head, lib=lib, threads=1)
    c.causal = 0
    attach_mask(c, "causal", 2)
    o, l = oracle.rows(c, tok, head, lib=lib, threads=1)
    assert np.array_equal(o, ref_o) and np.array_equal(l, ref_l)


def pin_mask_single_key(lib):
    """One allowed key per row: the row's output is that key's value row, its lse the
    key's scaled score (closed form)."""
    c = synth.make_case("prefill", batch=2, Hq=2, Hkv=1, d_qk=32, d_vo=32, page_size=8,
                        kv_lens=[17, 10], qo_lens=[4, 10], causal=0, seed=47)
    rng = np.random.default_rng(3)
    qo = c.qo_indptr.tolist()
    blocks, indptr, pick = [], [0], {}
    for b in range(c.batch):
        ql, L = qo[b + 1] - qo[b], c.kv_lens[b]
        g = np.zeros((ql, L), dtype=bool)
        for i in range(ql):
            pick[(b, i)] = int(rng.integers(0, L))
            g[i, pick[(b, i)]] = True
        blocks.append(np.packbits(g.ravel(), bitorder="little"))
        indptr.append(indptr[-1] + blocks[-1].size)
    c.mask = torch.from_numpy(np.concatenate(blocks))
    c.mask_indptr = torch.tensor(indptr, dtype=torch.int64)
    tok, head = _all_rows(c)
    o, l = oracle.rows(c, tok, head, lib=lib, threads=1)
    for r, (t, h) in enumerate(zip(tok, head)):
        b = 0 if t < qo[1] else 1
        j = pick[(b, int(t) - qo[b])]
        K, V = seq_kv(c, b, int(h) // c.group)
        q = c.q[int(t), int(h)].double().numpy()
        _close(o[r], V[j], what="single-key output")
        _close([l[r]], [c.sm_scale * float(K[j] @ q)], what="single-key lse")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
