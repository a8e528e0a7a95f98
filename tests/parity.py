"""Shared helpers of the GPU parity tests: build the library, run a synth.Case through the
C ABI, and compare with the fp64 oracle under the stated tolerance.

Tolerance: bf16 outputs |err| <= 1e-2 + 1e-2 * |ref| element by element; lse |err| <= 1e-3
(absolute, natural-log units); rows with no visible key must give out = 0, lse = -inf.
"""

import numpy as np
import torch

import oracle
import paged_gqa_attention_hd512_gb300 as pa
from paged_gqa_attention_hd512_gb300 import build as pa_build

OUT_ABS, OUT_REL, LSE_ABS = 1e-2, 1e-2, 1e-3

_built = False


def ensure_built():
    global _built
    if not _built:
        pa_build.build()
        pa.load()
        _built = True


def run_gpu(case_gpu, **extra):
    ensure_built()
    out, lse = pa.run_case(case_gpu, **extra)
    torch.cuda.synchronize()
    assert pa.paged_attn_check_device_error() == 0
    return out, lse


def compare(out_gpu, lse_gpu, ref_out, ref_lse, what=""):
    """out_gpu [n, d] bf16 (any device), lse_gpu [n]; ref_* fp64 numpy."""
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.float().cpu().numpy().astype(np.float64)
    ref_out = np.asarray(ref_out, dtype=np.float64).reshape(o.shape)
    ref_lse = np.asarray(ref_lse, dtype=np.float64).reshape(l.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - ref_out)
    bound = OUT_ABS + OUT_REL * np.abs(ref_out)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs out of tolerance, max err "
                           f"{err.max():.4g} at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    inf_ref = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), inf_ref), f"{what}: -inf lse mismatch"
    if (~inf_ref).any():
        le = np.abs(l[~inf_ref] - ref_lse[~inf_ref])
        assert le.max() <= LSE_ABS, f"{what}: lse max err {le.max():.4g}"
    return float(err.max()), float(np.abs(l[~inf_ref] - ref_lse[~inf_ref]).max()) if (~inf_ref).any() else 0.0


def check_full(case_cpu, what="", **extra):
    """Run the whole case on the GPU and compare every output row with the oracle."""
    ref_out, ref_lse = oracle.full(case_cpu)
    g = case_cpu.to("cuda")
    out, lse = run_gpu(g, **extra)
    n = case_cpu.total_q * case_cpu.Hq
    return compare(out.reshape(n, -1), lse.reshape(n), ref_out.reshape(n, -1), ref_lse.reshape(n), what)


def check_rows(case_gpu, rows_tok, rows_head, what="", case_cpu=None, **extra):
    """Run a (large) case on the GPU and compare the chosen rows with the oracle, which
    reads a host copy of the same input tensors."""
    out, lse = run_gpu(case_gpu, **extra)
    host = case_cpu if case_cpu is not None else case_gpu.to("cpu")
    ref_out, ref_lse = oracle.rows(host, rows_tok, rows_head)
    t = torch.as_tensor(np.asarray(rows_tok), dtype=torch.long)
    h = torch.as_tensor(np.asarray(rows_head), dtype=torch.long)
    return compare(out[t, h], lse[t, h], ref_out, ref_lse, what)
