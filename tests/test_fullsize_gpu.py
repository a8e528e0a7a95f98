"""Parity at the full sizes of the benchmark workloads, in the launch configuration bench.py
times (the same C-ABI call on the whole batch).

The oracle reads a compact host copy of the checked sequences (their pages, page table
and query rows, gathered from the device input tensors with plain torch indexing), so the
largest caches never need a full host copy; pages a sliding window hides are replaced by
one shared zero page, which the oracle never weighs.

Coverage:
  * decode: every sequence of the bf16 GQA decode (64) and of the sliding-window decode
    (256), every query head; the FP8 decode on 16 of its 128 sequences (12.5 %), spread
    over the batch and including the first and the last;
  * causal prefill (lengths 2048 / 3000 / 4096 / 6272): every sequence; per sequence the
    first and last row of every query tile (128 // group positions), every row of the
    last, ragged tile, and a seeded 10 % of the remaining rows, every query head;
  * NVFP4 asymmetric prefill: every sequence, with the same row choice.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_attention_hd512_gb300 as pa
import synth
from parity import compare, ensure_built

pytestmark = pytest.mark.gpu


def subcase(c, seqs):
    """Host synth.Case holding only sequences `seqs` of device case `c`.  Pages before a
    sliding window's first visible page (decode: the window of the one query token) map
    to a zero page shared by all of them."""
    ip = c.kv_indptr.tolist()
    qo = c.qo_indptr.tolist()
    page_bytes = c.page_bytes()
    pages_dev = c.kv_cache.view(c.num_pages, page_bytes)
    sf_dev = c.sf.view(c.num_pages, -1) if c.sf is not None else None
    host_pages = [torch.zeros(1, page_bytes, dtype=torch.uint8)]
    host_sf = [torch.zeros(1, sf_dev.shape[1], dtype=torch.uint8)] if sf_dev is not None else None
    new_ind, new_ip, new_qo = [], [0], [0]
    n_host = 1
    for b in seqs:
        np_b = ip[b + 1] - ip[b]
        first = 0
        if c.window_left >= 0 and c.phase == "decode":
            first = max(0, c.kv_lens[b] - 1 - c.window_left) // c.page_size
        ids = c.kv_indices[ip[b] + first:ip[b + 1]].long()
        host_pages.append(pages_dev[ids].cpu())
        if sf_dev is not None:
            host_sf.append(sf_dev[ids].cpu())
        new_ind += [0] * first + list(range(n_host, n_host + np_b - first))
        n_host += np_b - first
        new_ip.append(new_ip[-1] + np_b)
        new_qo.append(new_qo[-1] + qo[b + 1] - qo[b])
    q_rows = torch.cat([torch.arange(qo[b], qo[b + 1]) for b in seqs])
    s = synth.Case(**{k: getattr(c, k) for k in c.__dataclass_fields__})
    s.batch = len(seqs)
    s.num_pages = n_host
    s.kv_cache = torch.cat(host_pages).reshape(-1)
    s.sf = torch.cat(host_sf).reshape(-1) if host_sf is not None else None
    s.kv_indptr = torch.tensor(new_ip, dtype=torch.int32)
    s.kv_indices = torch.tensor(new_ind, dtype=torch.int32)
    s.kv_last_page_len = c.kv_last_page_len.cpu()[list(seqs)].clone()
    s.q = c.q[q_rows.to(c.q.device)].cpu()
    s.qo_indptr = torch.tensor(new_qo, dtype=torch.int32)
    s.kv_lens = [c.kv_lens[b] for b in seqs]
    s.qo_lens = [c.qo_lens[b] for b in seqs]
    return s


def run_full(c):
    ensure_built()
    pa.paged_attn_set_decode_chunk_pages(0)
    out, lse = pa.run_case(c)
    torch.cuda.synchronize()
    assert pa.paged_attn_check_device_error() == 0
    return out, lse


def check_rows(c, out, lse, seqs, rows_per_seq, what):
    """Compare the rows rows_per_seq(b) (query indices within sequence b, every head) of
    the sequences `seqs` with the oracle."""
    host = subcase(c, seqs)
    qo_host = host.qo_indptr.tolist()
    qo = c.qo_indptr.tolist()
    tok, head, gtok = [], [], []
    for k, b in enumerate(seqs):
        for i in rows_per_seq(b):
            for h in range(c.Hq):
                tok.append(qo_host[k] + i)
                gtok.append(qo[b] + i)
                head.append(h)
    ref_out, ref_lse = oracle.rows(host, tok, head)
    t = torch.tensor(gtok, dtype=torch.long)
    hh = torch.tensor(head, dtype=torch.long)
    compare(out[t, hh], lse[t, hh], ref_out, ref_lse, f"{what}: {len(tok)} rows")
    return len(tok)


@pytest.mark.parametrize("name,frac", [("gqa_decode_bf16", 1.0), ("sliding_decode_d256", 1.0),
                                       ("fp8_decode", 0.125)])
def test_fullsize_decode(name, frac):
    c = synth.workload(name, device="cuda")
    out, lse = run_full(c)
    B = c.batch
    n = max(1, int(round(B * frac)))
    seqs = sorted({int(x) for x in np.linspace(0, B - 1, n).round()})
    assert len(seqs) >= n * 0.99
    # in chunks of sequences, so that the host copy stays a few GB
    chunk = 16 if c.kv_dtype == synth.KV_FP8 else 64
    total = 0
    for i in range(0, len(seqs), chunk):
        total += check_rows(c, out, lse, seqs[i:i + chunk], lambda b: [0], name)
    assert total == len(seqs) * c.Hq
    del c
    torch.cuda.empty_cache()


def prefill_rows(c, frac=0.10, seed=0):
    """Per sequence: first and last row of every query tile, every row of the last
    (ragged) tile, and a seeded `frac` of the other rows."""
    P = 128 // c.group

    def rows(b):
        n = c.qo_lens[b]
        pick = set()
        for t0 in range(0, n, P):
            pick.add(t0)
            pick.add(min(n, t0 + P) - 1)
        last0 = (n - 1) // P * P
        pick |= set(range(last0, n))
        rest = np.array(sorted(set(range(n)) - pick), dtype=np.int64)
        if rest.size:
            rng = np.random.default_rng(seed * 1000 + b)
            k = int(np.ceil(frac * n))
            pick |= {int(x) for x in rng.choice(rest, size=min(k, rest.size), replace=False)}
        return sorted(pick)
    return rows


@pytest.mark.parametrize("name", ["causal_prefill_bf16", "nvfp4_asym_prefill"])
def test_fullsize_prefill(name):
    c = synth.workload(name, device="cuda")
    out, lse = run_full(c)
    rows = prefill_rows(c)
    seqs = list(range(c.batch))
    checked = check_rows(c, out, lse, seqs, rows, name)
    assert checked >= 0.10 * c.total_q * c.Hq
    del c
    torch.cuda.empty_cache()
