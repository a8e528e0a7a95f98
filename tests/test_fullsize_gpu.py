"""Parity at the full sizes of the benchmark workloads, in the launch configuration bench.py
times (the same C-ABI call on the whole batch), checked on sampled rows.

The oracle reads a compact host copy of the sampled sequences (their pages, page table
and query rows, gathered from the device input tensors with plain torch indexing), so the
largest caches never need a full host copy.  Rows are chosen to cover the first and last
sequences, the shortest and longest ones, tile and page boundaries and the last rows of
each sequence.
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
    """Host synth.Case holding only sequences `seqs` of device case `c`."""
    ip = c.kv_indptr.tolist()
    qo = c.qo_indptr.tolist()
    page_ids = torch.cat([c.kv_indices[ip[b]:ip[b + 1]].long() for b in seqs])
    pages = c.kv_cache.view(c.num_pages, c.page_bytes())[page_ids].cpu()
    sf = c.sf.view(c.num_pages, -1)[page_ids].cpu().reshape(-1) if c.sf is not None else None
    new_ip, new_qo = [0], [0]
    for b in seqs:
        new_ip.append(new_ip[-1] + ip[b + 1] - ip[b])
        new_qo.append(new_qo[-1] + qo[b + 1] - qo[b])
    q_rows = torch.cat([torch.arange(qo[b], qo[b + 1]) for b in seqs])
    s = synth.Case(**{k: getattr(c, k) for k in c.__dataclass_fields__})
    s.batch = len(seqs)
    s.num_pages = len(page_ids)
    s.kv_cache = pages.reshape(-1)
    s.sf = sf
    s.kv_indptr = torch.tensor(new_ip, dtype=torch.int32)
    s.kv_indices = torch.arange(len(page_ids), dtype=torch.int32)
    s.kv_last_page_len = c.kv_last_page_len.cpu()[list(seqs)].clone()
    s.q = c.q[q_rows.to(c.q.device)].cpu()
    s.qo_indptr = torch.tensor(new_qo, dtype=torch.int32)
    s.kv_lens = [c.kv_lens[b] for b in seqs]
    s.qo_lens = [c.qo_lens[b] for b in seqs]
    return s


def check_sampled(c, seqs, rows_per_seq):
    """rows_per_seq(b) -> query indices within sequence b (every head of each is checked)."""
    ensure_built()
    out, lse = pa.run_case(c)
    torch.cuda.synchronize()
    assert pa.paged_attn_check_device_error() == 0
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
    return compare(out[t, hh], lse[t, hh], ref_out, ref_lse, f"{len(tok)} sampled rows")


@pytest.mark.parametrize("name", ["gqa_decode_bf16", "fp8_decode", "sliding_decode_d256"])
def test_fullsize_decode(name):
    c = synth.workload(name, device="cuda")
    B = c.batch
    order = np.argsort(c.kv_lens)
    seqs = sorted({0, 1, B // 3, B // 2, B - 2, B - 1, int(order[0]), int(order[-1])})
    check_sampled(c, seqs, lambda b: [0])
    del c
    torch.cuda.empty_cache()


def _prefill_rows(c):
    P = 128 // c.group

    def rows(b):
        n = c.qo_lens[b]
        pick = {0, 1, P - 1, P, 127, 128, 255, 256, 257, n // 2, n - P - 1, n - P, n - 2, n - 1}
        rng = np.random.default_rng(b)
        pick |= {int(x) for x in rng.integers(0, n, 12)}
        return sorted(i for i in pick if 0 <= i < n)
    return rows


@pytest.mark.parametrize("name,seqs", [("causal_prefill_bf16", [0, 3]), ("nvfp4_asym_prefill", [0, 7])])
def test_fullsize_prefill(name, seqs):
    c = synth.workload(name, device="cuda")
    check_sampled(c, seqs, _prefill_rows(c))
    del c
    torch.cuda.empty_cache()
