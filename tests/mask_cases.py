"""Seeded custom masks for prefill cases (input generation only): per sequence a
[qo_len, kv_len] boolean grid, packed little-endian into bytes with numpy, each sequence's
block starting on a byte boundary."""

import numpy as np
import torch


def grid(kind: str, qo_len: int, kv_len: int, rng) -> np.ndarray:
    pos = kv_len - qo_len + np.arange(qo_len)[:, None]
    j = np.arange(kv_len)[None, :]
    if kind == "random":
        return rng.random((qo_len, kv_len)) < 0.7
    if kind == "spans":  # causal, plus bidirectional attention inside spans of the new tokens
        g = j <= pos
        start = kv_len - qo_len
        cuts = np.sort(rng.choice(np.arange(1, max(2, qo_len)), size=min(3, max(0, qo_len - 1)), replace=False)) \
            if qo_len > 2 else np.array([], dtype=int)
        edges = [0, *cuts.tolist(), qo_len]
        for a, e in zip(edges[:-1], edges[1:]):
            if rng.random() < 0.6:
                g[a:e, start + a:start + e] = True
        return g
    if kind == "sparse_rows":  # a few keys per row, some rows with none at all
        g = rng.random((qo_len, kv_len)) < 0.02
        g[rng.random(qo_len) < 0.2] = False
        return g
    if kind == "causal":
        return j <= pos
    if kind == "all":
        return np.ones((qo_len, kv_len), dtype=bool)
    raise ValueError(kind)


def attach(case, kind: str, seed: int):
    """Give a (CPU) synth prefill Case a custom mask of the given kind."""
    rng = np.random.default_rng(seed)
    qo = case.qo_indptr.cpu().tolist()
    blocks, indptr = [], [0]
    for b in range(case.batch):
        g = grid(kind, qo[b + 1] - qo[b], case.kv_lens[b], rng)
        packed = np.packbits(g.ravel(), bitorder="little")
        blocks.append(packed)
        indptr.append(indptr[-1] + packed.size)
    data = np.concatenate(blocks) if blocks else np.zeros(0, np.uint8)
    case.mask = torch.from_numpy(np.concatenate([data, np.zeros(max(1, 16 - data.size % 16), np.uint8)]))
    case.mask_indptr = torch.tensor(indptr, dtype=torch.int64)
    return case
