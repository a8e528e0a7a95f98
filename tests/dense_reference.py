"""An independent, contiguous-layout attention for pinning the oracle.

It reads the cache through torch reshapes of the pages' layout (not through the oracle's
address arithmetic), decodes FP8 with torch's float8_e4m3fn conversion and NVFP4 with a
literal e2m1 value table, and forms softmax with scipy's softmax/logsumexp.  Nothing here
is shared with oracle/paged_attn_oracle.c.
"""

import numpy as np
import scipy.special
import torch

import synth

# e2m1 magnitudes of codes 0..7 (OCP microscaling formats, FP4 E2M1)
E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def _e2m1_decode(nib: np.ndarray) -> np.ndarray:
    mag = E2M1_TABLE[nib & 7]
    return np.where(nib & 8, -mag, mag)


def seq_kv(case, b: int, kvh: int):
    """Dequantised (K [kv_len, d_qk], V [kv_len, d_vo]) of sequence b, kv head kvh."""
    H, ps, dq, dv = case.Hkv, case.page_size, case.d_qk, case.d_vo
    P = case.num_pages
    ip = case.kv_indptr.cpu().tolist()
    pages = case.kv_indices.cpu()[ip[b]:ip[b + 1]].long()
    L = case.kv_lens[b]
    raw = case.kv_cache.cpu()
    if case.kv_dtype == synth.KV_BF16:
        flat = raw.view(torch.bfloat16).view(P, H * ps * (dq + dv)).double()
        K = flat[:, :H * ps * dq].reshape(P, H, ps, dq)
        V = flat[:, H * ps * dq:].reshape(P, H, ps, dv)
    elif case.kv_dtype == synth.KV_FP8:
        flat = raw.view(torch.float8_e4m3fn).view(P, H * ps * (dq + dv)).double()
        K = flat[:, :H * ps * dq].reshape(P, H, ps, dq) * case.k_scale
        V = flat[:, H * ps * dq:].reshape(P, H, ps, dv) * case.v_scale
    else:
        by = raw.view(P, H * ps * (dq + dv) // 2).numpy()
        nib = np.stack([by & 15, by >> 4], axis=-1).reshape(P, -1)
        val = _e2m1_decode(nib)
        sfb = case.sf.cpu().view(torch.float8_e4m3fn).view(P, -1).double().numpy()
        sfe = np.repeat(sfb, 16, axis=1)
        K = torch.from_numpy((val[:, :H * ps * dq] * sfe[:, :H * ps * dq])
                             .reshape(P, H, ps, dq)) * case.k_scale
        V = torch.from_numpy((val[:, H * ps * dq:] * sfe[:, H * ps * dq:])
                             .reshape(P, H, ps, dv)) * case.v_scale
    Ks = K[pages, kvh].reshape(-1, dq)[:L].numpy()
    Vs = V[pages, kvh].reshape(-1, dv)[:L].numpy()
    return Ks, Vs


def attention_row(case, tok: int, h: int, key_range=None):
    """softmax(q K^T * sm_scale) V for one query row, with the causal / window mask."""
    qo = case.qo_indptr.cpu().tolist()
    b = max(i for i in range(case.batch) if qo[i] <= tok)
    i = tok - qo[b]
    qo_len = qo[b + 1] - qo[b]
    L = case.kv_lens[b]
    pos = L - qo_len + i
    kvh = h // case.group
    K, V = seq_kv(case, b, kvh)
    q = case.q.cpu()[tok, h].double().numpy()
    j = np.arange(L)
    ok = np.ones(L, dtype=bool)
    if case.causal:
        ok &= j <= pos
    if case.window_left >= 0:
        ok &= j >= pos - case.window_left
    if key_range is not None:
        ok &= (j >= key_range[0]) & (j < key_range[1])
    cm = getattr(case, "mask", None)
    if cm is not None:  # custom mask: numpy's little-endian unpacking of the sequence's bits
        m = cm.cpu().numpy() if hasattr(cm, "cpu") else np.asarray(cm)
        off = int(np.asarray(case.mask_indptr.cpu() if hasattr(case.mask_indptr, "cpu") else case.mask_indptr)[b])
        bits = np.unpackbits(m[off:off + (qo_len * L + 7) // 8], bitorder="little")
        ok &= bits[i * L:(i + 1) * L].astype(bool)
    if not ok.any():
        return np.zeros(case.d_vo), -np.inf
    s = (K[ok] @ q) * case.sm_scale
    p = scipy.special.softmax(s)
    return p @ V[ok], float(scipy.special.logsumexp(s))
