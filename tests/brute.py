"""Dense brute-force attention for tiny inputs (numpy float64) -- a pin for the
oracle, written with a different structure: K/V are first de-paged into dense
per-request arrays with fancy indexing, an explicit [q_len x seq_len] boolean
mask is built, and softmax(scale * Q K^T masked) V is taken as whole-matrix
operations.  Conversions to float64 go through torch dtypes (bfloat16,
float8_e4m3fn), not through the oracle's own bit-level decoders.

Semantics (page "[vLLM] FlashAttention": cache shape, GQA ratio,
varlen metadata; page "RBLN Attention modes": naive attention, causal mask,
sliding window): row i of request r sits at position ctx + i with
ctx = seq_len - query_len.
"""
import numpy as np
import torch


def to_f64_q(q):
    return q.detach().cpu().to(torch.float32).to(torch.float64).numpy()


def _as16(kv, kv_dtype):
    want = torch.float16 if kv_dtype == 2 else torch.bfloat16
    return kv if kv.dtype == want else kv.view(want)


def to_f64_kv(kv, kv_dtype, kv_scale):
    kv = kv.detach().cpu()
    if kv_dtype in (0, 2):
        return _as16(kv, kv_dtype).to(torch.float32).to(torch.float64).numpy()
    x = kv.view(torch.float8_e4m3fn).to(torch.float32).to(torch.float64).numpy()
    x = x.copy()
    x[0] *= float(kv_scale[0])
    x[1] *= float(kv_scale[1])
    return x


def brute_attention(q, kv_cache, block_table, seq_lens, query_start_loc, *, scale,
                    num_heads, num_kv_heads, head_size, block_size, window=0,
                    causal=1, kv_dtype=0, kv_scale=(1.0, 1.0), sinks=None, head_size_v=0):
    """Returns (out [T, H, d], lse [T, H]) in float64; rows of tokens outside
    every request stay NaN.  sinks: per-head sink logits, taken here as one
    more key column whose score is the sink and whose value row is zero.
    head_size_v > 0: kv_cache is [NB, bs, Hkv, head_size + head_size_v], each
    row K then V."""
    Q = to_f64_q(q)
    KV = to_f64_kv(kv_cache, kv_dtype, kv_scale)
    bt = np.asarray(block_table.cpu() if torch.is_tensor(block_table) else block_table)
    sl = np.asarray(seq_lens.cpu() if torch.is_tensor(seq_lens) else seq_lens)
    qsl = np.asarray(query_start_loc.cpu() if torch.is_tensor(query_start_loc)
                     else query_start_loc)
    T = Q.shape[0]
    G = num_heads // num_kv_heads
    dv = head_size_v or head_size
    out = np.full((T, num_heads, dv), np.nan)
    lse = np.full((T, num_heads), np.nan)
    bs = block_size
    for r in range(len(sl)):
        t0, t1 = int(qsl[r]), int(qsl[r + 1])
        ql, s = t1 - t0, int(sl[r])
        if ql == 0:
            continue
        nb = (s + bs - 1) // bs
        blocks = bt[r, :nb]
        if head_size_v:
            rows = KV[blocks].reshape(nb * bs, num_kv_heads, head_size + dv)[:s]
            K, V = rows[:, :, :head_size], rows[:, :, head_size:]
        else:
            K = KV[0][blocks].reshape(nb * bs, num_kv_heads, head_size)[:s]
            V = KV[1][blocks].reshape(nb * bs, num_kv_heads, head_size)[:s]
        pos = (s - ql) + np.arange(ql)[:, None]
        key = np.arange(s)[None, :]
        mask = np.ones((ql, s), dtype=bool)
        if causal:
            mask &= key <= pos
        if window > 0:
            mask &= (pos - key) < window
        for h in range(num_heads):
            g = h // G
            S = float(np.float32(scale)) * (Q[t0:t1, h, :] @ K[:, g, :].T)
            S = np.where(mask, S, -np.inf)
            Vh = V[:, g, :]
            if sinks is not None:
                S = np.concatenate([S, np.full((ql, 1), float(sinks[h]))], axis=1)
                Vh = np.concatenate([Vh, np.zeros((1, dv))], axis=0)
            m = S.max(axis=1, keepdims=True)
            W = np.exp(S - m)
            den = W.sum(axis=1, keepdims=True)
            out[t0:t1, h, :] = (W @ Vh) / den
            lse[t0:t1, h] = (m + np.log(den))[:, 0]
    return out, lse
