"""Small seeded case builders shared by the oracle tests and the GPU parity
tests (inputs only; no attention arithmetic here)."""
import random

import numpy as np
import torch

import workloads as W


def small_spec(seed, *, H=4, Hkv=2, d=16, bs=16, n_req=3, max_s=70, window=0,
               causal=1, kv_dtype=W.KV_BF16, kinds=("prefill", "decode", "chunk"),
               extra_pool=3, scale=None, unused_fill=0):
    """A random varlen batch: each request is a full prefill (q = s), a decode
    (q = 1) or a chunked prefill (1 < q < s), drawn with a Python RNG."""
    rng = random.Random(seed)
    q_lens, seq_lens = [], []
    for _ in range(n_req):
        kind = rng.choice(kinds)
        s = rng.randint(1, max_s)
        if kind == "prefill":
            q = s
        elif kind == "decode":
            q = 1
        elif kind == "empty":
            q = 0
        else:
            q = rng.randint(1, s)
        q_lens.append(q)
        seq_lens.append(s)
    need = sum((s + bs - 1) // bs for s in seq_lens)
    return W.CaseSpec(f"small{seed}", q_lens, seq_lens, H, Hkv, d, bs, window=window,
                      causal=causal, kv_dtype=kv_dtype, pool_blocks=need + extra_pool,
                      seed=seed, scale=scale, unused_fill=unused_fill)


def case_args(case):
    """Keyword arguments shared by the oracle, the brute force and the binding."""
    s = case.spec
    return dict(scale=case.scale, num_heads=s.num_heads, num_kv_heads=s.num_kv_heads,
                head_size=s.head_size, block_size=s.block_size, window=s.window,
                causal=s.causal, kv_dtype=s.kv_dtype, kv_scale=case.kv_scale)


def host_arrays(case):
    """(q bits, kv bits/bytes, block_table, seq_lens, qsl) as numpy arrays."""
    q = case.q.detach().cpu().view(torch.int16).numpy().view(np.uint16)
    kv = case.kv_cache.detach().cpu()
    if case.spec.kv_dtype in (W.KV_BF16, W.KV_F16):
        kv = kv.view(torch.int16).numpy().view(np.uint16)
    else:
        kv = kv.numpy()
    return (q, kv, case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(),
            case.query_start_loc.cpu().numpy())


def shuffle_blocks(case, seed):
    """Move every physical block to a new slot of the pool and rewrite the
    block table to match (the same logical cache)."""
    g = torch.Generator().manual_seed(seed)
    nb = case.kv_cache.shape[1]
    perm = torch.randperm(nb, generator=g)            # new position of block b
    kv = torch.empty_like(case.kv_cache)
    kv[:, perm.to(kv.device)] = case.kv_cache
    bt = case.block_table.cpu().clone()
    sl = case.seq_lens.cpu()
    for r in range(bt.shape[0]):
        s = int(sl[r])
        n = (s + case.spec.block_size - 1) // case.spec.block_size
        bt[r, :n] = perm[bt[r, :n].long()].to(torch.int32)
    return W.Case(spec=case.spec, q=case.q, kv_cache=kv,
                  block_table=bt.to(case.block_table.device),
                  seq_lens=case.seq_lens, query_start_loc=case.query_start_loc,
                  scale=case.scale, kv_scale=case.kv_scale)


class DiffKVCase:
    """A varlen batch over a cache in the DiffKV layout
    [num_blocks][block_size][num_kv_heads][dk + dv] (each row: K then V)."""

    def __init__(self, case, cache, dv):
        self.case, self.cache, self.dv = case, cache, dv
        self.spec = case.spec


def diffkv_case(seed, *, H=4, Hkv=2, dk=32, dv=64, bs=16, n_req=3, max_s=70, window=0,
                kv_dtype=W.KV_BF16, kinds=("prefill", "decode", "chunk"), device="cpu"):
    """Metadata and q (head size dk) from small_spec; a seeded N(0,1) cache in
    the DiffKV layout.  The standard-layout cache of the case is not used."""
    sp = small_spec(seed, H=H, Hkv=Hkv, d=dk, bs=bs, n_req=n_req, max_s=max_s,
                    window=window, kv_dtype=kv_dtype, kinds=kinds)
    case = W.make_case(sp, device=device)
    g = torch.Generator().manual_seed(seed + 7919)
    nb = case.kv_cache.shape[1]
    dt = torch.float16 if kv_dtype == W.KV_F16 else torch.bfloat16
    cache = torch.randn(nb, bs, Hkv, dk + dv, generator=g).to(dt).to(device)
    return DiffKVCase(case, cache, dv)
