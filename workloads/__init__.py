"""Seeded synthetic inputs for paged variable-length attention.

This module is shared by the oracle's tests and by the CUDA path's tests and
benchmark.  It only draws numbers and lays them out; it holds none of the
attention arithmetic.

Layouts (page "[vLLM] FlashAttention", FlashAttentionBackend.get_kv_cache_shape
and FlashAttentionMetadata):
  q               bf16  [T, H, d]
  kv_cache        [2, num_blocks, block_size, Hkv, d]; index 0 = K, 1 = V;
                  bf16, or e4m3 bytes (uint8) with one fp32 scale per tensor
  block_table     int32 [B, max_blocks_per_seq]
  seq_lens        int32 [B]          (context_len + query_len)
  query_start_loc int32 [B + 1]      (prefix sum of query lengths)

Recipe: integers (lengths, block permutation) come from a CPU
``torch.Generator`` seeded with ``seed``; bulk N(0, 1) values from a generator
on the target device seeded with ``seed`` too, drawn in fp32 and rounded to
bf16 (round to nearest even).  Physical blocks are handed to the requests in
order from a seeded permutation of the whole pool; the pool is filled whole.
FP8 tensors are quantised per tensor: scale = amax / 448, byte =
e4m3(x / scale) with saturation (torch.float8_e4m3fn).
"""
from dataclasses import dataclass, field
import math
from typing import List, Optional, Tuple

import torch

KV_BF16 = 0
KV_FP8_E4M3 = 1
KV_F16 = 2  # f16 cache, and q / out in f16 too
E4M3_MAX = 448.0


@dataclass
class CaseSpec:
    name: str
    q_lens: List[int]
    seq_lens: List[int]
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    window: int = 0
    causal: int = 1
    kv_dtype: int = KV_BF16
    pool_blocks: Optional[int] = None      # None: exactly the blocks needed
    max_blocks_per_seq: Optional[int] = None
    scale: Optional[float] = None          # None: 1/sqrt(head_size) as fp32
    num_splits: int = 0                    # 0: library chooses
    seed: int = 0
    unused_fill: int = 0                   # block_table entries past each request


@dataclass
class Case:
    spec: CaseSpec
    q: torch.Tensor
    kv_cache: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor
    scale: float
    kv_scale: Tuple[float, float] = (1.0, 1.0)

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.kv_cache.shape[1])

    @property
    def max_query_len(self) -> int:
        return max(self.spec.q_lens) if self.spec.q_lens else 0

    @property
    def max_seq_len(self) -> int:
        return max(self.spec.seq_lens) if self.spec.seq_lens else 0


def _randn_f16(shape, gen, device, chunk_elems=1 << 28):
    """N(0,1) drawn in fp32 chunk by chunk and rounded to f16."""
    out = torch.empty(shape, dtype=torch.float16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device,
                                dtype=torch.float32).to(torch.float16)
    return out


def _randn_bf16(shape, gen, device, chunk_elems=1 << 28):
    """N(0,1) drawn in fp32 chunk by chunk and rounded to bf16."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device,
                                dtype=torch.float32).to(torch.bfloat16)
    return out


def _randn_e4m3(shape, gen, device):
    """N(0,1) in fp32 quantised to e4m3 bytes with one per-tensor scale."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    amax = float(x.abs().max())
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    scale = float(torch.tensor(scale, dtype=torch.float32))
    codes = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    del x
    return codes, scale


def make_case(spec: CaseSpec, device="cpu") -> Case:
    device = torch.device(device)
    B = len(spec.q_lens)
    assert len(spec.seq_lens) == B
    bs = spec.block_size
    nblk = [(s + bs - 1) // bs for s in spec.seq_lens]
    need = sum(nblk)
    pool = spec.pool_blocks if spec.pool_blocks is not None else need
    assert pool >= need, "pool smaller than the blocks the requests need"
    mbps = spec.max_blocks_per_seq or max([1] + nblk)
    cpu = torch.Generator(device="cpu").manual_seed(spec.seed)
    perm = torch.randperm(pool, generator=cpu).to(torch.int32)
    bt = torch.full((B, mbps), spec.unused_fill, dtype=torch.int32)
    off = 0
    for r, n in enumerate(nblk):
        bt[r, :n] = perm[off:off + n]
        off += n
    qsl = torch.zeros(B + 1, dtype=torch.int32)
    if B:
        qsl[1:] = torch.cumsum(torch.tensor(spec.q_lens, dtype=torch.int64), 0).to(torch.int32)
    T = int(qsl[-1])
    gen = torch.Generator(device=device).manual_seed(spec.seed)
    H, Hkv, d = spec.num_heads, spec.num_kv_heads, spec.head_size
    q = _randn_bf16((T, H, d), gen, device)
    kv_scale = (1.0, 1.0)
    if spec.kv_dtype == KV_F16:
        q = _randn_f16((T, H, d), gen, device)
        kv = _randn_f16((2, pool, bs, Hkv, d), gen, device)
    elif spec.kv_dtype == KV_BF16:
        kv = _randn_bf16((2, pool, bs, Hkv, d), gen, device)
    else:
        k, ks = _randn_e4m3((pool, bs, Hkv, d), gen, device)
        v, vs = _randn_e4m3((pool, bs, Hkv, d), gen, device)
        kv = torch.stack([k, v], 0)
        del k, v
        kv_scale = (ks, vs)
    scale = spec.scale if spec.scale is not None else 1.0 / math.sqrt(d)
    scale = float(torch.tensor(scale, dtype=torch.float32))
    return Case(spec=spec, q=q, kv_cache=kv, block_table=bt.to(device),
                seq_lens=torch.tensor(spec.seq_lens, dtype=torch.int32, device=device),
                query_start_loc=qsl.to(device), scale=scale, kv_scale=kv_scale)


def _uniform_ints(lo, hi, n, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def config_spec(index: int) -> CaseSpec:
    """The five synthetic workloads, numbered 1..5.

    1 tiny mixed batch (prefill 8/8 + decode 1/40), H 4, Hkv 2, d 64, bs 16
    2 decode-only GQA: 64 x (q 1, s ~ U{512..4096}), H 32, Hkv 8, d 128, bs 16,
      20k-block pool
    3 varlen causal prefill: 8 x (q = s ~ U{1024..8192}), H 32, Hkv 8, d 128
    4 mixed chunked prefill + decode, window 4096: 4 x (q 2048, s 8192) then
      192 x (q 1, s ~ U{1024..32768}), H 64, Hkv 8, d 128, bs 16
    5 long split-KV decode, e4m3 KV: 8 x (q 1, s 131072), H 64, Hkv 8, d 128,
      bs 64, 16 partitions
    """
    seed = 1000 + index
    if index == 1:
        return CaseSpec("tiny_mixed", [8, 1], [8, 40], 4, 2, 64, 16,
                        pool_blocks=8, max_blocks_per_seq=3, seed=seed)
    if index == 2:
        s = _uniform_ints(512, 4096, 64, seed)
        return CaseSpec("decode_gqa", [1] * 64, s, 32, 8, 128, 16,
                        pool_blocks=20000, max_blocks_per_seq=256, seed=seed)
    if index == 3:
        L = _uniform_ints(1024, 8192, 8, seed)
        return CaseSpec("varlen_prefill", L, L, 32, 8, 128, 16,
                        max_blocks_per_seq=512, seed=seed)
    if index == 4:
        s = [8192] * 4 + _uniform_ints(1024, 32768, 192, seed)
        return CaseSpec("mixed_swa4096", [2048] * 4 + [1] * 192, s, 64, 8, 128, 16,
                        window=4096, max_blocks_per_seq=2048, seed=seed)
    if index == 5:
        return CaseSpec("long_split_fp8", [1] * 8, [131072] * 8, 64, 8, 128, 64,
                        kv_dtype=KV_FP8_E4M3, pool_blocks=16384,
                        max_blocks_per_seq=2048, num_splits=16, seed=seed)
    raise ValueError(f"no workload {index}")
