"""float64 CPU oracle for paged variable-length attention -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU
baseline and reference arm) may import this package.  The CUDA library never
imports it and must never fall back to it.

The arithmetic lives in ``pattn_ref.c`` (plain loops, float64).  This module
only marshals numpy arrays into that library through ctypes.

Definition followed (pages "[vLLM] FlashAttention": KV cache shape,
FlashAttentionImpl GQA ratio, FlashAttentionMetadata; "[vLLM] other attention
backends": TritonAttentionMetadata length meanings; "RBLN Attention modes":
naive attention, causal masking, sliding window, partition merge):
for each (token, head) row, scores over the visible keys of its request,
softmax, product with V; lse = ln of the softmax denominator after max shift.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def bind(path):
    """Open an oracle shared library at ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    lib.pattn_ref_rows.restype = ctypes.c_int
    lib.pattn_ref_rows.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int]
    lib.pattn_ref_e4m3_to_double.restype = ctypes.c_double
    lib.pattn_ref_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.pattn_ref_bf16_to_double.restype = ctypes.c_double
    lib.pattn_ref_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.pattn_ref_f16_to_double.restype = ctypes.c_double
    lib.pattn_ref_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.pattn_ref_e4m3_encode.restype = ctypes.c_uint8
    lib.pattn_ref_e4m3_encode.argtypes = [ctypes.c_float]
    lib.pattn_ref_reshape_and_cache_diffkv.restype = ctypes.c_int
    lib.pattn_ref_reshape_and_cache_diffkv.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.pattn_ref_reshape_and_cache.restype = ctypes.c_int
    lib.pattn_ref_reshape_and_cache.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_float, ctypes.c_float]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(_build.build())
    return _lib


class OracleError(RuntimeError):
    pass


_ERRORS = {1: "invalid argument", 2: "invalid metadata (q_len > seq_len, "
           "block id or slot out of range, or token outside every request)",
           3: "out of host memory"}


def e4m3_to_double(code: int, lib=None) -> float:
    """Decode one e4m3 byte with the oracle's own decoder."""
    return (lib or _load()).pattn_ref_e4m3_to_double(int(code) & 0xFF)


def f16_to_double(bits: int, lib=None) -> float:
    """Decode one IEEE binary16 pattern with the oracle's own decoder."""
    return (lib or _load()).pattn_ref_f16_to_double(int(bits) & 0xFFFF)


def bf16_to_double(bits: int, lib=None) -> float:
    return (lib or _load()).pattn_ref_bf16_to_double(int(bits) & 0xFFFF)


def e4m3_encode(x: float, lib=None) -> int:
    """Encode one fp32 value as an e4m3 byte with the oracle's own encoder
    (round to nearest even, saturating at +-448)."""
    return int((lib or _load()).pattn_ref_e4m3_encode(float(x)))


def reshape_and_cache(key_bits, value_bits, kv_cache, slot_mapping, *, num_kv_heads,
                      head_size, block_size, kv_dtype=0, kv_scale=None, lib=None):
    """Apply a KV-cache write to a host copy of the cache (numpy, updated in
    place and returned): bf16 key/value bits [T, Hkv, d], int64 slots [T]
    (negative: no write).  Raises OracleError for a slot beyond the pool."""
    lib = lib or _load()
    key_bits = _c(key_bits, np.uint16)
    value_bits = _c(value_bits, np.uint16)
    slots = _c(slot_mapping, np.int64)
    assert kv_cache.flags["C_CONTIGUOUS"]
    assert kv_cache.dtype == (np.uint8 if kv_dtype == 1 else np.uint16)
    ks, vs = (float(kv_scale[0]), float(kv_scale[1])) if kv_dtype == 1 else (1.0, 1.0)
    rc = lib.pattn_ref_reshape_and_cache(
        key_bits.ctypes.data, value_bits.ctypes.data, kv_cache.ctypes.data, slots.ctypes.data,
        int(slots.shape[0]), num_kv_heads, head_size, block_size, int(kv_cache.shape[1]),
        kv_dtype, ks, vs)
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"error {rc}"))
    return kv_cache


def reshape_and_cache_diffkv(key_bits, value_bits, kv_cache, slot_mapping, *, num_kv_heads,
                             head_size, head_size_v, block_size, lib=None):
    """Oracle cache write into the DiffKV layout: key_bits uint16 [T, Hkv,
    head_size], value_bits uint16 [T, Hkv, head_size_v], kv_cache uint16 [NB,
    bs, Hkv, head_size + head_size_v] updated in place and returned."""
    lib = lib or _load()
    key_bits = _c(key_bits, np.uint16)
    value_bits = _c(value_bits, np.uint16)
    slots = _c(slot_mapping, np.int64)
    assert kv_cache.dtype == np.uint16 and kv_cache.flags["C_CONTIGUOUS"]
    rc = lib.pattn_ref_reshape_and_cache_diffkv(
        key_bits.ctypes.data, value_bits.ctypes.data, kv_cache.ctypes.data, slots.ctypes.data,
        int(slots.shape[0]), num_kv_heads, head_size, head_size_v, block_size,
        int(kv_cache.shape[0]))
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"error {rc}"))
    return kv_cache


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def ref_rows(q_bits, kv_cache, block_table, seq_lens, query_start_loc, *, scale,
             num_heads, num_kv_heads, head_size, block_size, window=0, causal=1,
             kv_dtype=0, kv_scale=(1.0, 1.0), rows=None, num_splits=0,
             num_threads=None, sinks=None, head_size_v=0, lib=None):
    """Oracle output for selected (token, head) rows.

    q_bits        uint16 [T, H, d]   (bf16 bit patterns)
    kv_cache      uint16 (bf16 bits) or uint8 (e4m3 bytes) [2, NB, bs, Hkv, d];
                  with head_size_v > 0 the DiffKV layout [NB, bs, Hkv, d + head_size_v]
    block_table   int32 [B, max_blocks_per_seq]
    seq_lens      int32 [B];  query_start_loc int32 [B + 1]
    rows          int array [n, 2] of (token, head); None = every row
    sinks         float32 [H] attention-sink logits, or None
    lib           another oracle library opened with ``bind`` (tests only)
    Returns (out float64 [n, head_size_v or d], lse float64 [n]).
    """
    lib = lib or _load()
    q_bits = _c(q_bits, np.uint16)
    kv = _c(kv_cache, np.uint8 if kv_dtype == 1 else np.uint16)
    bt = _c(block_table, np.int32)
    if bt.ndim != 2:
        raise ValueError("block_table must be 2-D")
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    if rows is None:
        tok, hd = np.meshgrid(np.arange(int(qsl[0]), int(qsl[-1]), dtype=np.int32),
                              np.arange(num_heads, dtype=np.int32), indexing="ij")
        rows = np.stack([tok.ravel(), hd.ravel()], axis=1)
    rows = _c(rows, np.int32).reshape(-1, 2)
    rt = _c(rows[:, 0], np.int32)
    rh = _c(rows[:, 1], np.int32)
    n = rows.shape[0]
    dv = head_size_v if head_size_v > 0 else head_size
    nb = int(kv.shape[0]) if head_size_v > 0 else int(kv.shape[1])
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    ks = _c(np.asarray(kv_scale, dtype=np.float32).reshape(2), np.float32)
    if num_threads is None:
        num_threads = os.cpu_count() or 1
    sk = None
    if sinks is not None:
        sk = _c(np.asarray(sinks, dtype=np.float32).reshape(num_heads), np.float32)
    rc = lib.pattn_ref_rows(
        q_bits.ctypes.data, kv.ctypes.data, bt.ctypes.data, sl.ctypes.data,
        qsl.ctypes.data, int(sl.shape[0]), int(bt.shape[1]), nb,
        float(scale), int(num_heads), int(num_kv_heads), int(head_size),
        int(block_size), int(window), int(causal), int(kv_dtype), ks.ctypes.data,
        rt.ctypes.data, rh.ctypes.data, int(n), int(num_splits),
        int(num_threads), out.ctypes.data, lse.ctypes.data,
        sk.ctypes.data if sk is not None else None, int(head_size_v))
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"oracle error {rc}"))
    return out, lse


def ref_varlen(q_bits, kv_cache, block_table, seq_lens, query_start_loc, **kw):
    """Oracle output for every row: (out [T, H, d], lse [T, H]) in float64.
    Rows of tokens outside [qsl[0], qsl[B]) are NaN."""
    q_bits = np.asarray(q_bits)
    T, H, d = q_bits.shape
    qsl = np.asarray(query_start_loc)
    t0, t1 = int(qsl[0]), int(qsl[-1])
    o, l = ref_rows(q_bits, kv_cache, block_table, seq_lens, query_start_loc,
                    rows=None, **kw)
    dv = o.shape[1]
    out = np.full((T, H, dv), np.nan)
    lse = np.full((T, H), np.nan)
    out[t0:t1] = o.reshape(t1 - t0, H, dv)
    lse[t0:t1] = l.reshape(t1 - t0, H)
    return out, lse
