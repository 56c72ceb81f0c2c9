"""Python binding of libpattn -- paged variable-length attention for GB300.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libpattn.so`` (built by ``_build.build()``).  There is no CPU or
PyTorch fallback; if the library is missing, ``load()`` raises.

The names follow the C ABI in ``include/pattn.h``:
``pattn_varlen_fwd``, ``pattn_workspace_bytes``, ``pattn_decode_splits``,
``pattn_read_device_status``, ``pattn_status_string``, ``pattn_version``.
``forward(...)`` is a convenience wrapper for torch tensors that fills the
extension struct from the tensors' shapes and allocates the workspace with
torch (plumbing; the library itself allocates nothing).
"""
import ctypes
import os

from . import _build

KV_BF16 = 0
KV_FP8_E4M3 = 1
KV_F16 = 2  # f16 cache; q and out are f16 too
MAX_SPLITS = 64

STATUS = {0: "PATTN_OK", 1: "PATTN_ERR_INVALID_ARGUMENT", 2: "PATTN_ERR_UNSUPPORTED",
          3: "PATTN_ERR_WORKSPACE_TOO_SMALL", 4: "PATTN_ERR_CUDA",
          5: "PATTN_ERR_BAD_METADATA", 6: "PATTN_ERR_DEVICE_TIMEOUT"}

EXPORTS = ("pattn_varlen_fwd", "pattn_workspace_bytes", "pattn_decode_splits",
           "pattn_read_device_status", "pattn_status_string", "pattn_version",
           "pattn_decode_fwd_static", "pattn_reshape_and_cache",
           "pattn_reshape_and_cache_diffkv", "pattn_cascade_fwd",
           "pattn_cascade_workspace_bytes")
STATIC_SCRATCH_BYTES = 32 << 20


class PattnError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


class Ext(ctypes.Structure):
    """pattn_ext_t"""
    _fields_ = [("struct_size", ctypes.c_size_t), ("num_seqs", ctypes.c_int),
                ("num_tokens", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("max_query_len", ctypes.c_int),
                ("max_seq_len", ctypes.c_int), ("num_splits", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("stream", ctypes.c_void_p),
                ("timing_events", ctypes.POINTER(ctypes.c_void_p)),
                ("sinks", ctypes.c_void_p), ("head_size_v", ctypes.c_int)]

PHASES = ("plan", "prefill", "decode", "combine")


_lib = None


def library_path():
    return _build.LIB


def load(path=None):
    """Open libpattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise PattnError(4, f"{p} is missing; build it with __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.pattn_varlen_fwd.restype = i
    lib.pattn_varlen_fwd.argtypes = [vp, vp, vp, vp, vp, vp, f, i, i, i, i, i, i, i, vp,
                                     ctypes.POINTER(Ext)]
    lib.pattn_workspace_bytes.restype = ctypes.c_size_t
    lib.pattn_workspace_bytes.argtypes = [ctypes.POINTER(Ext), i, i, i, i]
    lib.pattn_decode_splits.restype = i
    lib.pattn_decode_splits.argtypes = [ctypes.POINTER(Ext), i, i, i, i]
    lib.pattn_read_device_status.restype = i
    lib.pattn_read_device_status.argtypes = [ctypes.POINTER(Ext)]
    lib.pattn_status_string.restype = ctypes.c_char_p
    lib.pattn_status_string.argtypes = [i]
    lib.pattn_version.restype = i
    lib.pattn_version.argtypes = []
    lib.pattn_decode_fwd_static.restype = i
    lib.pattn_decode_fwd_static.argtypes = [vp, vp, vp, vp, vp, vp, f, i, i, i, i, i, i, i, vp,
                                            i, i, i, i, i, i, vp]
    lib.pattn_cascade_fwd.restype = i
    lib.pattn_cascade_fwd.argtypes = [vp, vp, vp, vp, vp, vp, f, i, i, i, i, i, i, i, vp, i,
                                      ctypes.POINTER(Ext)]
    lib.pattn_cascade_workspace_bytes.restype = ctypes.c_size_t
    lib.pattn_cascade_workspace_bytes.argtypes = [ctypes.POINTER(Ext), i, i, i, i, i]
    lib.pattn_reshape_and_cache.restype = i
    lib.pattn_reshape_and_cache.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp, vp, vp]
    lib.pattn_reshape_and_cache_diffkv.restype = i
    lib.pattn_reshape_and_cache_diffkv.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp]
    if path is None:
        _lib = lib
    return lib


def pattn_reshape_and_cache(key, value, kv_cache, slot_mapping, num_tokens, num_kv_heads,
                            head_size, block_size, num_blocks, kv_dtype, kv_scale,
                            device_status, stream, lib=None):
    """Raw call of the KV-cache write with integer device pointers; returns
    the status code."""
    lib = lib or load()
    ks = None
    if kv_scale is not None:
        ks = (ctypes.c_float * 2)(float(kv_scale[0]), float(kv_scale[1]))
    return lib.pattn_reshape_and_cache(key, value, kv_cache, slot_mapping, int(num_tokens),
                                       int(num_kv_heads), int(head_size), int(block_size),
                                       int(num_blocks), int(kv_dtype), ks,
                                       int(device_status) or None, int(stream) or None)


def reshape_and_cache(key, value, kv_cache, slot_mapping, *, block_size, kv_dtype=KV_BF16,
                      kv_scale=None, device_status=None, stream=None):
    """pattn_reshape_and_cache on torch tensors: key/value bf16 [T, Hkv, d],
    kv_cache [2, num_blocks, block_size, Hkv, d] (bf16, or uint8 e4m3 codes),
    slot_mapping int64 [T].  ``device_status``: optional int32/uint32 tensor of
    one element that collects the out-of-pool bit.  Raises PattnError."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(key.device)
    st = pattn_reshape_and_cache(key.data_ptr(), value.data_ptr(), kv_cache.data_ptr(),
                                 slot_mapping.data_ptr(), key.shape[0], key.shape[1],
                                 key.shape[2], block_size, kv_cache.shape[1], kv_dtype, kv_scale,
                                 0 if device_status is None else device_status.data_ptr(),
                                 stream.cuda_stream)
    if st != 0:
        raise PattnError(st, "pattn_reshape_and_cache")
    return kv_cache


def reshape_and_cache_diffkv(key, value, kv_cache, slot_mapping, *, block_size,
                             kv_dtype=KV_BF16, device_status=None, stream=None):
    """pattn_reshape_and_cache_diffkv on torch tensors: key 16-bit [T, Hkv, dk],
    value [T, Hkv, dv], kv_cache [num_blocks, block_size, Hkv, dk + dv],
    slot_mapping int64 [T].  Raises PattnError."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(key.device)
    st = load().pattn_reshape_and_cache_diffkv(
        key.data_ptr(), value.data_ptr(), kv_cache.data_ptr(), slot_mapping.data_ptr(),
        int(key.shape[0]), int(key.shape[1]), int(key.shape[2]), int(value.shape[2]),
        int(block_size), int(kv_cache.shape[0]), int(kv_dtype),
        None if device_status is None else device_status.data_ptr(), stream.cuda_stream)
    if st != 0:
        raise PattnError(st, "pattn_reshape_and_cache_diffkv")
    return kv_cache


def pattn_cascade_workspace_bytes(ext, num_heads, num_kv_heads, head_size, block_size,
                                  common_prefix_len, lib=None):
    lib = lib or load()
    return lib.pattn_cascade_workspace_bytes(ctypes.byref(ext), int(num_heads), int(num_kv_heads),
                                             int(head_size), int(block_size),
                                             int(common_prefix_len))


def cascade_forward(q, kv_cache, block_table, seq_lens, query_start_loc, *, scale, num_heads,
                    num_kv_heads, head_size, block_size, common_prefix_len, window=0, causal=1,
                    kv_dtype=KV_BF16, kv_scale=None, max_query_len, max_seq_len, num_splits=0,
                    out=None, workspace=None, stream=None, sinks=None):
    """pattn_cascade_fwd on torch tensors: pattn_varlen_fwd for a batch whose
    requests share their first common_prefix_len keys (same blocks).
    ``sinks``: optional fp32 [num_heads] device tensor of attention-sink logits.
    Returns ``out``; raises PattnError."""
    import torch
    dev = q.device
    T = q.shape[0]
    if out is None:
        odt = torch.float16 if kv_dtype == KV_F16 else torch.bfloat16
        out = torch.empty((T, num_heads, head_size), dtype=odt, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    ext = make_ext(num_seqs=seq_lens.shape[0], num_tokens=T,
                   max_blocks_per_seq=block_table.shape[1], num_blocks=kv_cache.shape[1],
                   max_query_len=max_query_len, max_seq_len=max_seq_len,
                   num_splits=num_splits, stream=stream.cuda_stream,
                   sinks=_sinks_ptr(sinks, num_heads, dev))
    need = pattn_cascade_workspace_bytes(ext, num_heads, num_kv_heads, head_size, block_size,
                                         common_prefix_len)
    if need == 0:
        raise PattnError(1, "pattn_cascade_workspace_bytes")
    ws = (workspace or _default_ws).get(need, dev)
    ext.workspace = ws.data_ptr()
    ext.workspace_bytes = ws.numel()
    ks = None
    if kv_scale is not None:
        ks = (ctypes.c_float * 2)(float(kv_scale[0]), float(kv_scale[1]))
    st = load().pattn_cascade_fwd(q.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(),
                                  seq_lens.data_ptr(), query_start_loc.data_ptr(), out.data_ptr(),
                                  float(scale), int(num_heads), int(num_kv_heads), int(head_size),
                                  int(block_size), int(window), int(causal), int(kv_dtype), ks,
                                  int(common_prefix_len), ctypes.byref(ext))
    if st != 0:
        raise PattnError(st, "pattn_cascade_fwd")
    forward.last_ext = ext
    return out


def make_ext(*, num_seqs, num_tokens, max_blocks_per_seq, num_blocks, max_query_len,
             max_seq_len, num_splits=0, workspace=0, workspace_bytes=0, stream=0,
             timing_events=None, sinks=0, head_size_v=0):
    e = Ext()
    e.struct_size = ctypes.sizeof(Ext)
    e.num_seqs, e.num_tokens = int(num_seqs), int(num_tokens)
    e.max_blocks_per_seq, e.num_blocks = int(max_blocks_per_seq), int(num_blocks)
    e.max_query_len, e.max_seq_len = int(max_query_len), int(max_seq_len)
    e.num_splits = int(num_splits)
    e.workspace = int(workspace) or None
    e.workspace_bytes = int(workspace_bytes)
    e.stream = int(stream) or None
    e.sinks = int(sinks) or None
    e.head_size_v = int(head_size_v)
    if timing_events is not None:
        arr = (ctypes.c_void_p * 8)(*[int(x) for x in timing_events])
        e._events_keepalive = arr
        e.timing_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    return e


def pattn_varlen_fwd(q, kv_cache, block_table, seq_lens, query_start_loc, out, scale,
                     num_heads, num_kv_heads, head_size, block_size, window, causal,
                     kv_dtype, kv_scale, ext, lib=None):
    """Raw call with integer device pointers; returns the status code."""
    lib = lib or load()
    ks = None
    if kv_scale is not None:
        ks = (ctypes.c_float * 2)(float(kv_scale[0]), float(kv_scale[1]))
    return lib.pattn_varlen_fwd(q, kv_cache, block_table, seq_lens, query_start_loc, out,
                                float(scale), int(num_heads), int(num_kv_heads),
                                int(head_size), int(block_size), int(window), int(causal),
                                int(kv_dtype), ks, ctypes.byref(ext))


def pattn_decode_fwd_static(q, kv_cache, block_table, seq_lens, query_start_loc, out, scale,
                            num_heads, num_kv_heads, head_size, block_size, window, causal,
                            kv_dtype, kv_scale, num_seqs, num_tokens, max_blocks_per_seq,
                            num_blocks, max_seq_len, num_splits, stream, lib=None):
    """Raw call of the workspace-free decode entry point; returns the status.
    For callers that cannot allocate device memory (see include/pattn.h)."""
    lib = lib or load()
    ks = None
    if kv_scale is not None:
        ks = (ctypes.c_float * 2)(float(kv_scale[0]), float(kv_scale[1]))
    return lib.pattn_decode_fwd_static(q, kv_cache, block_table, seq_lens, query_start_loc,
                                       out, float(scale), int(num_heads), int(num_kv_heads),
                                       int(head_size), int(block_size), int(window),
                                       int(causal), int(kv_dtype), ks, int(num_seqs),
                                       int(num_tokens), int(max_blocks_per_seq),
                                       int(num_blocks), int(max_seq_len), int(num_splits),
                                       int(stream) or None)


def pattn_workspace_bytes(ext, num_heads, num_kv_heads, head_size, block_size, lib=None):
    return (lib or load()).pattn_workspace_bytes(ctypes.byref(ext), num_heads, num_kv_heads,
                                                 head_size, block_size)


def pattn_decode_splits(ext, num_heads, num_kv_heads, block_size, window, lib=None):
    return (lib or load()).pattn_decode_splits(ctypes.byref(ext), num_heads, num_kv_heads,
                                               block_size, window)


def pattn_read_device_status(ext, lib=None):
    return (lib or load()).pattn_read_device_status(ctypes.byref(ext))


def pattn_status_string(status, lib=None):
    return (lib or load()).pattn_status_string(int(status)).decode()


def pattn_version(lib=None):
    return (lib or load()).pattn_version()


class Workspace:
    """A torch-allocated device workspace, grown on demand (plumbing only)."""

    def __init__(self):
        self.buf = None

    def get(self, nbytes, device):
        import torch
        nbytes = max(256, int(nbytes))
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != torch.device(device):
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        return self.buf


_default_ws = Workspace()


def _sinks_ptr(sinks, num_heads, device):
    """Device pointer of an fp32 [num_heads] sink tensor (0 for None)."""
    if sinks is None:
        return 0
    import torch
    if (sinks.dtype != torch.float32 or sinks.device != torch.device(device) or
            sinks.numel() != num_heads or not sinks.is_contiguous()):
        raise ValueError("sinks must be a contiguous fp32 [num_heads] tensor on q's device")
    return sinks.data_ptr()


def forward(q, kv_cache, block_table, seq_lens, query_start_loc, *, scale, num_heads,
            num_kv_heads, head_size, block_size, window=0, causal=1, kv_dtype=KV_BF16,
            kv_scale=None, max_query_len, max_seq_len, num_splits=0, out=None,
            workspace=None, stream=None, timing_events=None, sinks=None, head_size_v=0,
            check=True, lib=None):
    """pattn_varlen_fwd on torch tensors (all on one CUDA device).

    max_query_len / max_seq_len are host ints (as in FlashAttentionMetadata):
    the library never reads device memory on the host.  ``timing_events``:
    optional 8 raw cudaEvent_t handles (see pattn_ext_t).  ``sinks``: optional
    fp32 [num_heads] device tensor of attention-sink logits.  ``head_size_v``:
    > 0 selects the DiffKV cache layout [num_blocks, block_size, num_kv_heads,
    head_size + head_size_v] and an output of head size head_size_v (see
    pattn_ext_t).  ``lib``: a library handle from ``load(path)`` (default: the
    built libpattn.so).  Returns ``out``.
    """
    import torch
    dev = q.device
    T = q.shape[0]
    if out is None:
        odt = torch.float16 if kv_dtype == KV_F16 else torch.bfloat16
        out = torch.empty((T, num_heads, head_size_v or head_size), dtype=odt, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    num_blocks = kv_cache.shape[0] if head_size_v else kv_cache.shape[1]
    ext = make_ext(num_seqs=seq_lens.shape[0], num_tokens=T,
                   max_blocks_per_seq=block_table.shape[1], num_blocks=num_blocks,
                   max_query_len=max_query_len, max_seq_len=max_seq_len,
                   num_splits=num_splits, stream=stream.cuda_stream,
                   timing_events=timing_events, sinks=_sinks_ptr(sinks, num_heads, dev),
                   head_size_v=head_size_v)
    need = pattn_workspace_bytes(ext, num_heads, num_kv_heads, head_size, block_size, lib=lib)
    if need == 0:
        raise PattnError(1, "pattn_workspace_bytes")
    ws = (workspace or _default_ws).get(need, dev)
    ext.workspace = ws.data_ptr()
    ext.workspace_bytes = ws.numel()
    st = pattn_varlen_fwd(q.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(),
                          seq_lens.data_ptr(), query_start_loc.data_ptr(), out.data_ptr(),
                          scale, num_heads, num_kv_heads, head_size, block_size, window,
                          causal, kv_dtype, kv_scale, ext, lib=lib)
    if check and st != 0:
        raise PattnError(st, "pattn_varlen_fwd")
    forward.last_ext = ext
    return out
