"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every entry point include/pattn.h declares, and
rejects invalid arguments before any CUDA work."""
import ctypes
import os
import re

import pytest

import paged_varlen_attention_attn_gb300 as pa
from paged_varlen_attention_attn_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pattn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pa.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pattn_[a-z_]+)\s*\(", src)))


def test_header_declares_the_binding_names():
    assert set(declared_functions()) == set(pa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_ext_struct_layout_matches_c():
    # size_t + 7 ints (padded) + void* + size_t + void* + void** + float* + int
    assert ctypes.sizeof(pa.Ext) == 88
    assert pa.Ext.workspace.offset == 40 and pa.Ext.stream.offset == 56
    assert pa.Ext.timing_events.offset == 64 and pa.Ext.sinks.offset == 72
    assert pa.Ext.head_size_v.offset == 80


def _ext(**kw):
    base = dict(num_seqs=2, num_tokens=9, max_blocks_per_seq=3, num_blocks=8,
                max_query_len=8, max_seq_len=40, num_splits=0)
    base.update(kw)
    return pa.make_ext(**base)


FAKE = 1 << 20  # a 256-aligned non-null value; never dereferenced by these calls


def _call(lib, ext, **kw):
    args = dict(q=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, qsl=FAKE, out=FAKE, scale=0.125, H=4,
                Hkv=2, D=64, bs=16, window=0, causal=1, kv_dtype=0, kv_scale=None)
    args.update(kw)
    return pa.pattn_varlen_fwd(args["q"], args["kv"], args["bt"], args["sl"], args["qsl"],
                               args["out"], args["scale"], args["H"], args["Hkv"], args["D"],
                               args["bs"], args["window"], args["causal"], args["kv_dtype"],
                               args["kv_scale"], ext, lib=lib)


@pytest.mark.parametrize("kw,status", [
    (dict(bs=24), 1),             # block_size not a multiple of 16 (get_kv_cache_shape)
    (dict(bs=0), 1),
    (dict(H=6, Hkv=4), 1),        # heads not divisible
    (dict(D=96), 2),              # head size not built
    (dict(H=64, Hkv=2), 2),       # GQA ratio above 16
    (dict(q=0), 1),               # NULL
    (dict(out=0), 1),
    (dict(scale=-1.0), 1),
    (dict(scale=float("nan")), 1),
    (dict(scale=float("inf")), 1),
    (dict(causal=0, window=16), 2),
    (dict(causal=2), 1),
    (dict(kv_dtype=7), 2),
    (dict(kv_dtype=1, kv_scale=None), 1),
    (dict(kv_dtype=1, kv_scale=(0.0, 1.0)), 1),
    (dict(kv=FAKE + 8), 1),       # misaligned cache pointer
])
def test_invalid_arguments_are_rejected_on_the_host(lib, kw, status):
    ws = 1 << 30
    ext = _ext(workspace=ws, workspace_bytes=1 << 30)
    assert _call(lib, ext, **kw) == status


def test_missing_workspace_is_rejected(lib):
    assert _call(lib, _ext()) == 1


def test_small_workspace_is_rejected(lib):
    ext = _ext()
    need = pa.pattn_workspace_bytes(ext, 4, 2, 64, 16, lib=lib)
    assert need > 0
    ext = _ext(workspace=FAKE, workspace_bytes=need - 1)
    assert _call(lib, ext) == 3


def test_bad_struct_size_is_rejected(lib):
    ext = _ext(workspace=FAKE, workspace_bytes=1 << 30)
    ext.struct_size = 8
    assert _call(lib, ext) == 1
    assert pa.pattn_workspace_bytes(ext, 4, 2, 64, 16, lib=lib) == 0
    ext.struct_size = 71  # one byte short of the struct before `sinks`
    assert pa.pattn_workspace_bytes(ext, 4, 2, 64, 16, lib=lib) == 0


def test_struct_without_the_sinks_field_is_accepted(lib):
    # a caller built against the header before `sinks` passes 72 bytes
    ext = _ext()
    full = pa.pattn_workspace_bytes(ext, 4, 2, 64, 16, lib=lib)
    ext.struct_size = 72
    assert pa.pattn_workspace_bytes(ext, 4, 2, 64, 16, lib=lib) == full > 0


def test_split_choice(lib):
    # forced
    assert pa.pattn_decode_splits(_ext(num_splits=16), 64, 8, 64, 0, lib=lib) == 16
    # automatic: bounded by the visible blocks, by the maximum, at least 1
    e = _ext(num_seqs=8, max_seq_len=131072, max_query_len=1)
    s = pa.pattn_decode_splits(e, 64, 8, 64, 0, lib=lib)
    assert 1 <= s <= pa.MAX_SPLITS
    e = _ext(num_seqs=64, max_seq_len=16, max_query_len=1)
    assert pa.pattn_decode_splits(e, 32, 8, 16, 0, lib=lib) == 1
    # a window caps the partitions at the blocks the window can see
    e = _ext(num_seqs=4, max_seq_len=32768, max_query_len=1)
    assert pa.pattn_decode_splits(e, 32, 8, 16, 32, lib=lib) <= 3


def test_workspace_grows_with_splits(lib):
    a = pa.pattn_workspace_bytes(_ext(num_splits=1), 4, 2, 64, 16, lib=lib)
    b = pa.pattn_workspace_bytes(_ext(num_splits=16), 4, 2, 64, 16, lib=lib)
    assert b > a > 0


def test_status_strings(lib):
    for code in range(7):
        assert pa.pattn_status_string(code, lib=lib)
    assert "unknown" in pa.pattn_status_string(99, lib=lib)


def test_empty_batch_is_a_no_op(lib):
    ext = _ext(num_seqs=0, num_tokens=0, workspace=FAKE, workspace_bytes=1 << 20)
    assert _call(lib, ext) == 0


# ------------------------------------------------------------------ cache write

def _cw(lib, **kw):
    a = dict(key=FAKE, value=FAKE, cache=FAKE, slots=FAKE, T=4, Hkv=2, d=128, bs=16, nb=8,
             kv_dtype=0, kv_scale=None)
    a.update(kw)
    return pa.pattn_reshape_and_cache(a["key"], a["value"], a["cache"], a["slots"], a["T"],
                                      a["Hkv"], a["d"], a["bs"], a["nb"], a["kv_dtype"],
                                      a["kv_scale"], 0, 0, lib=lib)


@pytest.mark.parametrize("kw,status", [
    (dict(key=0), 1),                     # NULL key
    (dict(slots=0), 1),                   # NULL slot mapping
    (dict(bs=20), 1),                     # block size not a multiple of 16
    (dict(T=-1), 1),                      # negative token count
    (dict(d=12), 2),                      # head size not a multiple of 8
    (dict(kv_dtype=3), 2),                # unknown cache dtype
    (dict(kv_dtype=1), 1),                # e4m3 without scales
    (dict(kv_dtype=1, kv_scale=(0.0, 1.0)), 1),
    (dict(value=FAKE + 8), 1),            # misaligned value pointer
])
def test_cache_write_arguments_are_rejected_on_the_host(lib, kw, status):
    assert _cw(lib, **kw) == status


def test_cache_write_of_no_tokens_is_a_no_op(lib):
    assert _cw(lib, T=0) == 0


# ------------------------------------------------------------------ cascade

def _casc(lib, prefix=32, **kw):
    args = dict(q=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, qsl=FAKE, out=FAKE, scale=0.125, H=4, Hkv=2,
                D=128, bs=16, window=0, causal=1, kv_dtype=0, kv_scale=None)
    args.update(kw)
    ext = _ext(workspace=FAKE, workspace_bytes=1 << 30)
    ks = None
    if args["kv_scale"] is not None:
        ks = (ctypes.c_float * 2)(*args["kv_scale"])
    return lib.pattn_cascade_fwd(args["q"], args["kv"], args["bt"], args["sl"], args["qsl"],
                                 args["out"], args["scale"], args["H"], args["Hkv"], args["D"],
                                 args["bs"], args["window"], args["causal"], args["kv_dtype"], ks,
                                 prefix, ctypes.byref(ext))


@pytest.mark.parametrize("prefix,kw,status", [
    (24, {}, 1),                                   # prefix not a multiple of block_size
    (0, {}, 1),                                    # no prefix
    (32, dict(causal=0), 2),                       # cascade is causal only
    (32, dict(window=64), 2),                      # no window
    (32, dict(kv_dtype=1), 1),                     # e4m3 cache without scales
])
def test_cascade_arguments_are_rejected_on_the_host(lib, prefix, kw, status):
    assert _casc(lib, prefix=prefix, **kw) == status


def test_cascade_workspace_covers_partials(lib):
    e = _ext(num_seqs=4, num_tokens=100, max_query_len=64, max_seq_len=2048)
    plain = pa.pattn_workspace_bytes(e, 8, 2, 128, 16, lib=lib)
    casc = pa.pattn_cascade_workspace_bytes(e, 8, 2, 128, 16, 512, lib=lib)
    assert casc >= plain + 2 * 100 * 8 * (128 + 1) * 4
    assert pa.pattn_cascade_workspace_bytes(e, 8, 2, 128, 16, 20, lib=lib) == 0


def test_diffkv_argument_checks(lib):
    # the DiffKV layout takes head sizes that are multiples of 32 up to 256
    ext = _ext(workspace=FAKE, workspace_bytes=1 << 30, head_size_v=96)
    assert pa.pattn_workspace_bytes(ext, 4, 2, 160, 16, lib=lib) > 0
    assert pa.pattn_workspace_bytes(ext, 4, 2, 48, 16, lib=lib) == 0   # head_size % 32
    ext.head_size_v = 288
    assert pa.pattn_workspace_bytes(ext, 4, 2, 64, 16, lib=lib) == 0
    ext.head_size_v = -1
    assert pa.pattn_workspace_bytes(ext, 4, 2, 64, 16, lib=lib) == 0
    # e4m3 caches are not served in the DiffKV layout (a decode-only call,
    # which e4m3 supports in the standard layout)
    ext.head_size_v = 64
    ext.max_query_len = 1
    assert _call(lib, ext, kv_dtype=1, kv_scale=(1.0, 1.0)) == 2
