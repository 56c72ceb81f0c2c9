"""Pins of the oracle's KV-cache write and e4m3 encoder (CPU only).

The encoder is checked against torch's float8_e4m3fn cast (round to nearest
even) wherever that cast is finite, on every exact tie between neighbouring
codes and on the values one fp32 ulp either side, plus the saturation and NaN
rules of the definition.  The cache write is checked against a numpy scatter
of the rows to their slots (and torch's cast for e4m3).  Planted mistakes in
the oracle's source must each fail one of these pins."""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
E4M3_MAX = 448.0
TORCH_NAN_FROM = 464.0  # torch's cast (not saturating) gives NaN above this


def _codes_as_float():
    c = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn)
    return c.to(torch.float64).numpy()  # magnitudes of codes 0x00..0x7E, ascending


def _probe_values():
    mags = _codes_as_float()
    mids = (mags[:-1] + mags[1:]) / 2.0          # exact ties (representable in fp32)
    pts = np.concatenate([mags, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(-np.inf))
    rng = np.random.default_rng(7)
    rnd = (rng.standard_normal(4000) * np.exp(rng.uniform(-9, 6, 4000))).astype(np.float32)
    v = np.concatenate([pts, up, dn, rnd, np.float32([0.0, 1e-30, 2.0 ** -10])])
    v = v[np.abs(v) < TORCH_NAN_FROM]
    return np.concatenate([v, -v]).astype(np.float32)


def encoder_failures(lib):
    bad = []
    v = _probe_values()
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x), lib=lib) for x in v], dtype=np.uint8)
    if not np.array_equal(got, ref):
        bad.append("encode-vs-torch")
    sat = [(448.0, 0x7E), (463.0, 0x7E), (500.0, 0x7E), (1e30, 0x7E), (np.inf, 0x7E),
           (-448.0, 0xFE), (-1e9, 0xFE), (-np.inf, 0xFE)]
    if any(oracle.e4m3_encode(x, lib=lib) != c for x, c in sat):
        bad.append("saturation")
    if oracle.e4m3_encode(float("nan"), lib=lib) & 0x7F != 0x7F:
        bad.append("nan")
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        if oracle.e4m3_encode(oracle.e4m3_to_double(c, lib=lib), lib=lib) != c:
            bad.append("round-trip")
            break
    return bad


def _cache_case(kv_dtype, seed=3, T=37, Hkv=2, d=16, bs=16, nb=9):
    rng = np.random.default_rng(seed)
    key = torch.randn(T, Hkv, d, generator=torch.Generator().manual_seed(seed)) * 3
    val = torch.randn(T, Hkv, d, generator=torch.Generator().manual_seed(seed + 1)) * 3
    key_bits = key.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    val_bits = val.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[::5] = -1                              # padding tokens write nothing
    if kv_dtype == 0:
        cache = rng.integers(0, 1 << 16, size=(2, nb, bs, Hkv, d), dtype=np.uint16)
    else:
        cache = rng.integers(0, 256, size=(2, nb, bs, Hkv, d), dtype=np.uint8)
    scale = (float(key.abs().max()) / E4M3_MAX, float(val.abs().max()) / E4M3_MAX)
    return key_bits, val_bits, slots, cache, scale


def _scatter_expected(key_bits, val_bits, slots, cache, kv_dtype, scale):
    exp = cache.copy()
    nb, bs, Hkv, d = cache.shape[1:]
    flat = exp.reshape(2, nb * bs, Hkv, d)
    ok = slots >= 0
    for kv, bits, sc in ((0, key_bits, scale[0]), (1, val_bits, scale[1])):
        if kv_dtype == 0:
            flat[kv, slots[ok]] = bits[ok]
        else:
            x = torch.from_numpy(bits[ok].view(np.int16)).view(torch.bfloat16).float()
            q = (x / torch.tensor(sc, dtype=torch.float32)).to(torch.float8_e4m3fn)
            flat[kv, slots[ok]] = q.view(torch.uint8).numpy()
    return exp


def cache_write_failures(lib):
    bad = []
    for kv_dtype in (0, 1):
        key_bits, val_bits, slots, cache, scale = _cache_case(kv_dtype)
        exp = _scatter_expected(key_bits, val_bits, slots, cache, kv_dtype, scale)
        got = oracle.reshape_and_cache(key_bits, val_bits, cache.copy(), slots, num_kv_heads=2,
                                       head_size=16, block_size=16, kv_dtype=kv_dtype,
                                       kv_scale=scale, lib=lib)
        if not np.array_equal(got, exp):
            bad.append(f"scatter-{kv_dtype}")
    key_bits, val_bits, slots, cache, scale = _cache_case(0)
    slots[3] = cache.shape[1] * cache.shape[2]  # one past the pool
    try:
        oracle.reshape_and_cache(key_bits, val_bits, cache, slots, num_kv_heads=2,
                                 head_size=16, block_size=16, lib=lib)
        bad.append("slot-range")
    except oracle.OracleError:
        pass
    return bad


def diffkv_write_failures(lib):
    """DiffKV layout: a numpy scatter of [K | V] rows to their slots."""
    bad = []
    rng = np.random.default_rng(17)
    T, Hkv, dk, dv, bs, nb = 29, 2, 16, 40, 16, 5
    key = rng.integers(0, 1 << 16, (T, Hkv, dk), dtype=np.uint16)
    val = rng.integers(0, 1 << 16, (T, Hkv, dv), dtype=np.uint16)
    cache = rng.integers(0, 1 << 16, (nb, bs, Hkv, dk + dv), dtype=np.uint16)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[::6] = -1
    exp = cache.copy()
    flat = exp.reshape(nb * bs, Hkv, dk + dv)
    ok = slots >= 0
    flat[slots[ok], :, :dk] = key[ok]
    flat[slots[ok], :, dk:] = val[ok]
    got = oracle.reshape_and_cache_diffkv(key, val, cache.copy(), slots, num_kv_heads=Hkv,
                                          head_size=dk, head_size_v=dv, block_size=bs, lib=lib)
    if not np.array_equal(got, exp):
        bad.append("diffkv-scatter")
    slots[1] = nb * bs
    try:
        oracle.reshape_and_cache_diffkv(key, val, cache.copy(), slots, num_kv_heads=Hkv,
                                        head_size=dk, head_size_v=dv, block_size=bs, lib=lib)
        bad.append("diffkv-slot-range")
    except oracle.OracleError:
        pass
    return bad


def test_diffkv_write_pins():
    assert diffkv_write_failures(None) == []


def test_encoder_pins():
    assert encoder_failures(None) == []


def test_cache_write_pins():
    assert cache_write_failures(None) == []


def test_cache_write_with_block_size_32_and_head_size_64():
    key_bits, val_bits, slots, cache, scale = _cache_case(1, seed=11, T=50, Hkv=4, d=64, bs=32,
                                                          nb=5)
    exp = _scatter_expected(key_bits, val_bits, slots, cache, 1, scale)
    got = oracle.reshape_and_cache(key_bits, val_bits, cache.copy(), slots, num_kv_heads=4,
                                   head_size=64, block_size=32, kv_dtype=1, kv_scale=scale)
    assert np.array_equal(got, exp)


MUTATIONS = {
    "ties_away_from_zero": ("c = (lo & 1) ? lo + 1 : lo;", "c = lo + 1;"),
    "overflow_to_nan": ("if (a >= 448.0) return (uint8_t)((sign << 7) | 0x7E);",
                        "if (a >= 448.0) return (uint8_t)((sign << 7) | 0x7F);"),
    "sign_dropped": ("return (uint8_t)((sign << 7) | c);", "return (uint8_t)c;"),
    "scale_multiplied": ("const float q = x / sc;", "const float q = x * sc;"),
    "block_and_slot_swapped": ("const int64_t blk = s / block_size, slot = s % block_size;",
                               "const int64_t blk = s % block_size, slot = s / block_size;"),
    "k_and_v_swapped": ("const uint16_t* src = kv ? value : key;",
                        "const uint16_t* src = kv ? key : value;"),
    "negative_slot_written": ("if (s < 0) continue;", "if (s < 0) s = 0;"),
    "diffkv_v_at_row_start": ("row[head_size + j] = value[", "row[j] = value["),
    "diffkv_row_width_k": ("* (int64_t)width;", "* (int64_t)head_size;"),
    "diffkv_value_stride_k": ("value[((int64_t)t * num_kv_heads + h) * head_size_v + j]",
                              "value[((int64_t)t * num_kv_heads + h) * head_size + j]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "pattn_ref.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found once"
    src = src.replace(old, new)
    if name == "negative_slot_written":
        src = src.replace("const int64_t s = slot_mapping[t];", "int64_t s = slot_mapping[t];", 1)
    (tmp_path / "mut.c").write_text(src)
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                    str(tmp_path / "mut.c"), "-lm"], check=True)
    lib = oracle.bind(str(so))
    assert (encoder_failures(lib) + cache_write_failures(lib) + diffkv_write_failures(lib)), \
        f"{name} went unnoticed"
