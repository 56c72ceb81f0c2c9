"""The e4m3 split of q (prefill scores over an e4m3 cache at head size 128)
rests on a property of the formats, pinned here exhaustively on the CPU: a
bf16 value v in a row whose largest magnitude has exponent E, scaled by
sc = 2^(7 - E) (so the maximum lands in [128, 256)), is y = v * sc; with
hi = e4m3(y) and lo = e4m3(y - hi), both rounded to nearest,

  - hi + lo == y exactly whenever |y| >= 2^-2 (v within 2^9 of the maximum):
    a bf16 value has 8 significant bits, hi keeps the top 4 and the
    remainder has at most 4;
  - otherwise |hi + lo - y| <= 2^-10, under 2^-16 of the maximum;
  - |y| < 256 never reaches e4m3's largest value (448).

(The kernel clamps the scale exponent to +-126, so rows whose largest
magnitude is below 2^-119 are scaled less; they are left out here.)  The
conversions are torch's float8_e4m3fn casts (round to nearest even), which
the OCP definition of e4m3 fixes; every bf16 bit pattern is tried against a
row maximum 0, 3, 8, 9, 12 and 20 binades above it."""
import numpy as np
import torch


def _split(y):
    t = torch.from_numpy(y.astype(np.float32))
    hi = t.to(torch.float8_e4m3fn).float()
    lo = (t - hi).to(torch.float8_e4m3fn).float()
    return hi.numpy().astype(np.float64), lo.numpy().astype(np.float64)


def test_two_e4m3_codes_hold_a_scaled_bf16_value():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32).astype(np.float64)
    v = v[np.isfinite(v) & (v != 0.0)]
    e_v = np.floor(np.log2(np.abs(v))).astype(np.int64)
    checked = 0
    for above in (0, 3, 8, 9, 12, 20):
        e_max = e_v + above
        keep = (e_max >= -119) & (e_max <= 127)
        y = v[keep] * np.exp2(7.0 - e_max[keep])   # exact: a power-of-two scaling
        assert np.all(np.abs(y) < 256.0)
        hi, lo = _split(y)
        assert np.all(np.isfinite(hi)) and np.all(np.isfinite(lo))
        big = np.abs(y) >= 0.25
        np.testing.assert_array_equal(hi[big] + lo[big], y[big])
        assert np.all(np.abs(hi[~big] + lo[~big] - y[~big]) <= 2.0 ** -10)
        checked += int(keep.sum())
    assert checked > 300000


def test_the_split_is_not_exact_below_the_bound():
    # the bound is tight: a value 2^10 below the row maximum with all 8
    # significant bits set loses its lowest bits to e4m3's smallest step
    y = np.array([(255.0 / 128.0) * 2.0 ** -4], dtype=np.float64)  # 1.1111111b x 2^-4
    hi, lo = _split(y)
    assert hi[0] + lo[0] != y[0]
    assert abs(hi[0] + lo[0] - y[0]) <= 2.0 ** -10
