"""Pins of the groupwise Int4 oracle ("loralei" README, QLoRA section: int4 base, group sizes 32,
64, 128 or 256) against facts that do not come from the oracle itself: exact round trips of
weights that lie on a 16-level grid, literal code bytes and bf16 scale bits for a hand-made row,
the nearest-level property, range coverage, and constant groups."""
import numpy as np
import pytest

from oracle import int4 as oi4

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_hand_made_row_codes_and_scale_bits():
    # one group of 32: (i - 8) / 2 for i = 0..15, then the same levels descending.  mn = -4,
    # mx = 3.5, so s = 7.5 / 15 = 0.5 (bf16 0x3F00) and z = -4 + 8 * 0.5 = 0 (bf16 0x0000);
    # the codes are i, packed high nibble first.
    lv = (np.arange(16) - 8) / 2.0
    w = np.concatenate([lv, lv[::-1]]).astype(np.float32)[None, :]
    codes, s, z, q = oi4.quantize(w, 32)
    assert list(codes[:8]) == [0x01, 0x23, 0x45, 0x67, 0x89, 0xAB, 0xCD, 0xEF]
    assert list(codes[8:]) == [0xFE, 0xDC, 0xBA, 0x98, 0x76, 0x54, 0x32, 0x10]
    sz = oi4.scale_zero_bits(s, z)
    assert sz.shape == (1, 1, 2) and sz[0, 0, 0] == 0x3F00 and sz[0, 0, 1] == 0x0000
    assert np.array_equal(oi4.dequantize(codes, s, z, 1, 32, 32), w)


@pytest.mark.parametrize("group", oi4.GROUPS)
def test_grid_weights_round_trip_exactly(group):
    # Each group lies on the grid (q - 8) * 2^e + k * 2^e with both end codes 0 and 15 present:
    # then mn = (k - 8) 2^e and mx = (k + 7) 2^e, the scale is exactly 2^e, the zero k 2^e, and
    # every value (a small integer times 2^e) is a bf16 value, so quantise -> dequantise is exact
    # and the codes are the chosen q.
    rng = np.random.default_rng(group)
    rows, cols = 6, 4 * group
    ng = cols // group
    e = rng.integers(-12, 4, size=(rows, ng)).astype(np.float64)
    k = rng.integers(-100, 100, size=(rows, ng)).astype(np.float64)
    q = rng.integers(0, 16, size=(rows, ng, group))
    q[:, :, 0], q[:, :, 1] = 0, 15
    w = ((q - 8) + k[:, :, None]) * np.exp2(e)[:, :, None]
    w32 = w.reshape(rows, cols).astype(np.float32)
    assert np.array_equal(oi4.bf16_round(w32), w32)
    codes, s, z, qq = oi4.quantize(w32, group)
    assert np.array_equal(s, np.exp2(e).astype(np.float32))
    assert np.array_equal(z, (k * np.exp2(e)).astype(np.float32))
    assert np.array_equal(qq, q.reshape(rows, cols).astype(np.uint8))
    assert np.array_equal(oi4.dequantize(codes, s, z, rows, cols, group), w32)
    # the stored layout is group-major: pair (g, i) belongs to row i, columns [g G, (g+1) G)
    sz = oi4.scale_zero_bits(s, z)
    g, i = ng - 1, rows - 2
    assert sz[g, i, 0] == oi4.bf16_bits(np.float32(np.exp2(e[i, g])))
    s2, z2 = oi4.split_scale_zero(sz)
    assert np.array_equal(s2, s) and np.array_equal(z2, z)


def _bf16_weights(rng, rows, cols, scale=0.05):
    return oi4.bf16_round((rng.standard_normal((rows, cols)) * scale).astype(np.float32))


@pytest.mark.parametrize("group", oi4.GROUPS)
def test_codes_pick_the_nearest_level(group):
    # Every code is the nearest of the 16 levels (q - 8) s + z of its group, up to the fp32
    # rounding of (w - z) / s; a wrong offset, sign or clamp breaks this.
    rng = np.random.default_rng(7 + group)
    rows, cols = 8, 2 * max(group, 64)
    w = _bf16_weights(rng, rows, cols)
    w[0, :group] += 3.0                      # an offset group: the zero point is far from 0
    w = oi4.bf16_round(w)
    codes, s, z, q = oi4.quantize(w, group)
    lv = (np.arange(16, dtype=np.float64) - 8)[None, None, :] * s[:, :, None].astype(np.float64) + z[:, :, None]
    wg = w.reshape(rows, cols // group, group).astype(np.float64)
    dist = np.abs(wg[:, :, :, None] - lv[:, :, None, :])
    got = np.take_along_axis(dist, q.reshape(rows, cols // group, group, 1).astype(np.int64), axis=3)[..., 0]
    slack = 1e-6 * s[:, :, None].astype(np.float64)
    assert np.all(got <= dist.min(axis=3) + slack)


@pytest.mark.parametrize("group", oi4.GROUPS)
def test_levels_cover_each_groups_range(group):
    # The 16 levels span [mn, mx]: both extremes reconstruct within half a step (plus the bf16
    # rounding of s and z), so nothing is clipped away.
    rng = np.random.default_rng(100 + group)
    rows, cols = 4, 4 * group
    w = _bf16_weights(rng, rows, cols, scale=1.0)
    codes, s, z, _ = oi4.quantize(w, group)
    wd = oi4.dequantize(codes, s, z, rows, cols, group).astype(np.float64)
    wg = w.reshape(rows, -1, group).astype(np.float64)
    dg = wd.reshape(rows, -1, group)
    err = np.abs(wg - dg)
    bound = 0.5 * s.astype(np.float64) * (1 + 2 ** -6) + 2 ** -8 * (np.abs(wg).max(axis=2) + 16 * s)
    assert np.all(err.max(axis=2) <= bound)
    amin, amax = wg.argmin(axis=2), wg.argmax(axis=2)
    for a in (amin, amax):
        e = np.take_along_axis(err, a[:, :, None], axis=2)[..., 0]
        assert np.all(e <= 0.5 * s * (1 + 2 ** -6) + 2 ** -8 * (np.abs(wg).max(axis=2) + 16 * s))


def test_constant_and_zero_groups():
    w = np.zeros((2, 64), dtype=np.float32)
    w[1, :32] = 0.375
    w[1, 32:] = -1.25
    codes, s, z, q = oi4.quantize(w, 32)
    assert np.all(s == 0) and np.all(q == 8)
    assert np.array_equal(z, np.array([[0.0, 0.0], [0.375, -1.25]], dtype=np.float32))
    assert np.array_equal(oi4.dequantize(codes, s, z, 2, 64, 32), w)


def test_rejects_bad_group_or_shape():
    with pytest.raises(ValueError):
        oi4.quantize(np.zeros((2, 64), np.float32), 16)
    with pytest.raises(ValueError):
        oi4.quantize(np.zeros((2, 96), np.float32), 64)
