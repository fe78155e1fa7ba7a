"""Pins for the NF4 oracle (CPU only): the published codebook, invariants of the block /
group scales, a brute-force nearest-code search in exact rational arithmetic, packing order
and requantisation stability."""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import nf4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _published():
    vals = []
    with open(os.path.join(GOLDEN, "nf4_codebook_qlora.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(float(line))
    return np.array(vals, dtype=np.float32)


def test_codebook_shape_and_anchors():
    cb = nf4.codebook()
    assert cb.dtype == np.float32 and cb.shape == (16,)
    assert np.all(np.diff(cb) > 0)
    assert cb[0] == -1.0 and cb[7] == 0.0 and cb[15] == 1.0
    assert np.sum(cb > 0) == 8 and np.sum(cb < 0) == 7


def test_codebook_equals_published_table_bitwise():
    assert np.array_equal(nf4.codebook().view(np.uint32), _published().view(np.uint32))


def _normal_weight(numel, seed=0, std=0.02):
    return (np.random.default_rng(seed).standard_normal(numel) * std).astype(np.float32)


def test_shape_rule():
    with pytest.raises(ValueError):
        nf4.quantize(np.zeros(64 * 255, np.float32))


def _brute_index(v32: np.float32, cb) -> int:
    """Nearest codebook entry by exact rational distance; ties to the lower index."""
    fv = Fraction(float(v32))
    best, bi = None, None
    for i, c in enumerate(cb):
        dd = abs(fv - Fraction(float(c)))
        if best is None or dd < best:
            best, bi = dd, i
    return bi


def test_indices_match_brute_force_including_ties():
    cb = nf4.codebook()
    rng = np.random.default_rng(11)
    x = rng.standard_normal(nf4.GROUP).astype(np.float32)
    # plant exact midpoints of neighbouring codes (ties) in block 0, whose absmax is 1
    mids = []
    for a, b in zip(cb[:-1], cb[1:]):
        m = (float(a) + float(b)) / 2
        if float(np.float32(m)) == m:
            mids.append(np.float32(m))
    assert len(mids) >= 3
    x[:64] = 0.01
    x[0] = 1.0
    x[1:1 + len(mids)] = mids
    codes, _, _ = nf4.quantize(x)
    idx = nf4.unpack_indices(codes)
    for i in range(0, 4096):
        blk = i // 64
        amax = np.max(np.abs(x[blk * 64:(blk + 1) * 64]))
        v = np.float32(x[i] / amax) if amax > 0 else np.float32(0)
        assert idx[i] == _brute_index(v, cb), i
    # ties go to the lower index
    for j, m in enumerate(mids):
        lo = int(np.searchsorted(cb, m)) - 1
        assert idx[1 + j] == lo


def test_pack_order_high_nibble_first():
    x = np.zeros(nf4.GROUP, np.float32)
    x[0] = 0.5          # block max -> code +1 (index 15)
    x[1] = -0.5         # -> code -1 (index 0)
    x[2] = 0.0          # -> index 7
    x[3] = 0.5
    codes, q, c = nf4.quantize(x)
    assert codes[0] == 0xF0 and codes[1] == 0x7F


def test_block_max_decodes_to_reconstructed_absmax():
    x = _normal_weight(4 * nf4.GROUP, seed=2)
    codes, q, c = nf4.quantize(x)
    w = nf4.dequantize(codes, q, c)
    amax_r = (q.astype(np.float32) * np.repeat(c, nf4.GROUP_BLOCKS)).astype(np.float32)
    xb, wb = x.reshape(-1, 64), w.reshape(-1, 64)
    at = np.argmax(np.abs(xb), axis=1)
    rows = np.arange(xb.shape[0])
    assert np.array_equal(np.abs(wb[rows, at]), amax_r)
    assert np.array_equal(np.sign(wb[rows, at]), np.sign(xb[rows, at]))
    # group max block is stored as 127
    assert np.all(q.reshape(-1, 256).max(axis=1) == 127)
    assert q.min() >= 0


def test_exact_scales_recover_absmax_exactly():
    """When every block absmax is an integer multiple of max/127 the double quantisation is
    exact, so the dequantised block maxima equal the true absmax bit for bit."""
    rng = np.random.default_rng(4)
    m = rng.integers(1, 128, size=256)
    m[17] = 127
    amax = (m * 2.0 ** -7).astype(np.float32)
    x = (rng.uniform(-1, 1, size=(256, 64)) * amax[:, None]).astype(np.float32)
    pos = rng.integers(0, 64, size=256)
    x[np.arange(256), pos] = amax * np.where(rng.random(256) < 0.5, -1, 1)
    codes, q, c = nf4.quantize(x.reshape(-1))
    assert c[0] == np.float32(2.0 ** -7)
    w = nf4.dequantize(codes, q, c).reshape(256, 64)
    assert np.array_equal(np.max(np.abs(w), axis=1), amax)


def test_error_bounds():
    x = _normal_weight(2 * nf4.GROUP, seed=8)
    codes, q, c = nf4.quantize(x)
    w = nf4.dequantize(codes, q, c)
    cb = nf4.codebook().astype(np.float64)
    half_gap = np.max(np.diff(cb)) / 2
    cc = np.repeat(c.astype(np.float64), nf4.GROUP_BLOCKS)
    amax = np.max(np.abs(x.reshape(-1, 64)), axis=1).astype(np.float64)
    amax_r = (q.astype(np.float32) * np.repeat(c, nf4.GROUP_BLOCKS)).astype(np.float64)
    # |amax' - absmax| <= c/2 + (division and product rounding) <= c (1/2 + 2^-15)
    assert np.all(np.abs(amax_r - amax) <= cc * (0.5 + 2.0 ** -15))
    err = np.abs(w.astype(np.float64) - x.astype(np.float64)).reshape(-1, 64)
    bound = (np.abs(amax_r - amax) + amax * (half_gap + 2.0 ** -23))[:, None] \
        + np.abs(w.astype(np.float64)).reshape(-1, 64) * 2.0 ** -23
    assert np.all(err <= bound)


def test_requantising_dequantised_weights_keeps_codes():
    x = _normal_weight(2 * nf4.GROUP, seed=9)
    codes, q, c = nf4.quantize(x)
    assert q.min() > 0
    w = nf4.dequantize(codes, q, c)
    codes2, _, _ = nf4.quantize(w)
    assert np.array_equal(codes, codes2)


def test_zero_blocks_and_zero_groups():
    x = np.zeros(nf4.GROUP, np.float32)
    codes, q, c = nf4.quantize(x)
    assert c[0] == 0 and np.all(q == 0)
    assert np.all(nf4.unpack_indices(codes) == 7)
    assert np.all(nf4.dequantize(codes, q, c) == 0)


def test_bf16_rounding_of_dequantised_base():
    x = _normal_weight(nf4.GROUP, seed=1)
    codes, q, c = nf4.quantize(x)
    w = nf4.dequantize(codes, q, c)
    wb = nf4.dequantize_bf16(codes, q, c)
    # bf16 values have zero low mantissa bits and lie within half a bf16 ulp of w
    assert np.all((wb.view(np.uint32) & 0xFFFF) == 0)
    nz = w != 0
    e = np.floor(np.log2(np.abs(w[nz]).astype(np.float64)))
    half_ulp = 2.0 ** (e - 8)          # bf16 keeps 8 significant bits
    assert np.all(np.abs(wb[nz].astype(np.float64) - w[nz]) <= half_ulp)
    assert np.all(wb[~nz] == 0)


def test_nearest_code_equals_argmin_of_exact_distances():
    """The midpoint count equals the plain argmin of |v - code| (first minimum = lower index),
    on random values, every midpoint (ties), the codes themselves and their fp32 neighbours."""
    cb = nf4.codebook()
    rng = np.random.default_rng(21)
    v = [rng.uniform(-1, 1, 20000).astype(np.float32)]
    mids = [np.float32((float(a) + float(b)) / 2) for a, b in zip(cb[:-1], cb[1:])]
    near = [np.nextafter(np.float32(m), np.float32(d)) for m in mids for d in (-2, 2)]
    v.append(np.array(mids + near + list(cb) + [0.0, -0.0], dtype=np.float32))
    v = np.concatenate(v)
    dist = np.abs(v.astype(np.float64)[:, None] - cb.astype(np.float64)[None, :])
    assert np.array_equal(nf4.nearest_code(v), np.argmin(dist, axis=1).astype(np.uint8))
