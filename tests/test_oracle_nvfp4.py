"""Pins of the NVFP4 oracle ("LoRA Optimizations", FP32 LoRA gradients: weight-only NVFP4 bases)
against facts that do not come from the oracle itself: the E2M1 value table and its tie cases as
literals, E4M3 decoding and rounding against PyTorch's float8_e4m3fn conversion, exact round trips
of weights built on the two-level grid, the nearest-level property, and the storage layout."""
import numpy as np
import pytest
import torch

from oracle import nvfp4 as nv


def test_e2m1_value_table():
    want = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(nv.e2m1_value(np.arange(8))) == want
    assert list(nv.e2m1_value(np.arange(8, 16))) == [-x for x in want]
    assert np.signbit(nv.e2m1_value(8))


def test_e2m1_rounding_ties_and_saturation():
    y = np.array([0.25, 0.2499, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.01, 7.0, 100.0, -0.25, -0.3, -6.5, 2.9, 0.0],
                 dtype=np.float32)
    want = [0, 0, 2, 2, 4, 4, 6, 6, 7, 7, 7, 8, 9, 15, 5, 0]
    assert list(nv.round_e2m1(y)) == want


def test_e4m3_matches_torch_float8():
    b = np.arange(255)
    b = b[b != 127]                               # S.1111.111 is NaN
    ref = torch.from_numpy(b.astype(np.uint8)).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(nv.e4m3_value(b).astype(np.float32), ref)
    assert nv.e4m3_value(126) == 448.0 and nv.e4m3_value(1) == 2.0 ** -9
    grid = nv.e4m3_value(np.arange(127))
    mids = (grid[:-1] + grid[1:]) / 2             # every tie
    rng = np.random.default_rng(3)
    x = np.concatenate([mids, grid, rng.uniform(0, 448, 20000), np.exp2(rng.uniform(-12, 8.8, 20000))])
    x = x[x <= 448].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(nv.round_e4m3(x), ref)
    assert list(nv.round_e4m3(np.array([464.0, 1e9], np.float32))) == [126, 126]   # saturation


def test_grid_weights_round_trip_exactly():
    # S_g = 2^k exactly (one block holds 6 * 448 * 2^k); each block's largest magnitude is
    # 6 * s_b * 2^k for a chosen E4M3 s_b, and every element is e2m1 * s_b * 2^k: quantisation
    # must give back s_b, the codes and the values exactly.
    rng = np.random.default_rng(5)
    rows, cols, k = 8, 256, -7
    nb = cols // 16
    sb = rng.integers(24, 127, size=(rows, nb)).astype(np.uint8)     # normal E4M3 scales
    sb[0, 0] = 126                                                   # 448: sets the tensor maximum
    q = rng.integers(0, 16, size=(rows, nb, 16)).astype(np.uint8)
    q[:, :, 0] = 7                                                   # +6 in every block
    q[:, :, 1] = 8                                                   # and a -0
    w = nv.e2m1_value(q) * nv.e4m3_value(sb)[:, :, None] * 2.0 ** k
    w32 = w.reshape(rows, cols).astype(np.float32)
    assert np.array_equal(w32.astype(np.float64), w.reshape(rows, cols))
    codes, sb2, sg, q2 = nv.quantize(w32)
    assert sg == np.float32(2.0 ** k)
    assert np.array_equal(sb2, sb)
    qq = q.reshape(rows, cols).copy()
    assert np.array_equal(q2, qq)
    back = nv.dequantize(codes, sb2, sg, rows, cols)
    assert np.array_equal(back, w32)
    assert np.array_equal(np.signbit(back), np.signbit(w32))


def test_codes_pick_the_nearest_level_and_error_bound():
    rng = np.random.default_rng(9)
    rows, cols = 16, 512
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    w[3, 64:80] *= 40.0                            # a loud block
    w[5, :16] = 0.0                                # a zero block
    codes, sb, sg, q = nv.quantize(w)
    S = (nv.e4m3_value(sb).astype(np.float32) * sg).astype(np.float32)
    y = (w.reshape(rows, -1, 16) / np.where(S > 0, S, 1)[:, :, None]).astype(np.float64)
    levels = nv.e2m1_value(np.arange(16))
    dist = np.abs(y[..., None] - levels)
    got = np.take_along_axis(dist, q.reshape(rows, -1, 16, 1).astype(np.int64), axis=3)[..., 0]
    live = (S > 0)[:, :, None]
    assert np.all(~live | (got <= dist.min(axis=3) + 1e-12))
    wd = nv.dequantize(codes, sb, sg, rows, cols).astype(np.float64).reshape(rows, -1, 16)
    err = np.abs(wd - w.reshape(rows, -1, 16))
    assert np.all(err <= S[:, :, None] * 1.0 + 1e-6 * np.abs(w.reshape(rows, -1, 16)))
    assert np.all(wd[5, 0] == 0)


def test_zero_tensor_and_layout():
    codes, sb, sg, q = nv.quantize(np.zeros((4, 64), np.float32))
    assert sg == 1.0 and not sb.any() and not codes.any()
    sb = np.arange(2 * 8, dtype=np.uint8).reshape(2, 8)            # 2 rows, 128 columns
    st = nv.scale_bytes(sb)
    assert st.shape == (2, 2, 4)
    assert st[1, 0, 2] == sb[0, 6] and st[0, 1, 3] == sb[1, 3]
    assert np.array_equal(nv.unscale_bytes(st), sb)
    c = nv.pack_codes(np.array([1, 2, 3, 15], np.uint8))
    assert list(c) == [0x21, 0xF3]                                  # element 2i in the low nibble
    assert list(nv.unpack_codes(c)) == [1, 2, 3, 15]


def test_rejects_bad_shape():
    with pytest.raises(ValueError):
        nv.quantize(np.zeros((2, 48), np.float32))
