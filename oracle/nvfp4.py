"""Exact oracle of the NVFP4 weight-only base: FP4 E2M1 codes with FP8 E4M3 scales per 16-element
block and one fp32 scale per tensor.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"LoRA Optimizations" (docs.axolotl.ai), FP32 LoRA gradients: native weight-only torchao
NVFP4Tensor bases keep their quantised forward, and dynamic NVFP4 activation quantisation is
rejected for training with the LoRA kernels -- so the activations stay bf16 and the base weight is
NVFP4.  The pages print no formulas; the readings taken here are the usual NVFP4 two-level scaling:

  * E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit, no inf/NaN): magnitudes
    0, 0.5, 1, 1.5, 2, 3, 4, 6.  E4M3 ("fn": 1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits, no inf, only S.1111.111 is NaN): largest finite 448, smallest subnormal 2^-9.
  * per tensor: S_g = fp32(amax / (6 * 448)), amax = max |w| (S_g = 1 when that is 0).
  * per block of 16 consecutive elements of a row: d = fp32(fp32(bmax / 6) / S_g), bmax the
    block's max |w|; s_b = E4M3(d), rounded to nearest with ties to even and saturated at 448.
  * per element: S = fp32(s_b * S_g); y = fp32(w / S); code = E2M1(y), rounded to nearest with
    ties to even (the even code, i.e. mantissa bit 0) and saturated at 6, sign bit = sign of w
    (so a negative w that rounds to zero is -0); every code is 0 when S == 0.
  * dequantisation: w' = fp32(e2m1(code) * fp32(s_b * S_g)), then bf16 for the matmul.
  * storage: codes row-major, element 2i in the LOW nibble of byte i (the PyTorch
    float4_e2m1fn_x2 order); block scales as E4M3 bytes in [cols/64][rows][4] -- the four
    16-element blocks of one 64-column span of a row in one 32-bit word, spans group-major -- and
    S_g as one fp32 value.
"""
from __future__ import annotations

import numpy as np

BLOCK = 16
E2M1_MAX = 6.0
E4M3_MAX = 448.0


def e2m1_value(code) -> np.ndarray:
    """Values of 4-bit E2M1 codes (fp64, exact), from the bit fields."""
    c = np.asarray(code, dtype=np.int64)
    e, m, s = (c >> 1) & 3, c & 1, (c >> 3) & 1
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return np.where(s == 1, -mag, mag)


def e4m3_value(byte) -> np.ndarray:
    """Values of E4M3 bytes (fp64, exact) for the finite encodings, from the bit fields."""
    b = np.asarray(byte, dtype=np.int64)
    e, m, s = (b >> 3) & 15, b & 7, (b >> 7) & 1
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    return np.where(s == 1, -mag, mag)


def _round_grid(a: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid value to each a >= 0 (grid ascending, exact in fp64); a tie goes
    to the even index (the encoding whose mantissa bit is 0); beyond the grid: the last index."""
    a = np.asarray(a, dtype=np.float64)
    hi = np.clip(np.searchsorted(grid, a, side="left"), 1, len(grid) - 1)
    lo = hi - 1
    dl, dh = a - grid[lo], grid[hi] - a
    pick_hi = (dh < dl) | ((dh == dl) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(a >= grid[-1], len(grid) - 1, idx)
    return np.where(a <= grid[0], 0, idx)


_E2M1_GRID = e2m1_value(np.arange(8))
_E4M3_GRID = e4m3_value(np.arange(127))      # bytes 0..126: 0 .. 448


def round_e4m3(d) -> np.ndarray:
    """E4M3 byte of non-negative values: nearest, ties to even, saturated at 448."""
    return _round_grid(d, _E4M3_GRID).astype(np.uint8)


def round_e2m1(y) -> np.ndarray:
    """E2M1 code of values: nearest magnitude, ties to even, saturated at 6; sign bit of y."""
    y = np.asarray(y, dtype=np.float32)
    mag = _round_grid(np.abs(y).astype(np.float64), _E2M1_GRID)
    return (mag | (np.signbit(y).astype(np.int64) << 3)).astype(np.uint8)


def quantize(w32: np.ndarray):
    """Quantise a (rows, cols) weight given as fp32 values (normally bf16 values); cols % 64 == 0.

    Returns (codes uint8 [rows*cols/2], sb uint8 [rows, cols/16] E4M3 block scales,
    S_g float32 scalar, q uint8 [rows, cols] codes)."""
    w = np.asarray(w32, dtype=np.float32)
    if w.ndim != 2 or w.shape[1] % 64:
        raise ValueError("NVFP4 here needs a 2-D weight whose column count is a multiple of 64")
    rows, cols = w.shape
    f = np.float32
    amax = f(np.abs(w).max()) if w.size else f(0.0)
    sg = f(amax / f(E2M1_MAX * E4M3_MAX))
    if not sg > 0:
        sg = f(1.0)
    blk = w.reshape(rows, cols // BLOCK, BLOCK)
    bmax = np.abs(blk).max(axis=2)
    d = ((bmax / f(E2M1_MAX)).astype(f) / sg).astype(f)
    sb = round_e4m3(d)
    S = (e4m3_value(sb).astype(f) * sg).astype(f)
    safe = np.where(S > 0, S, f(1.0)).astype(f)
    y = (blk / safe[:, :, None]).astype(f)
    q = np.where((S > 0)[:, :, None], round_e2m1(y), 0).astype(np.uint8).reshape(rows, cols)
    return pack_codes(q), sb, sg, q


def pack_codes(q: np.ndarray) -> np.ndarray:
    flat = np.asarray(q, dtype=np.uint8).reshape(-1)
    return (flat[0::2] | (flat[1::2] << 4)).astype(np.uint8)


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).reshape(-1)
    out = np.empty(c.size * 2, dtype=np.uint8)
    out[0::2] = c & 0x0F
    out[1::2] = c >> 4
    return out


def scale_bytes(sb: np.ndarray) -> np.ndarray:
    """The stored [cols/64][rows][4] uint8 array from [rows, cols/16] E4M3 block scales."""
    rows, nb = sb.shape
    return np.ascontiguousarray(np.asarray(sb, dtype=np.uint8).reshape(rows, nb // 4, 4).transpose(1, 0, 2))


def unscale_bytes(stored: np.ndarray) -> np.ndarray:
    a = np.asarray(stored, dtype=np.uint8)
    return np.ascontiguousarray(a.transpose(1, 0, 2).reshape(a.shape[1], a.shape[0] * 4))


def dequantize(codes, sb, sg, rows, cols) -> np.ndarray:
    """fp32 weights (rows, cols): w' = fp32(e2m1(code) * fp32(s_b * S_g))."""
    f = np.float32
    v = e2m1_value(unpack_codes(codes)).astype(f).reshape(rows, cols // BLOCK, BLOCK)
    S = (e4m3_value(sb).astype(f) * f(sg)).astype(f)
    return (v * S[:, :, None]).astype(f).reshape(rows, cols)


def dequantize_bf16(codes, sb, sg, rows, cols) -> np.ndarray:
    """The compute-dtype base weight: bf16(dequantize(...)), as fp32 values."""
    from oracle.int4 import bf16_round
    return bf16_round(dequantize(codes, sb, sg, rows, cols))
