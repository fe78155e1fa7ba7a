"""fp32-exact oracle of groupwise Int4 quantisation of a frozen base weight.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"loralei" README, QLoRA section: the alternative quantised base is int4 with groupwise scales,
group sizes 32, 64, 128 or 256 (the example uses 128), made from the bf16 weight by a tinygemm
style kernel; the input gradient is computed from the packed weight as well.  The pages print
no formula; the readings taken here are:

  * a group is G consecutive elements of one weight row (out feature i, in features
    [g*G, (g+1)*G)); cols must be a multiple of G.
  * asymmetric min/max affine quantisation with the zero point kept as a float in the weight's
    domain (the tinygemm convention): per group, with mn, mx the exact minimum and maximum,
        s = bf16(fp32((mx - mn) / 15))       scale, stored as bf16
        z = bf16(fp32(mn + 8 * s))           value of the middle code 8, stored as bf16
        q = clamp(rint(fp32(fp32(w - z) / s)) + 8, 0, 15)   (rint: half to even)
    and q = 8 for every element when s == 0 (a constant group).  Every step is one IEEE fp32
    operation followed, where stated, by a round-to-nearest-even to bf16.
  * dequantisation: w' = fp32((q - 8) * s + z).  (q - 8) * s is exact in fp32 (a 4-bit integer
    times an 8-bit significand), so this is one rounding of the exact value; the matmul operand
    is bf16(w').
  * storage: codes row-major, element 2i in the high nibble of byte i (as for NF4);
    scale_zero is [cols/G][rows][2] bf16 -- group-major, so the (s, z) pairs of one group of
    all rows are contiguous -- with s at [..][..][0] and z at [..][..][1].
"""
from __future__ import annotations

import numpy as np

GROUPS = (32, 64, 128, 256)


def bf16_round(x32: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even), returned as fp32 values (finite inputs)."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def bf16_bits(x32: np.ndarray) -> np.ndarray:
    """The bf16 bit patterns of fp32 values that are already bf16 values."""
    return (np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def quantize(w32: np.ndarray, group: int):
    """Quantise a (rows, cols) weight given as fp32 values (normally bf16 values).

    Returns (codes uint8 [rows*cols/2], s float32 [rows, cols/G], z float32 [rows, cols/G],
    q uint8 [rows, cols]); s and z hold bf16 values."""
    w = np.asarray(w32, dtype=np.float32)
    if w.ndim != 2 or group not in GROUPS or w.shape[1] % group:
        raise ValueError("int4 needs a 2-D weight whose column count is a multiple of the group")
    rows, cols = w.shape
    f = np.float32
    g = w.reshape(rows, cols // group, group)
    mn = g.min(axis=2)
    mx = g.max(axis=2)
    s = bf16_round(((mx - mn) / f(15.0)).astype(f))
    z = bf16_round((mn + f(8.0) * s).astype(f))
    nz = s > 0
    safe = np.where(nz, s, f(1.0)).astype(f)
    d = (g - z[:, :, None]).astype(f)
    ratio = (d / safe[:, :, None]).astype(f)
    q = np.clip(np.rint(ratio) + 8, 0, 15)
    q = np.where(nz[:, :, None], q, 8).astype(np.uint8).reshape(rows, cols)
    return pack_codes(q), s, z, q


def pack_codes(q: np.ndarray) -> np.ndarray:
    flat = np.asarray(q, dtype=np.uint8).reshape(-1)
    return ((flat[0::2] << 4) | flat[1::2]).astype(np.uint8)


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).reshape(-1)
    out = np.empty(c.size * 2, dtype=np.uint8)
    out[0::2] = c >> 4
    out[1::2] = c & 0x0F
    return out


def scale_zero_bits(s: np.ndarray, z: np.ndarray) -> np.ndarray:
    """The stored [cols/G][rows][2] uint16 array (bf16 bits of s, z) from [rows, cols/G] s, z."""
    out = np.empty((s.shape[1], s.shape[0], 2), dtype=np.uint16)
    out[:, :, 0] = bf16_bits(s).T
    out[:, :, 1] = bf16_bits(z).T
    return out


def split_scale_zero(sz_bits: np.ndarray):
    """[rows, cols/G] fp32 s and z from the stored [cols/G][rows][2] uint16 array."""
    a = np.asarray(sz_bits, dtype=np.uint16)
    s = (a[:, :, 0].astype(np.uint32) << 16).view(np.float32).T
    z = (a[:, :, 1].astype(np.uint32) << 16).view(np.float32).T
    return np.ascontiguousarray(s), np.ascontiguousarray(z)


def dequantize(codes: np.ndarray, s: np.ndarray, z: np.ndarray, rows: int, cols: int, group: int) -> np.ndarray:
    """fp32 weights (rows, cols): w' = fp32((q - 8) * s + z) per element of each group."""
    f = np.float32
    q = unpack_codes(codes).reshape(rows, cols // group, group).astype(f) - f(8.0)
    prod = (q * s[:, :, None]).astype(f)                     # exact
    return (prod + z[:, :, None]).astype(f).reshape(rows, cols)


def dequantize_bf16(codes, s, z, rows, cols, group) -> np.ndarray:
    """The compute-dtype base weight: bf16(dequantize(...)), as fp32 values."""
    return bf16_round(dequantize(codes, s, z, rows, cols, group))
