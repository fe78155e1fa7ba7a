"""fp32-exact oracle of NF4 quantisation with double-quantised block scales.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"loralei" README, QLoRA section: the frozen base is stored as NF4 with 64-element
blocks whose scales are themselves quantised per 256 blocks ("double-scale
reconstruction"); a weight's element count must be divisible by 64 * 256 and the
linear dimensions by 32.  The pages print neither the NF4 values nor the scale
format; the readings taken here are:

  * codebook: the NormalFloat-4 construction of the QLoRA paper (Dettmers et al.,
    2023, section 3): quantiles of N(0, 1) on an asymmetric grid -- 8 levels for
    the non-negative half (including an exact 0) and 7 for the negative half --
    normalised to [-1, 1].  The outermost grid point is the mean of the two
    quantile-estimator offsets 1/(2*16) and 1/(2*15), i.e. p = 1 - (1/32 + 1/30)/2.
    Values are rounded to fp32 (see ``codebook`` for the exact rounding steps,
    which reproduce the table printed in that paper's appendix bit for bit).
  * block absmax: max |x| over the 64 elements (exact in fp32).
  * double quantisation: per group of 256 blocks, c = fp32(max absmax / 127) and
    q_b = clamp(round_half_even(fp32(absmax_b / c)), 0, 127) stored as int8;
    symmetric, no mean subtraction; q_b = 0 when c == 0.
  * code index: x is normalised by its block's true absmax, v = fp32(x / absmax)
    (0 when absmax == 0), and mapped to the nearest codebook value by exact
    distance; an exact tie goes to the lower index.
  * packing: element 2i in the high nibble of byte i, element 2i+1 in the low one.
  * dequantisation: amax' = fp32(q_b * c), w = fp32(code[idx] * amax'), two
    separately rounded fp32 products.
"""
from __future__ import annotations

from statistics import NormalDist

import numpy as np

BLOCK = 64
GROUP_BLOCKS = 256
GROUP = BLOCK * GROUP_BLOCKS      # 16384 elements share one fp32 scale


def _fp32_grid(start: float, end: float, points: int) -> list:
    """``points`` evenly spaced fp32 values from start to end; the first half is stepped from
    ``start``, the second half back from ``end``, each point rounded to fp32."""
    f = np.float32
    a, b = f(start), f(end)
    step = f((b - a) / f(points - 1))
    half = points // 2
    return [float(f(a + f(i) * step)) if i < half else float(f(b - f(points - 1 - i) * step))
            for i in range(points)]


def codebook() -> np.ndarray:
    """The 16 NF4 values (fp32), ascending.

    The outer probability is 1 - (1/32 + 1/30)/2 = 0.96770833..., used at 7 digits
    (0.9677083) and on an fp32 grid, which is how the published NF4 table was made; the
    quantiles themselves are fp64 (statistics.NormalDist), rounded to fp32 and divided by
    the largest in fp32.
    """
    nd = NormalDist()
    p_hi = 0.9677083
    # 8 non-negative levels: quantiles at 9 grid points from p_hi to 1/2, the last (1/2 -> 0)
    # dropped here and added once below; 7 negative levels from 8 grid points likewise.
    pos = [nd.inv_cdf(p) for p in _fp32_grid(p_hi, 0.5, 9)[:-1]]
    neg = [-nd.inv_cdf(p) for p in _fp32_grid(p_hi, 0.5, 8)[:-1]]
    vals = np.array(sorted(pos + [0.0] + neg), dtype=np.float32)
    return (vals / vals.max()).astype(np.float32)


def _bf16_round(x32: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even), returned as fp32 values."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def quantize(w32: np.ndarray):
    """Quantise a weight (any shape, fp32 values) to NF4.

    Returns (codes uint8 [numel/2], absmax_q int8 [numel/64], scale float32 [numel/16384]).
    """
    x = np.ascontiguousarray(w32, dtype=np.float32).reshape(-1)
    if x.size % GROUP:
        raise ValueError("NF4 needs the element count divisible by 64*256")
    nb = x.size // BLOCK
    blocks = x.reshape(nb, BLOCK)
    absmax = np.max(np.abs(blocks), axis=1).astype(np.float32)            # exact
    groups = absmax.reshape(-1, GROUP_BLOCKS)
    gmax = np.max(groups, axis=1).astype(np.float32)
    scale = (gmax / np.float32(127.0)).astype(np.float32)                  # fp32 RN division
    q = np.zeros_like(groups, dtype=np.int8)
    nz = scale > 0
    ratio = (groups[nz] / scale[nz, None]).astype(np.float32)            # fp32 RN division
    q[nz] = np.clip(np.rint(ratio), 0, 127).astype(np.int8)               # half-even
    absmax_q = q.reshape(-1)

    safe = np.where(absmax > 0, absmax, np.float32(1.0)).astype(np.float32)
    idx = np.empty(x.size, dtype=np.uint8)
    chunk = 1 << 16                                                        # blocks per pass
    for b0 in range(0, nb, chunk):
        b1 = min(nb, b0 + chunk)
        v = (blocks[b0:b1] / safe[b0:b1, None]).astype(np.float32)       # fp32 RN division
        v = np.where(absmax[b0:b1, None] > 0, v, np.float32(0.0))
        idx[b0 * BLOCK:b1 * BLOCK] = nearest_code(v.reshape(-1))
    codes = ((idx[0::2] << 4) | idx[1::2]).astype(np.uint8)
    return codes, absmax_q, scale


def nearest_code(v32: np.ndarray) -> np.ndarray:
    """Index of the nearest codebook value to each fp32 v, an exact tie going to the lower index.

    The codebook is strictly increasing, so v is nearer to code[i+1] than to code[i] exactly
    when v exceeds their midpoint; the midpoints of two fp32 values are exact in fp64, and so is
    the comparison with an fp32 v.  The index is therefore the number of midpoints strictly
    below v (a tie, v equal to a midpoint, is not counted and stays with the lower code)."""
    cb = codebook().astype(np.float64)
    mids = 0.5 * (cb[:-1] + cb[1:])
    return np.searchsorted(mids, np.asarray(v32, dtype=np.float32).astype(np.float64), side="left").astype(np.uint8)


def unpack_indices(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.size * 2, dtype=np.uint8)
    out[0::2] = c >> 4
    out[1::2] = c & 0x0F
    return out


def dequantize(codes, absmax_q, scale) -> np.ndarray:
    """fp32 weights (flat) from NF4 codes, int8 block scales and fp32 group scales."""
    idx = unpack_indices(codes)
    cb = codebook()
    q = np.asarray(absmax_q, dtype=np.int8).astype(np.float32)
    c = np.repeat(np.asarray(scale, dtype=np.float32), GROUP_BLOCKS)
    amax = (q * c).astype(np.float32)                                     # fp32 RN product
    w = (cb[idx].reshape(-1, BLOCK) * amax[:, None]).astype(np.float32)  # fp32 RN product
    return w.reshape(-1)


def dequantize_bf16(codes, absmax_q, scale) -> np.ndarray:
    """The compute-dtype base weight: bf16(dequantize(...)), as fp32 values."""
    return _bf16_round(dequantize(codes, absmax_q, scale))
