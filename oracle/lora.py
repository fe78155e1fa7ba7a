"""fp64 oracle of the LoRA MLP, LoRA QKV and LoRA W (O) forward and backward.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Notation (PEFT nn.Linear layout; "Avoid recomputing LoRA B-projected gradient",
matmul_lora: out = X W^T plus the LoRA term; LoRA_W backward returns d_A.t(),
d_B.t()): W (out, in), A (r, in), B (out, r), s = alpha / r.  Activations are
(T, features) with T = batch * seq flattened.

Everything is evaluated in float64 from the exact fp64 widening of the bf16
inputs; no intermediate is rounded.  The backward is the chain rule of the
forward written out term by term; the B-projected gradient G = dOut . B is
formed once and used for both dA and dX (the hoist of the unsloth diff).
"""
from __future__ import annotations

import math

import numpy as np

_SQRT2 = math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


def from_bf16(bits: np.ndarray) -> np.ndarray:
    """Exact fp64 value of bf16 bit patterns (uint16)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of fp32 values, round to nearest with ties to even.

    fp32 LoRA parameters ("LoRA Optimizations", FP32 LoRA gradients: the trainable parameters
    stay fp32, the GEMMs take bf16 inputs) enter the computation as these bf16 values.  bf16 is
    the top 16 bits of an fp32; the dropped 16 bits decide the rounding: above half an ulp
    rounds up, below rounds down, exactly half rounds to the even (last kept bit 0) neighbour.
    Finite inputs only (an fp32 that rounds past the largest bf16 becomes infinity).
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    hi, lo = u >> np.uint64(16), u & np.uint64(0xFFFF)
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & np.uint64(1)) == 1))
    return (hi + up.astype(np.uint64)).astype(np.uint16)


# ----------------------------------------------------------------------------------------------
# Gated activations ("LoRA Optimizations", Triton kernels: SwiGLU and GeGLU forward / backward).
# SiLU(x) = x * sigmoid(x); GELU is the exact-erf form 0.5 x (1 + erf(x / sqrt 2)).
# ----------------------------------------------------------------------------------------------

def _erf(x: np.ndarray) -> np.ndarray:
    try:
        from scipy.special import erf
        return erf(x)
    except ImportError:  # pragma: no cover - exercised only where scipy is absent
        return np.vectorize(math.erf, otypes=[np.float64])(x)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    return x * sigmoid(x)


def silu_grad(x):
    sg = sigmoid(x)
    return sg * (1.0 + x * (1.0 - sg))


def normal_cdf(x):
    return 0.5 * (1.0 + _erf(x / _SQRT2))


def normal_pdf(x):
    return _INV_SQRT_2PI * np.exp(-0.5 * x * x)


def gelu_erf(x):
    return x * normal_cdf(x)


def gelu_erf_grad(x):
    return normal_cdf(x) + x * normal_pdf(x)


ACTS = {
    "swiglu": (silu, silu_grad),
    "geglu": (gelu_erf, gelu_erf_grad),
}


# ----------------------------------------------------------------------------------------------
# One LoRA projection (matmul_lora / LoRA_W): Y = X W^T + s (X A^T) B^T.
# ----------------------------------------------------------------------------------------------

def lora_w_forward(X, W, A, B, s):
    """Returns (Y, XA) with XA = X A^T (T, r)."""
    XA = X @ A.T
    Y = X @ W.T + s * (XA @ B.T)
    return Y, XA


def lora_w_backward(X, dY, W, A, B, s):
    """LoRA_W backward. Returns dict(dX, dA (r, in), dB (out, r), G = dY B).

    d/dA <dY, s X A^T B^T> = s G^T X,   d/dB = s dY^T (X A^T),   dX = dY W + s G A.
    """
    G = dY @ B                    # the B-projected gradient, formed once
    XA = X @ A.T
    dA = s * (G.T @ X)
    dB = s * (dY.T @ XA)
    dX = dY @ W + s * (G @ A)
    return {"dX": dX, "dA": dA, "dB": dB, "G": G}


def lora_w_lora_grads(X, dY, A, B, s):
    """dA and dB of lora_w_backward without its base-weight dX GEMM (O(T r (in + out)) work)."""
    G = dY @ B
    return {"dA": s * (G.T @ X), "dB": s * (dY.T @ (X @ A.T))}


# ----------------------------------------------------------------------------------------------
# LoRA MLP ("LoRA Optimizations": LoRA MLP autograd function; unsloth LoRA_MLP):
#   e = X Wg^T + sg (X Ag^T) Bg^T,  u = X Wu^T + su (X Au^T) Bu^T,
#   h = act(e) * u,                  y = h Wd^T + sd (h Ad^T) Bd^T.
# ----------------------------------------------------------------------------------------------

def mlp_forward(X, p, act="swiglu"):
    """p: dict with Wg, Ag, Bg, sg, Wu, Au, Bu, su, Wd, Ad, Bd, sd (fp64 arrays / floats)."""
    f, _ = ACTS[act]
    XAg = X @ p["Ag"].T
    XAu = X @ p["Au"].T
    e = X @ p["Wg"].T + p["sg"] * (XAg @ p["Bg"].T)
    u = X @ p["Wu"].T + p["su"] * (XAu @ p["Bu"].T)
    h = f(e) * u
    hA = h @ p["Ad"].T
    y = h @ p["Wd"].T + p["sd"] * (hA @ p["Bd"].T)
    return {"e": e, "u": u, "h": h, "y": y, "XAg": XAg, "XAu": XAu, "hA": hA}


def mlp_backward(X, dY, p, act="swiglu"):
    """Gradients of L = <dY, y> for X and every A, B.  Frozen W get no gradient.

    Down projection: Gd = dY Bd (hoisted), dh = dY Wd + sd Gd Ad,
                     dAd = sd Gd^T h, dBd = sd dY^T (h Ad^T).
    Activation:      de = dh * u * act'(e),  du = dh * act(e).
    Gate / up:       Gg = de Bg, Gu = du Bu (hoisted),
                     dAg = sg Gg^T X, dBg = sg de^T (X Ag^T)  (same for up),
                     dX = de Wg + du Wu + sg Gg Ag + su Gu Au.
    """
    f, fprime = ACTS[act]
    fw = mlp_forward(X, p, act)
    e, u, h = fw["e"], fw["u"], fw["h"]
    Gd = dY @ p["Bd"]
    dh = dY @ p["Wd"] + p["sd"] * (Gd @ p["Ad"])
    dAd = p["sd"] * (Gd.T @ h)
    dBd = p["sd"] * (dY.T @ fw["hA"])
    de = dh * u * fprime(e)
    du = dh * f(e)
    Gg = de @ p["Bg"]
    Gu = du @ p["Bu"]
    dAg = p["sg"] * (Gg.T @ X)
    dBg = p["sg"] * (de.T @ fw["XAg"])
    dAu = p["su"] * (Gu.T @ X)
    dBu = p["su"] * (du.T @ fw["XAu"])
    dX = de @ p["Wg"] + du @ p["Wu"] + p["sg"] * (Gg @ p["Ag"]) + p["su"] * (Gu @ p["Au"])
    return {"dX": dX, "dAg": dAg, "dBg": dBg, "dAu": dAu, "dBu": dBu, "dAd": dAd, "dBd": dBd,
            "de": de, "du": du, "dh": dh, "Gg": Gg, "Gu": Gu, "Gd": Gd, **fw}


# ----------------------------------------------------------------------------------------------
# Non-gated ReLU^2 MLP ("LoRA Optimizations", FP32 LoRA gradients: dense ReLU^2 MLPs with up/down
# LoRA projections and a fused ReLU^2 activation derivative).  ReLU^2(x) = max(x, 0)^2, its
# derivative 2 max(x, 0).
# ----------------------------------------------------------------------------------------------

def relu2(x):
    return np.square(np.maximum(x, 0.0))


def relu2_grad(x):
    return 2.0 * np.maximum(x, 0.0)


def relu2_mlp_forward(X, p):
    """p: dict with Wu, Au, Bu, su, Wd, Ad, Bd, sd.  u = X Wu^T + su (X Au^T) Bu^T, h = relu(u)^2,
    y = h Wd^T + sd (h Ad^T) Bd^T."""
    XAu = X @ p["Au"].T
    u = X @ p["Wu"].T + p["su"] * (XAu @ p["Bu"].T)
    h = relu2(u)
    hA = h @ p["Ad"].T
    y = h @ p["Wd"].T + p["sd"] * (hA @ p["Bd"].T)
    return {"u": u, "h": h, "y": y, "XAu": XAu, "hA": hA}


def relu2_mlp_backward(X, dY, p):
    """Gradients of L = <dY, y> for X and the four LoRA factors.

    Down: Gd = dY Bd (hoisted), dh = dY Wd + sd Gd Ad, dAd = sd Gd^T h, dBd = sd dY^T (h Ad^T).
    Activation: du = dh * 2 relu(u).
    Up: Gu = du Bu (hoisted), dAu = su Gu^T X, dBu = su du^T (X Au^T), dX = du Wu + su Gu Au.
    """
    fw = relu2_mlp_forward(X, p)
    u, h = fw["u"], fw["h"]
    Gd = dY @ p["Bd"]
    dh = dY @ p["Wd"] + p["sd"] * (Gd @ p["Ad"])
    dAd = p["sd"] * (Gd.T @ h)
    dBd = p["sd"] * (dY.T @ fw["hA"])
    du = dh * relu2_grad(u)
    Gu = du @ p["Bu"]
    dAu = p["su"] * (Gu.T @ X)
    dBu = p["su"] * (du.T @ fw["XAu"])
    dX = du @ p["Wu"] + p["su"] * (Gu @ p["Au"])
    return {"dX": dX, "dAu": dAu, "dBu": dBu, "dAd": dAd, "dBd": dBd, "du": du, "dh": dh, "Gu": Gu,
            "Gd": Gd, **fw}


def relu2_mlp_flops(T, d, n, r):
    """Algorithmic flops of one fwd+bwd of the ReLU^2 MLP: the up and down projections as two
    LoRA projections (base 4 T in out each, fwd + dX) plus the rank-r terms."""
    return lora_proj_flops(T, d, n, r) + lora_proj_flops(T, n, d, r)


def mlp_backward_columns(X, dY, p, cols, act="swiglu"):
    """dB_gate[cols], dB_up[cols] and dA_down[:, cols] of mlp_backward, for a subset of the n
    intermediate features.  Column c of e, u, h, dh, de, du depends only on row c of W_g, W_u, B_g,
    B_u and column c of W_d, A_d (plus the rank-r products X A^T and dY B_d), so these gradient
    entries cost O(T * d) per column instead of the full O(T * d * n) backward."""
    f, fprime = ACTS[act]
    cols = np.asarray(cols)
    XAg = X @ p["Ag"].T
    XAu = X @ p["Au"].T
    Gd = dY @ p["Bd"]
    e = X @ p["Wg"][cols].T + p["sg"] * (XAg @ p["Bg"][cols].T)
    u = X @ p["Wu"][cols].T + p["su"] * (XAu @ p["Bu"][cols].T)
    h = f(e) * u
    dh = dY @ p["Wd"][:, cols] + p["sd"] * (Gd @ p["Ad"][:, cols])
    de = dh * u * fprime(e)
    du = dh * f(e)
    return {"dBg": p["sg"] * (de.T @ XAg), "dBu": p["su"] * (du.T @ XAu), "dAd": p["sd"] * (Gd.T @ h)}


# ----------------------------------------------------------------------------------------------
# LoRA QKV (unsloth LoRA_QKV): three projections of one input X; dX is the sum of the three
# projections' input gradients.  Written out directly (not through lora_w_*), so that the
# equality with three LoRA_W runs is a real check.
# ----------------------------------------------------------------------------------------------

def qkv_forward(X, p):
    """p: dict with Wq, Aq, Bq, sq, Wk, Ak, Bk, sk, Wv, Av, Bv, sv."""
    out = {}
    for t in ("q", "k", "v"):
        XA = X @ p["A" + t].T
        out["XA" + t] = XA
        out[t.upper()] = X @ p["W" + t].T + p["s" + t] * (XA @ p["B" + t].T)
    return out


def qkv_backward(X, dQ, dK, dV, p):
    grads = {"q": dQ, "k": dK, "v": dV}
    res = {}
    dX = np.zeros_like(X)
    for t in ("q", "k", "v"):
        d = grads[t]
        G = d @ p["B" + t]
        XA = X @ p["A" + t].T
        res["dA" + t] = p["s" + t] * (G.T @ X)
        res["dB" + t] = p["s" + t] * (d.T @ XA)
        res["G" + t] = G
        dX += d @ p["W" + t] + p["s" + t] * (G @ p["A" + t])
    res["dX"] = dX
    return res


# ----------------------------------------------------------------------------------------------
# Adapter parameter count ("LoRA Optimizations", FP32 LoRA gradients): A is (r, in), B is
# (out, r), so one adapted projection holds r * (in + out) parameters.
# ----------------------------------------------------------------------------------------------

def adapter_param_count(projs, r, layers=1):
    """projs: iterable of (in_features, out_features)."""
    return layers * sum(r * (i + o) for i, o in projs)


# ----------------------------------------------------------------------------------------------
# Algorithmic flop counts (for the benchmark's TFLOP/s).  Base GEMMs: 2 T in out each for the
# forward and for the input gradient (frozen W have no weight gradient).  Rank-r work per
# projection: forward X A^T and (XA) B^T, backward G = dY B, dA, dB and G A (dX term).
# ----------------------------------------------------------------------------------------------

def lora_proj_flops(T, d_in, d_out, r):
    return 4 * T * d_in * d_out + 2 * T * r * (d_in + d_out) + 2 * T * r * (2 * d_in + 2 * d_out)


def mlp_flops(T, d, n, r):
    return (lora_proj_flops(T, d, n, r) * 2 + lora_proj_flops(T, n, d, r))
