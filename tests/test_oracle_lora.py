"""Pins for the fp64 LoRA oracle (CPU only).

Each check ties the oracle to something other than its own formulas: central finite
differences of L = <dY, y>, the merge identity W' = W + s B A (loralei README: merge_lora
folds the adapter into the base), closed forms at B = 0, s = 0 and A = 0, the identity
<A, dA> = <B, dB>, known values of the activations, the composition of LoRA_QKV from three
LoRA_W runs, and the adapter parameter count printed on the "LoRA Optimizations" page.
"""
import json
import math
import os
from statistics import NormalDist

import numpy as np
import pytest

from bwd_lora_mlp_gb300 import synth
from oracle import lora as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _mlp_params(inp, s):
    p = {}
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        p["W" + k] = O.from_bf16(inp["W_" + t])
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = s
    return p


def _small_mlp(T=48, d=32, n=80, r=8, alpha=16.0, act="swiglu", **kw):
    w = synth.mlp_workload("t", T, d, n, r, alpha, act=act)
    inp = synth.make_inputs(w, seed=99, **kw)
    p = _mlp_params(inp, w.s)
    X = O.from_bf16(inp["X"])
    dY = O.from_bf16(inp["dY"])
    return X, dY, p


def _loss(X, dY, p, act):
    return float(np.sum(dY * O.mlp_forward(X, p, act)["y"]))


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_mlp_backward_matches_finite_differences(act):
    X, dY, p = _small_mlp(act=act)
    # Make dY O(1) so the loss is not dominated by rounding.
    dY = dY * 100.0
    g = O.mlp_backward(X, dY, p, act)
    rng = np.random.default_rng(7)
    targets = [("X", None)] + [(k, "d" + k) for k in ("Ag", "Bg", "Au", "Bu", "Ad", "Bd")]
    for name, gname in targets:
        base = X if name == "X" else p[name]
        V = rng.standard_normal(base.shape)
        h = 1e-6 * max(1.0, float(np.sqrt(np.mean(base ** 2))))
        if name == "X":
            lp = _loss(X + h * V, dY, p, act)
            lm = _loss(X - h * V, dY, p, act)
            an = float(np.sum(g["dX"] * V))
        else:
            pp = dict(p); pp[name] = base + h * V
            pm = dict(p); pm[name] = base - h * V
            lp, lm = _loss(X, dY, pp, act), _loss(X, dY, pm, act)
            an = float(np.sum(g[gname] * V))
        fd = (lp - lm) / (2 * h)
        assert abs(fd - an) <= 1e-6 * max(abs(an), 1e-3), (name, fd, an)


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_merge_identity(act):
    """Factored LoRA equals the unfused computation on W + s B A (forward and dX)."""
    X, dY, p = _small_mlp(act=act)
    merged = dict(p)
    for k in ("g", "u", "d"):
        merged["W" + k] = p["W" + k] + p["s" + k] * (p["B" + k] @ p["A" + k])
        merged["A" + k] = np.zeros_like(p["A" + k])
        merged["B" + k] = np.zeros_like(p["B" + k])
    f1 = O.mlp_forward(X, p, act)
    f2 = O.mlp_forward(X, merged, act)
    for key in ("e", "u", "h", "y"):
        np.testing.assert_allclose(f1[key], f2[key], rtol=1e-12, atol=1e-13 * np.abs(f2[key]).max())
    b1 = O.mlp_backward(X, dY, p, act)
    b2 = O.mlp_backward(X, dY, merged, act)
    np.testing.assert_allclose(b1["dX"], b2["dX"], rtol=1e-11, atol=1e-12 * np.abs(b2["dX"]).max())


def _base_mlp(X, p, act):
    f, _ = O.ACTS[act]
    return (f(X @ p["Wg"].T) * (X @ p["Wu"].T)) @ p["Wd"].T


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_B_zero_closed_form(act):
    X, dY, p = _small_mlp(act=act, zero_B=True)
    fw = O.mlp_forward(X, p, act)
    np.testing.assert_allclose(fw["y"], _base_mlp(X, p, act), rtol=1e-13, atol=1e-15)
    g = O.mlp_backward(X, dY, p, act)
    for k in ("dAg", "dAu", "dAd"):
        assert np.all(g[k] == 0.0)
    # dB = s * (output gradient)^T (input A^T): nonzero in general
    assert np.abs(g["dBg"]).max() > 0


def test_s_zero_and_A_zero():
    X, dY, p = _small_mlp()
    p0 = dict(p); p0.update(sg=0.0, su=0.0, sd=0.0)
    g = O.mlp_backward(X, dY, p0)
    for k in ("dAg", "dBg", "dAu", "dBu", "dAd", "dBd"):
        assert np.all(g[k] == 0.0)
    np.testing.assert_allclose(g["y"], _base_mlp(X, p, "swiglu"), rtol=1e-13, atol=1e-15)
    X, dY, pA = _small_mlp(zero_A=True)
    g = O.mlp_backward(X, dY, pA)
    for k in ("dBg", "dBu", "dBd"):
        assert np.all(g[k] == 0.0)


def test_A_dA_equals_B_dB():
    X, dY, p = _small_mlp(act="geglu")
    g = O.mlp_backward(X, dY, p, "geglu")
    for k in ("g", "u", "d"):
        a = float(np.sum(p["A" + k] * g["dA" + k]))
        b = float(np.sum(p["B" + k] * g["dB" + k]))
        assert abs(a - b) <= 1e-12 * max(abs(a), abs(b)), (k, a, b)


def test_activation_values_and_derivatives():
    nd = NormalDist()
    xs = np.array([-3.0, -1.0, -0.25, 0.0, 0.5, 1.0, 2.5])
    np.testing.assert_allclose(O.gelu_erf(xs), [x * nd.cdf(x) for x in xs], rtol=1e-14, atol=1e-16)
    np.testing.assert_allclose(O.silu(xs), [x / (1 + math.exp(-x)) for x in xs], rtol=1e-15)
    assert O.gelu_erf(np.array(0.0)) == 0.0
    assert O.gelu_erf_grad(np.array(0.0)) == 0.5
    assert O.silu_grad(np.array(0.0)) == 0.5
    assert abs(O.silu(np.array(1.0)) - 0.7310585786300049) < 1e-15
    h = 1e-6
    for f, fp in (O.ACTS["swiglu"], O.ACTS["geglu"]):
        fd = (f(xs + h) - f(xs - h)) / (2 * h)
        np.testing.assert_allclose(fp(xs), fd, rtol=1e-8, atol=1e-9)


def _small_qkv(v=None):
    w = synth.qkv_workload("t", 40, 64, 64, 32, 8, 16.0, v=v)
    inp = synth.make_inputs(w, seed=5)
    p = {}
    for t in ("q", "k", "v"):
        p["W" + t] = O.from_bf16(inp["W_" + t])
        p["A" + t] = O.from_bf16(inp["A_" + t])
        p["B" + t] = O.from_bf16(inp["B_" + t])
        p["s" + t] = w.s
    dys = [O.from_bf16(inp["dY_" + t]) * 100 for t in ("q", "k", "v")]
    return O.from_bf16(inp["X"]), dys, p


@pytest.mark.parametrize("v", [None, 96])   # V as wide as K, or wider
def test_qkv_is_three_lora_w_with_summed_dX(v):
    X, (dQ, dK, dV), p = _small_qkv(v)
    assert dV.shape[1] == (32 if v is None else v)
    fw = O.qkv_forward(X, p)
    bw = O.qkv_backward(X, dQ, dK, dV, p)
    dX = np.zeros_like(X)
    for t, d in zip(("q", "k", "v"), (dQ, dK, dV)):
        Y, _ = O.lora_w_forward(X, p["W" + t], p["A" + t], p["B" + t], p["s" + t])
        np.testing.assert_allclose(fw[t.upper()], Y, rtol=1e-14, atol=1e-15)
        g = O.lora_w_backward(X, d, p["W" + t], p["A" + t], p["B" + t], p["s" + t])
        np.testing.assert_allclose(bw["dA" + t], g["dA"], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(bw["dB" + t], g["dB"], rtol=1e-13, atol=1e-15)
        dX += g["dX"]
    np.testing.assert_allclose(bw["dX"], dX, rtol=1e-13, atol=1e-14)


def test_lora_w_matches_finite_differences():
    X, (dY, _, _), p = _small_qkv()
    W, A, B, s = p["Wq"], p["Aq"], p["Bq"], p["sq"]
    g = O.lora_w_backward(X, dY, W, A, B, s)

    def L(X_, A_, B_):
        return float(np.sum(dY * O.lora_w_forward(X_, W, A_, B_, s)[0]))

    rng = np.random.default_rng(3)
    for name in ("X", "A", "B"):
        V = rng.standard_normal({"X": X, "A": A, "B": B}[name].shape)
        h = 1e-6
        args_p = [X, A, B]
        args_m = [X, A, B]
        i = ("X", "A", "B").index(name)
        args_p = list(args_p); args_m = list(args_m)
        args_p[i] = args_p[i] + h * V
        args_m[i] = args_m[i] - h * V
        fd = (L(*args_p) - L(*args_m)) / (2 * h)
        an = float(np.sum(g["d" + name] * V))
        assert abs(fd - an) <= 1e-6 * max(abs(an), 1e-3), (name, fd, an)


def test_adapter_param_count_matches_page():
    with open(os.path.join(GOLDEN, "qwen3_8b_adapter_params.json")) as f:
        gold = json.load(f)
    projs = [tuple(v) for v in gold["projections_in_out"].values()]
    n = O.adapter_param_count(projs, gold["rank"], gold["layers"])
    assert n == gold["adapter_params"]
    # two extra bytes per parameter for the weight and two for the gradient
    # "about 167 MiB": 43,646,976 * 4 B = 166.5 MiB
    assert abs(n * 4 / 2 ** 20 - gold["extra_mib_rounded"]) <= 0.5


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_column_sampled_gradients_equal_full_backward(act):
    X, dY, p = _small_mlp(act=act)
    full = O.mlp_backward(X, dY, p, act)
    cols = [0, 3, 17, 79]
    part = O.mlp_backward_columns(X, dY, p, cols, act)
    np.testing.assert_allclose(part["dBg"], full["dBg"][cols], rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(part["dBu"], full["dBu"][cols], rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(part["dAd"], full["dAd"][:, cols], rtol=1e-12, atol=1e-16)


def test_lora_grads_without_dX_equal_full_backward():
    X, (dY, _, _), p = _small_qkv()
    full = O.lora_w_backward(X, dY, p["Wq"], p["Aq"], p["Bq"], p["sq"])
    part = O.lora_w_lora_grads(X, dY, p["Aq"], p["Bq"], p["sq"])
    np.testing.assert_allclose(part["dA"], full["dA"], rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(part["dB"], full["dB"], rtol=1e-13, atol=1e-16)


def test_to_bf16_bits_rounds_to_nearest_even():
    """fp32 -> bf16 of fp32 LoRA parameters ("LoRA Optimizations", FP32 LoRA gradients: bf16 GEMM
    inputs): values fixed by the bf16 format, then brute force against the nearest neighbour."""
    f = lambda v: np.array(v, dtype=np.float32)
    # representable values are unchanged
    exact = np.array([0x3F80, 0xC020, 0x0000, 0x7F7F, 0x0001, 0x8001], dtype=np.uint16)
    back = (exact.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(O.to_bf16_bits(back), exact)
    # 1 + 2^-8 lies halfway between 1 (0x3F80, even) and 1 + 2^-7 (0x3F81): ties go to even
    assert O.to_bf16_bits(f([1 + 2.0 ** -8]))[0] == 0x3F80
    assert O.to_bf16_bits(f([-(1 + 2.0 ** -8)]))[0] == 0xBF80
    # 1 + 3 * 2^-8 lies halfway between 0x3F81 (odd) and 0x3F82 (even)
    assert O.to_bf16_bits(f([1 + 3 * 2.0 ** -8]))[0] == 0x3F82
    assert O.to_bf16_bits(f([-(1 + 3 * 2.0 ** -8)]))[0] == 0xBF82
    # just above / below half an ulp
    assert O.to_bf16_bits(f([1 + 2.0 ** -8 + 2.0 ** -20]))[0] == 0x3F81
    assert O.to_bf16_bits(f([1 + 2.0 ** -8 - 2.0 ** -20]))[0] == 0x3F80
    # the largest finite fp32 is above the largest bf16 by more than half an ulp: infinity
    assert O.to_bf16_bits(f([np.finfo(np.float32).max]))[0] == 0x7F80
    # brute force: the nearer of the two bf16 neighbours (fp64 distances), ties to the even one
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000))).astype(np.float32)
    down = (x.view(np.uint32) >> 16).astype(np.uint16)
    up = (down.astype(np.uint32) + 1).astype(np.uint16)
    vd, vu, vx = O.from_bf16(down), O.from_bf16(up), x.astype(np.float64)
    dd, du = np.abs(vx - vd), np.abs(vu - vx)
    want = np.where(dd < du, down, np.where(du < dd, up, np.where(down % 2 == 0, down, up)))
    assert np.array_equal(O.to_bf16_bits(x), want)
