"""Pins of the fp64 oracle of the non-gated ReLU^2 MLP ("LoRA Optimizations", FP32 LoRA
gradients: dense ReLU^2 MLPs with up/down LoRA projections and a fused ReLU^2 derivative).

ReLU^2(x) = max(x, 0)^2 with derivative 2 max(x, 0): fixed values, then the backward against
central finite differences of the forward, and the B = 0 closed form."""
import numpy as np

from bwd_lora_mlp_gb300 import synth
from oracle import lora as O


def test_relu2_values_and_derivative():
    x = np.array([3.0, -2.0, 0.0, 0.5, -1e-300, 7.25])
    assert np.array_equal(O.relu2(x), np.array([9.0, 0.0, 0.0, 0.25, 0.0, 52.5625]))
    assert np.array_equal(O.relu2_grad(x), np.array([6.0, 0.0, 0.0, 1.0, 0.0, 14.5]))


def _params(inp, s):
    p = {}
    for t, k in (("up", "u"), ("down", "d")):
        p["W" + k] = O.from_bf16(inp["W_" + t])
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = s
    return p


def _small(T=48, d=32, n=80, r=8, alpha=16.0, **kw):
    w = synth.relu2_workload("t", T, d, n, r, alpha)
    inp = synth.make_inputs(w, seed=77, **kw)
    return O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), _params(inp, w.s)


def _loss(X, dY, p):
    return float(np.sum(dY * O.relu2_mlp_forward(X, p)["y"]))


def test_relu2_backward_matches_finite_differences():
    X, dY, p = _small()
    dY = dY * 100.0
    g = O.relu2_mlp_backward(X, dY, p)
    assert (g["u"] > 0).any() and (g["u"] < 0).any()  # both branches of the activation occur
    rng = np.random.default_rng(11)
    for name, gname in [("X", "dX")] + [(k, "d" + k) for k in ("Au", "Bu", "Ad", "Bd")]:
        base = X if name == "X" else p[name]
        V = rng.standard_normal(base.shape)
        h = 1e-6 * max(1.0, float(np.sqrt(np.mean(base ** 2))))
        if name == "X":
            lp, lm = _loss(X + h * V, dY, p), _loss(X - h * V, dY, p)
        else:
            pp = dict(p); pp[name] = base + h * V
            pm = dict(p); pm[name] = base - h * V
            lp, lm = _loss(X, dY, pp), _loss(X, dY, pm)
        fd = (lp - lm) / (2 * h)
        an = float(np.sum(g[gname] * V))
        assert abs(fd - an) <= 1e-6 * max(abs(an), 1e-3), (name, fd, an)


def test_relu2_B_zero_closed_form():
    X, dY, p = _small(zero_B=True)
    # with B = 0 the adapters vanish from the forward: y = max(X Wu^T, 0)^2 Wd^T
    u = X @ p["Wu"].T
    y = np.square(np.maximum(u, 0.0)) @ p["Wd"].T
    fw = O.relu2_mlp_forward(X, p)
    np.testing.assert_allclose(fw["y"], y, rtol=1e-13, atol=1e-15)
    g = O.relu2_mlp_backward(X, dY, p)
    assert np.all(g["dAu"] == 0.0) and np.all(g["dAd"] == 0.0)
    assert np.abs(g["dBu"]).max() > 0 and np.abs(g["dBd"]).max() > 0
