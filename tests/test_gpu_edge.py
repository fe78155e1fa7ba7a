"""Edge cases of the fused paths against the fp64 oracle, through the C ABI:

* a different LoRA scale s for every projection (a swapped or shared scale shows at once),
* a single token for every entry point and base,
* the Llama-3-8B feature sizes with a ragged token count (partial 512-row tiles, split tail
  tiles and a long K in one launch), every output against the oracle in full,
* a token count of 50 row tiles with small features, every output against the oracle in full."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import lora as O
from oracle import nf4 as onf4

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu


def _base(bits, base):
    if base == "bf16":
        return O.from_bf16(bits)
    x = synth.bf16_bits_to_f32(bits).reshape(-1)
    return onf4.dequantize_bf16(*onf4.quantize(x)).astype(np.float64).reshape(bits.shape)


def _dev(inp, t, s, base):
    W = dev_bf16(inp["W_" + t])
    return L.Lora(L.nf4_pack(W) if base == "nf4" else W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), s)


def _mlp(inp, scales, base, act):
    Ls = {t: _dev(inp, t, scales[t], base) for t in ("gate", "up", "down")}
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, Ls["gate"], Ls["up"], Ls["down"], act=act)
    bw = L.lora_mlp_bwd(X, dY, fw, Ls["gate"], Ls["up"], Ls["down"], act=act)
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        p["W" + k] = _base(inp["W_" + t], base)
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = scales[t]
    return fw, bw, p


MLP_GRADS = (("dA_gate", "dAg"), ("dB_gate", "dBg"), ("dA_up", "dAu"), ("dB_up", "dBu"),
             ("dA_down", "dAd"), ("dB_down", "dBd"))


@pytest.mark.parametrize("base", ["bf16", "nf4"])
@pytest.mark.parametrize("T", [1, 333])
def test_mlp_distinct_scales(base, T):
    w = synth.mlp_workload("sc", T, 256, 512, 16, 32.0, act="geglu")
    inp = synth.make_inputs(w, seed=61)
    scales = {"gate": 0.5, "up": 3.0, "down": -1.25}
    fw, bw, p = _mlp(inp, scales, base, "geglu")
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, "geglu")
    for k in ("e", "u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in MLP_GRADS:
        check(k, host64(bw[k]), ref[rk])


@pytest.mark.parametrize("base", ["bf16", "nf4"])
@pytest.mark.parametrize("T", [1, 77])
def test_qkv_distinct_scales(base, T):
    w = synth.qkv_workload("qsc", T, 512, 512, 256, 16, 32.0)
    inp = synth.make_inputs(w, seed=67)
    scales = {"q": 0.25, "k": 2.0, "v": -3.0}
    Ls = {t: _dev(inp, t, scales[t], base) for t in ("q", "k", "v")}
    X = dev_bf16(inp["X"])
    dO = {t: dev_bf16(inp["dY_" + t]) for t in ("q", "k", "v")}
    fw = L.lora_qkv_fwd(X, Ls["q"], Ls["k"], Ls["v"])
    bw = L.lora_qkv_bwd(X, dO["q"], dO["k"], dO["v"], fw, Ls["q"], Ls["k"], Ls["v"])
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t in ("q", "k", "v"):
        p["W" + t] = _base(inp["W_" + t], base)
        p["A" + t] = O.from_bf16(inp["A_" + t])
        p["B" + t] = O.from_bf16(inp["B_" + t])
        p["s" + t] = scales[t]
    Xo = O.from_bf16(inp["X"])
    rf = O.qkv_forward(Xo, p)
    rb = O.qkv_backward(Xo, O.from_bf16(inp["dY_q"]), O.from_bf16(inp["dY_k"]), O.from_bf16(inp["dY_v"]), p)
    for t in ("Q", "K", "V"):
        check(t, host64(fw[t]), rf[t])
    check("dX", host64(bw["dX"]), rb["dX"])
    for t in ("q", "k", "v"):
        check("dA_" + t, host64(bw["dA_" + t]), rb["dA" + t])
        check("dB_" + t, host64(bw["dB_" + t]), rb["dB" + t])


@pytest.mark.parametrize("base", ["bf16", "nf4"])
def test_single_token_o_and_relu2(base):
    wo = synth.o_workload("o1", 1, 512, 256, 16, 32.0)
    io = synth.make_inputs(wo, seed=71)
    o = _dev(io, "o", wo.s, base)
    X, dY = dev_bf16(io["X"]), dev_bf16(io["dY"])
    f = L.lora_o_fwd(X, o)
    b = L.lora_o_bwd(X, dY, f, o)
    L.lm_workspace_check(f["ws"])
    Wo, Ao, Bo = _base(io["W_o"], base), O.from_bf16(io["A_o"]), O.from_bf16(io["B_o"])
    Xo, dYo = O.from_bf16(io["X"]), O.from_bf16(io["dY"])
    Y, _ = O.lora_w_forward(Xo, Wo, Ao, Bo, wo.s)
    g = O.lora_w_backward(Xo, dYo, Wo, Ao, Bo, wo.s)
    check("Y", host64(f["Y"]), Y)
    check("dX", host64(b["dX"]), g["dX"])
    check("dA", host64(b["dA"]), g["dA"])
    check("dB", host64(b["dB"]), g["dB"])

    w = synth.relu2_workload("r1", 1, 256, 512, 16, 32.0)
    inp = synth.make_inputs(w, seed=73)
    up, down = _dev(inp, "up", w.s, base), _dev(inp, "down", w.s, base)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_relu2_mlp_fwd(X, up, down)
    bw = L.lora_relu2_mlp_bwd(X, dY, fw, up, down)
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t, k in (("up", "u"), ("down", "d")):
        p["W" + k] = _base(inp["W_" + t], base)
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = w.s
    ref = O.relu2_mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p)
    for k in ("u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_up", "dAu"), ("dB_up", "dBu"), ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])


@pytest.mark.parametrize("base", ["bf16", "nf4"])
def test_8b_features_ragged_tokens(base):
    """The Llama-3-8B feature sizes with T = 2500 (a partial last 512-row tile and split tail tiles):
    every output and gradient against the full oracle."""
    T, d, n = 2500, 4096, 14336
    w = synth.mlp_workload("ragged8b", T, d, n, 16, 32.0)
    inp = synth.make_inputs(w, seed=79)
    scales = {"gate": w.s, "up": w.s, "down": w.s}
    fw, bw, p = _mlp(inp, scales, base, "swiglu")
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, "swiglu")
    for k in ("e", "u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in MLP_GRADS:
        check(k, host64(bw[k]), ref[rk])


@pytest.mark.parametrize("base", ["bf16", "nf4"])
def test_fifty_row_tiles_checked_in_full(base):
    """T = 50 x 128 - 37 tokens (many split-K units per rank-r projection, a ragged last tile) with
    feature sizes small enough for the oracle to check every output and gradient in full."""
    T = 50 * 128 - 37
    w = synth.mlp_workload("rows50", T, 256, 384, 16, 32.0, act="swiglu")
    inp = synth.make_inputs(w, seed=83)
    scales = {"gate": 0.75, "up": 2.5, "down": 1.5}
    fw, bw, p = _mlp(inp, scales, base, "swiglu")
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, "swiglu")
    for k in ("e", "u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in MLP_GRADS:
        check(k, host64(bw[k]), ref[rk])

    wq = synth.qkv_workload("rows50q", T, 256, 256, 128, 16, 32.0)
    iq = synth.make_inputs(wq, seed=89)
    Ls = {t: _dev(iq, t, wq.s, base) for t in ("q", "k", "v")}
    X = dev_bf16(iq["X"])
    dO = {t: dev_bf16(iq["dY_" + t]) for t in ("q", "k", "v")}
    fq = L.lora_qkv_fwd(X, Ls["q"], Ls["k"], Ls["v"])
    bq = L.lora_qkv_bwd(X, dO["q"], dO["k"], dO["v"], fq, Ls["q"], Ls["k"], Ls["v"])
    L.lm_workspace_check(fq["ws"])
    pq = {}
    for t in ("q", "k", "v"):
        pq["W" + t] = _base(iq["W_" + t], base)
        pq["A" + t] = O.from_bf16(iq["A_" + t])
        pq["B" + t] = O.from_bf16(iq["B_" + t])
        pq["s" + t] = wq.s
    Xo = O.from_bf16(iq["X"])
    rf = O.qkv_forward(Xo, pq)
    rb = O.qkv_backward(Xo, O.from_bf16(iq["dY_q"]), O.from_bf16(iq["dY_k"]), O.from_bf16(iq["dY_v"]), pq)
    for t in ("Q", "K", "V"):
        check(t, host64(fq[t]), rf[t])
    check("dX", host64(bq["dX"]), rb["dX"])
    for t in ("q", "k", "v"):
        check("dA_" + t, host64(bq["dA_" + t]), rb["dA" + t])
        check("dB_" + t, host64(bq["dB_" + t]), rb["dB" + t])
