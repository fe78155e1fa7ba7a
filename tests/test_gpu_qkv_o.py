"""GPU parity of lora_qkv_fwd/bwd and lora_o_fwd/bwd against the fp64 oracle (C ABI)."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import lora as O
from oracle import nf4 as onf4

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu


def _qkv(T, d, nq, nkv, r, alpha, seed, **kw):
    w = synth.qkv_workload("qkv", T, d, nq, nkv, r, alpha)
    inp = synth.make_inputs(w, seed=seed, **kw)
    Ls = {t: L.Lora(dev_bf16(inp["W_" + t]), dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), w.s)
          for t in ("q", "k", "v")}
    X = dev_bf16(inp["X"])
    fw = L.lora_qkv_fwd(X, Ls["q"], Ls["k"], Ls["v"])
    bw = L.lora_qkv_bwd(X, dev_bf16(inp["dY_q"]), dev_bf16(inp["dY_k"]), dev_bf16(inp["dY_v"]), fw,
                        Ls["q"], Ls["k"], Ls["v"])
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t in ("q", "k", "v"):
        p["W" + t] = O.from_bf16(inp["W_" + t])
        p["A" + t] = O.from_bf16(inp["A_" + t])
        p["B" + t] = O.from_bf16(inp["B_" + t])
        p["s" + t] = w.s
    Xo = O.from_bf16(inp["X"])
    rf = O.qkv_forward(Xo, p)
    rb = O.qkv_backward(Xo, O.from_bf16(inp["dY_q"]), O.from_bf16(inp["dY_k"]), O.from_bf16(inp["dY_v"]), p)
    return fw, bw, rf, rb


@pytest.mark.parametrize("T,d,nq,nkv,r", [(300, 256, 256, 64, 16), (512, 512, 512, 128, 8), (130, 128, 128, 32, 64),
                                            (200, 256, 256, 128, 32)])
def test_qkv_matches_oracle(T, d, nq, nkv, r):
    fw, bw, rf, rb = _qkv(T, d, nq, nkv, r, 2.0 * r, seed=31)
    for t in ("Q", "K", "V"):
        check(t, host64(fw[t]), rf[t])
    check("dX", host64(bw["dX"]), rb["dX"])
    for t in ("q", "k", "v"):
        check("dA_" + t, host64(bw["dA_" + t]), rb["dA" + t])
        check("dB_" + t, host64(bw["dB_" + t]), rb["dB" + t])


def test_qkv_lora_alone_with_zero_base():
    fw, bw, rf, rb = _qkv(256, 256, 256, 64, 16, 32.0, seed=9, zero_W=True)
    for t in ("Q", "K", "V"):
        check(t, host64(fw[t]), rf[t])
    check("dX", host64(bw["dX"]), rb["dX"])


@pytest.mark.parametrize("T,din,dout,r,zero_W", [(300, 256, 192, 16, False), (257, 512, 512, 64, False),
                                                   (200, 256, 256, 8, True)])
def test_o_matches_oracle(T, din, dout, r, zero_W):
    w = synth.o_workload("o", T, din, dout, r, 2.0 * r)
    inp = synth.make_inputs(w, seed=17, zero_W=zero_W)
    o = L.Lora(dev_bf16(inp["W_o"]), dev_bf16(inp["A_o"]), dev_bf16(inp["B_o"]), w.s)
    X = dev_bf16(inp["X"])
    fw = L.lora_o_fwd(X, o)
    bw = L.lora_o_bwd(X, dev_bf16(inp["dY"]), fw, o)
    L.lm_workspace_check(fw["ws"])
    Xo, dYo = O.from_bf16(inp["X"]), O.from_bf16(inp["dY"])
    W, A, B = (O.from_bf16(inp[k]) for k in ("W_o", "A_o", "B_o"))
    Y, _ = O.lora_w_forward(Xo, W, A, B, w.s)
    g = O.lora_w_backward(Xo, dYo, W, A, B, w.s)
    check("Y", host64(fw["Y"]), Y)
    check("dX", host64(bw["dX"]), g["dX"])
    check("dA", host64(bw["dA"]), g["dA"])
    check("dB", host64(bw["dB"]), g["dB"])


def _pack(bits, base):
    W = dev_bf16(bits)
    return L.nf4_pack(W) if base == "nf4" else W


def _base64(bits, base):
    if base == "bf16":
        return O.from_bf16(bits)
    x = synth.bf16_bits_to_f32(bits).reshape(-1)
    return onf4.dequantize_bf16(*onf4.quantize(x)).astype(np.float64).reshape(bits.shape)


@pytest.mark.parametrize("base", ["bf16", "nf4"])
@pytest.mark.parametrize("T,d,nq,nk,nv,r", [(300, 256, 256, 64, 192, 16), (200, 512, 256, 128, 32, 64),
                                            (517, 512, 512, 128, 256, 16)])
def test_qkv_k_and_v_of_different_widths(base, T, d, nq, nk, nv, r):
    """K and V of different widths (the ABI takes nq, nk and nv separately): a swapped width or a
    plan that indexes V by K's width shows at once."""
    w = synth.qkv_workload("qkvw", T, d, nq, nk, r, 2.0 * r, v=nv)
    inp = synth.make_inputs(w, seed=37)
    Ls = {t: L.Lora(_pack(inp["W_" + t], base), dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), w.s)
          for t in ("q", "k", "v")}
    X = dev_bf16(inp["X"])
    fw = L.lora_qkv_fwd(X, Ls["q"], Ls["k"], Ls["v"])
    bw = L.lora_qkv_bwd(X, dev_bf16(inp["dY_q"]), dev_bf16(inp["dY_k"]), dev_bf16(inp["dY_v"]), fw,
                        Ls["q"], Ls["k"], Ls["v"])
    L.lm_workspace_check(fw["ws"])
    assert tuple(fw["K"].shape) == (T, nk) and tuple(fw["V"].shape) == (T, nv)
    p = {}
    for t in ("q", "k", "v"):
        p["W" + t] = _base64(inp["W_" + t], base)
        p["A" + t] = O.from_bf16(inp["A_" + t])
        p["B" + t] = O.from_bf16(inp["B_" + t])
        p["s" + t] = w.s
    Xo = O.from_bf16(inp["X"])
    rf = O.qkv_forward(Xo, p)
    rb = O.qkv_backward(Xo, O.from_bf16(inp["dY_q"]), O.from_bf16(inp["dY_k"]), O.from_bf16(inp["dY_v"]), p)
    for t in ("Q", "K", "V"):
        check(t, host64(fw[t]), rf[t])
    check("dX", host64(bw["dX"]), rb["dX"])
    for t in ("q", "k", "v"):
        check("dA_" + t, host64(bw["dA_" + t]), rb["dA" + t])
        check("dB_" + t, host64(bw["dB_" + t]), rb["dB" + t])
