"""Parity at the full workload sizes (bf16, NF4, int4 and NVFP4 bases), in the launch configuration the
benchmark times, every element against the fp64 oracle.

Each MLP workload runs the whole oracle forward and backward on all of its tokens (about 6 TFLOP
of fp64 matmul for the Llama-3-8B shapes, 12 for the Llama-3-70B ones: seconds to tens of seconds
on the host's BLAS) and compares y, e, u, h, dX and all six LoRA gradients element by element, so
every 512 x 256 tile of the down and dX GEMMs -- including the split tail tiles that a
finalisation kernel sums -- and every column block of the gradient reductions is covered.  QKV and
O likewise, every output and gradient in full.  The identity <A, dA> = <B, dB> is checked on top.
"""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import lora as O
from oracle import int4 as oi4
from oracle import nf4 as onf4
from oracle import nvfp4 as onv

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu

_cache = {}

MLP_GRADS = (("dA_gate", "dAg"), ("dB_gate", "dBg"), ("dA_up", "dAu"), ("dB_up", "dBu"),
             ("dA_down", "dAd"), ("dB_down", "dBd"))


def _base64(bits, w):
    if w.int4_group:
        x = synth.bf16_bits_to_f32(bits).reshape(bits.shape)
        codes, s, z, _ = oi4.quantize(x, w.int4_group)
        return oi4.dequantize_bf16(codes, s, z, bits.shape[0], bits.shape[1], w.int4_group).astype(np.float64)
    if w.nvfp4:
        x = synth.bf16_bits_to_f32(bits).reshape(bits.shape)
        codes, sb, sg, _ = onv.quantize(x)
        return onv.dequantize_bf16(codes, sb, sg, bits.shape[0], bits.shape[1]).astype(np.float64)
    if not w.nf4:
        return O.from_bf16(bits)
    x = synth.bf16_bits_to_f32(bits).reshape(-1)
    return onf4.dequantize_bf16(*onf4.quantize(x)).astype(np.float64).reshape(bits.shape)


def _inputs(w):
    key = (tuple((p.d_in, p.d_out) for p in w.projs), w.T, w.r, w.nf4, w.int4_group, w.nvfp4)
    if key not in _cache:
        _cache.clear()
        inp = synth.make_inputs(w)
        p = {}
        for t, k in zip([q.name for q in w.projs], ["g", "u", "d"] if w.kind == "mlp" else [q.name for q in w.projs]):
            p["W" + k] = _base64(inp["W_" + t], w)
            p["A" + k] = O.from_bf16(inp["A_" + t])
            p["B" + k] = O.from_bf16(inp["B_" + t])
            p["s" + k] = w.s
        _cache[key] = (inp, p)
    return _cache[key]


def _dev_lora(inp, t, w):
    W = dev_bf16(inp["W_" + t])
    if w.nf4:
        W = L.nf4_pack(W)
    elif w.int4_group:
        W = L.int4_pack(W, w.int4_group)
    elif w.nvfp4:
        W = L.nvfp4_pack(W)
    return L.Lora(W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), w.s)


MLP = ["llama3_8b_mlp_bf16", "llama3_8b_mlp_nf4", "llama3_70b_mlp_nf4_swiglu", "llama3_70b_mlp_nf4_geglu",
       "llama3_8b_mlp_int4", "llama3_8b_mlp_nvfp4"]


@pytest.mark.parametrize("name", MLP)
def test_full_size_mlp(name):
    w = synth.WORKLOADS[name]
    inp, p = _inputs(w)
    gate, up, down = (_dev_lora(inp, t, w) for t in ("gate", "up", "down"))
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, gate, up, down, act=w.act)
    bw = L.lora_mlp_bwd(X, dY, fw, gate, up, down, act=w.act)
    L.lm_workspace_check(fw["ws"])
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, w.act)
    for k in ("e", "u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in MLP_GRADS:
        check(k, host64(bw[k]), ref[rk])
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        a = float(np.sum(p["A" + k] * host64(bw["dA_" + t])))
        b = float(np.sum(p["B" + k] * host64(bw["dB_" + t])))
        assert abs(a - b) <= 1e-2 * max(abs(a), abs(b)), (t, a, b)


@pytest.mark.parametrize("base", ["bf16", "nf4", "int4", "nvfp4"])
def test_full_size_qkv_and_o(base):
    w = synth.WORKLOADS["llama3_8b_qkv_" + base]
    inp, p = _inputs(w)
    Ls = {t: _dev_lora(inp, t, w) for t in ("q", "k", "v")}
    X = dev_bf16(inp["X"])
    dO = {t: dev_bf16(inp["dY_" + t]) for t in ("q", "k", "v")}
    fw = L.lora_qkv_fwd(X, Ls["q"], Ls["k"], Ls["v"])
    bw = L.lora_qkv_bwd(X, dO["q"], dO["k"], dO["v"], fw, Ls["q"], Ls["k"], Ls["v"])
    L.lm_workspace_check(fw["ws"])
    Xo = O.from_bf16(inp["X"])
    dOo = {t: O.from_bf16(inp["dY_" + t]) for t in ("q", "k", "v")}
    rf = O.qkv_forward(Xo, p)
    rb = O.qkv_backward(Xo, dOo["q"], dOo["k"], dOo["v"], p)
    for t in ("Q", "K", "V"):
        check(t, host64(fw[t]), rf[t])
    check("dX", host64(bw["dX"]), rb["dX"])
    for t in ("q", "k", "v"):
        check("dA_" + t, host64(bw["dA_" + t]), rb["dA" + t])
        check("dB_" + t, host64(bw["dB_" + t]), rb["dB" + t])

    wo = synth.WORKLOADS["llama3_8b_o_" + base]
    io, po = _inputs(wo)
    o = _dev_lora(io, "o", wo)
    Xd, dYd = dev_bf16(io["X"]), dev_bf16(io["dY"])
    f = L.lora_o_fwd(Xd, o)
    b = L.lora_o_bwd(Xd, dYd, f, o)
    L.lm_workspace_check(f["ws"])
    Xo, dYo = O.from_bf16(io["X"]), O.from_bf16(io["dY"])
    Wo, Ao, Bo, so = po["Wo"], po["Ao"], po["Bo"], po["so"]
    Y, _ = O.lora_w_forward(Xo, Wo, Ao, Bo, so)
    g = O.lora_w_backward(Xo, dYo, Wo, Ao, Bo, so)
    check("Y", host64(f["Y"]), Y)
    check("dX", host64(b["dX"]), g["dX"])
    check("dA", host64(b["dA"]), g["dA"])
    check("dB", host64(b["dB"]), g["dB"])
