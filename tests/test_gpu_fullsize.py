"""Parity at the full workload sizes (bf16, NF4, int4 and NVFP4 bases), in the launch configuration the
benchmark times.

The oracle cannot run a full-size backward in seconds, so it is checked where it can be
computed exactly and cheaply:
  * forward outputs and dX at sampled token rows (every one of them depends only on its own row
    of X and dY),
  * dB_gate, dB_up and dA_down at sampled intermediate features (column c needs only O(T d)
    work, oracle.lora.mlp_backward_columns),
  * dA_gate, dA_up and dB_down through the identity <A, dA> = <B, dB>, which holds at any size
    and ties them to the directly checked gradients,
  * for QKV and O every gradient in full (no activation: dA = s G^T X, dB = s dOut^T (X A^T)
    cost O(T r (in + out))).
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


def _rows(T, k=24, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, k)]))


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
    T, n = w.T, w.projs[0].d_out
    R = _rows(T)
    Xo, dYo = O.from_bf16(inp["X"]), O.from_bf16(inp["dY"])
    ref = O.mlp_backward(Xo[R], dYo[R], p, w.act)     # row-local: e, u, h, y, dX at rows R
    Rt = torch.from_numpy(R).cuda()
    for k in ("e", "u", "h", "y"):
        check(k, host64(fw[k].index_select(0, Rt)), ref[k])
    check("dX", host64(bw["dX"].index_select(0, Rt)), ref["dX"])
    C = _rows(n, k=14, seed=1)
    col = O.mlp_backward_columns(Xo, dYo, p, C, w.act)
    Ct = torch.from_numpy(C).cuda()
    check("dB_gate", host64(bw["dB_gate"].index_select(0, Ct)), col["dBg"])
    check("dB_up", host64(bw["dB_up"].index_select(0, Ct)), col["dBu"])
    check("dA_down", host64(bw["dA_down"].index_select(1, Ct)), col["dAd"])
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
    R = _rows(w.T)
    Rt = torch.from_numpy(R).cuda()
    Xo = O.from_bf16(inp["X"])
    dOo = {t: O.from_bf16(inp["dY_" + t]) for t in ("q", "k", "v")}
    rf = O.qkv_forward(Xo[R], p)
    rb = O.qkv_backward(Xo[R], dOo["q"][R], dOo["k"][R], dOo["v"][R], p)
    for t in ("Q", "K", "V"):
        check(t, host64(fw[t].index_select(0, Rt)), rf[t])
    check("dX", host64(bw["dX"].index_select(0, Rt)), rb["dX"])
    for t in ("q", "k", "v"):   # the LoRA gradients in full
        g = O.lora_w_lora_grads(Xo, dOo[t], p["A" + t], p["B" + t], p["s" + t])
        check("dA_" + t, host64(bw["dA_" + t]), g["dA"])
        check("dB_" + t, host64(bw["dB_" + t]), g["dB"])

    wo = synth.WORKLOADS["llama3_8b_o_" + base]
    io, po = _inputs(wo)
    o = _dev_lora(io, "o", wo)
    Xd, dYd = dev_bf16(io["X"]), dev_bf16(io["dY"])
    f = L.lora_o_fwd(Xd, o)
    b = L.lora_o_bwd(Xd, dYd, f, o)
    L.lm_workspace_check(f["ws"])
    Xo, dYo = O.from_bf16(io["X"]), O.from_bf16(io["dY"])
    Wo, Ao, Bo, so = po["Wo"], po["Ao"], po["Bo"], po["so"]
    Y, _ = O.lora_w_forward(Xo[R], Wo, Ao, Bo, so)
    g = O.lora_w_backward(Xo[R], dYo[R], Wo, Ao, Bo, so)
    check("Y", host64(f["Y"].index_select(0, Rt)), Y)
    check("dX", host64(b["dX"].index_select(0, Rt)), g["dX"])
    go = O.lora_w_lora_grads(Xo, dYo, Ao, Bo, so)
    check("dA", host64(b["dA"]), go["dA"])
    check("dB", host64(b["dB"]), go["dB"])
