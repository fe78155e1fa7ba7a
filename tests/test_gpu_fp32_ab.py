"""fp32 LoRA parameters as inputs ("LoRA Optimizations", FP32 LoRA gradients: the trainable A, B
stay fp32 and the GEMMs take bf16 inputs with fp32 gradient outputs).

Each call rounds fp32 A and B to bf16 (round to nearest even).  Two checks per projection kind:
  * the fp32-parameter run equals, bit for bit, the bf16 run on the rounded parameters (the
    oracle's own rounding, oracle.lora.to_bf16_bits), so the rounding is exactly RNE and the rest
    of the path is unchanged;
  * both match the fp64 oracle evaluated on those rounded parameters.
"""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from gpu_util import check, dev_bf16, host64
from oracle import lora as O

pytestmark = pytest.mark.gpu


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _same(name, a, b):
    assert torch.equal(a, b), name + ": fp32-parameter run differs from the bf16 run on rounded parameters"


@pytest.mark.parametrize("T", [512, 333])
def test_mlp_fp32_parameters(T):
    w = synth.scaled_workload(synth.WORKLOADS["tiny_mlp_swiglu"], T)
    inp = synth.make_inputs(w, seed=23)
    ab = synth.fp32_ab(w)
    rb = {k: O.to_bf16_bits(v) for k, v in ab.items()}
    W = {t: dev_bf16(inp["W_" + t]) for t in ("gate", "up", "down")}
    f32 = [L.Lora(W[t], _f32(ab["A_" + t]), _f32(ab["B_" + t]), w.s) for t in ("gate", "up", "down")]
    b16 = [L.Lora(W[t], dev_bf16(rb["A_" + t]), dev_bf16(rb["B_" + t]), w.s) for t in ("gate", "up", "down")]
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    out = []
    for ps in (f32, b16):
        fw = L.lora_mlp_fwd(X, *ps)
        bw = L.lora_mlp_bwd(X, dY, fw, *ps)
        L.lm_workspace_check(fw["ws"])
        out.append((fw, bw))
    torch.cuda.synchronize()
    (f1, b1), (f2, b2) = out
    for k in ("y", "e", "u", "h"):
        _same(k, f1[k], f2[k])
    for k in b1:
        _same(k, b1[k], b2[k])
    p = {}
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        p["W" + k] = O.from_bf16(inp["W_" + t])
        p["A" + k] = O.from_bf16(rb["A_" + t])
        p["B" + k] = O.from_bf16(rb["B_" + t])
        p["s" + k] = w.s
    Xo, dYo = O.from_bf16(inp["X"]), O.from_bf16(inp["dY"])
    ref = O.mlp_backward(Xo, dYo, p, "swiglu")
    check("y", host64(f1["y"]), ref["y"])
    check("dX", host64(b1["dX"]), ref["dX"])
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        check("dA_" + t, host64(b1["dA_" + t]), ref["dA" + k])
        check("dB_" + t, host64(b1["dB_" + t]), ref["dB" + k])


@pytest.mark.parametrize("nf4", [False, True])
def test_o_fp32_parameters(nf4):
    w = synth.o_workload("o", 300, 256, 256, 16, 32.0)
    inp = synth.make_inputs(w, seed=29)
    ab = synth.fp32_ab(w)
    rb = {k: O.to_bf16_bits(v) for k, v in ab.items()}
    Wd = dev_bf16(inp["W_o"])
    Wb = L.nf4_pack(Wd) if nf4 else Wd
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    out = []
    for A, B in ((_f32(ab["A_o"]), _f32(ab["B_o"])), (dev_bf16(rb["A_o"]), dev_bf16(rb["B_o"]))):
        o = L.Lora(Wb, A, B, w.s)
        fw = L.lora_o_fwd(X, o)
        bw = L.lora_o_bwd(X, dY, fw, o)
        L.lm_workspace_check(fw["ws"])
        out.append((fw, bw))
    torch.cuda.synchronize()
    (f1, b1), (f2, b2) = out
    _same("Y", f1["Y"], f2["Y"])
    for k in ("dX", "dA", "dB"):
        _same(k, b1[k], b2[k])
    Wo = O.from_bf16(inp["W_o"]) if not nf4 else None
    if Wo is not None:
        Xo, dYo = O.from_bf16(inp["X"]), O.from_bf16(inp["dY"])
        A, B = O.from_bf16(rb["A_o"]), O.from_bf16(rb["B_o"])
        Y, _ = O.lora_w_forward(Xo, Wo, A, B, w.s)
        g = O.lora_w_backward(Xo, dYo, Wo, A, B, w.s)
        check("Y", host64(f1["Y"]), Y)
        check("dX", host64(b1["dX"]), g["dX"])
        check("dA", host64(b1["dA"]), g["dA"])
        check("dB", host64(b1["dB"]), g["dB"])


def test_qkv_fp32_parameters():
    w = synth.qkv_workload("qkv", 256, 256, 256, 64, 16, 32.0)
    inp = synth.make_inputs(w, seed=37)
    ab = synth.fp32_ab(w)
    rb = {k: O.to_bf16_bits(v) for k, v in ab.items()}
    X = dev_bf16(inp["X"])
    dYs = [dev_bf16(inp["dY_" + t]) for t in ("q", "k", "v")]
    out = []
    for mk in ((lambda t: (_f32(ab["A_" + t]), _f32(ab["B_" + t]))),
               (lambda t: (dev_bf16(rb["A_" + t]), dev_bf16(rb["B_" + t])))):
        ps = [L.Lora(dev_bf16(inp["W_" + t]), *mk(t), w.s) for t in ("q", "k", "v")]
        fw = L.lora_qkv_fwd(X, *ps)
        bw = L.lora_qkv_bwd(X, *dYs, fw, *ps)
        L.lm_workspace_check(fw["ws"])
        out.append((fw, bw))
    torch.cuda.synchronize()
    (f1, b1), (f2, b2) = out
    for k in ("Q", "K", "V"):
        _same(k, f1[k], f2[k])
    for k in b1:
        _same(k, b1[k], b2[k])


@pytest.mark.parametrize("base", ["int4", "nvfp4"])
def test_mlp_fp32_parameters_over_int4_and_nvfp4_bases(base):
    """The conversion does not depend on the base: with an int4 (G = 64) or NVFP4 base the
    fp32-parameter run equals the bf16 run on the rounded parameters bit for bit."""
    w = synth.mlp_workload("ab32q", 300, 256, 512, 16, 32.0)
    inp = synth.make_inputs(w, seed=37)
    ab = synth.fp32_ab(w)
    rb = {k: O.to_bf16_bits(v) for k, v in ab.items()}
    pack = (lambda W: L.int4_pack(W, 64)) if base == "int4" else L.nvfp4_pack
    W = {t: pack(dev_bf16(inp["W_" + t])) for t in ("gate", "up", "down")}
    f32 = [L.Lora(W[t], _f32(ab["A_" + t]), _f32(ab["B_" + t]), w.s) for t in ("gate", "up", "down")]
    b16 = [L.Lora(W[t], dev_bf16(rb["A_" + t]), dev_bf16(rb["B_" + t]), w.s) for t in ("gate", "up", "down")]
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    out = []
    for ps in (f32, b16):
        fw = L.lora_mlp_fwd(X, *ps)
        bw = L.lora_mlp_bwd(X, dY, fw, *ps)
        L.lm_workspace_check(fw["ws"])
        out.append((fw, bw))
    torch.cuda.synchronize()
    (f1, b1), (f2, b2) = out
    for k in ("y", "e", "u", "h"):
        _same(k, f1[k], f2[k])
    for k in b1:
        _same(k, b1[k], b2[k])


def test_relu2_fp32_parameters():
    w = synth.relu2_workload("ab32r", 300, 256, 512, 16, 32.0)
    inp = synth.make_inputs(w, seed=39)
    ab = synth.fp32_ab(w)
    rb = {k: O.to_bf16_bits(v) for k, v in ab.items()}
    W = {t: dev_bf16(inp["W_" + t]) for t in ("up", "down")}
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    out = []
    for mk in (lambda t: (_f32(ab["A_" + t]), _f32(ab["B_" + t])), lambda t: (dev_bf16(rb["A_" + t]), dev_bf16(rb["B_" + t]))):
        up, down = (L.Lora(W[t], *mk(t), w.s) for t in ("up", "down"))
        fw = L.lora_relu2_mlp_fwd(X, up, down)
        bw = L.lora_relu2_mlp_bwd(X, dY, fw, up, down)
        L.lm_workspace_check(fw["ws"])
        out.append((fw, bw))
    torch.cuda.synchronize()
    (f1, b1), (f2, b2) = out
    for k in ("y", "u", "h"):
        _same(k, f1[k], f2[k])
    for k in b1:
        _same(k, b1[k], b2[k])
