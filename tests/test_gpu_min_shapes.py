"""The smallest shapes the ABI accepts: feature sizes of 32 (half of one 64-deep K block, so every
GEMM runs a single short K block and most of each tile is outside the tensors), r = 8, a handful
of tokens; bf16 bases, and NF4 at the smallest shapes its format allows (rows of whole 64-element
blocks, numel a multiple of 64 x 256).
Every output and gradient against the fp64 oracle."""
import pytest

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import lora as O
from oracle import nf4 as onf4

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu

GRADS = (("dA_gate", "dAg"), ("dB_gate", "dBg"), ("dA_up", "dAu"), ("dB_up", "dBu"), ("dA_down", "dAd"),
         ("dB_down", "dBd"))


def _w64(bits, base):
    if base == "bf16":
        return O.from_bf16(bits)
    x = synth.bf16_bits_to_f32(bits).reshape(-1)
    return onf4.dequantize_bf16(*onf4.quantize(x)).astype("float64").reshape(bits.shape)


def _dev(inp, t, s, base):
    W = dev_bf16(inp["W_" + t])
    return L.Lora(L.nf4_pack(W) if base == "nf4" else W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), s)


@pytest.mark.parametrize("T,d,n,base,act", [(7, 32, 32, "bf16", "swiglu"), (130, 32, 96, "bf16", "geglu"),
                                              (65, 64, 512, "nf4", "swiglu"), (3, 64, 256, "nf4", "geglu")])
def test_mlp_smallest_features(T, d, n, base, act):
    w = synth.mlp_workload("min", T, d, n, 8, 16.0, act=act)
    inp = synth.make_inputs(w, seed=91)
    gate, up, down = (_dev(inp, t, w.s, base) for t in ("gate", "up", "down"))
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, gate, up, down, act=act)
    bw = L.lora_mlp_bwd(X, dY, fw, gate, up, down, act=act)
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        p["W" + k] = _w64(inp["W_" + t], base)
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = w.s
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, act)
    for k in ("e", "u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in GRADS:
        check(k, host64(bw[k]), ref[rk])


def test_qkv_o_relu2_smallest_features():
    w = synth.qkv_workload("minq", 9, 32, 32, 32, 8, 16.0, v=64)
    inp = synth.make_inputs(w, seed=92)
    q, k, v = (_dev(inp, t, w.s, "bf16") for t in ("q", "k", "v"))
    X = dev_bf16(inp["X"])
    fw = L.lora_qkv_fwd(X, q, k, v)
    bw = L.lora_qkv_bwd(X, dev_bf16(inp["dY_q"]), dev_bf16(inp["dY_k"]), dev_bf16(inp["dY_v"]), fw, q, k, v)
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
    for t in ("Q", "K", "V"):
        check(t, host64(fw[t]), rf[t])
    check("dX", host64(bw["dX"]), rb["dX"])
    for t in ("q", "k", "v"):
        check("dA_" + t, host64(bw["dA_" + t]), rb["dA" + t])
        check("dB_" + t, host64(bw["dB_" + t]), rb["dB" + t])

    wo = synth.o_workload("mino", 5, 32, 32, 8, 16.0)
    io = synth.make_inputs(wo, seed=93)
    o = _dev(io, "o", wo.s, "bf16")
    X, dY = dev_bf16(io["X"]), dev_bf16(io["dY"])
    f = L.lora_o_fwd(X, o)
    b = L.lora_o_bwd(X, dY, f, o)
    L.lm_workspace_check(f["ws"])
    Wo, Ao, Bo = (O.from_bf16(io[k]) for k in ("W_o", "A_o", "B_o"))
    Xo, dYo = O.from_bf16(io["X"]), O.from_bf16(io["dY"])
    Y, _ = O.lora_w_forward(Xo, Wo, Ao, Bo, wo.s)
    g = O.lora_w_backward(Xo, dYo, Wo, Ao, Bo, wo.s)
    check("Y", host64(f["Y"]), Y)
    for k in ("dX", "dA", "dB"):
        check(k, host64(b[k]), g[k])

    wr = synth.relu2_workload("minr", 11, 32, 32, 8, 16.0)
    ir = synth.make_inputs(wr, seed=94)
    up, down = _dev(ir, "up", wr.s, "bf16"), _dev(ir, "down", wr.s, "bf16")
    X, dY = dev_bf16(ir["X"]), dev_bf16(ir["dY"])
    fr = L.lora_relu2_mlp_fwd(X, up, down)
    br = L.lora_relu2_mlp_bwd(X, dY, fr, up, down)
    L.lm_workspace_check(fr["ws"])
    p = {}
    for t, kk in (("up", "u"), ("down", "d")):
        p["W" + kk] = O.from_bf16(ir["W_" + t])
        p["A" + kk] = O.from_bf16(ir["A_" + t])
        p["B" + kk] = O.from_bf16(ir["B_" + t])
        p["s" + kk] = wr.s
    ref = O.relu2_mlp_backward(O.from_bf16(ir["X"]), O.from_bf16(ir["dY"]), p)
    for kk in ("u", "h", "y"):
        check(kk, host64(fr[kk]), ref[kk])
    check("dX", host64(br["dX"]), ref["dX"])
    for kk, rk in (("dA_up", "dAu"), ("dB_up", "dBu"), ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(kk, host64(br[kk]), ref[rk])
