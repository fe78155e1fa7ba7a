"""The dual rank-r reduction of the MLP, ReLU^2, QKV and O backward (one pass over an output gradient dOut for both its
B-projected gradient G = dOut B and its B gradient dB = dOut^T (s X A^T); "Avoid recomputing LoRA
B-projected gradient in fused-LoRA backward", LoRA_MLP.backward), against the fp64 oracle.

The planner takes the dual pass where it estimates it faster (the full-size workloads); here the
test hook forces it at small and ragged shapes -- T and the feature sizes not multiples of the
128 x 128 tile, ranks 8 to 64 (so 1 to 3 dB accumulators per unit), several row and column ranges
-- and checks every output and gradient, bitwise determinism of the backward, and agreement with
the separate passes."""
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import lora as O
from oracle import nf4 as onf4

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu

FORCE_DUAL = 16
GRADS = (("dA_gate", "dAg"), ("dB_gate", "dBg"), ("dA_up", "dAu"), ("dB_up", "dBu"), ("dA_down", "dAd"),
         ("dB_down", "dBd"))


def _base64(bits, base):
    if base == "bf16":
        return O.from_bf16(bits)
    x = synth.bf16_bits_to_f32(bits).reshape(-1)
    return onf4.dequantize_bf16(*onf4.quantize(x)).astype("float64").reshape(bits.shape)


def _bwd(X, dY, fw, Ls, act, force):
    assert L.call_status("lm_debug_inject", FORCE_DUAL if force else 0, 0) == L.LM_OK
    try:
        bw = L.lora_mlp_bwd(X, dY, fw, Ls["gate"], Ls["up"], Ls["down"], act=act)
    finally:
        assert L.call_status("lm_debug_inject", 0, 0) == L.LM_OK
    L.lm_workspace_check(fw["ws"])
    torch.cuda.synchronize()
    return bw


@pytest.mark.parametrize("base", ["bf16", "nf4"])
@pytest.mark.parametrize("T,d,n,r,act", [(517, 256, 704, 16, "swiglu"), (300, 384, 512, 64, "geglu"),
                                         (1000, 512, 1408, 8, "swiglu"), (6363, 256, 384, 32, "swiglu"),
                                         (5, 128, 256, 16, "geglu")])
def test_dual_reductions_match_oracle(base, T, d, n, r, act):
    w = synth.mlp_workload("dual", T, d, n, r, 2.0 * r, act=act)
    inp = synth.make_inputs(w, seed=113)
    Ls = {}
    for t in ("gate", "up", "down"):
        W = dev_bf16(inp["W_" + t])
        Ls[t] = L.Lora(L.nf4_pack(W) if base == "nf4" else W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), w.s)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, Ls["gate"], Ls["up"], Ls["down"], act=act)
    bw = _bwd(X, dY, fw, Ls, act, True)
    again = _bwd(X, dY, fw, Ls, act, True)
    for k in bw:
        assert torch.equal(bw[k], again[k]), k   # fixed-order reductions: bitwise reproducible
    sep = _bwd(X, dY, fw, Ls, act, False)
    p = {}
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        p["W" + k] = _base64(inp["W_" + t], base)
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = w.s
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, act)
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in GRADS:
        check(k, host64(bw[k]), ref[rk])
        check(k + " (separate passes)", host64(bw[k]), host64(sep[k]))


def _forced(fn):
    assert L.call_status("lm_debug_inject", FORCE_DUAL, 0) == L.LM_OK
    try:
        return fn()
    finally:
        assert L.call_status("lm_debug_inject", 0, 0) == L.LM_OK


@pytest.mark.parametrize("base", ["bf16", "nf4"])
@pytest.mark.parametrize("T,d,n,r", [(517, 256, 704, 16), (300, 384, 512, 64)])
def test_dual_relu2_matches_oracle(base, T, d, n, r):
    w = synth.relu2_workload("dual_relu2", T, d, n, r, 2.0 * r)
    inp = synth.make_inputs(w, seed=127)
    Ls = {}
    for t in ("up", "down"):
        W = dev_bf16(inp["W_" + t])
        Ls[t] = L.Lora(L.nf4_pack(W) if base == "nf4" else W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), w.s)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_relu2_mlp_fwd(X, Ls["up"], Ls["down"])
    bw = _forced(lambda: L.lora_relu2_mlp_bwd(X, dY, fw, Ls["up"], Ls["down"]))
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t, k in (("up", "u"), ("down", "d")):
        p["W" + k] = _base64(inp["W_" + t], base)
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = w.s
    ref = O.relu2_mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p)
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_up", "dAu"), ("dB_up", "dBu"), ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])


@pytest.mark.parametrize("base", ["bf16", "nf4"])
@pytest.mark.parametrize("T,d,nq,nk,nv,r", [(300, 256, 256, 64, 192, 16), (517, 512, 512, 128, 256, 48)])
def test_dual_qkv_and_o_match_oracle(base, T, d, nq, nk, nv, r):
    w = synth.qkv_workload("dual_qkv", T, d, nq, nk, r, 2.0 * r, v=nv)
    inp = synth.make_inputs(w, seed=131)
    Ls = {}
    for t in ("q", "k", "v"):
        W = dev_bf16(inp["W_" + t])
        Ls[t] = L.Lora(L.nf4_pack(W) if base == "nf4" else W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), w.s)
    X = dev_bf16(inp["X"])
    dO = {t: dev_bf16(inp["dY_" + t]) for t in ("q", "k", "v")}
    fw = L.lora_qkv_fwd(X, Ls["q"], Ls["k"], Ls["v"])
    bw = _forced(lambda: L.lora_qkv_bwd(X, dO["q"], dO["k"], dO["v"], fw, Ls["q"], Ls["k"], Ls["v"]))
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t in ("q", "k", "v"):
        p["W" + t] = _base64(inp["W_" + t], base)
        p["A" + t] = O.from_bf16(inp["A_" + t])
        p["B" + t] = O.from_bf16(inp["B_" + t])
        p["s" + t] = w.s
    Xo = O.from_bf16(inp["X"])
    rb = O.qkv_backward(Xo, O.from_bf16(inp["dY_q"]), O.from_bf16(inp["dY_k"]), O.from_bf16(inp["dY_v"]), p)
    check("dX", host64(bw["dX"]), rb["dX"])
    for t in ("q", "k", "v"):
        check("dA_" + t, host64(bw["dA_" + t]), rb["dA" + t])
        check("dB_" + t, host64(bw["dB_" + t]), rb["dB" + t])

    wo = synth.o_workload("dual_o", T, d, nq, r, 2.0 * r)
    io = synth.make_inputs(wo, seed=137)
    Wo = dev_bf16(io["W_o"])
    o = L.Lora(L.nf4_pack(Wo) if base == "nf4" else Wo, dev_bf16(io["A_o"]), dev_bf16(io["B_o"]), wo.s)
    Xd, dYd = dev_bf16(io["X"]), dev_bf16(io["dY"])
    f = L.lora_o_fwd(Xd, o)
    b = _forced(lambda: L.lora_o_bwd(Xd, dYd, f, o))
    L.lm_workspace_check(f["ws"])
    g = O.lora_w_backward(O.from_bf16(io["X"]), O.from_bf16(io["dY"]), _base64(io["W_o"], base), O.from_bf16(io["A_o"]),
                          O.from_bf16(io["B_o"]), wo.s)
    check("O dX", host64(b["dX"]), g["dX"])
    check("O dA", host64(b["dA"]), g["dA"])
    check("O dB", host64(b["dB"]), g["dB"])
