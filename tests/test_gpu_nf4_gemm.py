"""GPU parity of the NF4-base paths (codes decoded inside the GEMM mainloop) against the fp64
oracle run on the oracle's own NF4 reconstruction of the same bf16 weights.

The GPU packs W with nf4_pack; the oracle quantises the same bf16 bytes with oracle.nf4 and uses
bf16(dequantize(...)) as the base weight ("dequantise to compute dtype, then matmul")."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import lora as O
from oracle import nf4 as onf4

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu


def _oracle_base(bits):
    x = synth.bf16_bits_to_f32(bits).reshape(-1)
    codes, q, c = onf4.quantize(x)
    return onf4.dequantize_bf16(codes, q, c).astype(np.float64).reshape(bits.shape)


def _nf4_lora(inp, t, s):
    W = L.nf4_pack(dev_bf16(inp["W_" + t]))
    return L.Lora(W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), s)


NF4_MLP = [
    ("tiny_nf4_swiglu", 512, 256, 704, 8, 16.0, "swiglu", False),
    ("ragged_nf4_geglu", 300, 256, 448, 16, 32.0, "geglu", False),
    ("nf4_r64", 200, 128, 256, 64, 128.0, "swiglu", False),
    ("nf4_zero_base", 260, 256, 320, 16, 32.0, "geglu", True),
    # four K blocks per dh tile (the fewest with which its epilogue borrows a stage slot) and
    # 80 tiles, so that some CTA pairs run two
    ("nf4_four_kblocks", 2048, 192, 5120, 16, 32.0, "swiglu", False),
]


@pytest.mark.parametrize("name,T,d,n,r,alpha,act,zero_W", NF4_MLP, ids=[c[0] for c in NF4_MLP])
def test_mlp_nf4_matches_oracle(name, T, d, n, r, alpha, act, zero_W):
    w = synth.mlp_workload(name, T, d, n, r, alpha, act=act, nf4=True)
    inp = synth.make_inputs(w, seed=77, zero_W=zero_W)
    gate, up, down = (_nf4_lora(inp, t, w.s) for t in ("gate", "up", "down"))
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, gate, up, down, act=act)
    bw = L.lora_mlp_bwd(X, dY, fw, gate, up, down, act=act)
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        p["W" + k] = _oracle_base(inp["W_" + t])
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = w.s
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, act)
    for k in ("e", "u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_gate", "dAg"), ("dB_gate", "dBg"), ("dA_up", "dAu"), ("dB_up", "dBu"),
                  ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])


def test_mlp_nf4_equals_bf16_path_on_dequantised_weights():
    """The fused NF4 GEMMs and the bf16 GEMMs on nf4_dequant's bf16 output compute the same
    products of the same bf16 values; they agree far inside the oracle tolerance."""
    w = synth.mlp_workload("eq", 384, 256, 448, 16, 32.0, nf4=True)
    inp = synth.make_inputs(w, seed=5)
    nf = {t: _nf4_lora(inp, t, w.s) for t in ("gate", "up", "down")}
    bf = {}
    for t, Lr in nf.items():
        Wd = L.nf4_dequant(Lr.W, torch.bfloat16).view(Lr.W.rows, Lr.W.cols)
        bf[t] = L.Lora(Wd, Lr.A, Lr.B, Lr.s)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    f1 = L.lora_mlp_fwd(X, nf["gate"], nf["up"], nf["down"])
    b1 = L.lora_mlp_bwd(X, dY, f1, nf["gate"], nf["up"], nf["down"])
    f2 = L.lora_mlp_fwd(X, bf["gate"], bf["up"], bf["down"])
    b2 = L.lora_mlp_bwd(X, dY, f2, bf["gate"], bf["up"], bf["down"])
    torch.cuda.synchronize()
    for k in ("e", "u", "h", "y"):
        check(k, host64(f1[k]), host64(f2[k]), rel_fro=2e-3, max_abs=2e-2)
    for k in b1:
        check(k, host64(b1[k]), host64(b2[k]), rel_fro=2e-3, max_abs=2e-2)


def test_qkv_and_o_nf4_match_oracle():
    T, d, nq, nkv, r = 300, 256, 256, 64, 16
    w = synth.qkv_workload("qkv", T, d, nq, nkv, r, 32.0, nf4=True)
    inp = synth.make_inputs(w, seed=19)
    Ls = {t: _nf4_lora(inp, t, w.s) for t in ("q", "k", "v")}
    X = dev_bf16(inp["X"])
    fw = L.lora_qkv_fwd(X, Ls["q"], Ls["k"], Ls["v"])
    bw = L.lora_qkv_bwd(X, dev_bf16(inp["dY_q"]), dev_bf16(inp["dY_k"]), dev_bf16(inp["dY_v"]), fw,
                        Ls["q"], Ls["k"], Ls["v"])
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t in ("q", "k", "v"):
        p["W" + t] = _oracle_base(inp["W_" + t])
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

    wo = synth.o_workload("o", 257, 256, 256, 16, 32.0, nf4=True)
    io = synth.make_inputs(wo, seed=23)
    o = _nf4_lora(io, "o", wo.s)
    Xd = dev_bf16(io["X"])
    f = L.lora_o_fwd(Xd, o)
    b = L.lora_o_bwd(Xd, dev_bf16(io["dY"]), f, o)
    L.lm_workspace_check(f["ws"])
    Wb = _oracle_base(io["W_o"])
    A, B = O.from_bf16(io["A_o"]), O.from_bf16(io["B_o"])
    Y, _ = O.lora_w_forward(O.from_bf16(io["X"]), Wb, A, B, wo.s)
    g = O.lora_w_backward(O.from_bf16(io["X"]), O.from_bf16(io["dY"]), Wb, A, B, wo.s)
    check("Y", host64(f["Y"]), Y)
    check("dX", host64(b["dX"]), g["dX"])
    check("dA", host64(b["dA"]), g["dA"])
    check("dB", host64(b["dB"]), g["dB"])
