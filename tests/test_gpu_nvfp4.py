"""GPU parity of the NVFP4 weight-only base ("LoRA Optimizations", FP32 LoRA gradients: weight-only
NVFP4 bases with bf16 activations), through the C ABI.

nvfp4_pack and nvfp4_dequant must equal the oracle bit for bit (codes, E4M3 block scales, the fp32
tensor scale, the fp32 and bf16 reconstructions), including E2M1 rounding ties, blocks whose E4M3
scale is subnormal, and zero blocks.  The fused GEMMs decode the codes inside their mainloop; their
results are checked against the fp64 oracle run on the oracle's own bf16 reconstruction of the same
bf16 weights (MLP with both activations, QKV, O, ReLU^2 MLP)."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import int4 as oi4
from oracle import lora as O
from oracle import nvfp4 as nv

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu


def _oracle_base(bits):
    x = synth.bf16_bits_to_f32(bits).reshape(bits.shape)
    codes, sb, sg, _ = nv.quantize(x)
    return nv.dequantize_bf16(codes, sb, sg, bits.shape[0], bits.shape[1]).astype(np.float64)


def _lora(inp, t, s):
    return L.Lora(L.nvfp4_pack(dev_bf16(inp["W_" + t])), dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), s)


def _params(inp, s, names):
    p = {}
    for t, k in names:
        p["W" + k] = _oracle_base(inp["W_" + t])
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = s
    return p


def _special_weight(rows=64, cols=512, seed=3):
    x = synth.bf16_bits_to_f32(synth.normal_bf16((rows, cols), 0.02, seed)).reshape(rows, cols).copy()
    x[0, 100] = 2688.0 * 2.0 ** -10           # the tensor maximum: S_g = 2^-10 exactly
    ties = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5, -6])
    x[1, :16] = ties * 2.0 ** -6               # s_b = 2^4, S = 2^-6: every E2M1 tie, exactly
    x[2, 16:32] *= 1e-3                        # a block whose E4M3 scale is subnormal
    x[3, 32:48] = 0.0                          # a zero block
    x[4, 48:64] = -0.0
    x[5] *= 1e-6                               # a row of tiny values
    x = oi4.bf16_round(x.astype(np.float32))
    return x, oi4.bf16_bits(x)


@pytest.mark.parametrize("shape", [(64, 512), (96, 1024)])
def test_pack_and_dequant_bit_exact(shape):
    rows, cols = shape
    x, bits = _special_weight(rows, cols)
    codes, sb, sg, _ = nv.quantize(x)
    assert 0 < sb[2, 1] < 8                    # the subnormal-scale block really is one
    Wq = L.nvfp4_pack(dev_bf16(bits))
    torch.cuda.synchronize()
    assert np.array_equal(Wq.codes.cpu().numpy(), codes)
    assert np.array_equal(Wq.block_scale.cpu().numpy(), nv.scale_bytes(sb))
    assert Wq.global_scale.cpu().numpy().view(np.uint32)[0] == np.float32(sg).view(np.uint32)
    ref = nv.dequantize(codes, sb, sg, rows, cols)
    f32 = L.nvfp4_dequant(Wq, torch.float32).cpu().numpy()
    assert np.array_equal(f32.view(np.uint32), ref.view(np.uint32))
    b16 = L.nvfp4_dequant(Wq, torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(b16, oi4.bf16_bits(oi4.bf16_round(ref)))


def test_pack_of_a_zero_weight():
    Wq = L.nvfp4_pack(torch.zeros((32, 128), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert Wq.global_scale.item() == 1.0
    assert not Wq.codes.any().item() and not Wq.block_scale.any().item()


MLP = [
    # name, T, d, n, r, alpha, act, zero_W
    ("swiglu", 512, 256, 704, 8, 16.0, "swiglu", False),
    ("geglu_ragged", 300, 256, 448, 16, 32.0, "geglu", False),
    ("r64", 200, 128, 256, 64, 128.0, "swiglu", False),
    ("zero_base", 260, 256, 320, 16, 32.0, "geglu", True),
]


@pytest.mark.parametrize("name,T,d,n,r,alpha,act,zero_W", MLP, ids=[c[0] for c in MLP])
def test_mlp_nvfp4_matches_oracle(name, T, d, n, r, alpha, act, zero_W):
    w = synth.mlp_workload(name, T, d, n, r, alpha, act=act)
    inp = synth.make_inputs(w, seed=97, zero_W=zero_W)
    gate, up, down = (_lora(inp, t, w.s) for t in ("gate", "up", "down"))
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, gate, up, down, act=act)
    bw = L.lora_mlp_bwd(X, dY, fw, gate, up, down, act=act)
    L.lm_workspace_check(fw["ws"])
    p = _params(inp, w.s, (("gate", "g"), ("up", "u"), ("down", "d")))
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, act)
    for k in ("e", "u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_gate", "dAg"), ("dB_gate", "dBg"), ("dA_up", "dAu"), ("dB_up", "dBu"),
                  ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])


def test_mlp_nvfp4_equals_bf16_path_on_dequantised_weights():
    """The fused NVFP4 GEMMs and the bf16 GEMMs on nvfp4_dequant's bf16 output multiply the same
    bf16 values; they agree far inside the oracle tolerance."""
    w = synth.mlp_workload("eq", 384, 256, 512, 16, 32.0)
    inp = synth.make_inputs(w, seed=6)
    q4 = {t: _lora(inp, t, w.s) for t in ("gate", "up", "down")}
    bf = {t: L.Lora(L.nvfp4_dequant(Lr.W, torch.bfloat16), Lr.A, Lr.B, Lr.s) for t, Lr in q4.items()}
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    f1 = L.lora_mlp_fwd(X, q4["gate"], q4["up"], q4["down"])
    b1 = L.lora_mlp_bwd(X, dY, f1, q4["gate"], q4["up"], q4["down"])
    f2 = L.lora_mlp_fwd(X, bf["gate"], bf["up"], bf["down"])
    b2 = L.lora_mlp_bwd(X, dY, f2, bf["gate"], bf["up"], bf["down"])
    torch.cuda.synchronize()
    for k in ("e", "u", "h", "y"):
        check(k, host64(f1[k]), host64(f2[k]), rel_fro=2e-3, max_abs=2e-2)
    for k in ("dX", "dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down"):
        check(k, host64(b1[k]), host64(b2[k]), rel_fro=2e-3, max_abs=2e-2)


def test_qkv_and_o_nvfp4_match_oracle():
    w = synth.qkv_workload("qkv_fp4", 300, 512, 512, 256, 16, 32.0)
    inp = synth.make_inputs(w, seed=41)
    Ls = {t: _lora(inp, t, w.s) for t in ("q", "k", "v")}
    X = dev_bf16(inp["X"])
    dO = {t: dev_bf16(inp["dY_" + t]) for t in ("q", "k", "v")}
    fw = L.lora_qkv_fwd(X, Ls["q"], Ls["k"], Ls["v"])
    bw = L.lora_qkv_bwd(X, dO["q"], dO["k"], dO["v"], fw, Ls["q"], Ls["k"], Ls["v"])
    L.lm_workspace_check(fw["ws"])
    p = _params(inp, w.s, (("q", "q"), ("k", "k"), ("v", "v")))
    Xo = O.from_bf16(inp["X"])
    rf = O.qkv_forward(Xo, p)
    rb = O.qkv_backward(Xo, O.from_bf16(inp["dY_q"]), O.from_bf16(inp["dY_k"]), O.from_bf16(inp["dY_v"]), p)
    for t in ("Q", "K", "V"):
        check(t, host64(fw[t]), rf[t])
    check("dX", host64(bw["dX"]), rb["dX"])
    for t in ("q", "k", "v"):
        check("dA_" + t, host64(bw["dA_" + t]), rb["dA" + t])
        check("dB_" + t, host64(bw["dB_" + t]), rb["dB" + t])

    wo = synth.o_workload("o_fp4", 260, 512, 256, 16, 32.0)
    io = synth.make_inputs(wo, seed=43)
    o = _lora(io, "o", wo.s)
    Xd, dYd = dev_bf16(io["X"]), dev_bf16(io["dY"])
    f = L.lora_o_fwd(Xd, o)
    b = L.lora_o_bwd(Xd, dYd, f, o)
    L.lm_workspace_check(f["ws"])
    Wo = _oracle_base(io["W_o"])
    Ao, Bo = O.from_bf16(io["A_o"]), O.from_bf16(io["B_o"])
    Xo, dYo = O.from_bf16(io["X"]), O.from_bf16(io["dY"])
    Y, _ = O.lora_w_forward(Xo, Wo, Ao, Bo, wo.s)
    g = O.lora_w_backward(Xo, dYo, Wo, Ao, Bo, wo.s)
    check("Y", host64(f["Y"]), Y)
    check("dX", host64(b["dX"]), g["dX"])
    check("dA", host64(b["dA"]), g["dA"])
    check("dB", host64(b["dB"]), g["dB"])


def test_relu2_nvfp4_matches_oracle():
    w = synth.relu2_workload("relu2_fp4", 300, 256, 512, 16, 32.0)
    inp = synth.make_inputs(w, seed=47)
    up, down = _lora(inp, "up", w.s), _lora(inp, "down", w.s)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_relu2_mlp_fwd(X, up, down)
    bw = L.lora_relu2_mlp_bwd(X, dY, fw, up, down)
    L.lm_workspace_check(fw["ws"])
    p = _params(inp, w.s, (("up", "u"), ("down", "d")))
    ref = O.relu2_mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p)
    for k in ("u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_up", "dAu"), ("dB_up", "dBu"), ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])
