"""GPU parity of the groupwise int4 base ("loralei" README, QLoRA section: int4 with group sizes 32,
64, 128, 256; input gradients from the packed weight), through the C ABI.

int4_pack and int4_dequant must equal the oracle bit for bit (codes, bf16 scale and zero, the fp32
and bf16 reconstructions).  The fused GEMMs decode the codes inside their mainloop; their results
are checked against the fp64 oracle run on the oracle's own bf16 reconstruction of the same bf16
weights, for every group size, both activations, ragged token counts, the ReLU^2 MLP and the
QKV / O projections (whose input gradients read the weight MN-major)."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import int4 as oi4
from oracle import lora as O

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu


def _oracle_base(bits, group):
    x = synth.bf16_bits_to_f32(bits).reshape(bits.shape)
    codes, s, z, _ = oi4.quantize(x, group)
    return oi4.dequantize_bf16(codes, s, z, bits.shape[0], bits.shape[1], group).astype(np.float64)


def _lora(inp, t, s, group):
    W = L.int4_pack(dev_bf16(inp["W_" + t]), group)
    return L.Lora(W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), s)


def _params(inp, s, group, names):
    p = {}
    for t, k in names:
        p["W" + k] = _oracle_base(inp["W_" + t], group)
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = s
    return p


@pytest.mark.parametrize("group", oi4.GROUPS)
def test_pack_and_dequant_bit_exact(group):
    rows, cols = 96, 1024
    x = synth.bf16_bits_to_f32(synth.normal_bf16((rows, cols), 0.02, 11 + group)).reshape(rows, cols).copy()
    x[0, :group] += 3.0                 # a group far from zero
    x[1, group:2 * group] = -0.375      # a constant group (s = 0)
    x[2] = 0.0                          # an all-zero row
    x[3, :group] *= 1e-30               # a group of tiny values
    x = oi4.bf16_round(x.astype(np.float32))
    bits = oi4.bf16_bits(x)
    codes, s, z, _ = oi4.quantize(x, group)
    Wq = L.int4_pack(dev_bf16(bits), group)
    torch.cuda.synchronize()
    assert np.array_equal(Wq.codes.cpu().numpy(), codes)
    got_sz = Wq.scale_zero.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got_sz, oi4.scale_zero_bits(s, z))
    ref = oi4.dequantize(codes, s, z, rows, cols, group)
    f32 = L.int4_dequant(Wq, torch.float32).cpu().numpy()
    assert np.array_equal(f32.view(np.uint32), ref.view(np.uint32))
    b16 = L.int4_dequant(Wq, torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(b16, oi4.bf16_bits(oi4.bf16_round(ref)))


MLP = [
    # name, T, d, n, r, alpha, act, group, zero_W
    ("g32_swiglu", 300, 256, 512, 16, 32.0, "swiglu", 32, False),
    ("g64_geglu", 512, 256, 768, 8, 16.0, "geglu", 64, False),
    ("g128_swiglu", 260, 512, 384, 16, 32.0, "swiglu", 128, False),
    ("g256_geglu_r64", 200, 256, 512, 64, 128.0, "geglu", 256, False),
    ("g128_zero_base", 333, 256, 640, 16, 32.0, "swiglu", 128, True),
]


@pytest.mark.parametrize("name,T,d,n,r,alpha,act,group,zero_W", MLP, ids=[c[0] for c in MLP])
def test_mlp_int4_matches_oracle(name, T, d, n, r, alpha, act, group, zero_W):
    w = synth.mlp_workload(name, T, d, n, r, alpha, act=act)
    inp = synth.make_inputs(w, seed=91, zero_W=zero_W)
    gate, up, down = (_lora(inp, t, w.s, group) for t in ("gate", "up", "down"))
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, gate, up, down, act=act)
    bw = L.lora_mlp_bwd(X, dY, fw, gate, up, down, act=act)
    L.lm_workspace_check(fw["ws"])
    p = _params(inp, w.s, group, (("gate", "g"), ("up", "u"), ("down", "d")))
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, act)
    for k in ("e", "u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_gate", "dAg"), ("dB_gate", "dBg"), ("dA_up", "dAu"), ("dB_up", "dBu"),
                  ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])


@pytest.mark.parametrize("group", [32, 128])
def test_mlp_int4_equals_bf16_path_on_dequantised_weights(group):
    """The fused int4 GEMMs and the bf16 GEMMs on int4_dequant's bf16 output multiply the same
    bf16 values; they agree far inside the oracle tolerance."""
    w = synth.mlp_workload("eq", 384, 256, 512, 16, 32.0)
    inp = synth.make_inputs(w, seed=5)
    q4 = {t: _lora(inp, t, w.s, group) for t in ("gate", "up", "down")}
    bf = {t: L.Lora(L.int4_dequant(Lr.W, torch.bfloat16), Lr.A, Lr.B, Lr.s) for t, Lr in q4.items()}
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


@pytest.mark.parametrize("group", [32, 256])
def test_qkv_int4_matches_oracle(group):
    w = synth.qkv_workload("qkv_i4", 300, 512, 512, 256, 16, 32.0)
    inp = synth.make_inputs(w, seed=23)
    Ls = {t: _lora(inp, t, w.s, group) for t in ("q", "k", "v")}
    X = dev_bf16(inp["X"])
    dO = {t: dev_bf16(inp["dY_" + t]) for t in ("q", "k", "v")}
    fw = L.lora_qkv_fwd(X, Ls["q"], Ls["k"], Ls["v"])
    bw = L.lora_qkv_bwd(X, dO["q"], dO["k"], dO["v"], fw, Ls["q"], Ls["k"], Ls["v"])
    L.lm_workspace_check(fw["ws"])
    p = _params(inp, w.s, group, (("q", "q"), ("k", "k"), ("v", "v")))
    Xo = O.from_bf16(inp["X"])
    rf = O.qkv_forward(Xo, p)
    rb = O.qkv_backward(Xo, O.from_bf16(inp["dY_q"]), O.from_bf16(inp["dY_k"]), O.from_bf16(inp["dY_v"]), p)
    for t in ("Q", "K", "V"):
        check(t, host64(fw[t]), rf[t])
    check("dX", host64(bw["dX"]), rb["dX"])
    for t in ("q", "k", "v"):
        check("dA_" + t, host64(bw["dA_" + t]), rb["dA" + t])
        check("dB_" + t, host64(bw["dB_" + t]), rb["dB" + t])


@pytest.mark.parametrize("group", [64, 128])
def test_o_int4_matches_oracle(group):
    w = synth.o_workload("o_i4", 260, 512, 256, 16, 32.0)
    inp = synth.make_inputs(w, seed=29)
    o = _lora(inp, "o", w.s, group)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    f = L.lora_o_fwd(X, o)
    b = L.lora_o_bwd(X, dY, f, o)
    L.lm_workspace_check(f["ws"])
    Wo = _oracle_base(inp["W_o"], group)
    Ao, Bo = O.from_bf16(inp["A_o"]), O.from_bf16(inp["B_o"])
    Xo, dYo = O.from_bf16(inp["X"]), O.from_bf16(inp["dY"])
    Y, _ = O.lora_w_forward(Xo, Wo, Ao, Bo, w.s)
    g = O.lora_w_backward(Xo, dYo, Wo, Ao, Bo, w.s)
    check("Y", host64(f["Y"]), Y)
    check("dX", host64(b["dX"]), g["dX"])
    check("dA", host64(b["dA"]), g["dA"])
    check("dB", host64(b["dB"]), g["dB"])


@pytest.mark.parametrize("group", [32, 128])
def test_relu2_int4_matches_oracle(group):
    w = synth.relu2_workload("relu2_i4", 300, 256, 512, 16, 32.0)
    inp = synth.make_inputs(w, seed=31)
    up, down = _lora(inp, "up", w.s, group), _lora(inp, "down", w.s, group)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_relu2_mlp_fwd(X, up, down)
    bw = L.lora_relu2_mlp_bwd(X, dY, fw, up, down)
    L.lm_workspace_check(fw["ws"])
    p = _params(inp, w.s, group, (("up", "u"), ("down", "d")))
    ref = O.relu2_mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p)
    for k in ("u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_up", "dAu"), ("dB_up", "dBu"), ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])
