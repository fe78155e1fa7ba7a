"""Saturating gate values through the fused activation epilogues ("LoRA Optimizations", Triton
kernels: SwiGLU / GeGLU forward and backward), against the fp64 oracle through the C ABI.

W_gate is scaled by 128 (exact in bf16), so e = X W_g^T + ... spreads over about +-150 with a
standard deviation near 40: the SiLU and GELU tails, where exp(-e) overflows fp32 (e below about
-88.7), where 1 + exp(-e) passes 2^126 (the band -89 < e < -87), and where erf saturates to +-1,
all reach the forward (h = act(e) u) and backward (de = dh u act'(e), du = dh act(e)) epilogues.
Both the direct-load dh epilogue (bf16 base) and the staged one (NF4 base, four or more K blocks
per tile) run.  de and du stay in the workspace; they are checked through what they feed: dB_gate =
s de^T (X A_g^T) and dB_up column by column, dA_gate and dA_up through G = de B, and dX."""
import numpy as np
import pytest

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import lora as O
from oracle import nf4 as onf4

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu

GAIN = 128.0


def _base64(bits, base):
    if base == "bf16":
        return O.from_bf16(bits)
    x = synth.bf16_bits_to_f32(bits).reshape(-1)
    return onf4.dequantize_bf16(*onf4.quantize(x)).astype(np.float64).reshape(bits.shape)


@pytest.mark.parametrize("base", ["bf16", "nf4"])
@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_saturating_gate_values(base, act):
    T, d, n, r = 517, 256, 704, 16
    w = synth.mlp_workload("extreme", T, d, n, r, 32.0, act=act)
    inp = synth.make_inputs(w, seed=97)
    wg = synth.bf16_bits_to_f32(inp["W_gate"]).reshape(inp["W_gate"].shape) * np.float32(GAIN)
    inp["W_gate"] = synth.f32_to_bf16_bits(wg).reshape(wg.shape)
    Ls = {}
    for t in ("gate", "up", "down"):
        W = dev_bf16(inp["W_" + t])
        Ls[t] = L.Lora(L.nf4_pack(W) if base == "nf4" else W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), w.s)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, Ls["gate"], Ls["up"], Ls["down"], act=act)
    bw = L.lora_mlp_bwd(X, dY, fw, Ls["gate"], Ls["up"], Ls["down"], act=act)
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        p["W" + k] = _base64(inp["W_" + t], base)
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = w.s
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, act)
    e = ref["e"]
    # the inputs reach every band the epilogues treat specially
    assert (e > 100).any() and (e < -100).any()
    assert ((e > -89) & (e < -87)).any() and ((e > 87) & (e < 89)).any()
    for k in ("e", "u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_gate", "dAg"), ("dB_gate", "dBg"), ("dA_up", "dAu"), ("dB_up", "dBu"),
                  ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])
