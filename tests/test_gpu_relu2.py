"""GPU parity of the non-gated ReLU^2 LoRA MLP ("LoRA Optimizations", FP32 LoRA gradients: dense
ReLU^2 MLPs with up/down LoRA projections and a fused ReLU^2 derivative) against the fp64 oracle,
through the C ABI: bf16 and NF4 bases, ragged token counts, r 8 / 16 / 64, a zero base, B = 0,
and the 8B sizes in full."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import lora as O
from oracle import nf4 as onf4

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu


def _oracle_base(bits, nf4):
    if not nf4:
        return O.from_bf16(bits)
    x = synth.bf16_bits_to_f32(bits).reshape(-1)
    codes, q, c = onf4.quantize(x)
    return onf4.dequantize_bf16(codes, q, c).astype(np.float64).reshape(bits.shape)


def _run(w, inp, nf4):
    def mk(t):
        W = dev_bf16(inp["W_" + t])
        return L.Lora(L.nf4_pack(W) if nf4 else W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), w.s)
    up, down = mk("up"), mk("down")
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_relu2_mlp_fwd(X, up, down)
    bw = L.lora_relu2_mlp_bwd(X, dY, fw, up, down)
    L.lm_workspace_check(fw["ws"])
    torch.cuda.synchronize()
    return fw, bw


def _params(inp, s, nf4):
    p = {}
    for t, k in (("up", "u"), ("down", "d")):
        p["W" + k] = _oracle_base(inp["W_" + t], nf4)
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = s
    return p


CASES = [
    # name, T, d, n, r, alpha, nf4, zero_W, zero_B
    ("tiny", 512, 256, 704, 8, 16.0, False, False, False),
    ("ragged", 333, 256, 416, 16, 32.0, False, False, False),
    ("r64", 200, 512, 512, 64, 128.0, False, False, False),
    ("zero_base", 260, 256, 320, 16, 32.0, False, True, False),
    ("B_zero", 300, 256, 384, 16, 32.0, False, False, True),
    ("nf4_tiny", 512, 256, 768, 8, 16.0, True, False, False),
    ("nf4_ragged", 300, 256, 512, 16, 32.0, True, False, False),
    ("nf4_r64", 200, 128, 512, 64, 128.0, True, False, False),
]


@pytest.mark.parametrize("name,T,d,n,r,alpha,nf4,zero_W,zero_B", CASES, ids=[c[0] for c in CASES])
def test_relu2_mlp_matches_oracle(name, T, d, n, r, alpha, nf4, zero_W, zero_B):
    w = synth.relu2_workload(name, T, d, n, r, alpha, nf4=nf4)
    inp = synth.make_inputs(w, seed=41, zero_W=zero_W, zero_B=zero_B)
    fw, bw = _run(w, inp, nf4)
    ref = O.relu2_mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), _params(inp, w.s, nf4))
    assert (ref["u"] > 0).any() and (ref["u"] < 0).any()
    for k in ("u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_up", "dAu"), ("dB_up", "dBu"), ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])
    if zero_B:  # dA = s G^T Z with G = dOut B = 0: exact zeros
        assert torch.count_nonzero(bw["dA_up"]) == 0 and torch.count_nonzero(bw["dA_down"]) == 0


@pytest.mark.parametrize("nf4", [False, True])
def test_relu2_mlp_8b_sizes_in_full(nf4):
    """The 8B sizes (T 8192, d 4096, n 14336, r 16), as the benchmark runs them: every output and
    gradient against the full oracle."""
    w = synth.WORKLOADS["relu2_mlp_8b_nf4" if nf4 else "relu2_mlp_8b_bf16"]
    inp = synth.make_inputs(w)
    fw, bw = _run(w, inp, nf4)
    ref = O.relu2_mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), _params(inp, w.s, nf4))
    for k in ("u", "h", "y"):
        check(k, host64(fw[k]), ref[k])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_up", "dAu"), ("dB_up", "dBu"), ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])
