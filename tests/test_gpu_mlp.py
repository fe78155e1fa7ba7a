"""GPU parity of lora_mlp_fwd / lora_mlp_bwd against the fp64 oracle, through the C ABI.

Sizes span several 128-row and 128/256-column tiles with ragged tails; r covers 8 (padded to a
16-wide MMA step), 16 and 64 (two 64-wide K blocks in the rank-r segment)."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import synth
from oracle import lora as O

from gpu_util import check, dev_bf16, host64, mlp_oracle_params, run_mlp

pytestmark = pytest.mark.gpu


def _compare(w, inp, fw, bw, act):
    p = mlp_oracle_params(inp, w.s)
    X, dY = O.from_bf16(inp["X"]), O.from_bf16(inp["dY"])
    ref = O.mlp_backward(X, dY, p, act)
    check("e", host64(fw["e"]), ref["e"])
    check("u", host64(fw["u"]), ref["u"])
    check("h", host64(fw["h"]), ref["h"])
    check("y", host64(fw["y"]), ref["y"])
    check("dX", host64(bw["dX"]), ref["dX"])
    for k, rk in (("dA_gate", "dAg"), ("dB_gate", "dBg"), ("dA_up", "dAu"), ("dB_up", "dBu"),
                  ("dA_down", "dAd"), ("dB_down", "dBd")):
        check(k, host64(bw[k]), ref[rk])


CASES = [
    # name, T, d, n, r, alpha, act
    ("tiny_swiglu", 512, 256, 704, 8, 16.0, "swiglu"),
    ("ragged_geglu_r16", 300, 256, 416, 16, 32.0, "geglu"),
    ("ragged_swiglu_r64", 200, 192, 352, 64, 128.0, "swiglu"),
    ("rows5_r32", 5, 128, 160, 32, 64.0, "geglu"),
]


@pytest.mark.parametrize("name,T,d,n,r,alpha,act", CASES, ids=[c[0] for c in CASES])
def test_mlp_matches_oracle(name, T, d, n, r, alpha, act):
    w = synth.mlp_workload(name, T, d, n, r, alpha, act=act)
    inp = synth.make_inputs(w, seed=2024)
    fw, bw = run_mlp(inp, w.s, act)
    _compare(w, inp, fw, bw, act)


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_lora_term_alone_with_zero_base(act):
    """W = 0: every output is made by the rank-r terms, so they are checked at their own scale."""
    w = synth.mlp_workload("w0", 384, 256, 320, 16, 32.0, act=act)
    inp = synth.make_inputs(w, seed=7, zero_W=True)
    fw, bw = run_mlp(inp, w.s, act)
    _compare(w, inp, fw, bw, act)


def test_B_zero_gives_exact_zero_dA():
    w = synth.mlp_workload("b0", 256, 128, 192, 16, 32.0)
    inp = synth.make_inputs(w, seed=3, zero_B=True)
    fw, bw = run_mlp(inp, w.s, "swiglu")
    for k in ("dA_gate", "dA_up", "dA_down"):
        assert torch.count_nonzero(bw[k]).item() == 0, k
    _compare(w, inp, fw, bw, "swiglu")


def test_A_zero_gives_exact_zero_dB():
    """A = 0: every rank-r product X Aᵀ (and h A_dᵀ) vanishes, so dB = dOutᵀ (s X Aᵀ) is exactly zero
    while dA = s Gᵀ X is not."""
    w = synth.mlp_workload("a0", 256, 128, 192, 16, 32.0)
    inp = synth.make_inputs(w, seed=4, zero_A=True)
    fw, bw = run_mlp(inp, w.s, "geglu")
    for k in ("dB_gate", "dB_up", "dB_down"):
        assert torch.count_nonzero(bw[k]).item() == 0, k
    for k in ("dA_gate", "dA_up", "dA_down"):
        assert torch.count_nonzero(bw[k]).item() > 0, k
    _compare(w, inp, fw, bw, "geglu")


def test_zero_scale_is_the_base_mlp():
    """s = 0 (alpha = 0): the outputs are the base MLP's and every LoRA gradient is exactly zero."""
    w = synth.mlp_workload("s0", 300, 256, 320, 16, 0.0)
    assert w.s == 0.0
    inp = synth.make_inputs(w, seed=6)
    fw, bw = run_mlp(inp, w.s, "swiglu")
    for k in ("dA_gate", "dB_gate", "dA_up", "dB_up", "dA_down", "dB_down"):
        assert torch.count_nonzero(bw[k]).item() == 0, k
    _compare(w, inp, fw, bw, "swiglu")
    base = synth.make_inputs(w, seed=6, zero_B=True)  # the same W, X, dY with the LoRA term removed
    fw0, _ = run_mlp(base, 1.0, "swiglu")
    for k in ("y", "e", "u", "h"):
        assert torch.equal(fw[k], fw0[k]), k


def test_bitwise_deterministic():
    w = synth.mlp_workload("det", 640, 256, 448, 16, 32.0)
    inp = synth.make_inputs(w, seed=11)
    fw1, bw1 = run_mlp(inp, w.s, "swiglu")
    fw2, bw2 = run_mlp(inp, w.s, "swiglu")
    for k in ("y", "e", "u", "h"):
        assert torch.equal(fw1[k], fw2[k]), k
    for k in bw1:
        assert torch.equal(bw1[k], bw2[k]), k


def test_gradient_identity_A_dA_equals_B_dB():
    w = synth.mlp_workload("ident", 512, 256, 384, 16, 32.0)
    inp = synth.make_inputs(w, seed=5)
    fw, bw = run_mlp(inp, w.s, "swiglu")
    for t in ("gate", "up", "down"):
        A = O.from_bf16(inp["A_" + t])
        Bm = O.from_bf16(inp["B_" + t])
        a = float(np.sum(A * host64(bw["dA_" + t])))
        b = float(np.sum(Bm * host64(bw["dB_" + t])))
        assert abs(a - b) <= 2e-2 * max(abs(a), abs(b)), (t, a, b)
