"""Token counts whose activations pass 2^31 elements: T = 2^23 + 77 tokens at d = n = 256, r = 16
(T * n = 2 147 503 360), bf16 base, SwiGLU.  Row-wise outputs (e, u, h, y, dX) are compared with the
fp64 oracle on sampled rows, among them every row past element 2^31 of the T x n tensors; the
LoRA gradients, sums over all 8.4 M tokens, through the identity <A, dA> = <B, dB> of every
projection and against exact zero for none.  X and dY are drawn on the device from a seeded
generator and the sampled rows copied back, so the oracle sees the same bytes."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import synth
from bwd_lora_mlp_gb300 import lib as L
from oracle import lora as O

from gpu_util import check, host64, mlp_device_params, mlp_oracle_params

pytestmark = pytest.mark.gpu

T = (1 << 23) + 77
D = N = 256
R = 16


def _draw(rows, cols, std, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    step = 1 << 20
    for r0 in range(0, rows, step):  # in slices, to keep the fp32 draw small
        r1 = min(rows, r0 + step)
        out[r0:r1] = (torch.randn((r1 - r0, cols), generator=g, device="cuda") * std).to(torch.bfloat16)
    return out


def test_mlp_past_two_to_the_31_elements():
    w = synth.mlp_workload("large_t_params", 8, D, N, R, 32.0)
    inp = synth.make_inputs(w, seed=17)  # W, A, B (the small T of this workload is unused)
    gate, up, down = mlp_device_params(inp, w.s)
    X = _draw(T, D, 1.0, 1234)
    dY = _draw(T, D, 1e-2, 1235)
    fw = L.lora_mlp_fwd(X, gate, up, down)
    bw = L.lora_mlp_bwd(X, dY, fw, gate, up, down)
    torch.cuda.synchronize()
    L.lm_workspace_check(fw["ws"])
    assert (T * N) > (1 << 31)
    first_past = (1 << 31) // N  # first row with elements past 2^31
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(first_past - 40, T),
                                     np.linspace(0, T - 1, 200).astype(np.int64)]))
    idx = torch.from_numpy(rows).cuda()
    p = mlp_oracle_params(inp, w.s)
    ref = O.mlp_backward(host64(X[idx]), host64(dY[idx]), p, "swiglu")
    for name, key in (("e", "e"), ("u", "u"), ("h", "h"), ("y", "y")):
        check(name, host64(fw[name][idx]), ref[key])
    check("dX", host64(bw["dX"][idx]), ref["dX"])
    # LoRA gradients: every one finite, none all zero, and <A, dA> = <B, dB> per projection
    for t in ("gate", "up", "down"):
        dA, dB = host64(bw["dA_" + t]), host64(bw["dB_" + t])
        assert np.all(np.isfinite(dA)) and np.all(np.isfinite(dB)), t
        assert np.abs(dA).max() > 0 and np.abs(dB).max() > 0, t
        A = O.from_bf16(inp["A_" + t])
        Bm = O.from_bf16(inp["B_" + t])
        lhs, rhs = float(np.sum(A * dA)), float(np.sum(Bm * dB))
        assert abs(lhs - rhs) <= 1e-2 * max(abs(lhs), abs(rhs)), (t, lhs, rhs)
