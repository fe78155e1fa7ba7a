"""Calls with no tokens (T = 0) through the C ABI: a forward is a no-op, and a backward writes
every LoRA gradient as the empty sum over tokens, exactly zero, over whatever the destination
held; dX has no rows.  Every block entry point, bf16 and NF4 bases."""
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth

from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

NAN = float("nan")


def _proj(inp, key, s, base):
    W = dev_bf16(inp["W_" + key])
    if base == "nf4":
        W = L.nf4_pack(W)
    return L.Lora(W, dev_bf16(inp["A_" + key]), dev_bf16(inp["B_" + key]), s)


def _nan_like(shapes):
    return {k: torch.full(v, NAN, dtype=torch.float32, device="cuda") for k, v in shapes.items()}


def _all_zero(grads):
    for k, g in grads.items():
        assert torch.equal(g, torch.zeros_like(g)), k


@pytest.mark.parametrize("base", ["bf16", "nf4"])
def test_mlp_without_tokens(base):
    d, n, r = 256, 512, 16
    w = synth.mlp_workload("empty", 8, d, n, r, 32.0)
    inp = synth.make_inputs(w, seed=5)
    gate, up, down = (_proj(inp, k, w.s, base) for k in ("gate", "up", "down"))
    X = torch.empty((0, d), dtype=torch.bfloat16, device="cuda")
    dY = torch.empty((0, d), dtype=torch.bfloat16, device="cuda")
    fw = L.lora_mlp_fwd(X, gate, up, down)
    assert fw["y"].shape == (0, d) and fw["h"].shape == (0, n)
    grads = _nan_like({"dA_gate": (r, d), "dB_gate": (n, r), "dA_up": (r, d), "dB_up": (n, r),
                       "dA_down": (r, n), "dB_down": (d, r)})
    bw = L.lora_mlp_bwd(X, dY, fw, gate, up, down, grads=grads)
    torch.cuda.synchronize()
    L.lm_workspace_check(fw["ws"])
    assert bw["dX"].shape == (0, d)
    _all_zero(grads)


@pytest.mark.parametrize("base", ["bf16", "nf4"])
def test_relu2_mlp_without_tokens(base):
    d, n, r = 256, 512, 16
    w = synth.mlp_workload("empty", 8, d, n, r, 32.0)
    inp = synth.make_inputs(w, seed=6)
    up, down = (_proj(inp, k, w.s, base) for k in ("up", "down"))
    X = torch.empty((0, d), dtype=torch.bfloat16, device="cuda")
    fw = L.lora_relu2_mlp_fwd(X, up, down)
    grads = _nan_like({"dA_up": (r, d), "dB_up": (n, r), "dA_down": (r, n), "dB_down": (d, r)})
    bw = L.lora_relu2_mlp_bwd(X, torch.empty_like(X), fw, up, down, grads=grads)
    torch.cuda.synchronize()
    L.lm_workspace_check(fw["ws"])
    assert bw["dX"].shape == (0, d)
    _all_zero(grads)


@pytest.mark.parametrize("base", ["bf16", "nf4"])
def test_qkv_and_o_without_tokens(base):
    d, nq, nkv, r = 256, 256, 128, 16
    w = synth.qkv_workload("empty", 8, d, nq, nkv, r, 32.0)
    inp = synth.make_inputs(w, seed=7)
    q, k, v = (_proj(inp, x, w.s, base) for x in ("q", "k", "v"))
    X = torch.empty((0, d), dtype=torch.bfloat16, device="cuda")
    fw = L.lora_qkv_fwd(X, q, k, v)
    grads = _nan_like({"dA_q": (r, d), "dB_q": (nq, r), "dA_k": (r, d), "dB_k": (nkv, r), "dA_v": (r, d),
                       "dB_v": (nkv, r)})
    e = lambda c: torch.empty((0, c), dtype=torch.bfloat16, device="cuda")
    bw = L.lora_qkv_bwd(X, e(nq), e(nkv), e(nkv), fw, q, k, v, grads=grads)
    torch.cuda.synchronize()
    L.lm_workspace_check(fw["ws"])
    assert bw["dX"].shape == (0, d)
    _all_zero(grads)

    wo = synth.o_workload("empty", 8, d, d, r, 32.0)
    inp = synth.make_inputs(wo, seed=8)
    o = _proj(inp, "o", wo.s, base)
    fo = L.lora_o_fwd(X, o)
    for entry in (L.lora_o_bwd, L.lora_o_bwd_static):
        dA = torch.full((r, d), NAN, device="cuda")
        dB = torch.full((d, r), NAN, device="cuda")
        bo = entry(X, e(d), fo, o, dA=dA, dB=dB)
        torch.cuda.synchronize()
        assert bo["dX"].shape == (0, d)
        _all_zero({"dA": dA, "dB": dB})
    L.lm_workspace_check(fo["ws"])
