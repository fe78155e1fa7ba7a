"""Helpers shared by the GPU parity tests: moving seeded bf16 inputs to the device, building the
LoRA structs, running the fp64 oracle on the same bytes, and the acceptance check.

Acceptance (every bf16-computed output and fp32 gradient against the fp64 oracle):
relative Frobenius error <= 1e-2 and max-abs error <= 2e-2 * max|ref|.
"""
from __future__ import annotations

import numpy as np
import torch

from bwd_lora_mlp_gb300 import lib as L
from oracle import lora as O

REL_FRO = 1e-2
MAX_ABS = 2e-2


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check(name: str, got: np.ndarray, ref: np.ndarray, rel_fro: float = REL_FRO, max_abs: float = MAX_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), name + ": non-finite values"
    nref = np.linalg.norm(ref)
    err = np.linalg.norm(got - ref)
    scale = np.abs(ref).max()
    mabs = np.abs(got - ref).max()
    if nref == 0:
        assert mabs == 0, "%s: expected exact zeros, max |got| = %g" % (name, mabs)
        return
    assert err <= rel_fro * nref, "%s: relative Frobenius error %.3e > %.0e" % (name, err / nref, rel_fro)
    assert mabs <= max_abs * scale, "%s: max-abs error %.3e > %.0e * %.3e" % (name, mabs, max_abs, scale)


def mlp_device_params(inp: dict, s: float):
    def mk(t):
        return L.Lora(dev_bf16(inp["W_" + t]), dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), s)
    return mk("gate"), mk("up"), mk("down")


def mlp_oracle_params(inp: dict, s: float) -> dict:
    p = {}
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        p["W" + k] = O.from_bf16(inp["W_" + t])
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = s
    return p


def run_mlp(inp: dict, s: float, act: str):
    gate, up, down = mlp_device_params(inp, s)
    X = dev_bf16(inp["X"])
    dY = dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, gate, up, down, act=act)
    bw = L.lora_mlp_bwd(X, dY, fw, gate, up, down, act=act)
    L.lm_workspace_check(fw["ws"])
    torch.cuda.synchronize()
    return fw, bw
