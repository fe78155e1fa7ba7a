"""The fused MLP forward + backward captured into a CUDA graph: the calls allocate nothing, never
synchronise and launch with programmatic stream serialisation, so a whole step can be captured
once and replayed.  Every replay must reproduce the eager results bit for bit (the kernels are
deterministic), also after the inputs are overwritten in place."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth

from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu


def _lora(inp, t, s, base):
    W = dev_bf16(inp["W_" + t])
    return L.Lora(L.nf4_pack(W) if base == "nf4" else W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), s)


@pytest.mark.parametrize("base", ["bf16", "nf4"])
def test_mlp_step_replays_from_a_cuda_graph(base):
    w = synth.mlp_workload("graph", 1000, 256, 704, 16, 32.0, act="geglu")
    inp = synth.make_inputs(w, seed=101)
    gate, up, down = (_lora(inp, t, w.s, base) for t in ("gate", "up", "down"))
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, gate, up, down, act="geglu")
    bw = L.lora_mlp_bwd(X, dY, fw, gate, up, down, act="geglu")
    grads = {k: v for k, v in bw.items() if k != "dX"}

    def step():
        L.lora_mlp_fwd(X, gate, up, down, act="geglu", y=fw["y"], e=fw["e"], u=fw["u"], h=fw["h"],
                       saved=fw["saved"], ws=fw["ws"])
        L.lora_mlp_bwd(X, dY, fw, gate, up, down, act="geglu", dX=bw["dX"], grads=grads)

    outs = [fw[k] for k in ("y", "e", "u", "h")] + list(bw.values())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):          # warm-up on the side stream the capture will use
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in outs:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    L.lm_workspace_check(fw["ws"])
    for a, b in zip(outs, eager):
        assert torch.equal(a, b)

    # new inputs in the same buffers: the replay must match an eager step on them
    inp2 = synth.make_inputs(w, seed=202)
    X.copy_(dev_bf16(inp2["X"]))
    dY.copy_(dev_bf16(inp2["dY"]))
    g.replay()
    torch.cuda.synchronize()
    replayed = [t.clone() for t in outs]
    step()
    torch.cuda.synchronize()
    for a, b in zip(outs, replayed):
        assert torch.equal(a, b)
    assert not torch.equal(replayed[0], eager[0])
