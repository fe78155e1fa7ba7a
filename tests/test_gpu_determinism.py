"""Bitwise reproducibility and stream placement of the QKV, O and ReLU² entry points (the MLP's are
in test_gpu_mlp.py): the same call twice gives the same bits (every reduction has a fixed order),
and the same call issued on a side stream gives the same bits as on the default stream, with the
side stream's work ordered by the stream argument alone."""
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth

from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu


def _dev(inp, t, s, base):
    W = dev_bf16(inp["W_" + t])
    return L.Lora(L.nf4_pack(W) if base == "nf4" else W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), s)


def _qkv(inp, w, base, stream=None):
    q, k, v = (_dev(inp, t, w.s, base) for t in ("q", "k", "v"))
    X = dev_bf16(inp["X"])
    fw = L.lora_qkv_fwd(X, q, k, v, stream=stream)
    bw = L.lora_qkv_bwd(X, dev_bf16(inp["dY_q"]), dev_bf16(inp["dY_k"]), dev_bf16(inp["dY_v"]), fw, q, k, v,
                        stream=stream)
    return {**{t: fw[t] for t in ("Q", "K", "V")}, **bw}


def _o(inp, w, base, stream=None):
    o = _dev(inp, "o", w.s, base)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_o_fwd(X, o, stream=stream)
    bw = L.lora_o_bwd(X, dY, fw, o, stream=stream)
    return {"Y": fw["Y"], **bw}


def _relu2(inp, w, base, stream=None):
    up, down = _dev(inp, "up", w.s, base), _dev(inp, "down", w.s, base)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_relu2_mlp_fwd(X, up, down, stream=stream)
    bw = L.lora_relu2_mlp_bwd(X, dY, fw, up, down, stream=stream)
    return {"y": fw["y"], "u": fw["u"], "h": fw["h"], **bw}


CASES = {
    "qkv": (lambda: synth.qkv_workload("detq", 640, 512, 512, 128, 16, 32.0, v=256), _qkv, 51),
    "o": (lambda: synth.o_workload("deto", 640, 512, 384, 16, 32.0), _o, 52),
    "relu2": (lambda: synth.relu2_workload("detr", 640, 256, 768, 16, 32.0), _relu2, 53),
}


@pytest.mark.parametrize("base", ["bf16", "nf4"])
@pytest.mark.parametrize("kind", sorted(CASES))
def test_bitwise_twice_and_on_a_side_stream(kind, base):
    make, run, seed = CASES[kind]
    w = make()
    inp = synth.make_inputs(w, seed=seed)
    a = run(inp, w, base)
    b = run(inp, w, base)
    torch.cuda.synchronize()
    # everything of the third call -- its uploads, allocations and workspace zeroing, and the
    # library's launches through the stream argument -- on a side stream
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        c = run(inp, w, base, stream=side)
    side.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), (k, "second call")
        assert torch.equal(a[k], c[k]), (k, "side stream")


def test_two_streams_at_once_match_sequential_calls():
    """Two MLP fwd+bwd calls with their own workspaces issued on two streams without waiting for each
    other: each gives the bits it gives when run alone (the library keeps no shared device state)."""
    def setup(seed):
        w = synth.mlp_workload("conc", 600, 256, 512, 16, 32.0)
        inp = synth.make_inputs(w, seed=seed)
        ps = {t: _dev(inp, t, w.s, "bf16") for t in ("gate", "up", "down")}
        return w, dev_bf16(inp["X"]), dev_bf16(inp["dY"]), ps

    def call(X, dY, ps, stream=None):
        fw = L.lora_mlp_fwd(X, ps["gate"], ps["up"], ps["down"], stream=stream)
        bw = L.lora_mlp_bwd(X, dY, fw, ps["gate"], ps["up"], ps["down"], stream=stream)
        return {"y": fw["y"], **bw}

    jobs = [setup(61), setup(62)]
    alone = [call(X, dY, ps) for _, X, dY, ps in jobs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    together = []
    for (_, X, dY, ps), s in zip(jobs, streams):
        with torch.cuda.stream(s):
            together.append(call(X, dY, ps, stream=s))
    for s in streams:
        s.synchronize()
    for a, b in zip(alone, together):
        for k in a:
            assert torch.equal(a[k], b[k]), k
