"""The bounded-wait timeout path of every GEMM kernel family, made to run out without a fault.

lm_debug_inject makes the TMA producers of one kernel family issue no loads at all, so no copy is in
flight, and shortens every pipeline wait to 50 ms: the consumers' waits run out, the kernels
record LM_ERR_TIMEOUT (with their family) in the workspace's error word, drain what they issued,
free their tensor memory and return, and lm_workspace_check reports the status.  The same call
made again with the switch off must then match the fp64 oracle: the context stays usable.
Families: 1 the split-K rank-r kernel, 2 the bf16 CTA-pair kernel (gate/up, dh of a bf16 base),
3 the packed-base CTA-pair kernel (down and dX of every base; gate/up and dh of an NF4 base, whose
decode warps and staged dh epilogue then time out too), 4 the dual rank-r reduction (forced onto
this small case by the hook's flag 16)."""
import ctypes

import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import lora as O
from oracle import nf4 as onf4

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu

WAIT_NS = 50_000_000


def _inject(mask, wait_ns):
    assert L.call_status("lm_debug_inject", mask, wait_ns) == L.LM_OK


def _mlp(base, act="swiglu"):
    w = synth.mlp_workload("timeout", 300, 256, 512, 16, 32.0, act=act)
    inp = synth.make_inputs(w, seed=101)
    Ls = {}
    for t in ("gate", "up", "down"):
        W = dev_bf16(inp["W_" + t])
        Ls[t] = L.Lora(L.nf4_pack(W) if base == "nf4" else W, dev_bf16(inp["A_" + t]), dev_bf16(inp["B_" + t]), w.s)
    return w, inp, Ls


def _step(inp, Ls, act):
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_mlp_fwd(X, Ls["gate"], Ls["up"], Ls["down"], act=act)
    bw = L.lora_mlp_bwd(X, dY, fw, Ls["gate"], Ls["up"], Ls["down"], act=act)
    return fw, bw


@pytest.mark.parametrize("base,mask,family", [("bf16", 1, 1), ("bf16", 2, 2), ("bf16", 4, 3), ("nf4", 4, 3),
                                              ("bf16", 8 | 16, 4)])
def test_starved_family_reports_timeout_then_recovers(base, mask, family):
    w, inp, Ls = _mlp(base)
    _inject(mask, WAIT_NS)
    try:
        fw, bw = _step(inp, Ls, w.act)
    finally:
        _inject(0, 0)
    with pytest.raises(L.LmError) as ei:
        L.lm_workspace_check(fw["ws"])
    assert ei.value.status == L.LM_ERR_TIMEOUT
    assert "kernel family %d" % family in str(ei.value)
    L.lm_workspace_check(fw["ws"])  # the check cleared the word
    # the same call again, normally: the context is usable and the results are right
    fw, bw = _step(inp, Ls, w.act)
    L.lm_workspace_check(fw["ws"])
    p = {}
    for t, k in (("gate", "g"), ("up", "u"), ("down", "d")):
        if base == "bf16":
            p["W" + k] = O.from_bf16(inp["W_" + t])
        else:
            x = synth.bf16_bits_to_f32(inp["W_" + t]).reshape(-1)
            p["W" + k] = onf4.dequantize_bf16(*onf4.quantize(x)).astype("float64").reshape(inp["W_" + t].shape)
        p["A" + k] = O.from_bf16(inp["A_" + t])
        p["B" + k] = O.from_bf16(inp["B_" + t])
        p["s" + k] = w.s
    ref = O.mlp_backward(O.from_bf16(inp["X"]), O.from_bf16(inp["dY"]), p, w.act)
    check("y", host64(fw["y"]), ref["y"])
    check("dX", host64(bw["dX"]), ref["dX"])
    check("dA_gate", host64(bw["dA_gate"]), ref["dAg"])
    check("dB_down", host64(bw["dB_down"]), ref["dBd"])


def test_static_scratch_timeout_is_read_back():
    """lora_o_bwd_static's kernels report a timeout through lm_static_scratch_check."""
    w = synth.o_workload("o", 200, 256, 256, 16, 32.0)
    inp = synth.make_inputs(w, seed=43)
    o = L.Lora(dev_bf16(inp["W_o"]), dev_bf16(inp["A_o"]), dev_bf16(inp["B_o"]), w.s)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_o_fwd(X, o)
    L.lm_workspace_check(fw["ws"])
    dX = torch.empty_like(X)
    dA = torch.empty((o.r, X.shape[1]), dtype=torch.float32, device="cuda")
    dB = torch.empty((o.W.shape[0], o.r), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        Lc = o.c_struct()
        st = L.call_status("lora_o_bwd_static", X.shape[0], X.shape[1], o.W.shape[0], X.data_ptr(), dY.data_ptr(),
                           fw["saved"].data_ptr(), fw["saved"].numel(), ctypes.byref(Lc), dX.data_ptr(),
                           dA.data_ptr(), dB.data_ptr(), stream)
        assert st == L.LM_OK, L.last_error()

    _inject(1, WAIT_NS)
    try:
        call()
    finally:
        _inject(0, 0)
    assert L.call_status("lm_static_scratch_check", stream) == L.LM_ERR_TIMEOUT
    assert "kernel family 1" in L.last_error()
    call()
    assert L.call_status("lm_static_scratch_check", stream) == L.LM_OK, L.last_error()
    ref = L.lora_o_bwd(X, dY, fw, o)
    L.lm_workspace_check(fw["ws"])
    assert torch.equal(dX, ref["dX"]) and torch.equal(dA, ref["dA"]) and torch.equal(dB, ref["dB"])
