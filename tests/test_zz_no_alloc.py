"""lora_o_bwd_static, the entry point for callers that must not allocate device memory (for
example a plugin whose host framework owns the device memory pool, or a process under a hard
device-memory cap): its scratch is a fixed device array inside the library instead of a
caller-provided workspace.  Checked through the C ABI on two calls in a row (the array keeps the
previous call's contents): bit for bit against lora_o_bwd on the same inputs (the same kernels run
in the same order), element by element against the fp64 oracle, its error word read back clean
with lm_static_scratch_check, and across a call made after the first one neither a fall of the
device's free memory nor a rise of torch's allocated bytes.  This file is collected last so that a run stopping at its
first failure has already run every other test."""
import ctypes
import gc

import pytest
import torch

from bwd_lora_mlp_gb300 import build as B
from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import lora as O

from gpu_util import check, dev_bf16, host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    L.load()


def _static_call(X, dY, saved, o, dX, dA, dB):
    T, d_in = X.shape
    d_out = o.W.shape[0]
    Lc = o.c_struct()
    st = L.call_status("lora_o_bwd_static", T, d_in, d_out, X.data_ptr(), dY.data_ptr(), saved.data_ptr(),
                       saved.numel(), ctypes.byref(Lc), dX.data_ptr(), dA.data_ptr(), dB.data_ptr(),
                       torch.cuda.current_stream().cuda_stream)
    assert st == L.LM_OK, L.last_error()


def _usage():
    gc.collect()
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()


def _scratch_check():
    st = L.call_status("lm_static_scratch_check", torch.cuda.current_stream().cuda_stream)
    assert st == L.LM_OK, L.last_error()


@pytest.mark.parametrize("T,din,dout,r", [(300, 256, 192, 16), (1000, 512, 384, 64)])
def test_static_scratch_matches_workspace_entry_point(T, din, dout, r):
    w = synth.o_workload("o", T, din, dout, r, 2.0 * r)
    inp = synth.make_inputs(w, seed=41)
    o = L.Lora(dev_bf16(inp["W_o"]), dev_bf16(inp["A_o"]), dev_bf16(inp["B_o"]), w.s)
    X, dY = dev_bf16(inp["X"]), dev_bf16(inp["dY"])
    fw = L.lora_o_fwd(X, o)
    ref = L.lora_o_bwd(X, dY, fw, o)
    L.lm_workspace_check(fw["ws"])
    Xo, dYo = O.from_bf16(inp["X"]), O.from_bf16(inp["dY"])
    W, A, Bm = (O.from_bf16(inp[k]) for k in ("W_o", "A_o", "B_o"))
    g = O.lora_w_backward(Xo, dYo, W, A, Bm, w.s)
    outs = [{k: torch.full_like(ref[k], float("nan")) for k in ("dX", "dA", "dB")} for _ in range(2)]
    torch.cuda.synchronize()
    usage = []
    for i in range(2):
        usage.append(_usage())
        out = outs[i]
        _static_call(X, dY, fw["saved"], o, out["dX"], out["dA"], out["dB"])
        torch.cuda.synchronize()
        _scratch_check()
        for k in ("dX", "dA", "dB"):
            assert torch.equal(out[k], ref[k]), k
        check("dX", host64(out["dX"]), g["dX"])
        check("dA", host64(out["dA"]), g["dA"])
        check("dB", host64(out["dB"]), g["dB"])
    # the second call allocated nothing: neither the device's free memory fell nor torch's
    # allocated bytes grew across it (garbage left by earlier tests is collected before each
    # reading, so only a fall of the allocated bytes is possible otherwise)
    free_after, alloc_after = _usage()
    assert free_after >= usage[1][0] and alloc_after <= usage[1][1], (usage[1], (free_after, alloc_after))


def test_static_scratch_rejects_shapes_beyond_its_size():
    T, din, dout, r = 1 << 20, 4096, 4096, 64
    need = ctypes.c_size_t(0)
    assert L.call_status("lora_o_workspace_size", T, din, dout, r, ctypes.byref(need)) == L.LM_OK
    assert need.value > 64 << 20
    o = L.lm_lora()
    o.W.kind, o.W.rows, o.W.cols, o.W.w = L.LM_WEIGHT_BF16, dout, din, 1 << 32
    o.A, o.B, o.r, o.s = 1 << 33, 1 << 34, r, 2.0
    st = L.call_status("lora_o_bwd_static", T, din, dout, 1 << 35, 1 << 36, 1 << 37, 1 << 30, ctypes.byref(o),
                       1 << 38, 1 << 39, 1 << 40, None)
    assert st == L.LM_ERR_WORKSPACE
    assert "static scratch" in L.last_error()
