"""Bit-exact check of the in-GEMM decoders of every packed base (NF4, int4 for each group size,
NVFP4), in both operand layouts.

With X = I, B = 0 and dY = I, the LoRA O projection computes Y = X W^T = W^T (forward: the weight
read K-major) and dX = dY W = W (input gradient: the weight read MN-major).  Every output element
is a single product of a decoded bf16 weight and 1 accumulated in fp32 with zeros, so it must
equal the oracle's bf16 reconstruction of that weight element bit for bit: any decode slip (a
swapped nibble, a scale of the wrong block, a rounding difference) shows as a mismatch."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import int4 as oi4
from oracle import nf4 as onf4
from oracle import nvfp4 as onv

from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

N = 512   # d_in = d_out = T


def _weight_bits(seed):
    x = synth.bf16_bits_to_f32(synth.normal_bf16((N, N), 0.02, seed)).reshape(N, N).copy()
    x[7, :64] += 0.5        # a block or group far from the others
    x[9, 64:128] = 0.0      # a zero block
    x = oi4.bf16_round(x.astype(np.float32))
    return x, oi4.bf16_bits(x)


def _oracle_bf16_bits(fmt, x):
    if fmt == "nf4":
        codes, q, c = onf4.quantize(x.reshape(-1))
        w = onf4.dequantize_bf16(codes, q, c).reshape(N, N)
    elif fmt == "nvfp4":
        codes, sb, sg, _ = onv.quantize(x)
        w = onv.dequantize_bf16(codes, sb, sg, N, N)
    else:
        g = int(fmt[5:])
        codes, s, z, _ = oi4.quantize(x, g)
        w = oi4.dequantize_bf16(codes, s, z, N, N, g)
    return oi4.bf16_bits(w)


def _pack(fmt, Wd):
    if fmt == "nf4":
        return L.nf4_pack(Wd)
    if fmt == "nvfp4":
        return L.nvfp4_pack(Wd)
    return L.int4_pack(Wd, int(fmt[5:]))


def _bits(t):
    return _plus_zero(t.view(torch.int16).cpu().numpy().view(np.uint16))


def _plus_zero(b):
    # a decoded -0 (NVFP4 keeps the sign of a zero code) leaves the fp32 accumulator as +0
    return np.where(b == 0x8000, 0, b).astype(np.uint16)


@pytest.mark.parametrize("fmt", ["nf4", "int4_32", "int4_64", "int4_128", "int4_256", "nvfp4"])
def test_decoded_weight_is_exact_in_both_layouts(fmt):
    x, bits = _weight_bits(17)
    want = _plus_zero(_oracle_bf16_bits(fmt, x))
    Wq = _pack(fmt, dev_bf16(bits))
    eye = torch.eye(N, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((16, N), dtype=torch.bfloat16, device="cuda")
    A[0, 0] = 1.0                                   # any A: B = 0 removes the LoRA term exactly
    B = torch.zeros((N, 16), dtype=torch.bfloat16, device="cuda")
    o = L.Lora(Wq, A, B, 2.0)
    f = L.lora_o_fwd(eye, o)
    b = L.lora_o_bwd(eye, eye, f, o)
    L.lm_workspace_check(f["ws"])
    torch.cuda.synchronize()
    assert np.array_equal(_bits(f["Y"]), want.T), "forward (K-major) decode differs"
    assert np.array_equal(_bits(b["dX"]), want), "input-gradient (MN-major) decode differs"
