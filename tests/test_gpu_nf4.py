"""GPU nf4_pack / nf4_dequant against the NF4 oracle: bytes and fp32 values bit-exact."""
import numpy as np
import pytest
import torch

from bwd_lora_mlp_gb300 import lib as L
from bwd_lora_mlp_gb300 import synth
from oracle import nf4 as onf4

from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu


def _weight_bits(rows, cols, seed):
    return synth.normal_bf16((rows, cols), 0.02, seed)


def _check_pack(bits):
    Wd = dev_bf16(bits)
    pk = L.nf4_pack(Wd)
    f32 = L.nf4_dequant(pk, torch.float32)
    b16 = L.nf4_dequant(pk, torch.bfloat16)
    torch.cuda.synchronize()
    x = synth.bf16_bits_to_f32(bits).reshape(-1)
    codes, q, c = onf4.quantize(x)
    assert np.array_equal(pk.codes.cpu().numpy(), codes)
    assert np.array_equal(pk.absmax_q.cpu().numpy(), q)
    assert np.array_equal(pk.group_scale.cpu().numpy().view(np.uint32), c.view(np.uint32))
    ref = onf4.dequantize(codes, q, c)
    assert np.array_equal(f32.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    refb = onf4.dequantize_bf16(codes, q, c)
    got_b = b16.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    assert np.array_equal(got_b, refb.view(np.uint32))


def test_pack_dequant_bit_exact_random():
    _check_pack(_weight_bits(256, 512, 1))


def test_pack_zero_blocks_zero_groups_and_block_maxima():
    """All-zero blocks and groups, negative zero, and blocks whose maximum sits at either sign.
    (Exact ties between two codes cannot arise from bf16 inputs normalised by a bf16 absmax
    except by rare coincidence; the tie rule is pinned on the oracle side.)"""
    bits = _weight_bits(64, 1024, 2)
    x = synth.bf16_bits_to_f32(bits).reshape(-1).copy()
    x[64:128] = 0.0                 # an all-zero block
    x[16384:32768] = 0.0            # an all-zero group
    x[40000] = -0.0
    x[50000] = -1.0                 # block maximum with a negative sign
    x[50001] = 1.0
    _check_pack(synth.f32_to_bf16_bits(x).reshape(bits.shape))


def test_pack_every_group_of_a_full_size_weight():
    """A 14336 x 4096 weight (the Llama-3-8B gate projection): every code byte, block scale, group
    scale and dequantised value of all 3584 groups, bit for bit."""
    rows, cols = 14336, 4096
    bits = _weight_bits(rows, cols, 3)
    pk = L.nf4_pack(dev_bf16(bits))
    deq = L.nf4_dequant(pk, torch.float32)
    torch.cuda.synchronize()
    x = synth.bf16_bits_to_f32(bits).reshape(-1)
    codes, q, c = onf4.quantize(x)
    assert np.array_equal(pk.codes.cpu().numpy(), codes)
    assert np.array_equal(pk.absmax_q.cpu().numpy(), q)
    assert np.array_equal(pk.group_scale.cpu().numpy().view(np.uint32), c.view(np.uint32))
    assert np.array_equal(deq.cpu().numpy().view(np.uint32), onf4.dequantize(codes, q, c).view(np.uint32))
