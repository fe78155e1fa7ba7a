"""Seeded synthetic inputs for the LoRA MLP / QKV / O workloads.

This module only draws random numbers and rounds them to bf16 storage; it holds
none of the method's arithmetic, so both the CUDA path and the fp64 oracle can
take their inputs from it.

Distributions (the second parameter of N(.,.) is a standard deviation):
  W ~ N(0, 0.02), A ~ U(-1/sqrt(in), 1/sqrt(in)), B ~ N(0, 0.02),
  X ~ N(0, 1), dY ~ N(0, 0.01); every tensor drawn in fp32 from its own
  numpy PCG64 stream (seed = base + tensor index) and rounded to bf16 with
  round-to-nearest-even.

Layouts follow the PEFT ``nn.Linear`` convention: W is (out, in), A is (r, in),
B is (out, r), activations are (T, features) row-major.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BASE_SEED = 1234


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bits (uint16) to fp32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal_bf16(shape, std: float, seed: int) -> np.ndarray:
    g = _rng(seed)
    x = g.standard_normal(size=shape, dtype=np.float32)
    x *= np.float32(std)
    return f32_to_bf16_bits(x)


def uniform_bf16(shape, bound: float, seed: int) -> np.ndarray:
    g = _rng(seed)
    x = g.uniform(-bound, bound, size=shape).astype(np.float32)
    return f32_to_bf16_bits(x)


def fp32_ab(w: "Workload", seed: int = 4321) -> dict:
    """fp32 LoRA parameters for every projection of ``w`` (fp32 LoRA-parameter runs): A ~
    U(+-1/sqrt(in)), B ~ N(0, 0.02), drawn in fp32 and kept in fp32 (most are not bf16 values).
    Returns ``A_<name>``, ``B_<name>`` as float32 arrays."""
    out = {}
    for i, p in enumerate(w.projs):
        out["A_" + p.name] = _rng(seed + 2 * i).uniform(-1.0 / math.sqrt(p.d_in), 1.0 / math.sqrt(p.d_in),
                                                        size=(w.r, p.d_in)).astype(np.float32)
        out["B_" + p.name] = (_rng(seed + 2 * i + 1).standard_normal(size=(p.d_out, w.r), dtype=np.float32)
                              * np.float32(0.02))
    return out


@dataclass
class ProjSpec:
    """One LoRA projection: out = X W^T + s (X A^T) B^T, W (out, in)."""
    name: str
    d_in: int
    d_out: int


@dataclass
class Workload:
    """A named workload: the projections of one block plus the token count."""
    name: str
    kind: str            # "mlp", "relu2", "qkv", "o"
    T: int
    r: int
    alpha: float
    projs: list = field(default_factory=list)
    act: str = "swiglu"  # mlp only: "swiglu" or "geglu"
    nf4: bool = False
    ab_f32: bool = False  # LoRA A, B passed as fp32 parameters
    int4_group: int = 0   # > 0: groupwise int4 base with groups of this many elements
    nvfp4: bool = False   # NVFP4 weight-only base

    @property
    def s(self) -> float:
        return self.alpha / self.r


def mlp_workload(name, T, d, n, r, alpha, act="swiglu", nf4=False) -> Workload:
    return Workload(name, "mlp", T, r, alpha,
                    [ProjSpec("gate", d, n), ProjSpec("up", d, n), ProjSpec("down", n, d)],
                    act=act, nf4=nf4)


def relu2_workload(name, T, d, n, r, alpha, nf4=False) -> Workload:
    """Non-gated ReLU^2 MLP: up (d -> n) and down (n -> d) projections."""
    return Workload(name, "relu2", T, r, alpha, [ProjSpec("up", d, n), ProjSpec("down", n, d)], act="relu2",
                    nf4=nf4)


def qkv_workload(name, T, d, q, kv, r, alpha, nf4=False, v=None) -> Workload:
    """Q (d -> q), K (d -> kv) and V (d -> kv, or d -> v when given)."""
    return Workload(name, "qkv", T, r, alpha,
                    [ProjSpec("q", d, q), ProjSpec("k", d, kv), ProjSpec("v", d, kv if v is None else v)], nf4=nf4)


def o_workload(name, T, d_in, d_out, r, alpha, nf4=False) -> Workload:
    return Workload(name, "o", T, r, alpha, [ProjSpec("o", d_in, d_out)], nf4=nf4)


# The workloads the benchmark and the parity tests use.
WORKLOADS = {
    "tiny_mlp_swiglu": mlp_workload("tiny_mlp_swiglu", 512, 256, 704, 8, 16.0),
    "llama3_8b_mlp_bf16": mlp_workload("llama3_8b_mlp_bf16", 8192, 4096, 14336, 16, 32.0),
    "llama3_8b_mlp_nf4": mlp_workload("llama3_8b_mlp_nf4", 8192, 4096, 14336, 16, 32.0, nf4=True),
    "llama3_8b_qkv_bf16": qkv_workload("llama3_8b_qkv_bf16", 8192, 4096, 4096, 1024, 16, 32.0),
    "llama3_8b_o_bf16": o_workload("llama3_8b_o_bf16", 8192, 4096, 4096, 16, 32.0),
    "llama3_8b_qkv_nf4": qkv_workload("llama3_8b_qkv_nf4", 8192, 4096, 4096, 1024, 16, 32.0, nf4=True),
    "llama3_8b_o_nf4": o_workload("llama3_8b_o_nf4", 8192, 4096, 4096, 16, 32.0, nf4=True),
    "llama3_70b_mlp_nf4_swiglu": mlp_workload("llama3_70b_mlp_nf4_swiglu", 4096, 8192, 28672, 64, 128.0,
                                              nf4=True),
    "llama3_70b_mlp_nf4_geglu": mlp_workload("llama3_70b_mlp_nf4_geglu", 4096, 8192, 28672, 64, 128.0,
                                             act="geglu", nf4=True),
}
# the non-gated ReLU^2 MLP at the 8B MLP sizes (the pages give no sizes for it)
WORKLOADS["tiny_relu2_mlp"] = relu2_workload("tiny_relu2_mlp", 512, 256, 704, 8, 16.0)
WORKLOADS["relu2_mlp_8b_bf16"] = relu2_workload("relu2_mlp_8b_bf16", 8192, 4096, 14336, 16, 32.0)
WORKLOADS["relu2_mlp_8b_nf4"] = relu2_workload("relu2_mlp_8b_nf4", 8192, 4096, 14336, 16, 32.0, nf4=True)
# the 8B MLP with fp32 LoRA parameters (bf16 and NF4 base)
for _b in ("bf16", "nf4"):
    _w = mlp_workload("llama3_8b_mlp_%s_ab32" % _b, 8192, 4096, 14336, 16, 32.0, nf4=_b == "nf4")
    _w.ab_f32 = True
    WORKLOADS[_w.name] = _w
# groupwise int4 base: groups of 128 (the pages' example) and of 32 (the smallest offered)
for _w in (mlp_workload("llama3_8b_mlp_int4", 8192, 4096, 14336, 16, 32.0),
           mlp_workload("llama3_8b_mlp_int4_g32", 8192, 4096, 14336, 16, 32.0),
           qkv_workload("llama3_8b_qkv_int4", 8192, 4096, 4096, 1024, 16, 32.0),
           o_workload("llama3_8b_o_int4", 8192, 4096, 4096, 16, 32.0),
           relu2_workload("relu2_mlp_8b_int4", 8192, 4096, 14336, 16, 32.0)):
    _w.int4_group = 32 if _w.name.endswith("_g32") else 128
    WORKLOADS[_w.name] = _w
# NVFP4 weight-only base
for _w in (mlp_workload("llama3_8b_mlp_nvfp4", 8192, 4096, 14336, 16, 32.0),
           qkv_workload("llama3_8b_qkv_nvfp4", 8192, 4096, 4096, 1024, 16, 32.0),
           o_workload("llama3_8b_o_nvfp4", 8192, 4096, 4096, 16, 32.0),
           relu2_workload("relu2_mlp_8b_nvfp4", 8192, 4096, 14336, 16, 32.0)):
    _w.nvfp4 = True
    WORKLOADS[_w.name] = _w


def make_inputs(w: Workload, seed: int = BASE_SEED, zero_W: bool = False, zero_B: bool = False,
                zero_A: bool = False) -> dict:
    """Draw every input of workload ``w`` as bf16 bits (numpy uint16).

    Returns a dict with X (T, d_in of the first projection), dY (T, d_out of the
    last projection; for qkv one dY per projection) and per projection
    ``W_<name>``, ``A_<name>``, ``B_<name>``.
    """
    out = {}
    idx = 0

    def nxt():
        nonlocal idx
        idx += 1
        return seed + idx

    first, last = w.projs[0], w.projs[-1]
    out["X"] = normal_bf16((w.T, first.d_in), 1.0, nxt())
    for p in w.projs:
        sW, sA, sB = nxt(), nxt(), nxt()
        out["W_" + p.name] = (np.zeros((p.d_out, p.d_in), np.uint16) if zero_W
                              else normal_bf16((p.d_out, p.d_in), 0.02, sW))
        out["A_" + p.name] = (np.zeros((w.r, p.d_in), np.uint16) if zero_A
                              else uniform_bf16((w.r, p.d_in), 1.0 / math.sqrt(p.d_in), sA))
        out["B_" + p.name] = (np.zeros((p.d_out, w.r), np.uint16) if zero_B
                              else normal_bf16((p.d_out, w.r), 0.02, sB))
    if w.kind == "qkv":
        for p in w.projs:
            out["dY_" + p.name] = normal_bf16((w.T, p.d_out), 0.01, nxt())
    else:
        out["dY"] = normal_bf16((w.T, last.d_out), 0.01, nxt())
    return out


def scaled_workload(w: Workload, T: int | None = None, shrink: int = 1) -> Workload:
    """A copy of ``w`` with T replaced and every feature size divided by ``shrink``."""
    import copy
    w2 = copy.deepcopy(w)
    if T is not None:
        w2.T = T
    if shrink != 1:
        for p in w2.projs:
            p.d_in //= shrink
            p.d_out //= shrink
    return w2
