"""Plain, slow, fp64 CPU oracle for the fused LoRA MLP / QKV / O block and NF4.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this package: only the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline / reference leg use it.  It shares no code with the CUDA path; the
one thing both sides take from a common place is the seeded input generator
(``bwd_lora_mlp_gb300.synth``), which holds none of the method's arithmetic.

Sources (web pages the method is described on):
  * "LoRA Optimizations" (docs.axolotl.ai, lora_optims): the LoRA MLP / QKV / O
    autograd functions, SwiGLU / GeGLU activation kernels, FP32 LoRA gradients.
  * "Avoid recomputing LoRA B-projected gradient in fused-LoRA backward"
    (unsloth fast_lora diff): the backward of LoRA_MLP, LoRA_QKV, LoRA_W and
    matmul_lora, with the dY.B^T hoist.
  * "loralei" README, QLoRA section: NF4 base weights, block 64, scaler block 256,
    double-scale reconstruction; the groupwise int4 base (groups 32 to 256).
  * "LoRA Optimizations", FP32 LoRA gradients: weight-only NVFP4 bases (E2M1 codes, E4M3
    scales per 16 elements, one fp32 scale per tensor).

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (finite differences, closed forms, the merge
identity, NF4 invariants, the published NF4 table, int4 and NVFP4 grid round
trips and nearest-level checks, E4M3 against PyTorch's float8 conversion, the
adapter parameter count printed on the "LoRA Optimizations" page).  No function is "parity unpinned".
"""
