"""Host checks of bench.py's arithmetic: the algorithmic flop counts behind every TFLOP/s and
roofline figure it prints agree with the oracle's own counts, and the per-kernel counts of the
four base GEMMs of the MLP add up to the block's six base GEMMs plus their rank-r terms."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from bwd_lora_mlp_gb300 import synth  # noqa: E402
from oracle import lora as O  # noqa: E402


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_workload_flops_match_the_oracle(name):
    w = synth.WORKLOADS[name]
    T, r = w.T, w.r
    if w.kind == "mlp":
        want = O.mlp_flops(T, w.projs[0].d_in, w.projs[0].d_out, r)
    elif w.kind == "relu2":
        want = O.relu2_mlp_flops(T, w.projs[0].d_in, w.projs[0].d_out, r)
    else:
        want = sum(O.lora_proj_flops(T, p.d_in, p.d_out, r) for p in w.projs)
    assert bench.workload_flops(w) == want


def test_base_gemm_kernel_flops_cover_the_six_base_gemms():
    w = synth.WORKLOADS["llama3_8b_mlp_bf16"]
    T, d, n, r = w.T, 4096, 14336, w.r
    tags = ("mlp.gateup", "mlp.down", "mlp.dh", "mlp.dX")
    total = sum(bench.kernel_flops(t, w) for t in tags)
    # 6 base GEMMs of 2 T d n each; the rank-r (XA) B^T of gate, up, down in the forward, G_d A_d
    # inside dh, and G_g A_g + G_u A_u inside dX: 2 T r per output column each
    assert total == 12 * T * d * n + 2 * T * r * (2 * n + d + n + 2 * d)
    assert 5.8e12 < bench.workload_flops(w) < 5.83e12       # 710 MFLOP per token at the 8B sizes


def test_step_roofline_fractions():
    peaks, src = bench.load_peaks()
    r = bench.step_roofline(1600.0, peaks, src)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["peak"] == peaks["bf16_tflops"]                      # the headline: burst
    assert abs(r["frac"] * peaks["bf16_tflops"] - 1600.0) < 1e-9
    assert r["frac_of_burst"] == r["frac"]
    assert abs(r["frac_of_sustained"] * peaks["bf16_tflops_sustained"] - 1600.0) < 1e-9
    assert abs(r["frac_of_nominal"] - 1600.0 / 2250.0) < 1e-12
    assert r["frac_of_nominal"] < r["frac"] <= r["frac_of_sustained"]


def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on(monkeypatch):
    rec = bench.committed_traffic("mlp.gateup", "llama3_8b_mlp_bf16")
    assert rec is None or rec > 10 ** 9          # a full-size launch moves over a GB
    monkeypatch.setattr(bench, "src_digest", lambda: "0000000000000000")
    assert bench.committed_traffic("mlp.gateup", "llama3_8b_mlp_bf16") is None
    assert bench.committed_traffic("mlp.unknown", "llama3_8b_mlp_bf16") is None


def test_source_digest_ignores_comments(tmp_path, monkeypatch):
    src = tmp_path / "bwd_lora_mlp_gb300" / "csrc"
    src.mkdir(parents=True)
    names = ("lm_gemm.cuh", "lm_gemm2.cuh", "lm_gemm2_nf4.cuh", "lm_ptx.cuh")
    for n in names:
        (src / n).write_text("int a = 1;  // one\n\n// note\nint b = 2;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.src_digest()
    (src / names[0]).write_text("int a = 1;  // changed comment\n// another note\nint b = 2;   \n")
    assert bench.src_digest() == d0
    (src / names[0]).write_text("int a = 3;\nint b = 2;\n")
    assert bench.src_digest() != d0
