"""bench.py's output contract on a GPU: one JSON line with the metric, the
roofline and relayout objects, the pipelined end-to-end leg (whose host copy
of the result must equal the device result) and the launch count."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [line for line in out.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.gpu
def test_attention_workload_line():
    d = run_bench("--workload", "tiny", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-clocks")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "roofline", "relayout", "gpu_launches", "e2e"):
        assert key in d, key
    assert d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["steps"] == 3 and d["n_gpus"] == 1 and d["scaling"] == "weak"
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["achieved"] > 0 and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], abs=1e-4)  # rounded to 4 places
    assert d["gpu_launches"] > 0
    e = d["e2e"]
    assert e["readback_verified"] is True
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0 and e["value"] > 0
    # the layout-only workload beside the attention line: U = 4 pack + all-to-all + unpack
    p = d["pack"]
    assert p["workload"] == "pack" and p["unit"] == "GB/s" and p["bound"] == "hbm" and p["achieved"] > 0
    assert p["frac"] == pytest.approx(p["achieved"] / p["peak"], abs=1e-4)
    # the packs and the unpacks each read and write the 75.5 MB of all ranks' Q/K/V once
    assert p["algorithmic_bytes"] == {"pack": 2 * 3 * 4 * 1024 * 24 * 128 * 2, "unpack": 2 * 3 * 4 * 1024 * 24 * 128 * 2}
    assert p["gpu_launches_per_set"] == {"pack": 4, "unpack": 4}
    # the interleaved staging layout, timed the same way
    assert p["staging_layout"] == "tqkv" and p["staging"] == [4, 3, 1, 1024, 6, 128]
    pi = p["interleaved"]
    assert pi["staging"] == [4, 1, 1024, 6, 384] and pi["achieved"] > 0 and pi["pack_gbs"] > 0
    assert p["pack_gbs"] > 0 and p["unpack_gbs"] > 0 and p["step_gbs"] > 0 and p["copy_gbs"] > 0
    assert p["copy_per_rank_gbs"] > 0


@pytest.mark.gpu
def test_masked_workload_line():
    # the Qwen-like layer: the key-mask merge runs in the step, FLOPs count the valid keys only
    d = run_bench("--workload", "qwen", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-clocks",
                  "--no-pack")
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and "pack" not in d
    assert d["roofline"]["algorithmic_flops_per_launch"] < 4.0 * 24 * 4096 * 4352 * 128
    assert d["e2e"]["readback_verified"] is True


@pytest.mark.gpu
def test_layout_workload_line():
    d = run_bench("--workload", "pack", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-clocks")
    assert d["unit"] == "GB/s" and d["value"] > 0
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["workload"] == "pack" and d["value"] == r["achieved"]
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], abs=1e-4)
    assert "write-back inside the timed region" in r["timing"]
    assert d["step"]["bound"] == "hbm"   # the in-step figure, kept beside it
    assert d["config"]["l2"] == "flushed_between_steps"
    assert d["e2e"]["readback_verified"] is True
    assert d["e2e"]["unit"] == "GB/s"


@pytest.mark.gpu
def test_layout_workload_line_interleaved():
    d = run_bench("--workload", "pack", "--layout", "interleaved", "--steps", "3", "--warmup", "3",
                  "--no-cpu-baseline", "--no-clocks")
    r = d["roofline"]
    assert d["config"]["staging_layout"] == "interleaved"
    assert r["staging_layout"] == "interleaved" and r["staging"] == [4, 1, 1024, 6, 384]
    assert d["value"] == r["achieved"] > 0 and r["tqkv"]["staging"] == [4, 3, 1, 1024, 6, 128]
    assert d["e2e"]["readback_verified"] is True


@pytest.mark.gpu
def test_attention_output_two_copies():
    # U = 1: the attention output of one copy of the layer is read back while the other computes
    d = run_bench("--workload", "wan480", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-clocks")
    assert "two copies of the layer" in d["e2e"]["pipeline"]
    assert d["e2e"]["readback_verified"] is True
    assert d["roofline"]["algorithmic_flops_per_launch"] == pytest.approx(4.0 * 12 * 32760 * 32760 * 128)


@pytest.mark.gpu
def test_single_attention_call_line():
    # --kernel attn: one call of a given shape, L2 flushed before every timed launch
    d = run_bench("--kernel", "attn", "--attn-shape", "1,300,700,3,128", "--dtype", "fp16", "--steps", "3",
                  "--warmup", "3", "--no-cpu-baseline", "--no-clocks")
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["dtype"] == "fp16"
    assert d["config"]["l2"] == "flushed_between_steps"
    assert d["roofline"]["algorithmic_flops_per_launch"] == pytest.approx(4.0 * 3 * 300 * 700 * 128)
    assert d["e2e"]["h2d_bytes_per_step"] == 2 * 128 * 3 * (300 + 2 * 700)


@pytest.mark.gpu
def test_varlen_line_pipelined_e2e():
    # packed varlen documents: eight ranks' remap + attention; the e2e leg double-buffers
    d = run_bench("--kernel", "varlen", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-clocks")
    assert d["config"]["workload"] == "varlen" and d["value"] > 0
    assert d["e2e"]["readback_verified"] is True and "two buffer sets" in d["e2e"]["pipeline"]
    assert d["e2e"]["h2d_bytes_per_step"] == 3 * 32768 * 12 * 128 * 2
    assert d["one_rank"]["balanced_tflops"] > 0
