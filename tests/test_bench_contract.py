"""bench.py's output contract: one JSON line with the fields the measurement
protocol needs. The reference arm (the float64 oracle on the host cores) runs
on CPU; the GPU arm is checked on a short run."""
import io
import json
import contextlib

import pytest

import bench


def _line(argv):
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.main(argv) == 0
    return json.loads(buf.getvalue().strip().splitlines()[-1])


def test_reference_arm_line():
    d = _line(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("gpt2s_bf16")


def test_reference_arm_times_fwd_and_bwd_apart():
    d = _line(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    cb = d["cpu_baseline"]
    assert cb["fwd_tflops"] > 0 and cb["bwd_tflops"] > 0
    # fwd+bwd rate lies between the two separate rates
    assert min(cb["fwd_tflops"], cb["bwd_tflops"]) <= d["value"] <= max(cb["fwd_tflops"], cb["bwd_tflops"])
    assert "heads in order" in cb["sample"]


def test_gpus_flag_launch_plan():
    """--gpus N starts N ranks itself, runs as it is under torch.distributed.run
    with a matching WORLD_SIZE, and refuses a mismatched one."""
    assert bench.launch_plan(1, {}) == ("run", None)
    how, argv = bench.launch_plan(4, {})
    assert how == "spawn" and "--nproc-per-node=4" in argv and "127.0.0.1" in argv
    assert bench.launch_plan(4, {"WORLD_SIZE": "4"}) == ("run", None)
    how, why = bench.launch_plan(8, {"WORLD_SIZE": "2"})
    assert how == "refuse" and "WORLD_SIZE=2" in why
    assert bench.launch_plan(0, {})[0] == "refuse"


def test_mismatched_world_size_is_refused(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "4", "--steps", "1", "--warmup", "3"])


def test_warmup_below_three_is_refused():
    with pytest.raises(SystemExit):
        bench.main(["--steps", "1", "--warmup", "2"])


@pytest.mark.gpu
def test_gpu_arm_line():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _line(["--steps", "3", "--warmup", "3", "--no-cpu-baseline"])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["value"] > 0 and d["gpu_launches"] > 0
    r = d["roofline"]
    assert r["bound"] == "tensor" and 0 < r["frac"] < 1.5 and r["unit"] == "TFLOP/s"
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert set(d["kernels"]) == {"attn_fwd_kernel", "attn_bwd_pre", "attn_bwd_kernel", "attn_bwd_dq_out"}
