"""bench.py's JSON line, assembled on CPU: the GPU timing is replaced by a
stand-in result, so a change to the line (a key it reads, a field it writes)
is caught before a GPU run."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_default_line_has_the_contract_fields(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    fake = {"ms": 0.04, "e2e_ms": 0.045, "launches": 2, "kernel": "k", "copies": 2,
            "spot_ok": True, "h2d": 1064960, "d2h": 1105920, "l2": 132 << 20,
            "e2e_zero_copy": True, "e2e_same": True, "planes": True,
            "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}}
    monkeypatch.setattr(bench, "time_gpu", lambda args, wl: dict(fake))
    per = [{"config": "q4_0_gemv_960x960", "linear": "gemv", "path": "stream", "us": 3.0,
            "frac": 0.03},
           {"config": "qwen2.5_3b_ffn_q4_0_M64", "linear": "l", "path": "mma", "us": 9.0,
            "frac": 0.3, "tensor_pipe": {"frac_of_bf16_peak": 0.2}}]
    dep = {"workload": "w", "ms_per_step": 0.2, "calls_per_step": 128, "frac": 0.13}
    monkeypatch.setattr(bench, "time_per_config", lambda device, l2, stream: list(per))
    monkeypatch.setattr(bench, "time_dependent_step",
                        lambda device, l2, stream, steps, warmup: dict(dep))
    monkeypatch.setattr(bench, "time_step_x_int8",
                        lambda device, l2, stream, steps, warmup: {"ms_per_step": 0.03})
    import torch
    monkeypatch.setattr(torch.cuda, "Stream", lambda device=None: None)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--no-cpu-baseline", "--steps", "5",
                                      "--warmup", "3"])
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main()
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["steps"] == 5 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["gpu_launches"] == 10
    assert line["dtype"] == "int32+fp32"
    assert abs(line["ms_per_step"] - 0.04) < 1e-12
    assert abs(line["value"] - 179118080 / 40e-6 / 1e9) < 1e-6  # whole-step GB/s
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in line["roofline"], key
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] == 1064960 and e2e["d2h_bytes_per_step"] == 1105920
    assert e2e["matches_device_buffers"] is True
    assert line["config"]["workload"] == "smollm2_360m_q4_0_decode_stack_32L"
    # every other workload and the layer-order decode step ride on the same line
    assert [p["config"] for p in line["per_config"]] == [p["config"] for p in per]
    assert line["per_config"][1]["tensor_pipe"]["frac_of_bf16_peak"] == 0.2
    assert line["decode_step_layer_order"]["calls_per_step"] == 128
    assert line["decode_step_x_int8"]["ms_per_step"] == 0.03
