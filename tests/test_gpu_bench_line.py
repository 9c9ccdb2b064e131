"""bench.py's JSON line on a short run: every key the benchmark contract asks
for is present and consistent (a format check; the numbers are the bench's)."""
from __future__ import annotations

import contextlib
import io
import json

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("mode", ["fused", "deferred"])
def test_bench_line_keys(mode):
    import bench

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--layers", "2", "--steps", "5", "--warmup", "3", "--no-cpu-baseline", "--mode", mode])
    d = json.loads(buf.getvalue().strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["config"]["mode"] == mode
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 2 * 2 * 5  # two kernels per layer call, two layers, five timed steps
