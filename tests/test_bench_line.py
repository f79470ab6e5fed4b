"""The bench JSON line carries every key of the measurement contract, with the
roofline and end-to-end figures derived from the timings it is given (host
logic only: the library calls that need a device are stubbed)."""
import argparse
import io
import json
from contextlib import redirect_stdout

import numpy as np

import bench
import moe_expert_layer_scan_gb300 as mm
import workloads


class FakeMoE:
    h = None

    @staticmethod
    def launches(T):
        return 4


def make_line(monkeypatch, name, per_kernel, steps=10, e2e_ms=None):
    monkeypatch.setattr(mm, "mm_token_tile_width", lambda h, T: 16)
    w = workloads.CONFIGS[name]
    idx, _ = workloads.routing(w)
    counts = np.bincount(idx[idx >= 0].ravel(), minlength=w.Ep)
    alg = bench.algorithmic(w, counts)
    args = argparse.Namespace(steps=steps, warmup=3, schedule="auto", tiles=-1, no_cpu_baseline=True)
    clk = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.report(args, w, 1, 0.25 * steps, e2e_ms, 59648, 114688, per_kernel, alg, FakeMoE(), clk)
    return json.loads(buf.getvalue().strip().splitlines()[-1]), alg


def test_decode_line_has_every_contract_key(monkeypatch):
    pk = [{"route": 0.01, "gather": 0.01, "gemm": 0.25, "combine": 0.01}]
    line, alg = make_line(monkeypatch, "decode", pk, e2e_ms=2.4)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 10 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "decode" and line["data"] == "synthetic"
    assert abs(line["ms_per_step"] - 0.25) < 1e-12
    assert abs(line["value"] - 8 / 0.25e-3) < 1e-6                      # T = 8 tokens per step
    r = line["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    # decode is weight-stream bound: achieved = algorithmic bytes of the fused GEMM / its time
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - (alg["l1_bytes"] + alg["l2_bytes"]) / 0.25e-3 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    stored = bench.NCU_TRAFFIC["decode"]
    assert r["traffic"] in (None, stored["bytes"])
    if stored["src"] == bench.gemm_source_hash():
        assert r["traffic"] == stored["bytes"]
    e = line["e2e"]
    assert e["h2d_bytes_per_step"] == 59648 and e["d2h_bytes_per_step"] == 114688
    assert abs(e["ms_per_step"] - 0.24) < 1e-12 and e["unit"] == "tokens/s"
    assert line["gpu_launches"] == 4 * 10


def test_prefill_line_is_tensor_bound_on_the_l1_gemm(monkeypatch):
    pk = [{"route": 0.04, "gather": 0.26, "l1_gemm": 3.0, "l2_gemm": 1.6, "combine": 0.4}]
    line, alg = make_line(monkeypatch, "prefill", pk)
    r = line["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - alg["l1_flops"] / 3.0e-3 / 1e12) < 1e-6
    assert line["config"]["gemm_schedule"].startswith("split")
    assert line["e2e"] is None
