"""The bench JSON line carries every key of the measurement contract, with the
roofline and end-to-end figures derived from the timings it is given (host
logic only: nothing here needs a device)."""
import argparse
import io
import json
from contextlib import redirect_stdout

import bench
import numpy as np
import workloads


def timings(name, per_kernel, steps, e2e_ms=None):
    w = workloads.CONFIGS[name]
    idx, _ = workloads.routing(w)
    counts = np.bincount(idx[idx >= 0].ravel(), minlength=w.Ep)
    alg = bench.algorithmic(w, counts)
    main = dict(total_ms=sum(per_kernel[0].values()) * steps, e2e_ms=e2e_ms, h2d=59648, d2h=114688,
                per_kernel=per_kernel, alg=alg, tile_width=16, launches=4)
    return w, main, alg


def make_line(name, per_kernel, steps=10, e2e_ms=None, dec=None):
    w, main, alg = timings(name, per_kernel, steps, e2e_ms)
    args = argparse.Namespace(steps=steps, warmup=3, schedule="auto", tiles=-1, no_cpu_baseline=True)
    clk = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3, "in_window": 3}
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.report(args, w, 1, main, clk, dec=dec, dec_clk=clk if dec else None)
    return json.loads(buf.getvalue().strip().splitlines()[-1]), alg


def test_decode_line_has_every_contract_key():
    pk = [{"route": 0.01, "gather": 0.01, "gemm": 0.22, "combine": 0.01}]
    line, alg = make_line("decode", pk, e2e_ms=2.4)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 10 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "decode" and line["data"] == "synthetic"
    # the run shape stays out of the workload config
    for k in ("parallelism", "gemm_schedule", "token_tiles"):
        assert k not in line["config"] and k in line
    assert abs(line["ms_per_step"] - 0.25) < 1e-12
    assert abs(line["value"] - 8 / 0.25e-3) < 1e-6                      # T = 8 tokens per step
    r = line["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    # decode is weight-stream bound: achieved = algorithmic bytes of the fused GEMM / its time
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - (alg["l1_bytes"] + alg["l2_bytes"]) / 0.22e-3 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    stored = bench.NCU_TRAFFIC["decode"]
    assert r["traffic"] in (None, stored["bytes"])
    if stored["src"] == bench.gemm_source_hash():
        assert r["traffic"] == stored["bytes"]
    # whole forward: the same bytes over the step time
    rs = line["roofline_step"]
    assert rs["bound"] == "hbm"
    assert abs(rs["achieved"] - (alg["l1_bytes"] + alg["l2_bytes"]) / 0.25e-3 / 1e9) < 1e-6
    e = line["e2e"]
    assert e["h2d_bytes_per_step"] == 59648 and e["d2h_bytes_per_step"] == 114688
    assert abs(e["ms_per_step"] - 0.24) < 1e-12 and e["unit"] == "tokens/s"
    assert line["gpu_launches"] == 4 * 10
    assert abs(line["clocks"]["ms_per_step_x_sm_mhz"] - 0.25 * 2070.0) < 1e-9


def test_prefill_line_is_tensor_bound_on_the_l1_gemm_and_carries_the_decode_record():
    pk = [{"route": 0.04, "gather": 0.26, "l1_gemm": 3.0, "l2_gemm": 1.6, "combine": 0.4}]
    dw, dmain, dalg = timings("decode", [{"route": 0.01, "gather": 0.01, "gemm": 0.22, "combine": 0.01}],
                              bench.DECODE_RECORD_STEPS)
    dmain["w"] = dw
    line, alg = make_line("prefill", pk, dec=dmain)
    r = line["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - alg["l1_flops"] / 3.0e-3 / 1e12) < 1e-6
    rs = line["roofline_step"]
    assert rs["bound"] == "tensor" and abs(rs["achieved"] - alg["flops"] / 5.3e-3 / 1e12) < 1e-6
    assert line["gemm_schedule"].startswith("split")
    assert line["e2e"] is None
    d = line["decode"]
    assert d["config"]["workload"] == "decode" and d["steps"] == bench.DECODE_RECORD_STEPS
    assert abs(d["ms_per_step"] - 0.25) < 1e-12
    assert d["roofline"]["bound"] == "hbm"
    assert abs(d["roofline"]["achieved"] - (dalg["l1_bytes"] + dalg["l2_bytes"]) / 0.22e-3 / 1e9) < 1e-6


def test_clock_summary_keeps_the_samples_inside_the_timed_windows():
    c = bench.Clocks(0)
    row = lambda ts, mhz, cap: [ts, "0", str(mhz), "2070", "900.0", "0x0", "Not Active", "Not Active",
                                "Not Active", "Active" if cap else "Not Active"]
    c.rows = [row("2026/12/03 05:00:00.000", 1000, False), row("2026/12/03 05:00:00.100", 2070, True),
              row("2026/12/03 05:00:00.120", 2050, False), row("2026/12/03 05:00:01.000", 900, False)]
    t0 = bench.Clocks._epoch("2026/12/03 05:00:00.090")
    t1 = bench.Clocks._epoch("2026/12/03 05:00:00.130")
    s = c.summary([(t0, t1)])
    assert s["in_window"] == 2 and s["samples"] == 2
    assert s["sm_mhz"] == 2060.0 and s["reasons"] == ["sw_power_cap"]
    # a window shorter than the sampling interval falls back to the nearest sample
    t2 = bench.Clocks._epoch("2026/12/03 05:00:00.990")
    s2 = c.summary([(t2, t2 + 0.001)])
    assert s2["in_window"] == 0 and s2["sm_mhz"] == 900.0
