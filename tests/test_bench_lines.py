"""Every bench line, not only the default decode one, on CPU: bench.main runs each workload
family (16-bit decode, FP8 and INT4 decode, prefill, prefix caching, swap) with a stand-in
for the GPU run, and the printed line must be one JSON object with the keys every line
carries, a value equal to the family's algorithmic count over the step time, and the
roofline fraction equal to achieved / peak."""
import json

import pytest

import bench
import workloads

STEPS = 10
# fake per-step times (ms), small enough that the tiny workloads' values stay well above
# the lines' rounding
STEP, DECODE, TWO, E2E = 5e-4, 4e-4, 6e-4, 8e-4
CONTRACT = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
            "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches")


def fake_runner(wl_name, **extra):
    def run(args, rank, world, local_rank):
        res = {"wl": workloads.RECIPES[wl_name](), "step_ms": STEP, "decode_ms": DECODE,
               "two_calls_ms": TWO, "e2e_ms": E2E, "h2d": 1000, "d2h": 500, "clocks": None,
               "flags": 0}
        res.update(extra)
        return res
    return run


def line_of(capsys, workload, runner):
    bench.main(["--workload", workload, "--steps", str(STEPS), "--warmup", "3",
                "--cpu-baseline-seconds", "0"], runner=runner)
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    line = json.loads(out[0])
    for k in CONTRACT:
        assert k in line, (workload, k)
    assert line["n_gpus"] == 1 and line["steps"] == STEPS and line["warmup"] == 3
    assert line["ms_per_step"] == pytest.approx(STEP, rel=1e-3)
    r = line["roofline"]
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=2e-3, abs=6e-5)  # both rounded
    assert line["e2e"]["h2d_bytes_per_step"] == 1000 and line["e2e"]["d2h_bytes_per_step"] == 500
    return line


def test_decode_line(capsys):
    line = line_of(capsys, "tiny", fake_runner("tiny"))
    dec, resh, _ = bench.step_bytes(workloads.tiny())
    assert line["value"] == pytest.approx((dec + resh) / (STEP * 1e-3) / 1e9, rel=1e-3)
    assert line["roofline"]["achieved"] == pytest.approx(dec / (DECODE * 1e-3) / 1e9, rel=1e-3)


@pytest.mark.parametrize("name,fmt", [("kv8_tiny", "fp8"), ("kv4_tiny", "int4")])
def test_quantised_decode_lines(capsys, name, fmt):
    line = line_of(capsys, name, fake_runner("tiny"))
    dec, resh = bench.fp8_step_bytes(workloads.tiny(), fmt)
    assert line["value"] == pytest.approx((dec + resh) / (STEP * 1e-3) / 1e9, rel=1e-3)
    assert line["roofline"]["achieved"] == pytest.approx(dec / (DECODE * 1e-3) / 1e9, rel=1e-3)
    assert ("INT4" in line["metric"]) == (fmt == "int4")


def test_prefill_line(capsys):
    line = line_of(capsys, "prefill_tiny", fake_runner("prefill_tiny"))
    flops = bench.prefill_flops(workloads.prefill_tiny())
    assert line["unit"] == "TFLOP/s" and line["roofline"]["bound"] == "tensor"
    assert line["value"] == pytest.approx(flops / (STEP * 1e-3) / 1e12, rel=1e-3)


def test_prefix_line(capsys):
    wl = workloads.prefix_tiny()
    runner = fake_runner("prefix_tiny", cached_dev_ms=4.5e-4, hit=16, planning_us=50.0,
                         planning_hash_us=120.0, hash_us_per_request=30.0, rows=100)
    line = line_of(capsys, "prefix_tiny", runner)
    assert line["unit"] == "tokens/s"
    assert line["value"] == pytest.approx(int(wl.context_lens.sum()) / (STEP * 1e-3), rel=1e-3)
    assert line["uncached"]["speedup_from_cache"] == pytest.approx(TWO / STEP, rel=1e-2)


def test_beam_line(capsys):
    import numpy as np
    wl = workloads.beam()
    ctx = (wl.shared_tokens + wl.private_tokens).astype(np.int32)
    line = line_of(capsys, "beam", fake_runner("beam", ctx=ctx, pairs=14, used_blocks=146))
    dec, copy, rows, unique = bench.beam_bytes(wl, ctx, 14)
    assert line["value"] == pytest.approx((dec + copy + rows) / (STEP * 1e-3) / 1e9, rel=1e-3)
    assert line["roofline"]["achieved"] == pytest.approx(dec / (DECODE * 1e-3) / 1e9, rel=1e-3)
    assert unique < dec
    assert line["kv_memory"]["blocks_used"] == 146


def test_swap_line(capsys):
    line = line_of(capsys, "swap_llama31_8b",
                   fake_runner("llama31_8b", moved=123_000_000, blocks=4454))
    assert line["unit"] == "GB/s"
    assert line["value"] == pytest.approx(2 * 123e6 / (STEP * 1e-3) / 1e9, rel=1e-3)
