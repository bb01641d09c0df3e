"""The bench's multi-rank host path on CPU: two gloo ranks run bench.main with a stand-in
for the GPU run that reports different per-rank times.  Rank 0 alone prints one JSON line;
its times are the maximum over ranks, and its value is the whole-job aggregate of
independent replicas (weak scaling: world x step bytes / slowest rank's step time)."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_CODE = r"""
import os, sys
sys.path.insert(0, {root!r})
import bench, workloads

def fake_run(args, rank, world, local_rank):
    wl = workloads.RECIPES[args.workload]()
    slow = 1.0 + rank  # rank 1 takes twice as long as rank 0
    return {{"wl": wl, "step_ms": 0.05 * slow, "decode_ms": 0.04 * slow,
            "two_calls_ms": 0.06 * slow, "e2e_ms": 0.08 * slow, "h2d": 1000, "d2h": 500,
            "clocks": None, "flags": 0}}

bench.main(["--gpus", "2", "--steps", "10", "--warmup", "3", "--cpu-baseline-seconds", "0",
            "--workload", "tiny"], runner=fake_run, backend="gloo")
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_report_the_slowest_rank():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_CODE.format(root=ROOT)],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e[-2000:]
    assert outs[1][0].strip() == ""  # only rank 0 prints
    line = json.loads(outs[0][0].strip().splitlines()[-1])

    sys.path.insert(0, ROOT)
    import bench
    import workloads
    wl = workloads.RECIPES["tiny"]()
    dec_b, resh_b, _ = bench.step_bytes(wl)
    step_s = 0.05 * 2.0 / 1e3  # rank 1's step time
    assert line["n_gpus"] == 2 and line["scaling"] == "weak"
    assert abs(line["ms_per_step"] - 0.1) < 1e-9
    assert abs(line["value"] - round(2 * (dec_b + resh_b) / step_s / 1e9, 1)) < 1e-6
    assert abs(line["roofline"]["decode_us"] - 80.0) < 1e-6  # 0.04 ms x 2
    assert abs(line["e2e"]["us_per_step"] - 160.0) < 1e-6
    assert line["config"]["parallelism"] == "replicas x2"
