"""Benchmark: paged decode on the Llama-3.1-8B-shaped batch, one JSON line.

A step is one pass of the whole hot path over one batch: the cache write of each
sequence's newest token followed by paged decode attention over every sequence,
contexts including that token.  The step runs as one kernel (pa_decode_append: one
persistent kernel; the last CTA to finish a pair cut between CTAs merges its split-KV
pieces); the same step as two calls (pa_reshape_and_cache, then pa_decode) is timed
too and reported beside it.  The decode kernel's own duration is timed separately:
--steps launches of pa_decode back to back in the same clock-sampled window.

Workload (seeded, synthetic; no dataset, no weights): 64 sequences, 32 query / 8 kv
heads, head_dim 128, bf16, block_size 16, context lengths uniform in
[128, 2048], K/V ~ N(0,1), blocks placed through the block pool from a shuffled
16384-block free list.  Three such batches live in disjoint blocks and steps rotate
through them, so every step reads K/V that the previous two steps did not touch
(each batch's K/V alone is larger than the 129 MB L2).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]

Under torchrun (N > 1) every rank runs its own replica on its own GPU (weak scaling; no
collective on the data path, only a barrier and a max-reduce of the elapsed time).
``--impl reference`` times the CPU oracle instead (rank 0 only).
"""
import argparse
import hashlib
import itertools
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV GB/s and % of GB300 HBM peak; µs per decode step"
FALLBACK_HBM_GBS = 6800.0
ROTATE = 3
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_llama31_8b_traffic.json")
KERNEL_SOURCES = ["paged_kv_cache_149_gb300/csrc/pa_decode_kernel.cuh",
                  "paged_kv_cache_149_gb300/csrc/pa_arrive.h",
                  "paged_kv_cache_149_gb300/csrc/pa_decode.cu",
                  "paged_kv_cache_149_gb300/csrc/pa_common.cuh"]


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def step_bytes(wl):
    """Algorithmic bytes of one step: K and V of every valid token (the newest included),
    q and out, the block table entries used and the context lengths (decode); plus the
    newest tokens' K/V rows written to the cache (cache write)."""
    e = 2
    n, hq, hkv, d, bs = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    ctx = [int(c) for c in wl.context_lens]
    kv = sum(ctx) * hkv * d * e * 2
    qo = 2 * n * hq * d * e
    table = sum(-(-c // bs) for c in ctx) * 4 + 4 * n
    decode = kv + qo + table
    reshape = n * hkv * d * e * 2
    padded_kv = sum(-(-c // bs) * bs for c in ctx) * hkv * d * e * 2
    return decode, reshape, padded_kv


def decode_config(wl, world):
    """The `config` of a 16-bit decode line (the native arm's and the reference arm's)."""
    dec_b = step_bytes(wl)[0]
    return {
        "workload": (f"{wl.name}: {wl.num_seqs} seqs, ctx {int(wl.context_lens.min())}..."
                     f"{int(wl.context_lens.max())} (sum {int(wl.context_lens.sum())}), "
                     f"{wl.num_q_heads} q / {wl.num_kv_heads} kv heads, head_dim {wl.head_dim}, "
                     f"block_size {wl.block_size}, pool {rotation_pool(wl, ROTATE)[0]} blocks; step = "
                     f"cache write of {wl.num_seqs} new tokens + paged decode, one kernel "
                     f"(pa_decode_append)"),
        "l2": f"each batch's K/V ({dec_b / 1e6:.0f} MB) exceeds L2; {ROTATE} batches in "
              "disjoint blocks rotated every step",
        "parallelism": f"replicas x{world}",
    }


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if the kernel source
    is unchanged since it was captured."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock and throttle samples, taken while the timed region runs."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"pa_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15]
        use = inside or rows[-3:]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        mhz = sorted(r[1] for r in use)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use),
                "window": "timed region" if inside else "after the timed region (too short to sample)"}


def rotation_pool(wl, rotate):
    """Blocks and free order of a pool that holds `rotate` copies of the batch: the
    workload's own pool when it is large enough, else one sized for the copies (a seeded
    shuffle, like the workload's)."""
    import numpy as np
    need = rotate * sum(-(-int(c) // wl.block_size) for c in wl.context_lens)
    if need <= wl.num_blocks:
        return wl.num_blocks, wl.free_order
    return need, np.random.default_rng(1).permutation(need).astype(np.int32)


# Timed loops: each timed loop runs exactly --steps steps between a barrier plus a device
# synchronise and the next; a line reports the median over REPEATS-many such loops, the
# count chosen so that each kind of loop runs for about LOOP_SECONDS in all.
LOOP_SECONDS = 0.4
MAX_REPEATS = 400


FIXED_REPEATS = None  # --repeats: a fixed count (profiling runs), else sized by LOOP_SECONDS


def repeats_for(ms_per_step, steps):
    if FIXED_REPEATS:
        return FIXED_REPEATS
    return int(min(MAX_REPEATS, max(5, round(LOOP_SECONDS * 1e3 / max(1e-3, ms_per_step * steps)))))


def timed_median(fn, steps, stream, device, world, repeats):
    """Median (and all) of the ms per step of `repeats` loops of `steps` calls fn(i), CUDA
    events on `stream` around each loop, a barrier and a synchronise on both sides."""
    import torch
    per = []
    for _ in range(repeats):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize(device)
        per.append(e0.elapsed_time(e1) / steps)
    return float(np.median(per)), per


def estimate_ms(fn, stream, device, n=5):
    """A rough ms per call (to size the repeats)."""
    import torch
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1) / n


def kv_memory(wl, used_blocks):
    """KV memory use of the batch's placement: the paged pool's slots against the tokens
    held (effective utilisation, aiqz.cc section 新旧方案对比), and the fragmentation of a
    contiguous allocator that reserves the recipe's maximum context per sequence
    (aiqz.cc section 连续分配之殇)."""
    tokens = int(sum(int(c) for c in wl.context_lens))
    slots = used_blocks * wl.block_size
    reserved = wl.num_seqs * wl.max_blocks_per_seq * wl.block_size
    return {"tokens": tokens, "paged_slots": slots,
            "paged_utilisation": round(tokens / slots, 5),
            "paged_waste_tokens": slots - tokens,
            "contiguous_reserved_tokens": reserved,
            "contiguous_fragmentation": round(1.0 - tokens / reserved, 5)}


def build_batches(wl, device, rotate, identity=False):
    """Place `rotate` copies of the batch in disjoint blocks of one pool and write every
    token except each sequence's newest one (the step writes those).  identity=True takes
    blocks in physical order (each sequence's blocks consecutive: the contiguous case)
    instead of the shuffled free list.  Returns the caches, the batches and the blocks one
    copy holds."""
    import numpy as np
    import torch

    import paged_kv_cache_149_gb300 as pa
    dt = {"fp16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(dt)

    nb, order = rotation_pool(wl, rotate)
    if identity:
        order = np.arange(nb, dtype=np.int32)
    shape = (nb, wl.num_kv_heads, wl.block_size, wl.head_dim)
    k_cache = torch.zeros(shape, dtype=dt, device=device)
    v_cache = torch.zeros(shape, dtype=dt, device=device)
    pool = pa.BlockPool(nb, wl.block_size, order)
    n, T = wl.num_seqs, wl.max_blocks_per_seq
    keys, values = up(wl.keys), up(wl.values)
    last_rows = torch.from_numpy(wl.seq_start[1:] - 1).to(device)
    batches = []
    free0 = pool.num_free()
    for r in range(rotate):
        if r == 1:
            used = free0 - pool.num_free()
        tables = np.full((n, T), 0, dtype=np.int32)
        slots = []
        for s in range(n):
            sid = r * n + s
            c = int(wl.context_lens[s])
            pool.allocate(sid, c)
            t = pool.block_table(sid)
            tables[s, :len(t)] = t
            slots.append(pool.slots(sid, 0, c))
        all_slots = torch.from_numpy(np.concatenate(slots)).to(device)
        pa.reshape_and_cache(keys, values, k_cache, v_cache, all_slots)
        new_slots = torch.from_numpy(np.array([sl[-1] for sl in slots], dtype=np.int64)).to(device)
        batches.append({
            "q": up(wl.q), "tables": torch.from_numpy(tables).to(device),
            "ctx": torch.from_numpy(np.ascontiguousarray(wl.context_lens, np.int32)).to(device),
            "slots": new_slots, "key": keys[last_rows].contiguous(),
            "value": values[last_rows].contiguous(),
            "out": torch.empty((n, wl.num_q_heads, wl.head_dim), dtype=dt, device=device),
        })
    if rotate == 1:
        used = free0 - pool.num_free()
    return k_cache, v_cache, batches, used


E2E_METHOD = ("each step: its inputs copied from pinned host memory, the public call "
              "(decode steps: a Launch planned once per staging slot), its output copied to "
              "pinned host memory.  Steps are independent, so they are staged in groups: one "
              "upload of a group's inputs on an upload stream, the group's calls back to back "
              "on the compute stream (no stream wait between them), one download of the "
              "group's outputs on a download stream; two groups of staging slots, so each "
              "group's copies overlap the neighbouring groups' kernels")

E2E_GROUP_BYTES = 8 << 20  # inputs staged together: about this many bytes, 1..10 steps


def pipelined_e2e(batches, names, make_launch, out_like, device, steps, warmup, repeats=1,
                  group=None):
    """Steps end to end from pinned host memory: every step's inputs (`names` of its batch,
    packed) come from pinned host memory, the step runs (`make_launch(dev_inputs, dev_out)`
    gives a callable taking the stream, made once per staging slot), and its output goes
    back to pinned host memory.  Consecutive steps are independent, so they are staged
    `group` at a time: a group's inputs go up in one copy on an upload stream, its calls
    run back to back on the compute stream (so each kernel may start while the one before
    it drains), and its outputs come down in one copy on a download stream.  Two groups of
    slots: the upload of group g + 2 waits for group g's kernels, group g + 2's kernels for
    group g's download.  Each timed run is `steps` steps; returns (the median ms per step
    over `repeats` runs, H2D bytes per step, D2H bytes per step)."""
    import torch

    align = 256
    layout, off = {}, 0
    for k in names:
        t = batches[0][k]
        layout[k] = (off, t.shape, t.dtype, t.numel() * t.element_size())
        off += -(-layout[k][3] // align) * align
    if group is None:  # small steps in groups of up to 10, large ones one at a time
        group = int(min(10, max(1, E2E_GROUP_BYTES // max(1, off))))
    S = max(1, group)
    nrot = len(batches)
    # a group's inputs, step after step (step k of a group uses rotation k % nrot; a group
    # starting at step i uses rotations i .. i + S - 1, so the host buffer is built per
    # starting rotation)
    def packed(first_rot):
        h = torch.empty(S * off, dtype=torch.uint8).pin_memory()
        for k_ in range(S):
            b = batches[(first_rot + k_) % nrot]
            for k in names:
                o, _, _, nb = layout[k]
                h[k_ * off + o:k_ * off + o + nb].copy_(b[k].contiguous().view(-1).view(torch.uint8).cpu())
        return h
    host = [packed(r) for r in range(nrot)]
    dev = [torch.empty(S * off, dtype=torch.uint8, device=device) for _ in range(2)]
    nout = out_like.numel()
    outs = [torch.empty((S,) + tuple(out_like.shape), dtype=out_like.dtype, device=device)
            for _ in range(2)]
    host_out = [torch.empty((S,) + tuple(out_like.shape), dtype=out_like.dtype).pin_memory()
                for _ in range(2)]
    launches = []
    for g in range(2):
        row = []
        for k_ in range(S):
            v = {k: dev[g][k_ * off + o:k_ * off + o + nb].view(dt).view(shape)
                 for k, (o, shape, dt, nb) in layout.items()}
            row.append(make_launch(v, outs[g][k_]))
        launches.append(row)
    comp, up_s, down_s = (torch.cuda.Stream(device) for _ in range(3))
    del nout

    def run(n):
        ng = -(-n // S)
        up = [torch.cuda.Event() for _ in range(ng)]
        done = [torch.cuda.Event() for _ in range(ng)]
        down = [torch.cuda.Event() for _ in range(ng)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(comp)
        up_s.wait_event(start)
        down_s.wait_event(start)

        def upload(g):
            if g >= 2:
                up_s.wait_event(done[g - 2])
            with torch.cuda.stream(up_s):
                dev[g % 2].copy_(host[(g * S) % nrot], non_blocking=True)
            up[g].record(up_s)
        for g in range(min(2, ng)):
            upload(g)
        for g in range(ng):
            m = min(S, n - g * S)
            comp.wait_event(up[g])
            if g >= 2:
                comp.wait_event(down[g - 2])
            for k_ in range(m):
                launches[g % 2][k_](comp)
            done[g].record(comp)
            down_s.wait_event(done[g])
            with torch.cuda.stream(down_s):
                host_out[g % 2][:m].copy_(outs[g % 2][:m], non_blocking=True)
            down[g].record(down_s)
            if g + 2 < ng:
                upload(g + 2)
        comp.wait_event(down[ng - 1])
        end.record(comp)
        torch.cuda.synchronize(device)
        return start.elapsed_time(end) / n

    run(max(3, warmup))
    ms = float(np.median([run(max(1, min(steps, 2000))) for _ in range(max(1, repeats))]))
    d2h = out_like.numel() * out_like.element_size()
    return ms, sum(layout[k][3] for k in names), d2h


def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch

    import paged_kv_cache_149_gb300 as pa
    import workloads
    from paged_kv_cache_149_gb300 import build as _build

    _build.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = workloads.RECIPES[args.workload]()
    k_cache, v_cache, batches, used = build_batches(wl, device, ROTATE)
    # the same batches placed contiguously (identity tables), for the paging overhead
    k_id, v_id, batches_id, _ = build_batches(wl, device, ROTATE, identity=True)
    ws = pa.make_workspace(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, device)
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)
    pa.get_device_error()

    def step(i):
        b = batches[i % ROTATE]
        pa.decode_append(b["q"], b["key"], b["value"], k_cache, v_cache, b["tables"], b["ctx"],
                         wl.scale, out=b["out"], workspace=ws, stream=stream)

    def step_two_calls(i):
        b = batches[i % ROTATE]
        pa.reshape_and_cache(b["key"], b["value"], k_cache, v_cache, b["slots"], stream=stream)
        pa.decode(b["q"], k_cache, v_cache, b["tables"], b["ctx"], wl.scale, out=b["out"],
                  workspace=ws, stream=stream)

    def decode_only(i):
        b = batches[i % ROTATE]
        pa.decode(b["q"], k_cache, v_cache, b["tables"], b["ctx"], wl.scale, out=b["out"],
                  workspace=ws, stream=stream)

    def decode_identity(i):
        b = batches_id[i % ROTATE]
        pa.decode(b["q"], k_id, v_id, b["tables"], b["ctx"], wl.scale, out=b["out"],
                  workspace=ws, stream=stream)

    for i in range(args.warmup):
        step(i)
        decode_only(i)
        step_two_calls(i)
        decode_identity(i)
    torch.cuda.synchronize(device)
    if pa.get_device_error(stream=stream):
        raise RuntimeError("device error flags set during warm-up")
    K = args.steps
    R = repeats_for(estimate_ms(step, stream, device), K)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t0 = time.time()
    # the step loop: nothing between the launches, so each kernel may start while the one
    # before it drains (programmatic dependent launch)
    step_ms, step_all = timed_median(step, K, stream, device, world, R)
    # the decode alone (decode kernel + merge kernel), back to back on the same stream
    decode_ms, _ = timed_median(decode_only, K, stream, device, world, R)
    # the same step as two calls
    two_calls_ms, _ = timed_median(step_two_calls, K, stream, device, world, R)
    # the decode over the same batches placed contiguously
    identity_ms, _ = timed_median(decode_identity, K, stream, device, world, R)
    t1 = time.time()
    clocks = sampler.stop(t0, t1) if sampler else None
    flags = pa.get_device_error(stream=stream)

    # end to end through the binding with host buffers: inputs from pinned host memory
    # every step, the output read back every step (copies pipelined with the kernels)
    def e2e_launch(d, out):
        return pa.decode_append(d["q"], d["key"], d["value"], k_cache, v_cache, d["tables"],
                                d["ctx"], wl.scale, out=out, workspace=ws, plan=True).run
    e2e_ms, h2d, d2h = pipelined_e2e(batches, ("q", "tables", "ctx", "key", "value"), e2e_launch,
                                     batches[0]["out"], device, K, args.warmup,
                                     repeats=max(5, R // 4))
    flags |= pa.get_device_error()
    return {"wl": wl, "step_ms": step_ms, "decode_ms": decode_ms, "e2e_ms": e2e_ms,
            "two_calls_ms": two_calls_ms, "identity_ms": identity_ms, "repeats": R,
            "step_ms_spread": [round(min(step_all), 5), round(max(step_all), 5)],
            "used_blocks": used,
            "h2d": h2d, "d2h": d2h, "clocks": clocks, "flags": flags}


def oracle_sample(name, budget_s, max_seqs, seed_seq=0):
    """Time the CPU oracle's paged decode on sequences of the workload until `budget_s`
    of CPU time is spent (at least one sequence).  Runs in a fresh single-threaded process."""
    code = f"""
import json, os, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import workloads
from oracle import attention, cache_ops, formats
from oracle.block_pool import BlockPool
wl = workloads.RECIPES[{name!r}]()
pool = BlockPool(wl.num_blocks, wl.block_size, wl.free_order)
n, T = wl.num_seqs, wl.max_blocks_per_seq
tables = np.full((n, T), -1, dtype=np.int32)
slots = []
for s in range(n):
    c = int(wl.context_lens[s]); pool.allocate(s, c)
    t = pool.block_table(s); tables[s, :len(t)] = t
    slots += [pool.slot(s, i) for i in range(c)]
shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
nan = formats.FORMATS[wl.dtype]["qnan"]
kc = np.full(shape, nan, dtype=np.uint16); vc = kc.copy()
kc, vc = cache_ops.reshape_and_cache(kc, vc, wl.keys, wl.values, np.array(slots, dtype=np.int64))
order = [({seed_seq} + i) % n for i in range(n)]
per, t0 = [], time.process_time()
while time.process_time() - t0 < {budget_s} and len(per) < {max_seqs}:
    s = order[len(per) % n]
    a = time.process_time()
    attention.paged_decode_bits(wl.q, kc, vc, tables, wl.context_lens, wl.scale,
                                wl.block_size, wl.dtype, seqs=[s])
    c = int(wl.context_lens[s])
    nb = (c * wl.num_kv_heads * wl.head_dim * 2 * 2 + 2 * wl.num_q_heads * wl.head_dim * 2
          + (-(-c // wl.block_size)) * 4 + 4)
    per.append((time.process_time() - a, nb))
print(json.dumps({{"seqs": len(per), "seconds": sum(p[0] for p in per),
                  "bytes": sum(p[1] for p in per), "per_seq": per}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle baseline failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_parallel(name, passes=3):
    """The same oracle sharded by sequence over every host core: the batch's paged caches
    are built once in a CUDA-free process, then worker processes forked from it (fork is
    safe there: no CUDA in that process) decode disjoint sequence sets.  Wall time of
    `passes` whole-batch passes."""
    code = f"""
import json, os, sys, time
sys.path.insert(0, {ROOT!r})
import multiprocessing as mp
import numpy as np
import workloads
from oracle import attention, cache_ops, formats
from oracle.block_pool import BlockPool
wl = workloads.RECIPES[{name!r}]()
pool = BlockPool(wl.num_blocks, wl.block_size, wl.free_order)
n, T = wl.num_seqs, wl.max_blocks_per_seq
tables = np.full((n, T), -1, dtype=np.int32)
slots = []
for s in range(n):
    c = int(wl.context_lens[s]); pool.allocate(s, c)
    t = pool.block_table(s); tables[s, :len(t)] = t
    slots += [pool.slot(s, i) for i in range(c)]
shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
nan = formats.FORMATS[wl.dtype]["qnan"]
kc = np.full(shape, nan, dtype=np.uint16); vc = kc.copy()
kc, vc = cache_ops.reshape_and_cache(kc, vc, wl.keys, wl.values, np.array(slots, dtype=np.int64))
def work(seqs):
    attention.paged_decode_bits(wl.q, kc, vc, tables, wl.context_lens, wl.scale,
                                wl.block_size, wl.dtype, seqs=seqs)
    return len(seqs)
cores = len(os.sched_getaffinity(0))
shards = [list(range(k, n, cores)) for k in range(cores) if k < n]
nbytes = sum(int(c) * wl.num_kv_heads * wl.head_dim * 4 + 2 * wl.num_q_heads * wl.head_dim * 2
             + (-(-int(c) // wl.block_size)) * 4 + 4 for c in wl.context_lens)
with mp.get_context("fork").Pool(len(shards)) as p:
    p.map(work, shards)  # warm-up
    t0 = time.time()
    for _ in range({passes}):
        p.map(work, shards)
    wall = (time.time() - t0) / {passes}
print(json.dumps({{"cores": cores, "workers": len(shards), "seconds": wall, "bytes": nbytes}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("parallel oracle baseline failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def prefill_flops(wl):
    """Algorithmic FLOPs of one prefill pass: every query row at position p scores p + 1
    keys (2 d FLOPs each) and sums as many V rows (2 d FLOPs each), for every query head."""
    qlen = np.diff(wl.query_start)
    total = 0
    for s in range(wl.num_seqs):
        c, n = int(wl.context_lens[s]), int(qlen[s])
        # positions c - n .. c - 1 attend to p + 1 keys each
        total += n * (2 * c - n + 1) // 2
    return 4 * wl.head_dim * wl.num_q_heads * total


def run_gpu_prefill(args, rank, world, local_rank):
    """K prefill passes over ROTATE batches in disjoint blocks (each batch's q alone is
    larger than L2), CUDA events around the loop; then end to end with host buffers."""
    import torch

    import paged_kv_cache_149_gb300 as pa
    import workloads
    from paged_kv_cache_149_gb300 import build as _build

    _build.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = workloads.RECIPES[args.workload]()
    dt = {"fp16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(dt)

    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    k_cache = torch.zeros(shape, dtype=dt, device=device)
    v_cache = torch.zeros(shape, dtype=dt, device=device)
    pool = pa.BlockPool(wl.num_blocks, wl.block_size, wl.free_order)
    n, T = wl.num_seqs, wl.max_blocks_per_seq
    keys, values, q = up(wl.keys), up(wl.values), up(wl.q)
    qs = torch.from_numpy(wl.query_start.astype(np.int32)).to(device)
    maxq = int(np.diff(wl.query_start).max())
    batches = []
    for r in range(ROTATE):
        tables = np.full((n, T), 0, dtype=np.int32)
        slots = []
        for s in range(n):
            c = int(wl.context_lens[s])
            pool.allocate(r * n + s, c)
            t = pool.block_table(r * n + s)
            tables[s, :len(t)] = t
            slots.append(pool.slots(r * n + s, 0, c))
        pa.reshape_and_cache(keys, values, k_cache, v_cache,
                             torch.from_numpy(np.concatenate(slots)).to(device))
        batches.append({"q": q if r == 0 else q.clone(), "tables": torch.from_numpy(tables).to(device),
                        "ctx": torch.from_numpy(np.ascontiguousarray(wl.context_lens, np.int32)).to(device),
                        "out": torch.empty_like(q)})
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)
    pa.get_device_error()

    def step(i):
        b = batches[i % ROTATE]
        pa.prefill(b["q"], k_cache, v_cache, b["tables"], b["ctx"], qs, wl.scale, maxq,
                   out=b["out"], stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(device)
    K = args.steps
    R = repeats_for(estimate_ms(step, stream, device), K)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t0 = time.time()
    step_ms, _ = timed_median(step, K, stream, device, world, R)
    t1 = time.time()
    clocks = sampler.stop(t0, t1) if sampler else None
    flags = pa.get_device_error(stream=stream)
    # end to end: q from pinned host memory, out read back, every pass (copies pipelined)
    b0 = batches[0]

    def e2e_launch(d, out):
        return lambda st: pa.prefill(d["q"], k_cache, v_cache, b0["tables"], b0["ctx"], qs, wl.scale,
                                     maxq, out=out, stream=st)
    e2e_ms, h2d, d2h = pipelined_e2e([b0], ("q",), e2e_launch, b0["out"], device, min(K, 50),
                                     args.warmup, repeats=max(3, R // 4))
    return {"wl": wl, "step_ms": step_ms, "decode_ms": step_ms, "repeats": R,
            "two_calls_ms": step_ms, "e2e_ms": e2e_ms,
            "h2d": h2d, "d2h": d2h, "clocks": clocks, "flags": flags}


def oracle_prefill_sample(name, budget_s):
    """The prefill oracle on a bounded sample: the first k tokens of the first sequence
    (a prompt from scratch of k tokens: the same rows and keys), k doubled while the
    single-threaded run stays within budget_s."""
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import workloads
from oracle import cache_ops, formats, prefill
from oracle.block_pool import BlockPool
wl = workloads.RECIPES[{name!r}]()
c0 = int(wl.context_lens[0]); q0 = int(wl.query_start[1] - wl.query_start[0])
best = None
k = 64
while True:
    k = min(k, q0)
    shape = (k // wl.block_size + 2, wl.num_kv_heads, wl.block_size, wl.head_dim)
    kc = np.zeros(shape, np.uint16); vc = np.zeros(shape, np.uint16)
    pool = BlockPool(shape[0], wl.block_size, np.arange(shape[0], dtype=np.int32))
    pool.allocate(0, k)
    tab = np.array([pool.block_table(0) + [0] * 2], dtype=np.int32)
    a = int(wl.seq_start[0]) + (c0 - q0)
    kc, vc = cache_ops.reshape_and_cache(kc, vc, wl.keys[a:a + k], wl.values[a:a + k],
                                         np.array([pool.slot(0, i) for i in range(k)], np.int64))
    q = wl.q[int(wl.query_start[0]):int(wl.query_start[0]) + k]
    t = time.process_time()
    prefill.paged_prefill(q, kc, vc, tab, np.array([k], np.int32), np.array([0, k]), wl.scale,
                          wl.block_size, wl.dtype)
    dt = time.process_time() - t
    best = (k, dt)
    if k >= q0 or dt * 4 > {budget_s}:
        break
    k *= 2
k, dt = best
flops = 4 * wl.head_dim * wl.num_q_heads * k * (k + 1) // 2
print(json.dumps({{"tokens": k, "seconds": dt, "flops": flops}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("prefill oracle baseline failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def prefill_line(args, res, world):
    wl = res["wl"]
    flops = prefill_flops(wl)
    step_s = res["step_ms"] / 1e3
    value = world * flops / step_s / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16, burst)"
    except (OSError, KeyError, ValueError):
        peak, kind = 1900.0, "fallback"
    cpu = oracle_prefill_sample(args.workload, args.cpu_baseline_seconds) \
        if args.cpu_baseline_seconds > 0 else None
    qlen = np.diff(wl.query_start)
    return {
        "metric": "paged prefill attention TFLOP/s (causal, over the block table)",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(res["step_ms"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded normals; no dataset or weights)",
        "config": {
            "workload": (f"{wl.name}: {wl.num_seqs} seqs, ctx {int(wl.context_lens.min())}.."
                         f"{int(wl.context_lens.max())}, new tokens {int(qlen.min())}.."
                         f"{int(qlen.max())} (sum {int(qlen.sum())}), {wl.num_q_heads} q / "
                         f"{wl.num_kv_heads} kv heads, head_dim {wl.head_dim}, block_size "
                         f"{wl.block_size}"),
            "l2": f"{ROTATE} batches in disjoint blocks rotated every pass; each batch's q "
                  "alone exceeds L2",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {"bound": "tensor", "kernel": "prefill_kernel (pa_prefill)",
                     "achieved": round(value / world, 2), "peak": peak, "peak_kind": kind,
                     "unit": "TFLOP/s", "frac": round(value / world / peak, 4), "traffic": None,
                     "algorithmic_flops": flops},
        "cpu_baseline": None if cpu is None else {
            "value": round(cpu["flops"] / cpu["seconds"] / 1e12, 6), "unit": "TFLOP/s",
            "cores": 1, "kind": "oracle",
            "sample": f"float64 NumPy prefill oracle, single thread, the first {cpu['tokens']} "
                      f"tokens of sequence 0 (a {cpu['tokens']}-token prompt)"},
        "e2e": {"value": round(world * flops / (res["e2e_ms"] / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "us_per_step": round(1e3 * res["e2e_ms"], 2), "method": E2E_METHOD},
        "clocks": res["clocks"],
        "gpu_launches": res.get("repeats", 1) * 1 * args.steps,
        "device_error_flags": res["flags"],
    }


SWAP_WORKLOADS = {"swap_llama31_8b": "llama31_8b", "swap_llama7b_mha": "llama7b_mha"}


def run_gpu_swap(args, rank, world, local_rank):
    """Preemption of a whole decode batch: swap-out of every sequence's blocks from the
    device pool to a pinned CPU pool, then swap-in to fresh device blocks -- one
    pa_swap_blocks launch per direction.  Timed three ways: the two launches alone on
    planned pair lists (CUDA events around K steps); the same bytes as two contiguous
    cudaMemcpyAsync copies (copy engines, the link's reference rate in this run); and end
    to end through the public API (pool planning, pair upload, both launches)."""
    import torch

    import paged_kv_cache_149_gb300 as pa
    import workloads
    from paged_kv_cache_149_gb300 import build as _build

    _build.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = workloads.RECIPES[SWAP_WORKLOADS[args.workload]]()
    dt = {"fp16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]
    n = wl.num_seqs
    used = sum(-(-int(c) // wl.block_size) for c in wl.context_lens)
    ncpu = used + 64
    pool = pa.BlockPool(wl.num_blocks, wl.block_size, wl.free_order, num_cpu_blocks=ncpu)
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    cshape = (ncpu,) + shape[1:]
    k_cache = torch.zeros(shape, dtype=dt, device=device)
    v_cache = torch.zeros(shape, dtype=dt, device=device)
    hk = torch.zeros(cshape, dtype=dt).pin_memory()
    hv = torch.zeros(cshape, dtype=dt).pin_memory()
    slots = []
    for s in range(n):
        pool.allocate(s, int(wl.context_lens[s]))
        slots.append(pool.slots(s, 0, int(wl.context_lens[s])))

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(dt)
    pa.reshape_and_cache(up(wl.keys), up(wl.values), k_cache, v_cache,
                         torch.from_numpy(np.concatenate(slots)).to(device))
    seqs = list(range(n))
    # planned pairs of one out / in cycle (the pool's own plan, uploaded once)
    out_pairs = pool.swap_out(seqs)
    in_pairs = pool.swap_in(seqs)  # (resident again; the end-to-end steps plan afresh)
    d_out = torch.from_numpy(out_pairs).to(device)
    d_in = torch.from_numpy(in_pairs).to(device)
    block_bytes = 2 * wl.num_kv_heads * wl.block_size * wl.head_dim * 2  # K and V
    moved = len(out_pairs) * block_bytes  # per direction
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)
    pa.get_device_error()

    def step(i):
        pa.swap_blocks(k_cache, v_cache, hk, hv, d_out, stream=stream, device=device)
        pa.swap_blocks(hk, hv, k_cache, v_cache, d_in, stream=stream, device=device)

    def timed(fn, K):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        e0.record(stream)
        for i in range(K):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1)

    for i in range(args.warmup):
        step(i)
    K = args.steps
    R = repeats_for(estimate_ms(step, stream, device, n=2), K)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t0 = time.time()
    step_ms, _ = timed_median(step, K, stream, device, world, R)
    t1 = time.time()
    clocks = sampler.stop(t0, t1) if sampler else None
    flags = pa.get_device_error(stream=stream)
    # the link's reference rate: the same bytes as one contiguous copy each way
    flat_dev = torch.empty(moved // 2, dtype=torch.int16, device=device)
    flat_host = torch.empty(moved // 2, dtype=torch.int16).pin_memory()

    def ce_step(i):
        with torch.cuda.stream(stream):
            flat_host.copy_(flat_dev, non_blocking=True)
            flat_dev.copy_(flat_host, non_blocking=True)
    for i in range(3):
        ce_step(i)
    ce_ms = timed(ce_step, max(3, min(K, 20))) / max(3, min(K, 20))
    # end to end through the public API: plan on the host, upload the pairs, move
    pin_pairs = torch.zeros((2, len(out_pairs) + 8, 2), dtype=torch.int32).pin_memory()
    dev_pairs = torch.zeros((2, len(out_pairs) + 8, 2), dtype=torch.int32, device=device)

    def e2e_step(i):
        # the swap-in is planned on the host while the swap-out copy runs
        for j, (fn, src, dst) in enumerate(((pool.swap_out, (k_cache, v_cache), (hk, hv)),
                                            (pool.swap_in, (hk, hv), (k_cache, v_cache)))):
            pairs = fn(seqs)
            m = len(pairs)
            pin_pairs[j, :m].numpy()[:] = pairs
            with torch.cuda.stream(stream):
                dev_pairs[j, :m].copy_(pin_pairs[j, :m], non_blocking=True)
            pa.swap_blocks(*src, *dst, dev_pairs[j, :m], stream=stream, device=device)
        stream.synchronize()  # (the pinned pair buffers are refilled next step)
    for i in range(3):
        e2e_step(i)
    ke = max(3, min(K, 20))
    torch.cuda.synchronize(device)
    w0 = time.perf_counter()
    for i in range(ke):
        e2e_step(i)
    torch.cuda.synchronize(device)
    e2e_ms = (time.perf_counter() - w0) * 1e3 / ke
    flags |= pa.get_device_error(stream=stream)
    return {"wl": wl, "step_ms": step_ms, "decode_ms": step_ms, "two_calls_ms": ce_ms, "repeats": R,
            "e2e_ms": e2e_ms, "h2d": moved + 8 * (len(out_pairs) + len(in_pairs)), "d2h": moved,
            "moved": moved, "blocks": len(out_pairs), "clocks": clocks, "flags": flags}


def oracle_swap_sample(name, budget_s):
    """The oracle's swap_blocks on a bounded sample of the batch's blocks (both
    directions), block count doubled while the single-threaded run stays within budget."""
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import workloads
from oracle import cache_ops
wl = workloads.RECIPES[{SWAP_WORKLOADS[name]!r}]()
rng = np.random.default_rng(0)
m = 16
while True:
    shape = (m, wl.num_kv_heads, wl.block_size, wl.head_dim)
    dk = rng.integers(0, 65535, size=shape, dtype=np.uint16)
    dv = rng.integers(0, 65535, size=shape, dtype=np.uint16)
    ck, cv = np.zeros_like(dk), np.zeros_like(dv)
    pairs = np.stack([np.arange(m), rng.permutation(m)], axis=1)
    t = time.process_time()
    ck, cv = cache_ops.swap_blocks(dk, dv, ck, cv, pairs)
    dk, dv = cache_ops.swap_blocks(ck, cv, dk, dv, pairs[:, ::-1])
    dt = time.process_time() - t
    if dt * 4 > {budget_s} or m >= 4096:
        break
    m *= 2
print(json.dumps({{"blocks": m, "seconds": dt, "bytes": 2 * dk.nbytes * 2}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("swap oracle baseline failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def swap_line(args, res, world):
    wl = res["wl"]
    step_bytes_ = 2 * res["moved"]  # out and in
    step_s = res["step_ms"] / 1e3
    value = world * step_bytes_ / step_s / 1e9
    link = step_bytes_ / (res["two_calls_ms"] / 1e3) / 1e9
    cpu = oracle_swap_sample(args.workload, args.cpu_baseline_seconds) \
        if args.cpu_baseline_seconds > 0 else None
    return {
        "metric": "paged KV swap GB/s (device pool -> pinned CPU pool -> device pool, "
                  "through the block tables)",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(res["step_ms"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16 (bit copy)",
        "data": "synthetic (seeded normals; no dataset or weights)",
        "config": {
            "workload": (f"{args.workload}: the {wl.name} batch ({wl.num_seqs} seqs, "
                         f"{res['blocks']} blocks of {wl.num_kv_heads} kv heads x "
                         f"{wl.block_size} x {wl.head_dim}, K and V) swapped out and back in "
                         "every step"),
            "l2": f"{res['moved'] / 1e6:.0f} MB each way per step (above L2)",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {"bound": "c2c", "kernel": "block_copy_kernel (pa_swap_blocks)",
                     "achieved": round(value / world, 1), "peak": round(link, 1),
                     "peak_kind": "measured in this run: the same bytes as one contiguous "
                                  "cudaMemcpyAsync each way (copy engines)",
                     "unit": "GB/s", "frac": round(value / world / link, 4), "traffic": None},
        "cpu_baseline": None if cpu is None else {
            "value": round(cpu["bytes"] / cpu["seconds"] / 1e9, 3), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"NumPy oracle swap_blocks (exact 16-bit copies), single thread, "
                      f"{cpu['blocks']} blocks out and back in"},
        "e2e": {"value": round(world * step_bytes_ / (res["e2e_ms"] / 1e3) / 1e9, 1),
                "unit": "GB/s", "h2d_bytes_per_step": res["h2d"],
                "d2h_bytes_per_step": res["d2h"], "us_per_step": round(1e3 * res["e2e_ms"], 2),
                "includes": "host planning by the C++ pool, pair upload, both launches"},
        "clocks": res["clocks"],
        "gpu_launches": res.get("repeats", 1) * 2 * args.steps,
        "device_error_flags": res["flags"],
    }


PREFIX_WORKLOADS = ("prefix_llama31_8b", "prefix_tiny")


def run_gpu_prefix(args, rank, world, local_rank):
    """Serving prompts that share a system prompt, warm prefix cache.  A step serves every
    request of the batch: the C++ pool looks up each prompt's full blocks by digest
    (pa_pool_allocate_prefix), one pa_reshape_and_cache writes the K/V rows of the
    tokens not found cached, one pa_prefill computes attention for those tokens over
    their whole context, and the requests end (their blocks stay cached in the free
    list).  The same batch served without the cache (every token written and
    prefilled) is timed beside it.  Each arm's write and prefill are marshalled once
    (plan=True) and run every step.  Host planning is inside the timed region; inputs
    (the new tokens' q and K/V rows, as a model's projection would produce them) are
    resident, and again from pinned host memory for the end-to-end number."""
    import torch

    import paged_kv_cache_149_gb300 as pa
    import workloads
    from paged_kv_cache_149_gb300 import build as _build

    _build.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = workloads.RECIPES[args.workload]()
    dt = {"fp16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]
    n, T, B = wl.num_seqs, wl.max_blocks_per_seq, wl.block_size
    L = wl.context_lens.astype(np.int64)
    toks = [wl.tokens[int(wl.seq_start[s]):int(wl.seq_start[s + 1])] for s in range(n)]
    hit = (wl.system_len // B) * B
    own = L - hit

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(dt)

    def rows_of(arr, first):   # rows first_s .. end of every request, concatenated
        return np.concatenate([arr[int(wl.seq_start[s]) + int(first[s]):int(wl.seq_start[s + 1])]
                               for s in range(n)])
    shape = (wl.num_blocks, wl.num_kv_heads, B, wl.head_dim)
    ctx = torch.from_numpy(L.astype(np.int32)).to(device)
    arms = {}
    for name, first in (("cached", np.full(n, hit)), ("uncached", np.zeros(n, np.int64))):
        cnt = L - first
        qs = np.zeros(n + 1, dtype=np.int32)
        np.cumsum(cnt, out=qs[1:])
        qsel = np.concatenate([np.arange(wl.query_start[s] + first[s], wl.query_start[s + 1])
                               for s in range(n)])
        # each arm has its own pool and caches: the uncached arm must not evict or
        # overwrite what the cached arm has cached
        arms[name] = {"first": first, "qs": torch.from_numpy(qs).to(device),
                      "q": up(wl.q[qsel]), "k": up(rows_of(wl.keys, first)),
                      "v": up(rows_of(wl.values, first)), "maxq": int(cnt.max()),
                      "rows": int(cnt.sum()),
                      "pool": pa.BlockPool(wl.num_blocks, B, wl.free_order),
                      "kc": torch.zeros(shape, dtype=dt, device=device),
                      "vc": torch.zeros(shape, dtype=dt, device=device)}
        arms[name]["out"] = torch.empty_like(arms[name]["q"])
    stream = torch.cuda.Stream(device)
    bufs = [{"slots": torch.zeros(int(L.sum()), dtype=torch.int64).pin_memory(),
             "tables": torch.zeros((n, T), dtype=torch.int32).pin_memory(),
             "ev": torch.cuda.Event()} for _ in range(2)]
    dslots = torch.zeros(int(L.sum()), dtype=torch.int64, device=device)
    dtables = torch.zeros((n, T), dtype=torch.int32, device=device)
    vocab = 128256
    base_tokens = np.ascontiguousarray(wl.tokens, dtype=np.int64)
    own_mask = np.ones(len(base_tokens), dtype=bool)
    for s in range(n):
        own_mask[int(wl.seq_start[s]):int(wl.seq_start[s]) + wl.system_len] = False
    token_start = wl.seq_start.astype(np.int64)
    ids = np.arange(n, dtype=np.int64)
    # The batches requests arrive in: every request is the shared system prompt followed by
    # its own tokens.  Made before the timing (arrival is not the engine's work); 24 sets,
    # used in turn, so a set comes back only after the pool's FIFO free list has cycled
    # (12 steps at 512 own blocks per step in 6144 blocks) and its own blocks are evicted:
    # every step is new requests, not repeats.
    prompt_sets = [np.where(own_mask, (base_tokens + 7919 * (k + 1)) % vocab,
                            base_tokens).astype(np.int32) for k in range(24)]
    # each request's block digests, computed when it arrives (as its tokens are)
    digest_sets = [b"".join(d for s_ in range(n)
                            for d in pa.block_hashes(ps[int(token_start[s_]):int(token_start[s_ + 1])], B))
                   for ps in prompt_sets]
    n_tokens = L.astype(np.int32)

    def prompts(i):
        return prompt_sets[i % len(prompt_sets)]

    fresh = itertools.count()
    cached_out = np.zeros(n, dtype=np.int32)

    def serve(arm, i, host_inputs=None):
        a = arms[arm]
        pool, kc, vc = a["pool"], a["kc"], a["vc"]
        buf = bufs[i % 2]
        buf["ev"].synchronize()          # the copy that last read this buffer is done
        slots, tables = buf["slots"].numpy(), buf["tables"].numpy()
        if arm == "cached":
            # one call: lookups by the digests computed at arrival, allocation, slots of
            # the uncached tokens and the block tables
            _, sl, _ = pool.allocate_hashed_batch(ids, n_tokens, digest_sets[next(fresh) % 24], T,
                                                  out=(cached_out, slots, tables))
            if not np.array_equal(cached_out, a["first"]):
                raise RuntimeError(f"cached tokens {cached_out.tolist()}, expected {a['first'][0]}")
            o = len(sl)
        else:
            o = 0
            for s in range(n):
                pool.allocate(s, int(L[s]))
                slots[o:o + int(L[s])] = pool.slots(s, 0, int(L[s]))
                o += int(L[s])
                t = pool.block_table(s)
                tables[s, :len(t)] = t
        with torch.cuda.stream(stream):
            dslots[:o].copy_(buf["slots"][:o], non_blocking=True)
            dtables.copy_(buf["tables"], non_blocking=True)
            buf["ev"].record(stream)
            q, k, v = a["q"], a["k"], a["v"]
            if host_inputs is not None:
                hq, hk, hv, hout = host_inputs[arm]
                q.copy_(hq, non_blocking=True)
                k.copy_(hk, non_blocking=True)
                v.copy_(hv, non_blocking=True)
        # the write and the prefill, marshalled once per arm (a serving loop's launch plan:
        # the buffers stay, their contents change every step)
        if a.get("plan_rows") != o:
            a["plans"] = (pa.reshape_and_cache(k, v, kc, vc, dslots[:o], plan=True),
                          pa.prefill(q, kc, vc, dtables, ctx, a["qs"], wl.scale, a["maxq"],
                                     out=a["out"], plan=True))
            a["plan_rows"] = o
        a["plans"][0].run(stream)
        a["plans"][1].run(stream)
        if host_inputs is not None:
            with torch.cuda.stream(stream):
                host_inputs[arm][3].copy_(a["out"], non_blocking=True)
        pool.free_batch(ids)

    def timed(arm, K, host_inputs=None):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0 = time.perf_counter()
        e0.record(stream)
        for i in range(K):
            serve(arm, i, host_inputs)
        e1.record(stream)
        torch.cuda.synchronize(device)
        return (time.perf_counter() - w0) * 1e3 / K, e0.elapsed_time(e1) / K

    # cold pass: the first request finds nothing cached and writes every row; the system
    # prompt's full blocks are cached from then on
    ca, ua = arms["cached"], arms["uncached"]   # ua's k / v hold every row of every request
    slot_all = []
    first_prompts = np.ascontiguousarray(base_tokens.astype(np.int32))
    for s in range(n):
        c = ca["pool"].allocate_prefix(s, first_prompts[int(token_start[s]):int(token_start[s + 1])])
        sl = np.full(int(L[s]), -1, dtype=np.int64)
        sl[c:] = ca["pool"].slots(s, c, int(L[s]) - c)
        slot_all.append(sl)
    pa.reshape_and_cache(ua["k"], ua["v"], ca["kc"], ca["vc"],
                         torch.from_numpy(np.concatenate(slot_all)).to(device), stream=stream)
    for s in range(n):
        ca["pool"].free(s)
    torch.cuda.synchronize(device)
    pa.get_device_error()
    for arm in ("cached", "uncached"):
        for i in range(args.warmup):
            serve(arm, i)
    # kernel-only: the prefill launch of a cached step, timed alone on its planned inputs
    K = args.steps
    serve("cached", K + 1)
    torch.cuda.synchronize(device)
    kev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    kev[0].record(stream)
    for i in range(K):
        pa.prefill(ca["q"], ca["kc"], ca["vc"], dtables, ctx, ca["qs"], wl.scale, ca["maxq"],
                   out=ca["out"], stream=stream)
    kev[1].record(stream)
    torch.cuda.synchronize(device)
    prefill_ms = kev[0].elapsed_time(kev[1]) / K
    R = repeats_for(timed("cached", 3)[0], K)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t0 = time.time()
    runs = [timed("cached", K) for _ in range(R)]   # (wall, device) ms per step
    cached_ms = float(np.median([r_[0] for r_ in runs]))
    cached_dev_ms = float(np.median([r_[1] for r_ in runs]))
    t1 = time.time()
    clocks = sampler.stop(t0, t1) if sampler else None
    uncached_ms, _ = timed("uncached", max(3, K // 4))
    # the host planning of a cached step alone (lookups, slots, tables, free), and the
    # same with the hashing done in the step (the library's parallel batch hashing); the
    # hashing of one request's blocks alone, serial
    hb = bufs[0]
    h0 = time.perf_counter()
    for _ in range(20):
        ca["pool"].allocate_hashed_batch(ids, n_tokens, digest_sets[next(fresh) % 24], T,
                                         out=(cached_out, hb["slots"].numpy(), hb["tables"].numpy()))
        ca["pool"].free_batch(ids)
    planning_us = (time.perf_counter() - h0) * 1e6 / 20
    h0 = time.perf_counter()
    for _ in range(20):
        ca["pool"].allocate_prefix_batch(ids, prompts(next(fresh)), token_start, table_width=T,
                                         out=(cached_out, hb["slots"].numpy(), hb["tables"].numpy()))
        ca["pool"].free_batch(ids)
    planning_hash_us = (time.perf_counter() - h0) * 1e6 / 20
    h0 = time.perf_counter()
    for k in range(4):
        ps = prompt_sets[k]
        for s_ in range(n):
            pa.block_hashes(ps[int(token_start[s_]):int(token_start[s_ + 1])], B)
    hash_us_per_request = (time.perf_counter() - h0) * 1e6 / (4 * n)
    host = {}
    for arm in arms:
        x = arms[arm]
        host[arm] = tuple(t.cpu().pin_memory() for t in (x["q"], x["k"], x["v"], x["out"]))
    e2e_ms, _ = timed("cached", max(3, min(K, 20)), host)
    flags = pa.get_device_error(stream=stream)
    h = host["cached"]
    return {"wl": wl, "step_ms": cached_ms, "decode_ms": prefill_ms, "repeats": R,
            "two_calls_ms": uncached_ms, "e2e_ms": e2e_ms, "cached_dev_ms": cached_dev_ms,
            "h2d": sum(t.numel() * t.element_size() for t in h[:3]) + int(own.sum()) * 8 + n * T * 4,
            "d2h": h[3].numel() * h[3].element_size(), "hit": hit,
            "rows": ca["rows"], "clocks": clocks, "flags": flags, "planning_us": planning_us,
            "planning_hash_us": planning_hash_us, "hash_us_per_request": hash_us_per_request}


def oracle_prefix_sample(name, budget_s):
    """The oracle serving request 1 of the batch warm: its pool finds the system prompt
    cached (request 0 placed first), then its prefill computes the first k own tokens
    over the cached prefix, k doubled while the single-threaded run stays within budget.
    Tokens served = the cached prefix + k."""
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import workloads
from oracle import cache_ops, prefill
from oracle.block_pool import BlockPool
wl = workloads.RECIPES[{name!r}]()
B = wl.block_size
toks = [wl.tokens[int(wl.seq_start[s]):int(wl.seq_start[s + 1])] for s in range(2)]
k = 16
while True:
    t0 = time.process_time()
    pool = BlockPool(wl.num_blocks, B, wl.free_order)
    shape = (wl.num_blocks, wl.num_kv_heads, B, wl.head_dim)
    kc = np.zeros(shape, np.uint16); vc = np.zeros(shape, np.uint16)
    pool.allocate_prefix(0, toks[0])
    a = int(wl.seq_start[0])
    kc, vc = cache_ops.reshape_and_cache(kc, vc, wl.keys[a:a + len(toks[0])],
                                         wl.values[a:a + len(toks[0])],
                                         np.array([pool.slot(0, i) for i in range(len(toks[0]))]))
    t = time.process_time()
    c = pool.allocate_prefix(1, toks[1][:wl.system_len + k])
    a = int(wl.seq_start[1])
    kc, vc = cache_ops.reshape_and_cache(kc, vc, wl.keys[a + c:a + c + k], wl.values[a + c:a + c + k],
                                         np.array([pool.slot(1, c + i) for i in range(k)]))
    tab = np.array([pool.block_table(1)], dtype=np.int32)
    q = wl.q[int(wl.query_start[1]) + c:int(wl.query_start[1]) + c + k]
    prefill.paged_prefill(q, kc, vc, tab, np.array([c + k], np.int32), np.array([0, k]),
                          wl.scale, B, wl.dtype)
    dt = time.process_time() - t
    if dt * 4 > {budget_s} or c + k >= len(toks[1]):
        break
    k *= 2
print(json.dumps({{"tokens": c + k, "own": k, "seconds": dt}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("prefix oracle baseline failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def prefix_line(args, res, world):
    wl = res["wl"]
    n = wl.num_seqs
    tokens = int(wl.context_lens.sum())
    step_s = res["step_ms"] / 1e3
    value = world * tokens / step_s
    # FLOPs of the prefill launch: each uncached row at position p scores p + 1 keys
    flops = 0
    for s in range(n):
        c, L = res["hit"], int(wl.context_lens[s])
        flops += (L - c) * (L + c + 1) // 2
    flops *= 4 * wl.head_dim * wl.num_q_heads
    achieved = flops / (res["decode_ms"] / 1e3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16, burst)"
    except (OSError, KeyError, ValueError):
        peak, kind = 1900.0, "fallback"
    uncached = world * tokens / (res["two_calls_ms"] / 1e3)
    cpu = oracle_prefix_sample(args.workload, args.cpu_baseline_seconds) \
        if args.cpu_baseline_seconds > 0 else None
    return {
        "metric": "prompt tokens served per second with a warm prefix cache (shared system "
                  "prompt; host lookup by block digests computed at arrival + cache write + "
                  "paged prefill of the uncached tokens)",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(res["step_ms"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded normals and token ids; no dataset or weights)",
        "config": {
            "workload": (f"{wl.name}: {n} requests x ({wl.system_len} shared + "
                         f"{int(wl.context_lens[0]) - wl.system_len} own tokens), "
                         f"{wl.num_q_heads} q / {wl.num_kv_heads} kv heads, head_dim "
                         f"{wl.head_dim}, block_size {wl.block_size}; {res['hit']} tokens of "
                         "each prompt found cached"),
            "l2": "no flush: the shared system prompt's K/V (a few MB) stays in L2 across "
                  "steps, as it does in serving; each step's new rows are written fresh",
            "parallelism": f"replicas x{world}",
        },
        "host_planning_us": round(res["planning_us"], 1),
        "host_planning_with_hashing_us": round(res["planning_hash_us"], 1),
        "hashing_us_per_request_at_arrival": round(res["hash_us_per_request"], 1),
        "uncached": {"value": round(uncached, 1), "unit": "tokens/s",
                     "ms_per_step": round(res["two_calls_ms"], 4),
                     "speedup_from_cache": round(value / uncached, 3)},
        "roofline": {"bound": "tensor", "kernel": "prefill_kernel (pa_prefill, uncached rows)",
                     "achieved": round(achieved, 2), "peak": peak, "peak_kind": kind,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "prefill_us": round(1e3 * res["decode_ms"], 2),
                     "device_ms_per_step": round(res["cached_dev_ms"], 4)},
        "cpu_baseline": None if cpu is None else {
            "value": round(cpu["tokens"] / cpu["seconds"], 1), "unit": "tokens/s", "cores": 1,
            "kind": "oracle",
            "sample": f"the oracle pool and float64 prefill oracle serving request 1 warm: "
                      f"{cpu['tokens'] - cpu['own']} tokens found cached, {cpu['own']} own "
                      "tokens written and prefilled, single thread"},
        "e2e": {"value": round(world * tokens / (res["e2e_ms"] / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "us_per_step": round(1e3 * res["e2e_ms"], 2)},
        "clocks": res["clocks"],
        "gpu_launches": res.get("repeats", 1) * 2 * args.steps,
        "device_error_flags": res["flags"],
    }


FP8_WORKLOADS = {"kv8_llama31_8b": "llama31_8b", "kv8_llama7b_mha": "llama7b_mha",
                 "kv8_tiny": "tiny"}
INT4_WORKLOADS = {"kv4_llama31_8b": "llama31_8b", "kv4_llama7b_mha": "llama7b_mha",
                  "kv4_tiny": "tiny"}
FP8_SCALE = 0.0123   # k_scale = v_scale: about max|N(0,1) draw| / 448 for these batches


def quant_recipe(name):
    """(format, batch recipe) of a quantised-KV workload name."""
    return ("int4", INT4_WORKLOADS[name]) if name in INT4_WORKLOADS else ("fp8", FP8_WORKLOADS[name])


def row_bytes(fmt, d):
    """Cached bytes of one token of one kv head, K or V: one byte a code for FP8; a nibble
    a code plus the float32 scale for INT4."""
    return d if fmt == "fp8" else d // 2 + 4


def fp8_step_bytes(wl, fmt="fp8"):
    """Algorithmic bytes of one quantised-KV step: decode reads the valid tokens' K/V rows
    (codes, and INT4 scales), q, the table entries and lengths, and writes out; the cache
    write reads the newest rows (16-bit) and writes their codes (and scales)."""
    n, hq, hkv, d, bs = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    ctx = [int(c) for c in wl.context_lens]
    rb = row_bytes(fmt, d)
    decode = sum(ctx) * hkv * rb * 2 + 2 * n * hq * d * 2 + sum(-(-c // bs) for c in ctx) * 4 + 4 * n
    reshape = n * hkv * (2 * d + rb) * 2
    return decode, reshape


def run_gpu_fp8(args, rank, world, local_rank):
    """The decode step over FP8 (or INT4) blocks: pa_decode_append_fp8 / _int4, one kernel
    that quantises the newest tokens' rows into the cache and decodes over the codes; the
    decode kernel alone and the two-call step timed beside it; end to end with host
    buffers.  ROTATE batches in disjoint blocks."""
    import torch

    import paged_kv_cache_149_gb300 as pa
    import workloads
    from paged_kv_cache_149_gb300 import build as _build

    _build.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    fmt, recipe = quant_recipe(args.workload)
    wl = workloads.RECIPES[recipe]()
    dt = {"fp16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]
    ks = vs = FP8_SCALE

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(dt)
    nb, order = rotation_pool(wl, ROTATE)
    d_bytes = wl.head_dim if fmt == "fp8" else wl.head_dim // 2
    shape = (nb, wl.num_kv_heads, wl.block_size, d_bytes)
    k8 = torch.zeros(shape, dtype=torch.uint8, device=device)
    v8 = torch.zeros(shape, dtype=torch.uint8, device=device)
    if fmt == "int4":
        k4s = torch.zeros(shape[:3], dtype=torch.float32, device=device)
        v4s = torch.zeros(shape[:3], dtype=torch.float32, device=device)

    def cache_write(key, value, slots):
        if fmt == "fp8":
            pa.reshape_and_cache_fp8(key, value, k8, v8, slots, ks, vs, stream=stream)
        else:
            pa.reshape_and_cache_int4(key, value, k8, v8, k4s, v4s, slots, stream=stream)

    def decode(b, out):
        if fmt == "fp8":
            pa.decode_fp8(b["q"], k8, v8, b["tables"], b["ctx"], wl.scale, ks, vs, out=out,
                          workspace=ws, stream=stream)
        else:
            pa.decode_int4(b["q"], k8, v8, k4s, v4s, b["tables"], b["ctx"], wl.scale, out=out,
                           workspace=ws, stream=stream)
    stream = None
    pool = pa.BlockPool(nb, wl.block_size, order)
    n, T = wl.num_seqs, wl.max_blocks_per_seq
    keys, values = up(wl.keys), up(wl.values)
    last_rows = torch.from_numpy(wl.seq_start[1:] - 1).to(device)
    batches = []
    for r in range(ROTATE):
        tables = np.full((n, T), 0, dtype=np.int32)
        slots = []
        for s in range(n):
            pool.allocate(r * n + s, int(wl.context_lens[s]))
            t = pool.block_table(r * n + s)
            tables[s, :len(t)] = t
            slots.append(pool.slots(r * n + s, 0, int(wl.context_lens[s])))
        cache_write(keys, values, torch.from_numpy(np.concatenate(slots)).to(device))
        batches.append({
            "q": up(wl.q), "tables": torch.from_numpy(tables).to(device),
            "ctx": torch.from_numpy(np.ascontiguousarray(wl.context_lens, np.int32)).to(device),
            "slots": torch.from_numpy(np.array([sl[-1] for sl in slots], np.int64)).to(device),
            "key": keys[last_rows].contiguous(), "value": values[last_rows].contiguous(),
            "out": torch.empty((n, wl.num_q_heads, wl.head_dim), dtype=dt, device=device)})
    del keys, values
    ws = pa.make_workspace(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, device)
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)
    pa.get_device_error()

    def step(i, b=None):
        b = b or batches[i % ROTATE]
        if fmt == "fp8":
            pa.decode_append_fp8(b["q"], b["key"], b["value"], k8, v8, b["tables"], b["ctx"],
                                 wl.scale, ks, vs, out=b["out"], workspace=ws, stream=stream)
        else:
            pa.decode_append_int4(b["q"], b["key"], b["value"], k8, v8, k4s, v4s, b["tables"],
                                  b["ctx"], wl.scale, out=b["out"], workspace=ws, stream=stream)

    def step_two_calls(i):
        b = batches[i % ROTATE]
        cache_write(b["key"], b["value"], b["slots"])
        decode(b, b["out"])

    def decode_only(i):
        b = batches[i % ROTATE]
        decode(b, b["out"])

    for i in range(args.warmup):
        step(i)
        decode_only(i)
        step_two_calls(i)
    torch.cuda.synchronize(device)
    if pa.get_device_error(stream=stream):
        raise RuntimeError("device error flags set during warm-up")
    K = args.steps
    R = repeats_for(estimate_ms(step, stream, device), K)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t0 = time.time()
    step_ms, _ = timed_median(step, K, stream, device, world, R)
    decode_ms, _ = timed_median(decode_only, K, stream, device, world, R)
    two_calls_ms, _ = timed_median(step_two_calls, K, stream, device, world, R)
    t1 = time.time()
    clocks = sampler.stop(t0, t1) if sampler else None
    flags = pa.get_device_error(stream=stream)
    # end to end with host buffers: every step's inputs from pinned host memory, its
    # output read back (copies pipelined with the kernels)
    def e2e_launch(d, out):
        if fmt == "fp8":
            return pa.decode_append_fp8(d["q"], d["key"], d["value"], k8, v8, d["tables"], d["ctx"],
                                        wl.scale, ks, vs, out=out, workspace=ws, plan=True).run
        return pa.decode_append_int4(d["q"], d["key"], d["value"], k8, v8, k4s, v4s, d["tables"],
                                     d["ctx"], wl.scale, out=out, workspace=ws, plan=True).run
    e2e_ms, h2d, d2h = pipelined_e2e(batches, ("q", "tables", "ctx", "key", "value"), e2e_launch,
                                     batches[0]["out"], device, K, args.warmup,
                                     repeats=max(5, R // 4))
    flags |= pa.get_device_error()
    return {"wl": wl, "step_ms": step_ms, "decode_ms": decode_ms, "repeats": R,
            "two_calls_ms": two_calls_ms, "e2e_ms": e2e_ms, "h2d": h2d, "d2h": d2h,
            "clocks": clocks, "flags": flags}


def oracle_fp8_sample(name, budget_s):
    """The FP8 (or INT4) decode oracle on whole sequences of the batch (codes made by the
    oracle's own cache write), single thread, until budget_s of CPU time is spent."""
    fmt, recipe = quant_recipe(name)
    if fmt == "int4":
        return oracle_int4_sample(recipe, budget_s)
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import workloads
from oracle import fp8
from oracle.block_pool import BlockPool
wl = workloads.RECIPES[{recipe!r}]()
pool = BlockPool(wl.num_blocks, wl.block_size, wl.free_order)
n, T = wl.num_seqs, wl.max_blocks_per_seq
tables = np.full((n, T), -1, dtype=np.int32)
slots = []
for s in range(n):
    c = int(wl.context_lens[s]); pool.allocate(s, c)
    t = pool.block_table(s); tables[s, :len(t)] = t
    slots += [pool.slot(s, i) for i in range(c)]
shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
k8 = np.zeros(shape, np.uint8); v8 = k8.copy()
k8, v8 = fp8.reshape_and_cache(k8, v8, wl.keys, wl.values, np.array(slots), {FP8_SCALE},
                               {FP8_SCALE}, wl.dtype)
done, nbytes, t0 = 0, 0, time.process_time()
while time.process_time() - t0 < {budget_s} and done < n:
    fp8.paged_decode_bits(wl.q, k8, v8, tables, wl.context_lens, wl.scale, {FP8_SCALE},
                          {FP8_SCALE}, wl.block_size, wl.dtype, seqs=[done])
    c = int(wl.context_lens[done])
    nbytes += c * wl.num_kv_heads * wl.head_dim * 2 + 2 * wl.num_q_heads * wl.head_dim * 2
    done += 1
print(json.dumps({{"seqs": done, "seconds": time.process_time() - t0, "bytes": nbytes}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("fp8 oracle baseline failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_int4_sample(recipe, budget_s):
    """The INT4 decode oracle on whole sequences of the batch, as oracle_fp8_sample."""
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import workloads
from oracle import int4
from oracle.block_pool import BlockPool
wl = workloads.RECIPES[{recipe!r}]()
pool = BlockPool(wl.num_blocks, wl.block_size, wl.free_order)
n, T = wl.num_seqs, wl.max_blocks_per_seq
tables = np.full((n, T), -1, dtype=np.int32)
slots = []
for s in range(n):
    c = int(wl.context_lens[s]); pool.allocate(s, c)
    t = pool.block_table(s); tables[s, :len(t)] = t
    slots += [pool.slot(s, i) for i in range(c)]
kc = np.zeros((wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim // 2), np.uint8)
ks = np.zeros((wl.num_blocks, wl.num_kv_heads, wl.block_size), np.float32)
kc, vc, ks, vs = int4.reshape_and_cache(kc, kc.copy(), ks, ks.copy(), wl.keys, wl.values,
                                        np.array(slots), wl.dtype)
done, nbytes, t0 = 0, 0, time.process_time()
while time.process_time() - t0 < {budget_s} and done < n:
    int4.paged_decode_bits(wl.q, kc, vc, ks, vs, tables, wl.context_lens, wl.scale,
                           wl.block_size, wl.dtype, seqs=[done])
    c = int(wl.context_lens[done])
    nbytes += c * wl.num_kv_heads * (wl.head_dim // 2 + 4) * 2 + 2 * wl.num_q_heads * wl.head_dim * 2
    done += 1
print(json.dumps({{"seqs": done, "seconds": time.process_time() - t0, "bytes": nbytes}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("int4 oracle baseline failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def fp8_line(args, res, world):
    wl = res["wl"]
    fmt, _ = quant_recipe(args.workload)
    dec_b, resh_b = fp8_step_bytes(wl, fmt)
    fp8 = fmt == "fp8"
    step_s = res["step_ms"] / 1e3
    value = world * (dec_b + resh_b) / step_s / 1e9
    peak, peak_kind = measured_peak()
    achieved = dec_b / (res["decode_ms"] / 1e3) / 1e9
    cpu = oracle_fp8_sample(args.workload, args.cpu_baseline_seconds) \
        if args.cpu_baseline_seconds > 0 else None
    ctx = wl.context_lens
    return {
        "metric": ("paged decode KV GB/s over FP8 (E4M3) blocks and % of GB300 HBM peak; "
                   "µs per decode step" if fp8 else
                   "paged decode KV GB/s over INT4 blocks (4-bit codes + a float32 scale per "
                   "row) and % of GB300 HBM peak; µs per decode step"),
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(res["step_ms"], 5),
        "us_per_step": round(1e3 * res["step_ms"], 2),
        "us_per_step_two_calls": round(1e3 * res["two_calls_ms"], 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (f"e4m3 K/V, {wl.dtype} q/out, f16 MMA" if fp8 else
                  f"int4 K/V codes + f32 row scales, {wl.dtype} q/out, f16 MMA"),
        "data": "synthetic (seeded normals; no dataset or weights)",
        "config": {
            "workload": (f"{args.workload}: the {wl.name} batch ({wl.num_seqs} seqs, ctx "
                         f"{int(ctx.min())}..{int(ctx.max())}, sum {int(ctx.sum())}, "
                         f"{wl.num_q_heads} q / {wl.num_kv_heads} kv heads, head_dim "
                         f"{wl.head_dim}, block_size {wl.block_size}) with "
                         + (f"E4M3 K/V blocks, k_scale = v_scale = {FP8_SCALE}" if fp8 else
                            "INT4 K/V blocks (codes in [-7, 7], scale max|x| / 7 per row)")),
            "l2": f"{ROTATE} batches in disjoint blocks rotated every step "
                  f"({dec_b / 1e6:.0f} MB of decode bytes per batch)",
            "parallelism": f"replicas x{world}",
            "step": (f"pa_decode_append_{fmt}: one kernel quantises each sequence's newest "
                     "rows into their slots and decodes (the two-call step is "
                     f"pa_reshape_and_cache_{fmt} + pa_decode_{fmt})"),
        },
        "roofline": {"bound": "hbm", "kernel": (f"decode_kernel<{'F8' if fp8 else 'INT4'}> "
                                                f"(pa_decode_{fmt})"),
                     "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (copy bandwidth)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "decode_us": round(1e3 * res["decode_ms"], 2),
                     "algorithmic_bytes_per_launch": dec_b},
        "cpu_baseline": None if cpu is None else {
            "value": round(cpu["bytes"] / cpu["seconds"] / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"float64 {fmt.upper()} decode oracle, single thread, {cpu['seqs']} "
                      "whole sequences of the batch"},
        "e2e": {"value": round(world * (dec_b + resh_b) / (res["e2e_ms"] / 1e3) / 1e9, 1),
                "unit": "GB/s", "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "us_per_step": round(1e3 * res["e2e_ms"], 2), "method": E2E_METHOD},
        "clocks": res["clocks"],
        # per timed loop: steps (1 kernel each), decode alone (1), two-call steps (2)
        "gpu_launches": res.get("repeats", 1) * 4 * args.steps,
        "repeats": res.get("repeats", 1),
        "device_error_flags": res["flags"],
    }


# ---------------------------------------------------------------- shared-prefix beams

BEAM_WORKLOADS = ("beam",)
DECODE16_WORKLOADS = ("tiny", "llama31_8b", "llama7b_mha", "long_b8", "long_b16", "long_b32")


def beam_place(pool, wl, base):
    """Shared-prefix beams through the block pool (sequence ids base ..): each prompt's
    parent holds the prefix and one generated token, forks into its beams, and each beam
    then writes its private tokens; a beam's first write into the shared, partly filled
    last block plans a copy.  Returns (slots and rows of the shared tokens per prompt,
    the copy pairs, the private tokens' slots, block tables, context lengths)."""
    import numpy as np
    shared = []
    for p in range(wl.prompts):
        root = base + p * wl.beams
        pool.allocate(root, wl.shared_tokens - 1)
        slots = list(pool.slots(root, 0, wl.shared_tokens - 1))
        s_new, cow = pool.append_slot(root)
        assert cow is None
        shared.append(np.array(slots + [s_new], dtype=np.int64))
        for b in range(1, wl.beams):
            pool.fork(root, root + b)
    cows, slots = [], []
    for k in range(wl.prompts * wl.beams):
        for _ in range(int(wl.private_tokens[k])):
            s_, cow = pool.append_slot(base + k)
            if cow:
                cows.append(cow)
            slots.append(s_)
    n = wl.prompts * wl.beams
    tables = np.zeros((n, wl.max_blocks_per_seq), dtype=np.int32)
    ctx = np.zeros(n, dtype=np.int32)
    for k in range(n):
        t = pool.block_table(base + k)
        tables[k, :len(t)] = t
        ctx[k] = pool.context_len(base + k)
    return shared, cows, np.array(slots, dtype=np.int64), tables, ctx


def beam_bytes(wl, ctx, n_pairs):
    """Algorithmic bytes of a beam step: the decode's (every sequence reads its whole
    context, shared blocks once per sequence), the copy-on-write block copies (read and
    written, both caches) and the private rows written; and the distinct K/V bytes the
    decode touches (shared blocks once)."""
    e, hkv, d, B = 2, wl.num_kv_heads, wl.head_dim, wl.block_size
    n = wl.prompts * wl.beams
    kv = int(ctx.sum()) * hkv * d * e * 2
    decode = kv + 2 * n * wl.num_q_heads * d * e + sum(-(-int(c) // B) for c in ctx) * 4 + 4 * n
    copy = n_pairs * 2 * hkv * B * d * e * 2
    rows = int(wl.private_tokens.sum()) * hkv * d * e * 2
    unique_kv = (wl.prompts * wl.shared_tokens + int(wl.private_tokens.sum())) * hkv * d * e * 2
    return decode, copy, rows, unique_kv


def run_gpu_beam(args, rank, world, local_rank):
    """The beam step (config of 2 prompts x 8 beams over a shared 1024-token prefix): the
    copy-on-write copies of the shared last blocks (pa_copy_blocks), the beams' private
    rows written (pa_reshape_and_cache), then decode over all 16 sequences (pa_decode).
    Every step redoes the same copies and writes, so steps are identical.  ROTATE
    placements in disjoint blocks of one pool rotate every step."""
    import torch

    import paged_kv_cache_149_gb300 as pa
    import workloads
    from paged_kv_cache_149_gb300 import build as _build

    _build.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = workloads.beam()
    dt = {"fp16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(dt)
    nb = ROTATE * wl.num_blocks
    order = np.random.default_rng(1).permutation(nb).astype(np.int32)
    pool = pa.BlockPool(nb, wl.block_size, order)
    shape = (nb, wl.num_kv_heads, wl.block_size, wl.head_dim)
    k_cache = torch.zeros(shape, dtype=dt, device=device)
    v_cache = torch.zeros(shape, dtype=dt, device=device)
    n = wl.prompts * wl.beams
    pk = up(np.concatenate(wl.private_keys))
    pv = up(np.concatenate(wl.private_values))
    free0 = pool.num_free()
    batches = []
    for r in range(ROTATE):
        shared, cows, slots, tables, ctx = beam_place(pool, wl, r * n)
        if r == 0:
            used = free0 - pool.num_free()
        for p in range(wl.prompts):
            pa.reshape_and_cache(up(wl.shared_keys[p]), up(wl.shared_values[p]), k_cache, v_cache,
                                 torch.from_numpy(shared[p]).to(device))
        pa.check_block_mapping(cows, nb)
        batches.append({"pairs": torch.tensor(cows, dtype=torch.int32, device=device),
                        "slots": torch.from_numpy(slots).to(device), "ctx_np": ctx,
                        "tables": torch.from_numpy(tables).to(device),
                        "ctx": torch.from_numpy(ctx).to(device), "q": up(wl.q),
                        "out": torch.empty((n, wl.num_q_heads, wl.head_dim), dtype=dt, device=device)})
    ws = pa.make_workspace(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, device)
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)
    pa.get_device_error()

    def step(i):
        b = batches[i % ROTATE]
        pa.copy_blocks(k_cache, v_cache, b["pairs"], stream=stream)
        pa.reshape_and_cache(pk, pv, k_cache, v_cache, b["slots"], stream=stream)
        pa.decode(b["q"], k_cache, v_cache, b["tables"], b["ctx"], wl.scale, out=b["out"],
                  workspace=ws, stream=stream)

    def decode_only(i):
        b = batches[i % ROTATE]
        pa.decode(b["q"], k_cache, v_cache, b["tables"], b["ctx"], wl.scale, out=b["out"],
                  workspace=ws, stream=stream)

    for i in range(args.warmup):
        step(i)
        decode_only(i)
    torch.cuda.synchronize(device)
    if pa.get_device_error(stream=stream):
        raise RuntimeError("device error flags set during warm-up")
    K = args.steps
    R = repeats_for(estimate_ms(step, stream, device), K)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t0 = time.time()
    step_ms, _ = timed_median(step, K, stream, device, world, R)
    decode_ms, _ = timed_median(decode_only, K, stream, device, world, R)
    t1 = time.time()
    clocks = sampler.stop(t0, t1) if sampler else None
    flags = pa.get_device_error(stream=stream)

    # end to end: q, tables, lengths, private rows, slots and pairs from pinned host memory,
    # the output read back
    for b in batches:
        b["pk"], b["pv"] = pk, pv

    def e2e_launch(d, out):
        def run(st):
            pa.copy_blocks(k_cache, v_cache, d["pairs"], stream=st)
            pa.reshape_and_cache(d["pk"], d["pv"], k_cache, v_cache, d["slots"], stream=st)
            pa.decode(d["q"], k_cache, v_cache, d["tables"], d["ctx"], wl.scale, out=out,
                      workspace=ws, stream=st)
        return run
    e2e_ms, h2d, d2h = pipelined_e2e(batches, ("q", "tables", "ctx", "pairs", "slots", "pk", "pv"),
                                     e2e_launch, batches[0]["out"], device, K, args.warmup,
                                     repeats=max(5, R // 4))
    flags |= pa.get_device_error()
    return {"wl": wl, "ctx": batches[0]["ctx_np"], "pairs": int(batches[0]["pairs"].shape[0]),
            "step_ms": step_ms, "decode_ms": decode_ms, "two_calls_ms": step_ms, "repeats": R,
            "e2e_ms": e2e_ms, "h2d": h2d, "d2h": d2h, "used_blocks": used, "clocks": clocks,
            "flags": flags}


def oracle_beam_sample(budget_s):
    """The oracle's side of the beam step, single thread: its pool, cache writes and
    copy-on-write copies, then its decode of whole beams until budget_s of CPU time."""
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import workloads
from oracle import attention, cache_ops, formats
from oracle.block_pool import BlockPool
wl = workloads.beam()
B = wl.block_size
pool = BlockPool(wl.num_blocks, B, wl.free_order)
shape = (wl.num_blocks, wl.num_kv_heads, B, wl.head_dim)
kc = np.zeros(shape, np.uint16); vc = kc.copy()
for p in range(wl.prompts):
    root = p * wl.beams
    pool.allocate(root, wl.shared_tokens - 1)
    sl = [pool.slot(root, t) for t in range(wl.shared_tokens - 1)]
    s_new, _ = pool.append_slot(root)
    kc, vc = cache_ops.reshape_and_cache(kc, vc, wl.shared_keys[p], wl.shared_values[p],
                                         np.array(sl + [s_new], np.int64))
    for b in range(1, wl.beams):
        pool.fork(root, root + b)
n = wl.prompts * wl.beams
cows, slots, keys, values = [], [], [], []
for k in range(n):
    for i in range(int(wl.private_tokens[k])):
        s_, cow = pool.append_slot(k)
        if cow:
            cows.append(cow)
        slots.append(s_); keys.append(wl.private_keys[k][i]); values.append(wl.private_values[k][i])
kc, vc = cache_ops.copy_blocks(kc, vc, cows)
kc, vc = cache_ops.reshape_and_cache(kc, vc, np.stack(keys), np.stack(values), np.array(slots, np.int64))
tables = np.zeros((n, wl.max_blocks_per_seq), np.int32); ctx = np.zeros(n, np.int32)
for k in range(n):
    t = pool.block_table(k); tables[k, :len(t)] = t; ctx[k] = pool.context_len(k)
per, t0 = [], time.process_time()
while time.process_time() - t0 < {budget_s} or not per:
    s = len(per) % n
    a = time.process_time()
    attention.paged_decode_bits(wl.q, kc, vc, tables, ctx, wl.scale, B, wl.dtype, seqs=[s])
    c = int(ctx[s])
    nb = c * wl.num_kv_heads * wl.head_dim * 4 + 2 * wl.num_q_heads * wl.head_dim * 2 + (-(-c // B)) * 4 + 4
    per.append((time.process_time() - a, nb))
print(json.dumps({{"seqs": len(per), "seconds": sum(p[0] for p in per), "bytes": sum(p[1] for p in per)}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("beam oracle baseline failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def beam_line(args, res, world):
    wl = res["wl"]
    dec_b, copy_b, rows_b, unique_kv = beam_bytes(wl, res["ctx"], res["pairs"])
    step_b = dec_b + copy_b + rows_b
    value = world * step_b / (res["step_ms"] / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    achieved = dec_b / (res["decode_ms"] / 1e3) / 1e9
    cpu = oracle_beam_sample(args.cpu_baseline_seconds) if args.cpu_baseline_seconds > 0 else None
    n = wl.prompts * wl.beams
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["step_ms"], 5),
        "us_per_step": round(1e3 * res["step_ms"], 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded normals; no dataset or weights)",
        "config": {
            "workload": (f"beam: {wl.prompts} prompts x {wl.beams} beams sharing a "
                         f"{wl.shared_tokens - 1}-token prefix + 1 shared token (65 blocks, "
                         f"reference count {wl.beams}), 1..15 private tokens per beam (ctx "
                         f"{int(res['ctx'].min())}..{int(res['ctx'].max())}), "
                         f"{wl.num_q_heads} q / {wl.num_kv_heads} kv heads, head_dim "
                         f"{wl.head_dim}, block_size {wl.block_size}; step = "
                         f"{res['pairs']} copy-on-write block copies + the private rows "
                         "written + decode over every beam"),
            "l2": f"{ROTATE} placements in disjoint blocks rotated every step; a step's "
                  f"distinct K/V ({unique_kv / 1e6:.0f} MB) fits in L2, and the beams of a "
                  "prompt read the same prefix blocks, so L2 serves part of the decode",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {"bound": "hbm", "kernel": "decode_kernel (pa_decode)",
                     "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (HBM copy)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "algorithmic_bytes": dec_b, "distinct_kv_bytes": unique_kv,
                     "decode_us": round(1e3 * res["decode_ms"], 2),
                     "note": "algorithmic bytes count each beam's reads of the shared prefix; "
                             "L2 absorbs the repeats, so the fraction can pass 1"},
        "cpu_baseline": None if cpu is None else {
            "value": round(cpu["bytes"] / cpu["seconds"] / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"float64 NumPy oracle, single thread, {cpu['seqs']} beams decoded"},
        "e2e": {"value": round(world * step_b / (res["e2e_ms"] / 1e3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "us_per_step": round(1e3 * res["e2e_ms"], 2), "method": E2E_METHOD},
        "clocks": res["clocks"],
        # per timed loop: steps (copy + write + decode), decode alone (1)
        "gpu_launches": res.get("repeats", 1) * 4 * args.steps,
        "repeats": res.get("repeats", 1),
        "device_error_flags": res["flags"],
        "kv_memory": {"beams": n, "blocks_used": res["used_blocks"],
                      "blocks_without_sharing": int(sum(-(-int(c) // wl.block_size)
                                                        for c in res["ctx"])),
                      "saved": round(1 - res["used_blocks"] /
                                     sum(-(-int(c) // wl.block_size) for c in res["ctx"]), 4)},
    }
    return line


def max_over_ranks(values):
    """Element-wise maximum of per-rank floats over the process group (NCCL on GPUs, or any
    other backend on CPU tensors)."""
    import torch
    dev = (torch.device("cuda", torch.cuda.current_device())
           if torch.distributed.get_backend() == "nccl" else torch.device("cpu"))
    t = torch.tensor(values, dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


# per-rank times that the JSON line takes as the maximum over ranks
RANK_TIMES = ("step_ms", "decode_ms", "two_calls_ms", "e2e_ms")


def timeline_phases(a, b):
    """Phases of launch `a` and the gap to launch `b` from their pa_decode_timeline stamps
    ([cta][warp][k] ns: k = 0 the programmatic wait released, 1 the warp's streaming done,
    2 its end; a CTA with no work left zeros), in µs from the first release of `a`."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    live = (a > 0).all(axis=(1, 2))
    a = a[live]
    t0 = a[:, :, 0].min()
    rel = lambda x: (x - t0) / 1e3
    release = rel(a[:, :, 0].min(axis=1))
    stream_end = rel(a[:, :, 1].max(axis=1))
    cta_end = rel(a[:, :, 2].max(axis=1))
    tail = cta_end - stream_end
    pct = lambda x, q: [round(float(v), 2) for v in np.percentile(x, q)]
    bl = b[(b[:, :, 0] > 0).all(axis=1)]  # (only the release stamps of `b` are read)
    nxt = rel(bl[:, :, 0].min()) if len(bl) else None
    return {
        "ctas": int(live.sum()),
        "release_spread_us": round(float(release.max()), 2),
        "stream_end_us": dict(zip(("p10", "p50", "p90", "max"), pct(stream_end, [10, 50, 90, 100]))),
        "cta_end_us": dict(zip(("p50", "max"), pct(cta_end, [50, 100]))),
        "end_phase_us": dict(zip(("p50", "max"), pct(tail, [50, 100]))),
        "longest_end_phases": [{"cta": int(np.flatnonzero(live)[c]), "released": round(float(release[c]), 2),
                                "stream_end": round(float(stream_end[c]), 2),
                                "end": round(float(cta_end[c]), 2)}
                               for c in np.argsort(tail)[::-1][:3]],
        "latest_released": [{"cta": int(np.flatnonzero(live)[c]), "released": round(float(release[c]), 2),
                             "stream_end": round(float(stream_end[c]), 2)}
                            for c in np.argsort(release)[::-1][:6]],
        "next_release_us": None if nxt is None else round(float(nxt), 2),
        "gap_after_last_end_us": None if nxt is None else round(float(nxt - cta_end.max()), 2),
    }


def run_timeline(args):
    """--timeline: the decode kernel alone, --steps launches back to back on one stream as
    in the roofline loop; the last two run the stamped copy of the kernel
    (pa_decode_timeline).  Prints one JSON line with the phases of the second-to-last launch
    and the gap to the last one."""
    import torch

    import paged_kv_cache_149_gb300 as pa
    import workloads
    from paged_kv_cache_149_gb300 import build as _build

    _build.build()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    wl = workloads.RECIPES[args.workload]()
    k_cache, v_cache, batches, _ = build_batches(wl, device, ROTATE)
    ws = pa.make_workspace(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, device)
    stream = torch.cuda.Stream(device)
    nsm = torch.cuda.get_device_properties(device).multi_processor_count
    bufs = [torch.zeros(nsm * 8 * 3, dtype=torch.int64, device=device) for _ in range(2)]
    torch.cuda.synchronize(device)

    def launch(i):
        b = batches[i % ROTATE]
        pa.decode(b["q"], k_cache, v_cache, b["tables"], b["ctx"], wl.scale, out=b["out"],
                  workspace=ws, stream=stream)

    for i in range(args.warmup):
        launch(i)
    try:  # the stamped kernel once too, so that loading it is not timed
        pa.decode_timeline(bufs[0])
        launch(0)
    finally:
        pa.decode_timeline(None)
    torch.cuda.synchronize(device)
    bufs[0].zero_()
    K = max(3, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K - 2):
        launch(i)
    try:
        pa.decode_timeline(bufs[0])
        launch(K - 2)
        pa.decode_timeline(bufs[1])
        launch(K - 1)
    finally:
        pa.decode_timeline(None)
    e1.record(stream)
    torch.cuda.synchronize(device)
    if pa.get_device_error(stream=stream):
        raise RuntimeError("device error flags set")
    a, b = (x.view(nsm, 8, 3).cpu().numpy() for x in bufs)
    print(json.dumps({"workload": args.workload, "launches": K,
                      "us_per_launch": round(e0.elapsed_time(e1) * 1e3 / K, 2),
                      "phases": timeline_phases(a, b)}))


def main(argv=None, runner=None, backend="nccl"):
    """One JSON line on rank 0.  `runner` (default: the GPU run) and `backend` are
    parameters so that the multi-rank host logic can run on CPU ranks."""
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="llama31_8b")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    ap.add_argument("--repeats", type=int, default=0,
                    help="timed loops of --steps steps each (default: enough for ~0.4 s)")
    ap.add_argument("--timeline", action="store_true",
                    help="16-bit decode workloads: print the phase stamps of a launch instead")
    args = ap.parse_args(argv)
    global FIXED_REPEATS
    FIXED_REPEATS = args.repeats if args.repeats > 0 else None
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        reference_arm(args)
        return
    if args.timeline:
        if args.workload not in DECODE16_WORKLOADS:
            ap.error("--timeline takes a 16-bit decode workload")
        run_timeline(args)
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group(backend)
    is_prefill = args.workload.startswith("prefill")
    is_swap = args.workload in SWAP_WORKLOADS
    is_prefix = args.workload in PREFIX_WORKLOADS
    is_fp8 = args.workload in FP8_WORKLOADS or args.workload in INT4_WORKLOADS
    is_beam = args.workload in BEAM_WORKLOADS
    default_runner = (run_gpu_prefill if is_prefill else run_gpu_swap if is_swap else
                      run_gpu_prefix if is_prefix else run_gpu_fp8 if is_fp8 else
                      run_gpu_beam if is_beam else run_gpu)
    res = (runner or default_runner)(args, rank, world, local_rank)
    if world > 1:
        res.update(zip(RANK_TIMES, max_over_ranks([res[k] for k in RANK_TIMES])))
    if rank != 0:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
        return
    if is_prefill or is_swap or is_prefix or is_fp8 or is_beam:
        line = (prefill_line if is_prefill else swap_line if is_swap else
                prefix_line if is_prefix else fp8_line if is_fp8 else beam_line)
        print(json.dumps(line(args, res, world)))
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
        return
    wl = res["wl"]
    dec_b, resh_b, padded = step_bytes(wl)
    step_s = res["step_ms"] / 1e3
    value = world * (dec_b + resh_b) / step_s / 1e9
    peak, peak_kind = measured_peak()
    achieved = dec_b / (res["decode_ms"] / 1e3) / 1e9
    traffic = recorded_traffic()
    cpu = (oracle_sample(args.workload, args.cpu_baseline_seconds, 10 ** 9)
           if args.cpu_baseline_seconds > 0 else None)
    cpu_par = oracle_parallel(args.workload) if args.cpu_baseline_seconds > 0 else None
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(res["step_ms"], 5),
        "us_per_step": round(1e3 * res["step_ms"], 2),
        "us_per_step_two_calls": round(1e3 * res["two_calls_ms"], 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded normals; no dataset or weights)",
        "config": decode_config(wl, world),
        "roofline": {
            "bound": "hbm",
            "kernel": "decode_kernel (pa_decode: persistent paged decode with in-kernel split-KV merge)",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} (HBM copy)",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes": dec_b,
            "padded_block_bytes": padded,
            "decode_us": round(1e3 * res["decode_ms"], 2),
            "decode_timing": "decode kernel alone, --steps launches back to back on the bench "
                             "stream, CUDA events around the loop (same clock window)",
        },
        "cpu_baseline": None if cpu is None else {
            "value": round(cpu["bytes"] / cpu["seconds"] / 1e9, 4),
            "unit": "GB/s",
            "cores": 1,
            "kind": "oracle",
            "sample": f"float64 NumPy oracle, single thread, {cpu['seqs']} sequences of the same "
                      f"batch in {cpu['seconds']:.1f} s of CPU time",
        },
        "cpu_baseline_parallel": None if cpu_par is None else {
            "value": round(cpu_par["bytes"] / cpu_par["seconds"] / 1e9, 4),
            "unit": "GB/s",
            "cores": cpu_par["workers"],
            "kind": "oracle",
            "sample": f"float64 NumPy oracle, the whole batch sharded by sequence over "
                      f"{cpu_par['workers']} processes ({cpu_par['cores']} host cores), "
                      f"{cpu_par['seconds'] * 1e3:.0f} ms per batch (wall)",
        },
        "e2e": {
            "value": round(world * (dec_b + resh_b) / (res["e2e_ms"] / 1e3) / 1e9, 1),
            "unit": "GB/s",
            "h2d_bytes_per_step": res["h2d"],
            "d2h_bytes_per_step": res["d2h"],
            "us_per_step": round(1e3 * res["e2e_ms"], 2),
            "method": E2E_METHOD,
        },
        "clocks": res["clocks"],
        # per timed loop: steps (1 kernel each), decode alone (1 each), two-call steps (2
        # each), decode over contiguous placement (1 each)
        "gpu_launches": res.get("repeats", 1) * 5 * args.steps,
        "repeats": res.get("repeats", 1),
        "timing": "median over `repeats` timed loops of exactly `steps` steps (each loop "
                  "between a synchronise on both sides)",
        "device_error_flags": res["flags"],
    }
    if "identity_ms" in res:
        # the cost of paging: the same decode over the same batches placed in shuffled
        # blocks (the step's placement) against each sequence's blocks in physical order
        line["paged_overhead"] = {
            "shuffled_us": round(1e3 * res["decode_ms"], 2),
            "contiguous_us": round(1e3 * res["identity_ms"], 2),
            "ratio": round(res["decode_ms"] / res["identity_ms"], 4),
            "method": "pa_decode on identity block tables (each sequence's blocks consecutive "
                      "in memory) against the shuffled pool placement; same kernel, same batch",
        }
    if "used_blocks" in res:
        line["kv_memory"] = kv_memory(wl, res["used_blocks"])
    print(json.dumps(line))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


def reference_arm(args):
    """The oracle as it stands, timed on the host cores: each step decodes a bounded
    sample of the same batch."""
    import workloads
    wl = workloads.RECIPES.get(args.workload, lambda: None)()
    if not isinstance(wl, workloads.DecodeWorkload) or isinstance(wl, workloads.PrefillWorkload):
        raise SystemExit(f"--impl reference times the 16-bit decode oracle; {args.workload!r} "
                         "is not a 16-bit decode workload")
    # calibrate: the per-sequence cost sets how many sequences fit in one step
    cal = oracle_sample(args.workload, 1.0, 4)
    per_seq = cal["seconds"] / max(1, cal["seqs"])
    budget = 120.0
    per_step = max(1, min(wl.num_seqs, int(budget / (args.steps + args.warmup) / per_seq)))
    t0 = time.time()
    res = oracle_sample(args.workload, 1e9, per_step * (args.steps + args.warmup))
    wall = time.time() - t0
    timed = res["per_seq"][per_step * args.warmup:]      # warm-up steps are not counted
    secs = sum(p[0] for p in timed)
    nbytes = sum(p[1] for p in timed)
    value = nbytes / secs / 1e9
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": decode_config(wl, args.gpus),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} sequence(s) of the batch per step, single thread; "
                                   f"{wall:.0f} s wall including setup"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
