"""The bench's algorithmic byte and FLOP counts, which every roofline fraction divides by,
checked against what the workload's own arrays hold: the bytes of the rows a step reads
and writes, the oracle's quantised rows for the FP8/INT4 formats, and a brute-force count
of the causal (query, key) pairs for prefill.  Also the pool that holds the bench's
rotated copies of a batch, and the reference arm's line (the oracle timed on the host),
which names the same workload config as the native decode line."""
import json

import numpy as np
import pytest

import bench
import workloads
from oracle import int4


def table_and_length_bytes(wl):
    blocks = sum(-(-int(c) // wl.block_size) for c in wl.context_lens)
    return 4 * blocks + 4 * wl.num_seqs


def test_decode_step_bytes_are_the_arrays_it_touches():
    for wl in (workloads.tiny(), workloads.llama31_8b(num_seqs=6)):
        decode, reshape, padded = bench.step_bytes(wl)
        # every logical K/V row is read once; q read and out written, both [n, Hq, d]
        assert decode == (wl.keys.nbytes + wl.values.nbytes + 2 * wl.q.nbytes
                          + table_and_length_bytes(wl))
        # the newest row of every sequence, K and V, written to the cache
        newest = wl.seq_start[1:] - 1
        assert reshape == wl.keys[newest].nbytes + wl.values[newest].nbytes
        # whole blocks: the rows of a block are contiguous, a block is B rows of every head
        row = wl.keys[0].nbytes // wl.num_kv_heads
        blocks = sum(-(-int(c) // wl.block_size) for c in wl.context_lens)
        assert padded == 2 * blocks * wl.block_size * wl.num_kv_heads * row
        assert padded >= decode - 2 * wl.q.nbytes - table_and_length_bytes(wl)


def test_quantised_step_bytes_match_the_oracle_rows():
    wl = workloads.custom("acct", [3, 17, 40], "bf16", 8, 2, 64, 16, 16, 64, seed=3)
    n, hkv = wl.num_seqs, wl.num_kv_heads
    fixed = 2 * wl.q.nbytes + table_and_length_bytes(wl)
    newest16 = 2 * wl.keys[wl.seq_start[1:] - 1].nbytes

    codes, scales = int4.quantize_rows(wl.keys, wl.dtype)
    decode, reshape = bench.fp8_step_bytes(wl, "int4")
    assert decode == 2 * (codes.nbytes + scales.nbytes) + fixed
    per_row = (codes.nbytes + scales.nbytes) // (codes.shape[0] * hkv)
    assert reshape == newest16 + 2 * n * hkv * per_row

    # one byte a code, no scale array per row (the FP8 scale is one number a tensor)
    decode, reshape = bench.fp8_step_bytes(wl, "fp8")
    assert decode == wl.keys.size + wl.values.size + fixed
    assert reshape == newest16 + 2 * n * hkv * wl.head_dim


def test_prefill_flops_count_the_causal_pairs():
    for wl in (workloads.prefill_tiny(), workloads.prefill_chunked(num_seqs=2, chunk=64)):
        qlen = np.diff(wl.query_start)
        pairs = 0
        for s in range(wl.num_seqs):
            c, n = int(wl.context_lens[s]), int(qlen[s])
            pos = np.arange(c - n, c)[:, None]          # positions of the new tokens
            pairs += int((np.arange(c)[None, :] <= pos).sum())
        # QK^T and PV: 2 d FLOPs each per (query head, query, key)
        assert bench.prefill_flops(wl) == pairs * 4 * wl.head_dim * wl.num_q_heads


def test_rotation_pool_holds_disjoint_copies():
    wl = workloads.tiny()
    need = sum(-(-int(c) // wl.block_size) for c in wl.context_lens)
    nb, order = bench.rotation_pool(wl, 1)
    assert nb == wl.num_blocks and order is wl.free_order
    rotate = wl.num_blocks // need + 2
    nb, order = bench.rotation_pool(wl, rotate)
    assert nb == rotate * need
    assert np.array_equal(np.sort(order), np.arange(nb))
    assert order.dtype == np.int32


def test_reference_arm_line_names_the_native_config(capsys, monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["config"] == bench.decode_config(workloads.tiny(), 1)
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    # another rank of a multi-rank launch does no work and prints nothing
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_reference_arm_rejects_what_it_does_not_time(monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    for name in ("prefill_tiny", "kv8_llama31_8b"):
        with pytest.raises(SystemExit):
            bench.main(["--impl", "reference", "--workload", name, "--steps", "3", "--warmup", "3"])
