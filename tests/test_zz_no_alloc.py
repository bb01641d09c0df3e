"""pa_decode_fixed_scratch: decode for callers that cannot allocate device memory.

Such callers (a server that reserved nearly all HBM for the KV block pool, a host
framework that owns every device buffer) cannot pass pa_decode a workspace; this entry
point uses a fixed scratch array inside the library instead.  These tests call it
through the C ABI and check it against pa_decode on the same inputs, twice in a row
(the second call runs on scratch the first one left behind): the same kernels in the
same order, so the same bits.  They also check that the calls allocate nothing: torch's
allocator is untouched, and the device's free memory does not change across a call once
the library's scratch array is loaded.  The file is named to be collected last.
"""
import ctypes
import gc

import numpy as np
import pytest
import torch

import workloads
from gpu_harness import TOL, GpuBatch, device_error, max_err, oracle_seq_bits, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()


def fixed_scratch_call(lib, gb, out):
    wl = gb.wl
    stream = torch.cuda.current_stream().cuda_stream
    return lib.pa_decode_fixed_scratch(
        gb.q.data_ptr(), gb.k_cache.data_ptr(), gb.v_cache.data_ptr(), gb.tables.data_ptr(),
        gb.tables.shape[1], gb.ctx.data_ptr(), wl.num_seqs, wl.num_q_heads, wl.num_kv_heads,
        wl.head_dim, wl.block_size, wl.num_blocks, ctypes.c_float(wl.scale), out.data_ptr(),
        1 if wl.dtype == "bf16" else 0, ctypes.c_void_p(stream))


def memory_state():
    """(torch's allocated bytes, its reserved bytes, the device's free bytes), with Python's
    garbage collected first so that no unrelated tensor is freed in between."""
    gc.collect()
    torch.cuda.synchronize()
    return (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(),
            torch.cuda.mem_get_info()[0])


@pytest.mark.parametrize("recipe", ["llama31_8b", "long_cut"])
def test_fixed_scratch_matches_pa_decode_twice(libpa, recipe):
    if recipe == "llama31_8b":
        wl = workloads.llama31_8b()
    else:  # one long sequence cut across many CTAs: the scratch carries the split pieces
        wl = workloads.custom("long_cut", [20000, 300, 4096], "fp16", 8, 2, 128, 16, 1600, 20480, seed=21)
    gb = GpuBatch(wl)
    ref = to_bits(gb.decode())
    lib = libpa.lib()
    outs = [torch.full_like(gb.q, float("nan")) for _ in range(2)]
    states = []
    for out in outs:
        states.append(memory_state())
        assert fixed_scratch_call(lib, gb, out) == libpa.PA_OK
        states.append(memory_state())
        np.testing.assert_array_equal(to_bits(out), ref)
        assert device_error() == 0
    # torch's allocator grew by nothing over either call
    for before, after in ((states[0], states[1]), (states[2], states[3])):
        assert after[0] <= before[0] and after[1] <= before[1]
    # and the device lost no memory over the second call (the first one may load the
    # library's scratch array, where CUDA loads modules lazily)
    assert states[3][2] >= states[2][2]
    got = to_bits(outs[1])
    worst = max(max_err(got[s], oracle_seq_bits(wl, s), wl.dtype) for s in range(wl.num_seqs))
    assert worst <= TOL[wl.dtype]


def test_fixed_scratch_rejects_bad_arguments(libpa):
    lib = libpa.lib()
    # head_dim 96 is not supported: rejected on the host, nothing launched
    st = lib.pa_decode_fixed_scratch(None, None, None, None, 8, None, 4, 4, 2, 96, 16, 64,
                                     ctypes.c_float(0.1), None, 0, None)
    assert st == libpa.PA_ERR_ARG
