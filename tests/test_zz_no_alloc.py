"""pa_decode_fixed_scratch: decode for callers that cannot allocate device memory.

Such callers (a server that reserved nearly all HBM for the KV block pool, a host
framework that owns every device buffer) cannot pass pa_decode a workspace; this entry
point uses a fixed scratch array inside the library instead.  These tests call it
through the C ABI and check it against pa_decode on the same inputs, twice in a row
(the second call runs on scratch the first one left behind).  The file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_harness import TOL, GpuBatch, device_error, max_err, to_bits

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


@pytest.mark.parametrize("recipe", ["llama31_8b", "long_cut"])
def test_fixed_scratch_matches_pa_decode_twice(libpa, recipe):
    if recipe == "llama31_8b":
        wl = workloads.llama31_8b()
    else:  # one long sequence cut across many CTAs: the scratch carries the split pieces
        wl = workloads.custom("long_cut", [20000, 300, 4096], "fp16", 8, 2, 128, 16, 1600, 20480, seed=21)
    gb = GpuBatch(wl)
    ref = to_bits(gb.decode())
    lib = libpa.lib()
    for _ in range(2):
        out = torch.full_like(gb.q, float("nan"))
        assert fixed_scratch_call(lib, gb, out) == libpa.PA_OK
        got = to_bits(out)
        assert max_err(got, ref, wl.dtype) <= TOL[wl.dtype]
        assert device_error() == 0


def test_fixed_scratch_rejects_bad_arguments(libpa):
    lib = libpa.lib()
    # head_dim 96 is not supported: rejected on the host, nothing launched
    st = lib.pa_decode_fixed_scratch(None, None, None, None, 8, None, 4, 4, 2, 96, 16, 64,
                                     ctypes.c_float(0.1), None, 0, None)
    assert st == libpa.PA_ERR_ARG
