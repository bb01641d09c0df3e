"""Empty work through every device call: no sequences, no tokens, no block pairs, or
sequences with no new tokens.  Each call returns success, leaves the caches as they were,
sets no device error bit and, where it has an output, returns zero rows."""
import pytest
import torch

import paged_kv_cache_149_gb300 as pa
from gpu_harness import device_error

pytestmark = pytest.mark.gpu

NB, HQ, HKV, B, D, T = 8, 8, 2, 16, 128, 4


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    device_error()


def filled(shape, dtype):
    g = torch.Generator(device="cpu").manual_seed(sum(shape))
    if dtype in (torch.float16, torch.bfloat16):
        return torch.randn(shape, generator=g).to(dtype).cuda()
    if dtype == torch.float32:
        return torch.rand(shape, generator=g).cuda()
    return torch.randint(0, 256, shape, generator=g, dtype=torch.int32).to(dtype).cuda()


def unchanged(*pairs):
    torch.cuda.synchronize()
    for before, after in pairs:
        assert torch.equal(before.view(torch.uint8), after.view(torch.uint8))


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_empty_16_bit_calls(dt):
    kc, vc = filled((NB, HKV, B, D), dt), filled((NB, HKV, B, D), dt)
    k0, v0 = kc.clone(), vc.clone()
    none3 = torch.empty((0, HKV, D), dtype=dt, device="cuda")
    q = torch.empty((0, HQ, D), dtype=dt, device="cuda")
    tables = torch.empty((0, T), dtype=torch.int32, device="cuda")
    lens = torch.empty((0,), dtype=torch.int32, device="cuda")
    slots = torch.empty((0,), dtype=torch.int64, device="cuda")
    pairs = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    pa.reshape_and_cache(none3, none3, kc, vc, slots)
    assert pa.decode(q, kc, vc, tables, lens, 0.1).shape == (0, HQ, D)
    assert pa.decode_append(q, none3, none3, kc, vc, tables, lens, 0.1).shape == (0, HQ, D)
    assert pa.decode_fixed_scratch(q, kc, vc, tables, lens, 0.1).shape == (0, HQ, D)
    pa.copy_blocks(kc, vc, pairs)
    host_k = torch.zeros((NB, HKV, B, D), dtype=dt).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    pa.swap_blocks(kc, vc, host_k, host_v, pairs)
    out = pa.prefill(q, kc, vc, tables, lens, torch.zeros(1, dtype=torch.int32, device="cuda"),
                     0.1, 0)
    assert out.shape == (0, HQ, D)
    unchanged((k0, kc), (v0, vc))
    assert not host_k.any() and not host_v.any()
    assert device_error() == 0


def test_prefill_with_no_new_tokens():
    """Sequences whose query spans are all empty (max_query_len 0): nothing is computed."""
    dt = torch.bfloat16
    kc, vc = filled((NB, HKV, B, D), dt), filled((NB, HKV, B, D), dt)
    tables = torch.arange(2 * T, dtype=torch.int32, device="cuda").view(2, T) % NB
    lens = torch.tensor([5, 17], dtype=torch.int32, device="cuda")
    q = torch.empty((0, HQ, D), dtype=dt, device="cuda")
    out = pa.prefill(q, kc, vc, tables, lens, torch.zeros(3, dtype=torch.int32, device="cuda"),
                     0.1, 0)
    assert out.shape == (0, HQ, D) and device_error() == 0


def test_empty_quantised_calls():
    dt = torch.bfloat16
    none3 = torch.empty((0, HKV, D), dtype=dt, device="cuda")
    q = torch.empty((0, HQ, D), dtype=dt, device="cuda")
    tables = torch.empty((0, T), dtype=torch.int32, device="cuda")
    lens = torch.empty((0,), dtype=torch.int32, device="cuda")
    slots = torch.empty((0,), dtype=torch.int64, device="cuda")
    pairs = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    # FP8 (E4M3 codes as bytes, per-tensor scales)
    k8, v8 = filled((NB, HKV, B, D), torch.uint8), filled((NB, HKV, B, D), torch.uint8)
    k80, v80 = k8.clone(), v8.clone()
    pa.reshape_and_cache_fp8(none3, none3, k8, v8, slots, 0.5, 0.25)
    assert pa.decode_fp8(q, k8, v8, tables, lens, 0.1, 0.5, 0.25).shape == (0, HQ, D)
    assert pa.decode_append_fp8(q, none3, none3, k8, v8, tables, lens, 0.1, 0.5,
                                0.25).shape == (0, HQ, D)
    # INT4 (two codes a byte, a float32 scale a row)
    k4, v4 = filled((NB, HKV, B, D // 2), torch.uint8), filled((NB, HKV, B, D // 2), torch.uint8)
    ks, vs = filled((NB, HKV, B), torch.float32), filled((NB, HKV, B), torch.float32)
    saved = [t.clone() for t in (k4, v4, ks, vs)]
    pa.reshape_and_cache_int4(none3, none3, k4, v4, ks, vs, slots)
    assert pa.decode_int4(q, k4, v4, ks, vs, tables, lens, 0.1).shape == (0, HQ, D)
    assert pa.decode_append_int4(q, none3, none3, k4, v4, ks, vs, tables, lens,
                                 0.1).shape == (0, HQ, D)
    pa.copy_blocks_int4(k4, v4, ks, vs, pairs)
    unchanged((k80, k8), (v80, v8), *zip(saved, (k4, v4, ks, vs)))
    assert device_error() == 0
