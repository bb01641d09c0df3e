"""Host-side logic of the Python binding, on CPU with no GPU work: a planned launch
(plan=True on the decode step functions) holds every tensor its marshalled device
addresses point into, including a workspace the call created itself, for as long as the
launch object lives.  The device checks are replaced by address lookups so that the
marshalling runs on CPU tensors; nothing is launched."""
import gc
import weakref

import pytest
import torch

N, HQ, HKV, D, NB, B, T = 3, 8, 2, 64, 8, 16, 4


@pytest.fixture
def cpu_marshal(libpa, monkeypatch):
    made = []

    def workspace(hq, hkv, d, device=None):
        w = torch.empty(256, dtype=torch.uint8)
        made.append(weakref.ref(w))
        return w
    monkeypatch.setattr(libpa, "_dev", lambda t, name, dtype=None: t.data_ptr())
    monkeypatch.setattr(libpa, "_fp8_cache", lambda t, name: t.data_ptr())
    monkeypatch.setattr(libpa, "_int4_cache", lambda c, s, name: (c.data_ptr(), s.data_ptr()))
    monkeypatch.setattr(libpa, "make_workspace", workspace)
    return libpa, made


def step_inputs(dtype=torch.bfloat16):
    return dict(q=torch.zeros(N, HQ, D, dtype=dtype),
                key_new=torch.zeros(N, HKV, D, dtype=dtype),
                value_new=torch.zeros(N, HKV, D, dtype=dtype),
                block_tables=torch.zeros(N, T, dtype=torch.int32),
                context_lens=torch.ones(N, dtype=torch.int32))


def plans(pa):
    i = step_inputs()
    yield "16-bit", lambda: pa.decode_append(
        i["q"], i["key_new"], i["value_new"], torch.zeros(NB, HKV, B, D, dtype=torch.bfloat16),
        torch.zeros(NB, HKV, B, D, dtype=torch.bfloat16), i["block_tables"], i["context_lens"],
        0.125, plan=True)
    yield "fp8", lambda: pa.decode_append_fp8(
        i["q"], i["key_new"], i["value_new"], torch.zeros(NB, HKV, B, D, dtype=torch.uint8),
        torch.zeros(NB, HKV, B, D, dtype=torch.uint8), i["block_tables"], i["context_lens"],
        0.125, 0.5, 0.5, plan=True)
    yield "int4", lambda: pa.decode_append_int4(
        i["q"], i["key_new"], i["value_new"], torch.zeros(NB, HKV, B, D // 2, dtype=torch.uint8),
        torch.zeros(NB, HKV, B, D // 2, dtype=torch.uint8), torch.zeros(NB, HKV, B),
        torch.zeros(NB, HKV, B), i["block_tables"], i["context_lens"], 0.125, plan=True)


def test_planned_launch_holds_its_tensors(cpu_marshal):
    pa, made = cpu_marshal
    for name, make in plans(pa):
        made.clear()
        launch = make()
        gc.collect()
        assert isinstance(launch, pa.Launch), name
        # the workspace the call made is alive while the launch is
        assert len(made) == 1 and made[0]() is not None, name
        # every tensor address in the marshalled arguments is one the launch holds
        held = {t.data_ptr() for t in launch._keep}
        ptrs = [a for a in launch._args if isinstance(a, int) and a in held]
        assert made[0]().data_ptr() in ptrs and launch.out.data_ptr() in ptrs, name
        assert len(ptrs) >= 9, name
        del launch
        gc.collect()
        assert made[0]() is None, name


def test_argument_checks_name_the_argument(libpa):
    """The checks in front of the library raise ValueError naming the bad argument (their
    messages are built only on failure)."""
    import numpy as np
    t = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError, match="slot_mapping must be a CUDA tensor"):
        libpa._dev(t, "slot_mapping", torch.int64)
    with pytest.raises(ValueError, match="tables must be a writeable C-contiguous int32"):
        libpa._host_out(np.zeros(8, np.int64), np.int32, 4, "tables")
    with pytest.raises(ValueError, match="slots holds 3 entries, 4 needed"):
        libpa._host_out(np.zeros(3, np.int64), np.int64, 4, "slots")
    ro = np.zeros(8, np.int32)
    ro.flags.writeable = False
    with pytest.raises(ValueError, match="cached must be a writeable"):
        libpa._host_out(ro, np.int32, 4, "cached")
    a = np.zeros(8, np.int32)
    assert libpa._host_out(a, np.int32, 8, "cached") is a
    with pytest.raises(ValueError, match="k codes must be uint8"):
        libpa._int4_cache(torch.zeros(2, 2, 2, 2, dtype=torch.int8), torch.zeros(2, 2, 2), "k")
    with pytest.raises(ValueError, match="v scales must be float32"):
        libpa._int4_cache(torch.zeros(2, 2, 2, 2, dtype=torch.uint8),
                          torch.zeros(2, 2, 2, dtype=torch.float16), "v")
    with pytest.raises(ValueError, match="must hold E4M3 codes"):
        libpa._fp8_cache(torch.zeros(2, dtype=torch.float16), "k_cache")
    with pytest.raises(ValueError, match="must be a CUDA tensor or a pinned CPU tensor"):
        libpa._reachable(t, "src_k")


def test_calls_run_on_their_tensors_device(libpa, monkeypatch):
    """A call on tensors of another device than the current one makes that device current
    for the call (the library's per-device state is the current device's)."""
    pa = libpa
    entered = []

    class FakeDevice:
        def __init__(self, dev):
            self.dev = dev

        def __enter__(self):
            entered.append(self.dev)

        def __exit__(self, *exc):
            return False

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "device", FakeDevice)

    class T:
        def __init__(self, index):
            self.device = torch.device("cuda", index)

    seen = []
    fn = pa._runs_on(lambda t: t.device)(lambda t: seen.append(len(entered)))
    fn(T(0))
    assert entered == [] and seen == [0]
    fn(T(1))
    assert entered == [torch.device("cuda", 1)] and seen == [0, 1]
    # every device call of the binding is wrapped so
    for name in ("reshape_and_cache", "decode", "decode_append", "decode_fp8", "decode_int4",
                 "decode_append_fp8", "decode_append_int4", "prefill", "decode_fixed_scratch",
                 "copy_blocks", "copy_blocks_int4", "swap_blocks", "swap_blocks_int4",
                 "reshape_and_cache_fp8", "reshape_and_cache_int4"):
        assert hasattr(getattr(pa, name), "__wrapped__"), name
    # pools: the device named, else the CUDA side of the copy (a pinned CPU pool has none)
    class P:
        def __init__(self, index):
            self.device = torch.device("cuda", index) if index is not None else torch.device("cpu")
            self.is_cuda = index is not None
    assert pa._pool_device(P(None), P(2)) == torch.device("cuda", 2)
    assert pa._pool_device((P(3),), (P(None),)) == torch.device("cuda", 3)
    assert pa._pool_device(P(3), P(None), device="cuda:1") == torch.device("cuda", 1)
