"""The C ABI library loads on a CPU-only host and exports every function that
include/pa.h declares (no GPU work is done here)."""
import os
import re

from conftest import ROOT


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("pa_decode", "pa_reshape_and_cache", "pa_copy_blocks", "pa_get_device_error",
              "pa_decode_workspace_size", "pa_pool_create", "pa_pool_append_slot"):
        assert n in names


def test_every_declared_symbol_is_exported(libpa):
    lib = libpa.lib()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing


def test_binding_covers_every_symbol(libpa):
    assert set(declared_functions()) == set(libpa.SIGNATURES)


def test_status_strings(libpa):
    assert libpa.status_string(0) == "ok"
    assert "exhausted" in libpa.status_string(libpa.PA_ERR_POOL_EXHAUSTED)


def test_host_argument_checks_need_no_gpu(libpa):
    lib = libpa.lib()
    # shape errors are rejected on the host before any CUDA call
    assert lib.pa_decode(None, None, None, None, 8, None, 4, 4, 3, 128, 16, 64, 0.1, None, None,
                         0, 0, None) == libpa.PA_ERR_ARG          # 4 % 3 != 0
    assert lib.pa_decode(None, None, None, None, 8, None, 4, 4, 2, 96, 16, 64, 0.1, None, None,
                         0, 0, None) == libpa.PA_ERR_ARG          # head_dim 96
    assert lib.pa_decode(None, None, None, None, 8, None, 4, 4, 2, 64, 12, 64, 0.1, None, None,
                         0, 0, None) == libpa.PA_ERR_ARG          # block_size 12
    assert lib.pa_decode(None, None, None, None, 8, None, 4, 4, 2, 64, 16, 64, float("nan"),
                         None, None, 0, 0, None) == libpa.PA_ERR_ARG
    assert lib.pa_decode(None, None, None, None, 8, None, 0, 4, 2, 64, 16, 64, 0.1, None, None,
                         0, 0, None) == libpa.PA_OK               # empty batch: no-op
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, 64, 2, 64, 16, 0,
                                    None) == libpa.PA_OK
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 3, 64, 2, 64, 16, 0,
                                    None) == libpa.PA_ERR_ARG
    assert lib.pa_copy_blocks(None, None, None, 0, 64, 2, 64, 16, 1, None) == libpa.PA_OK
    assert lib.pa_copy_blocks(None, None, None, 2, 64, 2, 64, 16, 7, None) == libpa.PA_ERR_ARG


def test_check_block_mapping(libpa):
    libpa.check_block_mapping([(0, 3), (1, 4)], 8)
    import pytest
    for bad in ([(0, 3), (1, 3)], [(0, 3), (3, 4)], [(0, 8)], [(-1, 2)]):
        with pytest.raises(libpa.PagedAttentionError):
            libpa.check_block_mapping(bad, 8)


def test_build_compiles_every_source():
    """build() compiles the sources it lists and nothing else, on whichever host builds the
    library: every .cu / .cpp under csrc must be listed."""
    from paged_kv_cache_149_gb300 import build as b
    on_disk = sorted(f for f in os.listdir(b.CSRC) if f.endswith((".cu", ".cpp")))
    assert sorted(b.SOURCES) == on_disk


def test_each_decode_variant_is_instantiated_once():
    """Every (K/V format, fused step or not) set of decode kernels is explicitly
    instantiated in exactly one translation unit, and declared extern everywhere else."""
    from paged_kv_cache_149_gb300 import build as b
    found = {}
    for f in b.SOURCES:
        src = open(os.path.join(b.CSRC, f)).read()
        for kv, new in re.findall(r"^\s*template int launch_format<(\w+), (true|false)>", src, re.M):
            found.setdefault((kv, new), []).append(f)
    want = {(kv, new) for kv in ("kKv16", "kKvFp8", "kKvInt4") for new in ("true", "false")}
    assert set(found) == want
    assert all(len(v) == 1 for v in found.values()), found
    hdr = open(os.path.join(b.CSRC, "pa_decode_kernel.cuh")).read()
    externs = set(re.findall(r"extern template int launch_format<(\w+), (true|false)>", hdr))
    assert externs == want
