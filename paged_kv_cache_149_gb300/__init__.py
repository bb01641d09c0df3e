"""Python binding of libpa.so: paged KV-cache decode attention on GB300 (sm_103a).

Argument marshalling only.  Every computation runs in the library's CUDA kernels (or,
for the block pool, its C++ host code); PyTorch supplies device memory and streams.
The functions take torch tensors, check dtypes/devices/shapes, pass raw pointers and
the current CUDA stream to the C ABI (include/pa.h) and raise ``PagedAttentionError``
on a negative status.  If libpa.so is missing the import of this package still works
but every call raises: there is no fallback path.

Layouts (row-major):
    q, out        [num_seqs, num_q_heads, head_dim]            fp16 / bf16
    k_cache       [num_blocks, num_kv_heads, block_size, head_dim]
    v_cache       [num_blocks, num_kv_heads, block_size, head_dim]
    block_tables  [num_seqs, max_blocks_per_seq] int32
    context_lens  [num_seqs] int32
    key, value    [num_tokens, num_kv_heads, head_dim]
    slot_mapping  [num_tokens] int64
    block_mapping [num_pairs, 2] int32
"""
import ctypes
import functools
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_OK = 0
PA_ERR_ARG = -1
PA_ERR_WORKSPACE = -2
PA_ERR_CUDA = -3
PA_ERR_POOL_EXHAUSTED = -4
PA_ERR_UNKNOWN_SEQ = -5
PA_ERR_WRONG_TIER = -6

DEVERR_BAD_BLOCK = 0x1
DEVERR_BAD_CONTEXT = 0x2
DEVERR_BAD_SLOT = 0x4
DEVERR_BAD_PAIR = 0x8
DEVERR_TIMEOUT = 0x10

PA_FP16 = 0
PA_BF16 = 1
PA_FP8_E4M3 = 2

_c = ctypes
_vp, _i32, _i64, _sz, _f32 = _c.c_void_p, _c.c_int, _c.c_int64, _c.c_size_t, _c.c_float

# name -> (restype, argtypes); mirrors include/pa.h
SIGNATURES = {
    "pa_reshape_and_cache": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp]),
    "pa_decode": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                         _f32, _vp, _vp, _sz, _i32, _vp]),
    "pa_decode_append": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                _i32, _i32, _f32, _vp, _vp, _sz, _i32, _vp]),
    "pa_decode_fp8": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                             _f32, _f32, _f32, _vp, _vp, _sz, _i32, _vp]),
    "pa_decode_append_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                    _i32, _i32, _i32, _f32, _f32, _f32, _vp, _vp, _sz, _i32,
                                    _vp]),
    "pa_reshape_and_cache_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                        _f32, _f32, _i32, _vp]),
    "pa_reshape_and_cache_int4": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                         _i32, _i32, _i32, _vp]),
    "pa_decode_int4": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                              _i32, _i32, _f32, _vp, _vp, _sz, _i32, _vp]),
    "pa_decode_append_int4": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32,
                                     _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _sz, _i32,
                                     _vp]),
    "pa_copy_blocks_int4": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp]),
    "pa_swap_blocks_int4": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                   _i32, _i32, _i32, _vp]),
    "pa_prefill": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                          _i32, _i32, _f32, _vp, _i32, _vp]),
    "pa_decode_workspace_size": (_sz, [_i32, _i32, _i32]),
    "pa_decode_timeline": (_i32, [_vp, _sz]),
    "pa_decode_fixed_scratch": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                       _i32, _f32, _vp, _i32, _vp]),
    "pa_copy_blocks": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp]),
    "pa_swap_blocks": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                              _vp]),
    "pa_check_block_mapping": (_i32, [_vp, _i32, _i32]),
    "pa_get_device_error": (_i32, [_vp, _c.POINTER(_c.c_uint32)]),
    "pa_status_string": (_c.c_char_p, [_i32]),
    "pa_pool_create": (_vp, [_i32, _i32, _vp]),
    "pa_pool_create_tiered": (_vp, [_i32, _i32, _vp, _i32, _vp]),
    "pa_pool_destroy": (None, [_vp]),
    "pa_pool_allocate": (_i32, [_vp, _i64, _i32]),
    "pa_pool_append_slot": (_i32, [_vp, _i64, _c.POINTER(_i64), _c.POINTER(_c.c_int32),
                                   _c.POINTER(_c.c_int32)]),
    "pa_pool_fork": (_i32, [_vp, _i64, _i64]),
    "pa_pool_free": (_i32, [_vp, _i64]),
    "pa_pool_block_table": (_i32, [_vp, _i64, _vp, _i32]),
    "pa_pool_context_len": (_i32, [_vp, _i64]),
    "pa_pool_slots": (_i32, [_vp, _i64, _i32, _i32, _vp]),
    "pa_pool_num_free": (_i32, [_vp]),
    "pa_pool_free_list": (_i32, [_vp, _vp, _i32]),
    "pa_pool_refcount": (_i32, [_vp, _c.c_int32]),
    "pa_pool_swap_out": (_i32, [_vp, _vp, _i32, _vp, _i32]),
    "pa_pool_swap_in": (_i32, [_vp, _vp, _i32, _vp, _i32]),
    "pa_pool_is_swapped": (_i32, [_vp, _i64]),
    "pa_pool_num_free_cpu": (_i32, [_vp]),
    "pa_pool_cpu_free_list": (_i32, [_vp, _vp, _i32]),
    "pa_pool_cpu_refcount": (_i32, [_vp, _c.c_int32]),
    "pa_pool_allocate_prefix": (_i32, [_vp, _i64, _vp, _i32, _vp, _i32, _c.POINTER(_c.c_int)]),
    "pa_pool_num_cached": (_i32, [_vp]),
    "pa_pool_table_width": (_i32, [_vp, _i32, _vp]),
    "pa_pool_allocate_prefix_batch": (_i32, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                             _i32, _c.POINTER(_c.c_int)]),
    "pa_pool_allocate_hashed_batch": (_i32, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                             _c.POINTER(_c.c_int)]),
    "pa_pool_free_batch": (_i32, [_vp, _vp, _i32]),
    "pa_pool_block_digest": (_i32, [_vp, _c.c_int32, _vp]),
    "pa_prefix_block_hashes": (_i32, [_vp, _i32, _i32, _vp, _i32, _vp, _i32]),
    "pa_sha256": (_i32, [_vp, _sz, _vp]),
}

_lib = None


class PagedAttentionError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else status_string(status))


class PoolExhausted(PagedAttentionError):
    pass


class UnknownSequence(PagedAttentionError):
    pass


class WrongTier(PagedAttentionError):
    pass


def lib():
    """The loaded libpa.so (ctypes), with argument types set.  Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_149_gb300.build` "
                "(nvcc, sm_103a).  There is no CPU or PyTorch fallback.")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def status_string(status):
    return lib().pa_status_string(int(status)).decode()


def _check(status, what):
    if status < 0:
        if status == PA_ERR_POOL_EXHAUSTED:
            raise PoolExhausted(status, what)
        if status == PA_ERR_UNKNOWN_SEQ:
            raise UnknownSequence(status, what)
        if status == PA_ERR_WRONG_TIER:
            raise WrongTier(status, what)
        raise PagedAttentionError(status, what)
    return status


def _switch_to(dev):
    """The device to make current for a call on tensors of `dev`, or None when it already
    is (the library works on the current device: its SM count, error word and scratch)."""
    import torch
    if dev is None or dev.type != "cuda" or dev.index is None:
        return None
    return None if dev.index == torch.cuda.current_device() else dev


def _runs_on(pick):
    """Decorator: run the call with the device `pick(*args, **kw)` current."""
    def deco(fn):
        @functools.wraps(fn)
        def wrapped(*args, **kw):
            dev = _switch_to(pick(*args, **kw))
            if dev is None:
                return fn(*args, **kw)
            import torch
            with torch.cuda.device(dev):
                return fn(*args, **kw)
        return wrapped
    return deco


# the device of the call's first tensor argument
_on_first = _runs_on(lambda t, *args, **kw: t.device)


def _pool_device(src, dst, *args, device=None, **kw):
    """The device of a copy between pools that may be pinned CPU memory."""
    import torch
    if device is not None:
        return torch.device(device)
    firsts = (src[0], dst[0]) if isinstance(src, (tuple, list)) else (src, dst)
    return next((t.device for t in firsts if t.is_cuda), None)


class Launch:
    """A library call whose arguments were checked and marshalled once (``plan=True`` on
    the decode step functions, prefill and reshape_and_cache): ``run(stream)`` issues it
    again on ``stream`` over the
    same buffers, whose contents may change between runs.  For serving loops that launch
    the same step shape many times; the per-call cost is one foreign call.  The marshalled
    arguments are raw device addresses, so the Launch holds a reference to every tensor
    they point into (a workspace the call created included): none is freed, and its
    memory reused, while the Launch can still run.  Drop the Launch only after its last
    run has finished, or ordered before later work on the stream it ran on.  A run makes
    the planned tensors' device current if another one is."""

    def __init__(self, name, args, out, keep=()):
        self._fn = getattr(lib(), name)
        self._name = name
        self._args = args
        self._keep = tuple(keep)
        self.out = out
        self.device = out.device

    def run(self, stream):
        dev = _switch_to(self.device)
        if dev is None:
            st = self._fn(*self._args, stream.cuda_stream)
        else:
            import torch
            with torch.cuda.device(dev):
                st = self._fn(*self._args, stream.cuda_stream)
        if st < 0:
            _check(st, self._name)
        return self.out


# ----------------------------------------------------------------- device calls

def _dtype_code(t):
    import torch
    if t.dtype == torch.float16:
        return PA_FP16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; expected float16 or bfloat16")


def _cache_code(t):
    """dtype code of a K/V cache tensor: 16-bit floats, or FP8 E4M3 codes (uint8 or
    torch.float8_e4m3fn)."""
    import torch
    if t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        return PA_FP8_E4M3
    return _dtype_code(t)


def _stream_ptr(stream, device):
    import torch
    s = torch.cuda.current_stream(device) if stream is None else stream
    return s.cuda_stream


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _host_out(arr, dtype, size, name):
    """A caller's host array the library writes `size` elements of: a writeable C-contiguous
    NumPy array of `dtype` with room for them."""
    import numpy as np
    # (messages are formatted only on failure: these checks run on every serving step)
    if not (isinstance(arr, np.ndarray) and arr.dtype == dtype and arr.flags.c_contiguous
            and arr.flags.writeable):
        raise ValueError(f"{name} must be a writeable C-contiguous {np.dtype(dtype).name} array")
    if arr.size < size:
        raise ValueError(f"{name} holds {arr.size} entries, {size} needed")
    return arr


def _dev(t, name, dtype=None):
    if not (t.is_cuda and t.is_contiguous() and (dtype is None or t.dtype == dtype)):
        _need(t.is_cuda, f"{name} must be a CUDA tensor")
        _need(t.is_contiguous(), f"{name} must be contiguous")
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


@_on_first
def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, stream=None, plan=False):
    """k_cache[slot // B, h, slot % B] = key[i, h] (and V) for every slot >= 0.  plan=True
    returns a Launch (whose run writes the rows the buffers hold then) instead of writing."""
    import torch
    n, hkv, d = key.shape
    nb, hkv2, bs, d2 = k_cache.shape
    _need(value.shape == key.shape and v_cache.shape == k_cache.shape, "shape mismatch")
    _need(hkv == hkv2 and d == d2 and slot_mapping.shape == (n,), "shape mismatch")
    _need(key.dtype == value.dtype == k_cache.dtype == v_cache.dtype, "dtype mismatch")
    args = (_dev(key, "key"), _dev(value, "value"), _dev(k_cache, "k_cache"),
            _dev(v_cache, "v_cache"), _dev(slot_mapping, "slot_mapping", torch.int64), n, nb, hkv,
            d, bs, _dtype_code(key))
    if plan:
        return Launch("pa_reshape_and_cache", args, k_cache,
                      keep=(key, value, v_cache, slot_mapping))
    st = lib().pa_reshape_and_cache(*args, _stream_ptr(stream, key.device))
    _check(st, "pa_reshape_and_cache")


def decode_workspace_size(num_q_heads, num_kv_heads, head_dim):
    """Bytes of workspace pa_decode needs on the current device."""
    n = lib().pa_decode_workspace_size(num_q_heads, num_kv_heads, head_dim)
    if n == 0:
        raise PagedAttentionError(PA_ERR_ARG, "pa_decode_workspace_size")
    return n


def decode_timeline(buffer=None):
    """Diagnostics (pa_decode_timeline): while `buffer` is set -- a device int64 tensor of
    at least SM count x 8 x 3 entries -- every 16-bit decode launch from this thread writes
    its warps' phase stamps into it, [cta][warp][k]; None clears the setting."""
    if buffer is None:
        _check(lib().pa_decode_timeline(None, 0), "pa_decode_timeline")
        return
    import torch
    if buffer.dtype != torch.int64 or not buffer.is_cuda or not buffer.is_contiguous():
        raise PagedAttentionError(PA_ERR_ARG, "pa_decode_timeline: a contiguous device int64 tensor")
    _check(lib().pa_decode_timeline(buffer.data_ptr(), buffer.numel() * 8), "pa_decode_timeline")


def make_workspace(num_q_heads, num_kv_heads, head_dim, device=None):
    import torch
    return torch.empty(decode_workspace_size(num_q_heads, num_kv_heads, head_dim),
                       dtype=torch.uint8, device=device or "cuda")


def _scratch(num_q_heads, num_kv_heads, head_dim, device, stream):
    """A workspace for one call launched on `stream`, allocated on that stream: the caching
    allocator then reuses its memory, once the call returns and the tensor is dropped, only
    for work ordered after the call on that stream."""
    import torch
    if stream is None:
        return make_workspace(num_q_heads, num_kv_heads, head_dim, device)
    with torch.cuda.stream(stream):
        return make_workspace(num_q_heads, num_kv_heads, head_dim, device)


@_on_first
def decode(q, k_cache, v_cache, block_tables, context_lens, scale, out=None, workspace=None,
           stream=None):
    """Paged decode attention; returns ``out`` [num_seqs, num_q_heads, head_dim]."""
    import torch
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    _need(v_cache.shape == k_cache.shape and d == d2, "shape mismatch")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == n, "block_tables must be [num_seqs, T]")
    _need(context_lens.shape == (n,), "context_lens must be [num_seqs]")
    _need(q.dtype == k_cache.dtype == v_cache.dtype, "dtype mismatch")
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        workspace = _scratch(hq, hkv, d, q.device, stream)
    st = lib().pa_decode(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), n, hq, hkv, d, bs, nb, float(scale),
        _dev(out, "out"), _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dtype_code(q), _stream_ptr(stream, q.device))
    _check(st, "pa_decode")
    return out


@_on_first
def decode_append(q, key_new, value_new, k_cache, v_cache, block_tables, context_lens, scale,
                  out=None, workspace=None, stream=None, plan=False):
    """One decode step in one kernel: writes each sequence's newest token (``key_new`` /
    ``value_new`` [num_seqs, num_kv_heads, head_dim], at position context_lens[s] - 1) into
    the caches and returns attention over contexts that include it.  Same results as
    reshape_and_cache into those slots followed by decode.  plan=True returns a Launch
    instead of launching."""
    import torch
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    _need(v_cache.shape == k_cache.shape and d == d2, "shape mismatch")
    _need(key_new.shape == (n, hkv, d) and value_new.shape == (n, hkv, d),
          "key_new / value_new must be [num_seqs, num_kv_heads, head_dim]")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == n, "block_tables must be [num_seqs, T]")
    _need(context_lens.shape == (n,), "context_lens must be [num_seqs]")
    _need(q.dtype == k_cache.dtype == v_cache.dtype == key_new.dtype == value_new.dtype,
          "dtype mismatch")
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        workspace = _scratch(hq, hkv, d, q.device, stream)
    args = (_dev(q, "q"), _dev(key_new, "key_new"), _dev(value_new, "value_new"),
            _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
            _dev(context_lens, "context_lens", torch.int32), n, hq, hkv, d, bs, nb, float(scale),
            _dev(out, "out"), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _dtype_code(q))
    if plan:
        return Launch("pa_decode_append", args, out,
                      keep=(q, key_new, value_new, k_cache, v_cache, block_tables,
                            context_lens, out, workspace))
    _check(lib().pa_decode_append(*args, _stream_ptr(stream, q.device)), "pa_decode_append")
    return out


def _fp8_cache(t, name):
    import torch
    if t.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        raise ValueError(f"{name} must hold E4M3 codes (uint8 or float8_e4m3fn), got {t.dtype}")
    return _dev(t, name)


@_on_first
def reshape_and_cache_fp8(key, value, k_cache, v_cache, slot_mapping, k_scale, v_scale,
                          stream=None):
    """FP8 cache write: k_cache[slot // B, h, slot % B] = E4M3(key[i, h] / k_scale) (and V)."""
    import torch
    n, hkv, d = key.shape
    nb, hkv2, bs, d2 = k_cache.shape
    _need(value.shape == key.shape and v_cache.shape == k_cache.shape, "shape mismatch")
    _need(hkv == hkv2 and d == d2 and slot_mapping.shape == (n,), "shape mismatch")
    _need(key.dtype == value.dtype, "dtype mismatch")
    st = lib().pa_reshape_and_cache_fp8(
        _dev(key, "key"), _dev(value, "value"), _fp8_cache(k_cache, "k_cache"),
        _fp8_cache(v_cache, "v_cache"), _dev(slot_mapping, "slot_mapping", torch.int64), n, nb,
        hkv, d, bs, float(k_scale), float(v_scale), _dtype_code(key),
        _stream_ptr(stream, key.device))
    _check(st, "pa_reshape_and_cache_fp8")


@_on_first
def decode_fp8(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale,
               out=None, workspace=None, stream=None):
    """Paged decode over FP8 E4M3 blocks (codes times k_scale / v_scale); q and out are
    fp16 or bf16."""
    import torch
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    _need(v_cache.shape == k_cache.shape and d == d2, "shape mismatch")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == n, "block_tables must be [num_seqs, T]")
    _need(context_lens.shape == (n,), "context_lens must be [num_seqs]")
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        workspace = _scratch(hq, hkv, d, q.device, stream)
    st = lib().pa_decode_fp8(
        _dev(q, "q"), _fp8_cache(k_cache, "k_cache"), _fp8_cache(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), n, hq, hkv, d, bs, nb, float(scale),
        float(k_scale), float(v_scale), _dev(out, "out"), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dtype_code(q), _stream_ptr(stream, q.device))
    _check(st, "pa_decode_fp8")
    return out


@_on_first
def decode_append_fp8(q, key_new, value_new, k_cache, v_cache, block_tables, context_lens,
                      scale, k_scale, v_scale, out=None, workspace=None, stream=None, plan=False):
    """One FP8 decode step in one kernel: each sequence's newest K/V row is quantised into
    its slot at position ctx - 1 (read from the block tables) and attended (= bit for bit
    reshape_and_cache_fp8 + decode_fp8).  plan=True returns a Launch instead of launching."""
    import torch
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    _need(v_cache.shape == k_cache.shape and d == d2, "shape mismatch")
    _need(key_new.shape == (n, hkv, d) and value_new.shape == key_new.shape, "key_new must be [n, Hkv, d]")
    _need(key_new.dtype == value_new.dtype == q.dtype, "dtype mismatch")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == n, "block_tables must be [num_seqs, T]")
    _need(context_lens.shape == (n,), "context_lens must be [num_seqs]")
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        workspace = _scratch(hq, hkv, d, q.device, stream)
    args = (_dev(q, "q"), _dev(key_new, "key_new"), _dev(value_new, "value_new"),
            _fp8_cache(k_cache, "k_cache"), _fp8_cache(v_cache, "v_cache"),
            _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
            _dev(context_lens, "context_lens", torch.int32), n, hq, hkv, d, bs, nb, float(scale),
            float(k_scale), float(v_scale), _dev(out, "out"), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _dtype_code(q))
    if plan:
        return Launch("pa_decode_append_fp8", args, out,
                      keep=(q, key_new, value_new, k_cache, v_cache, block_tables,
                            context_lens, out, workspace))
    _check(lib().pa_decode_append_fp8(*args, _stream_ptr(stream, q.device)), "pa_decode_append_fp8")
    return out


@_on_first
def prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
            max_query_len, out=None, stream=None, plan=False):
    """Causal attention of each sequence's newest tokens (q rows query_start[s] ..
    query_start[s+1]-1, at positions ctx - q_len .. ctx - 1, their K/V already in the cache)
    over its paged context; returns ``out`` shaped like q.  plan=True returns a Launch
    instead of launching: its runs read the tables, lengths and offsets the buffers hold
    then, so max_query_len must stay an upper bound of the query counts."""
    import torch
    ntok, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    n = context_lens.shape[0]
    _need(v_cache.shape == k_cache.shape and d == d2, "shape mismatch")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == n, "block_tables must be [num_seqs, T]")
    _need(query_start.shape == (n + 1,), "query_start must be [num_seqs + 1]")
    _need(q.dtype == k_cache.dtype == v_cache.dtype, "dtype mismatch")
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    args = (_dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
            _dev(context_lens, "context_lens", torch.int32),
            _dev(query_start, "query_start", torch.int32), n, int(max_query_len), hq, hkv, d, bs,
            nb, float(scale), _dev(out, "out"), _dtype_code(q))
    if plan:
        return Launch("pa_prefill", args, out,
                      keep=(q, k_cache, v_cache, block_tables, context_lens, query_start))
    st = lib().pa_prefill(*args, _stream_ptr(stream, q.device))
    _check(st, "pa_prefill")
    return out


@_on_first
def decode_fixed_scratch(q, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                         stream=None):
    """Paged decode that allocates nothing on the device: its scratch is a fixed array
    inside the library (see pa_decode_fixed_scratch in include/pa.h).  For callers that
    cannot allocate device memory; calls whose GPU work overlaps race on that scratch."""
    import torch
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    _need(v_cache.shape == k_cache.shape and d == d2, "shape mismatch")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == n, "block_tables must be [num_seqs, T]")
    _need(context_lens.shape == (n,), "context_lens must be [num_seqs]")
    _need(q.dtype == k_cache.dtype == v_cache.dtype, "dtype mismatch")
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    st = lib().pa_decode_fixed_scratch(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), n, hq, hkv, d, bs, nb, float(scale),
        _dev(out, "out"), _dtype_code(q), _stream_ptr(stream, q.device))
    _check(st, "pa_decode_fixed_scratch")
    return out


def _int4_cache(codes, scales, name):
    import torch
    if codes.dtype != torch.uint8:
        raise ValueError(f"{name} codes must be uint8 (two 4-bit codes a byte)")
    if scales.dtype != torch.float32:
        raise ValueError(f"{name} scales must be float32")
    if not (codes.dim() == 4 and scales.shape == codes.shape[:3]):
        raise ValueError(f"{name}: codes [NB, Hkv, B, d/2] and scales [NB, Hkv, B]")
    return _dev(codes, name), _dev(scales, name + " scales")


@_on_first
def reshape_and_cache_int4(key, value, k_codes, v_codes, k_scales, v_scales, slot_mapping,
                           stream=None):
    """INT4 cache write: the row key[i, h] gets s = max|x| / 7 and codes rint(x / s) in
    [-7, 7] at slot_mapping[i] (and V likewise)."""
    import torch
    n, hkv, d = key.shape
    nb, hkv2, bs, d2 = k_codes.shape
    _need(value.shape == key.shape and v_codes.shape == k_codes.shape, "shape mismatch")
    _need(hkv == hkv2 and d == 2 * d2 and slot_mapping.shape == (n,), "shape mismatch")
    _need(key.dtype == value.dtype, "dtype mismatch")
    kc, ks = _int4_cache(k_codes, k_scales, "k")
    vc, vs = _int4_cache(v_codes, v_scales, "v")
    st = lib().pa_reshape_and_cache_int4(
        _dev(key, "key"), _dev(value, "value"), kc, vc, ks, vs,
        _dev(slot_mapping, "slot_mapping", torch.int64), n, nb, hkv, d, bs, _dtype_code(key),
        _stream_ptr(stream, key.device))
    _check(st, "pa_reshape_and_cache_int4")


@_on_first
def decode_int4(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, scale,
                out=None, workspace=None, stream=None):
    """Paged decode over INT4 blocks (codes [NB, Hkv, B, d/2] uint8, scales [NB, Hkv, B])."""
    import torch
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_codes.shape
    _need(v_codes.shape == k_codes.shape and d == 2 * d2, "shape mismatch")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == n, "block_tables must be [num_seqs, T]")
    _need(context_lens.shape == (n,), "context_lens must be [num_seqs]")
    kc, ks = _int4_cache(k_codes, k_scales, "k")
    vc, vs = _int4_cache(v_codes, v_scales, "v")
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        workspace = _scratch(hq, hkv, d, q.device, stream)
    st = lib().pa_decode_int4(
        _dev(q, "q"), kc, vc, ks, vs, _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), n, hq, hkv, d, bs,
        nb, float(scale), _dev(out, "out"), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dtype_code(q), _stream_ptr(stream, q.device))
    _check(st, "pa_decode_int4")
    return out


@_on_first
def decode_append_int4(q, key_new, value_new, k_codes, v_codes, k_scales, v_scales, block_tables,
                       context_lens, scale, out=None, workspace=None, stream=None, plan=False):
    """One INT4 decode step in one kernel: each sequence's newest K/V row is quantised into
    its slot at position ctx - 1 and attended (= bit for bit reshape_and_cache_int4 +
    decode_int4).  plan=True returns a Launch instead of launching."""
    import torch
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_codes.shape
    _need(v_codes.shape == k_codes.shape and d == 2 * d2, "shape mismatch")
    _need(key_new.shape == (n, hkv, d) and value_new.shape == key_new.shape, "key_new must be [n, Hkv, d]")
    _need(key_new.dtype == value_new.dtype == q.dtype, "dtype mismatch")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == n, "block_tables must be [num_seqs, T]")
    _need(context_lens.shape == (n,), "context_lens must be [num_seqs]")
    kc, ks = _int4_cache(k_codes, k_scales, "k")
    vc, vs = _int4_cache(v_codes, v_scales, "v")
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        workspace = _scratch(hq, hkv, d, q.device, stream)
    args = (_dev(q, "q"), _dev(key_new, "key_new"), _dev(value_new, "value_new"), kc, vc, ks, vs,
            _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
            _dev(context_lens, "context_lens", torch.int32), n, hq, hkv, d, bs, nb, float(scale),
            _dev(out, "out"), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _dtype_code(q))
    if plan:
        return Launch("pa_decode_append_int4", args, out,
                      keep=(q, key_new, value_new, k_codes, v_codes, k_scales, v_scales,
                            block_tables, context_lens, out, workspace))
    _check(lib().pa_decode_append_int4(*args, _stream_ptr(stream, q.device)), "pa_decode_append_int4")
    return out


@_on_first
def copy_blocks_int4(k_codes, v_codes, k_scales, v_scales, block_mapping, stream=None):
    """copy_blocks for INT4 blocks: codes and scales of each (src, dst) pair."""
    import torch
    nb, hkv, bs, d2 = k_codes.shape
    _need(v_codes.shape == k_codes.shape, "shape mismatch")
    _need(block_mapping.dim() == 2 and block_mapping.shape[1] == 2, "block_mapping must be [n, 2]")
    kc, ks = _int4_cache(k_codes, k_scales, "k")
    vc, vs = _int4_cache(v_codes, v_scales, "v")
    st = lib().pa_copy_blocks_int4(kc, vc, ks, vs, _dev(block_mapping, "block_mapping", torch.int32),
                                   block_mapping.shape[0], nb, hkv, 2 * d2, bs,
                                   _stream_ptr(stream, k_codes.device))
    _check(st, "pa_copy_blocks_int4")


@_runs_on(_pool_device)
def swap_blocks_int4(src, dst, block_mapping, stream=None, device=None):
    """swap_blocks for INT4 blocks; src and dst are (k_codes, v_codes, k_scales, v_scales)
    pools, CUDA tensors or pinned CPU tensors."""
    import torch
    nbs, hkv, bs, d2 = src[0].shape
    nbd = dst[0].shape[0]
    _need(all(t.shape == src[0].shape for t in src[:2]) and all(t.shape == dst[0].shape for t in dst[:2]),
          "shape mismatch")
    _need(dst[0].shape[1:] == src[0].shape[1:], "pools must share Hkv, B, d")
    _need(all(t.dtype == torch.uint8 for t in (src[0], src[1], dst[0], dst[1])) and
          all(t.dtype == torch.float32 and t.shape == c.shape[:3]
              for t, c in ((src[2], src[0]), (src[3], src[0]), (dst[2], dst[0]), (dst[3], dst[0]))),
          "codes uint8 [NB, Hkv, B, d/2], scales float32 [NB, Hkv, B]")
    _need(block_mapping.dim() == 2 and block_mapping.shape[1] == 2, "block_mapping must be [n, 2]")
    if device is None:
        device = next((t.device for t in (src[0], dst[0]) if t.is_cuda), torch.device("cuda"))
    names = ("k", "v", "k scales", "v scales")
    st = lib().pa_swap_blocks_int4(
        *[_reachable(t, "src " + nm) for t, nm in zip(src, names)],
        *[_reachable(t, "dst " + nm) for t, nm in zip(dst, names)],
        _reachable(block_mapping, "block_mapping", torch.int32), block_mapping.shape[0], nbs, nbd,
        hkv, 2 * d2, bs, _stream_ptr(stream, device))
    _check(st, "pa_swap_blocks_int4")


@_on_first
def copy_blocks(k_cache, v_cache, block_mapping, stream=None):
    """k_cache[dst] = k_cache[src] and v_cache[dst] = v_cache[src] for each (src, dst)."""
    import torch
    nb, hkv, bs, d = k_cache.shape
    _need(v_cache.shape == k_cache.shape, "shape mismatch")
    _need(block_mapping.dim() == 2 and block_mapping.shape[1] == 2, "block_mapping must be [n, 2]")
    st = lib().pa_copy_blocks(
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_mapping, "block_mapping", torch.int32), block_mapping.shape[0], nb, hkv, d, bs,
        _cache_code(k_cache), _stream_ptr(stream, k_cache.device))
    _check(st, "pa_copy_blocks")


def _reachable(t, name, dtype=None):
    """A CUDA tensor, or a page-locked (pinned) CPU tensor that the GPU can address."""
    if not ((t.is_cuda or t.is_pinned()) and t.is_contiguous()
            and (dtype is None or t.dtype == dtype)):
        _need(t.is_cuda or t.is_pinned(), f"{name} must be a CUDA tensor or a pinned CPU tensor")
        _need(t.is_contiguous(), f"{name} must be contiguous")
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


@_runs_on(_pool_device)
def swap_blocks(src_k, src_v, dst_k, dst_v, block_mapping, stream=None, device=None):
    """dst_k[d] = src_k[s] and dst_v[d] = src_v[s] for each (s, d) of block_mapping, in one
    kernel launch.  Pools and mapping may be CUDA tensors or pinned CPU tensors (swap-out:
    device pool -> pinned CPU pool; swap-in: the reverse)."""
    import torch
    nbs, hkv, bs, d = src_k.shape
    nbd = dst_k.shape[0]
    _need(src_v.shape == src_k.shape and dst_v.shape == dst_k.shape, "shape mismatch")
    _need(dst_k.shape[1:] == src_k.shape[1:], "pools must share Hkv, B, d")
    _need(src_k.dtype == src_v.dtype == dst_k.dtype == dst_v.dtype, "dtype mismatch")
    _need(block_mapping.dim() == 2 and block_mapping.shape[1] == 2, "block_mapping must be [n, 2]")
    if device is None:
        device = next((t.device for t in (src_k, dst_k) if t.is_cuda), torch.device("cuda"))
    st = lib().pa_swap_blocks(
        _reachable(src_k, "src_k"), _reachable(src_v, "src_v"), _reachable(dst_k, "dst_k"),
        _reachable(dst_v, "dst_v"), _reachable(block_mapping, "block_mapping", torch.int32),
        block_mapping.shape[0], nbs, nbd, hkv, d, bs, _cache_code(src_k),
        _stream_ptr(stream, device))
    _check(st, "pa_swap_blocks")


def check_block_mapping(pairs, num_blocks):
    """Host check of a copy_blocks pair list (sequence of (src, dst)); raises on aliasing."""
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    st = lib().pa_check_block_mapping(arr.ctypes.data, arr.shape[0], num_blocks)
    _check(st, "pa_check_block_mapping")


def get_device_error(stream=None, device=None):
    """Synchronise the stream, then read and clear the error word of `device` (default:
    the stream's device, else the current one)."""
    import torch
    if device is None:
        dev = stream.device if stream is not None else torch.device("cuda", torch.cuda.current_device())
    else:
        dev = torch.device(device)
    sw = _switch_to(dev)
    v = ctypes.c_uint32(0)
    if sw is None:
        st = lib().pa_get_device_error(_stream_ptr(stream, dev), ctypes.byref(v))
    else:
        with torch.cuda.device(sw):
            st = lib().pa_get_device_error(_stream_ptr(stream, dev), ctypes.byref(v))
    _check(st, "pa_get_device_error")
    return v.value


# ------------------------------------------------------------------ block pool

def sha256(data):
    """SHA-256 digest of a bytes object, computed by the library (FIPS 180-4)."""
    buf = ctypes.create_string_buffer(bytes(data), max(len(data), 1))
    out = ctypes.create_string_buffer(32)
    _check(lib().pa_sha256(buf, len(data), out), "pa_sha256")
    return out.raw


def block_hashes(tokens, block_size, extra=b""):
    """The chained digests (list of 32-byte strings) of the full blocks of a token list."""
    import numpy as np
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    m = len(tok) // int(block_size)
    out = ctypes.create_string_buffer(32 * max(m, 1))
    ex = bytes(extra)
    n = _check(lib().pa_prefix_block_hashes(tok.ctypes.data, len(tok), int(block_size), ex or None,
                                            len(ex), out, m), "pa_prefix_block_hashes")
    return [out.raw[32 * i:32 * (i + 1)] for i in range(n)]


class BlockPool:
    """Host block pool (C++): ordered free list, refcounts, fork, copy-on-write planning,
    and an optional CPU pool for swap-out / swap-in."""

    def __init__(self, num_blocks, block_size, initial_free_order=None, num_cpu_blocks=0,
                 cpu_free_order=None):
        import numpy as np
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.num_cpu_blocks = int(num_cpu_blocks)

        def order_ptr(order, n, name):
            if order is None:
                return None, None
            arr = np.ascontiguousarray(np.asarray(order, dtype=np.int32))
            _need(arr.shape == (n,), f"{name} must have {n} entries")
            return arr, arr.ctypes.data
        self._order, order = order_ptr(initial_free_order, self.num_blocks, "initial_free_order")
        self._cpu_order, cpu_order = order_ptr(cpu_free_order, self.num_cpu_blocks, "cpu_free_order")
        self._h = lib().pa_pool_create_tiered(self.num_blocks, self.block_size, order,
                                              self.num_cpu_blocks, cpu_order)
        if not self._h:
            raise PagedAttentionError(PA_ERR_ARG, "pa_pool_create_tiered")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.pa_pool_destroy(h)
            self._h = None

    def allocate(self, seq, n_tokens):
        _check(lib().pa_pool_allocate(self._h, int(seq), int(n_tokens)), "allocate")

    def append_slot(self, seq):
        """Returns (slot, cow) with cow None or the (src, dst) pair to copy before writing."""
        slot = ctypes.c_int64(0)
        src = ctypes.c_int32(-1)
        dst = ctypes.c_int32(-1)
        st = _check(lib().pa_pool_append_slot(self._h, int(seq), ctypes.byref(slot),
                                              ctypes.byref(src), ctypes.byref(dst)), "append_slot")
        return slot.value, ((src.value, dst.value) if st == 1 else None)

    def fork(self, parent, child):
        _check(lib().pa_pool_fork(self._h, int(parent), int(child)), "fork")

    def free(self, seq):
        _check(lib().pa_pool_free(self._h, int(seq)), "free")

    def block_table(self, seq):
        import numpy as np
        n = _check(lib().pa_pool_block_table(self._h, int(seq), None, 0), "block_table")
        out = np.zeros(n, dtype=np.int32)
        _check(lib().pa_pool_block_table(self._h, int(seq), out.ctypes.data, n), "block_table")
        return out

    def context_len(self, seq):
        return _check(lib().pa_pool_context_len(self._h, int(seq)), "context_len")

    def slots(self, seq, first, count):
        import numpy as np
        out = np.zeros(count, dtype=np.int64)
        _check(lib().pa_pool_slots(self._h, int(seq), int(first), int(count), out.ctypes.data), "slots")
        return out

    def num_free(self):
        return _check(lib().pa_pool_num_free(self._h), "num_free")

    def free_list(self):
        import numpy as np
        n = self.num_free()
        out = np.zeros(n, dtype=np.int32)
        _check(lib().pa_pool_free_list(self._h, out.ctypes.data, n), "free_list")
        return out

    def refcount(self, block):
        return _check(lib().pa_pool_refcount(self._h, int(block)), "refcount")

    def _move(self, fn, seqs, what):
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(list(seqs), dtype=np.int64))
        cap = sum(len(self.block_table(int(s))) for s in set(ids.tolist())) if ids.size else 0
        pairs = np.zeros((max(cap, 1), 2), dtype=np.int32)
        n = _check(fn(self._h, ids.ctypes.data, ids.size, pairs.ctypes.data, cap), what)
        return pairs[:n]

    def swap_out(self, seqs):
        """Move a group of resident sequences to the CPU pool; returns the (device block,
        CPU block) pairs [n, 2] int32 to copy with swap_blocks."""
        return self._move(lib().pa_pool_swap_out, seqs, "swap_out")

    def swap_in(self, seqs):
        """Bring a group of swapped-out sequences back; returns (CPU block, device block)
        pairs."""
        return self._move(lib().pa_pool_swap_in, seqs, "swap_in")

    def is_swapped(self, seq):
        return bool(_check(lib().pa_pool_is_swapped(self._h, int(seq)), "is_swapped"))

    def num_free_cpu(self):
        return _check(lib().pa_pool_num_free_cpu(self._h), "num_free_cpu")

    def cpu_free_list(self):
        import numpy as np
        n = self.num_free_cpu()
        out = np.zeros(max(n, 1), dtype=np.int32)
        _check(lib().pa_pool_cpu_free_list(self._h, out.ctypes.data, n), "cpu_free_list")
        return out[:n]

    def cpu_refcount(self, block):
        return _check(lib().pa_pool_cpu_refcount(self._h, int(block)), "cpu_refcount")

    def allocate_prefix(self, seq, tokens, extra=b""):
        """Prefill with prefix caching; returns the number of leading tokens whose K/V
        the reused blocks already hold."""
        import numpy as np
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        ex = bytes(extra)
        cached = ctypes.c_int(0)
        _check(lib().pa_pool_allocate_prefix(self._h, int(seq), tok.ctypes.data, len(tok),
                                             ex or None, len(ex), ctypes.byref(cached)),
               "allocate_prefix")
        return cached.value

    def num_cached(self):
        return _check(lib().pa_pool_num_cached(self._h), "num_cached")

    def block_digest(self, block):
        out = ctypes.create_string_buffer(32)
        st = _check(lib().pa_pool_block_digest(self._h, int(block), out), "block_digest")
        return out.raw if st == 1 else None

    def allocate_prefix_batch(self, seq_ids, tokens, token_start, extras=None, extra_start=None,
                              table_width=None, out=None):
        """Place a batch of prompts through the prefix cache in one call (see
        pa_pool_allocate_prefix_batch).  tokens: int32 [total], token_start: int64 [n + 1].
        Returns (cached [n] int32, slots of the uncached tokens int64, tables [n, width]
        int32).  `out` may pass (cached, slots, tables) arrays to fill."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = ids.size
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        ts = np.ascontiguousarray(np.asarray(token_start, dtype=np.int64))
        _need(ts.shape == (n + 1,), "token_start must have n + 1 entries")
        lens = np.diff(ts)
        if table_width is None:
            table_width = _check(lib().pa_pool_table_width(self._h, n, ts.ctypes.data),
                                 "pa_pool_table_width")
        _need(n == 0 or (ts[0] >= 0 and ts[-1] <= tok.size and (lens >= 0).all()),
              "token_start must be non-decreasing within tokens")
        if out is None:
            cached = np.zeros(n, dtype=np.int32)
            slots = np.zeros(int(lens.sum()), dtype=np.int64)
            tables = np.zeros((n, table_width), dtype=np.int32)
        else:
            cached, slots, tables = out
            _host_out(cached, np.int32, n, "cached")
            _host_out(slots, np.int64, int(lens.sum()), "slots")
            _host_out(tables, np.int32, n * int(table_width), "tables")
        ex = es = None
        if extras is not None:
            ex = np.ascontiguousarray(np.frombuffer(bytes(extras), dtype=np.uint8)) if not \
                isinstance(extras, np.ndarray) else np.ascontiguousarray(extras, dtype=np.uint8)
            es = np.ascontiguousarray(np.asarray(extra_start, dtype=np.int64))
            _need(es.shape == (n + 1,), "extra_start must have n + 1 entries")
            _need(n == 0 or (es[0] >= 0 and es[-1] <= ex.size and (np.diff(es) >= 0).all()),
                  "extra_start must be non-decreasing within extras")
        done = ctypes.c_int(0)
        _check(lib().pa_pool_allocate_prefix_batch(
            self._h, n, ids.ctypes.data, tok.ctypes.data, ts.ctypes.data,
            None if ex is None else ex.ctypes.data, None if es is None else es.ctypes.data,
            cached.ctypes.data, slots.ctypes.data, tables.ctypes.data, int(table_width),
            ctypes.byref(done)), "allocate_prefix_batch")
        used = int((lens - cached).sum())
        return cached, slots[:used], tables

    def allocate_hashed_batch(self, seq_ids, n_tokens, digests, table_width, out=None):
        """Place a batch from digests computed earlier (bytes or uint8 array holding every
        request's full-block digests in order, as block_hashes returns them joined).
        Returns (cached, slots of the uncached tokens, tables)."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = ids.size
        nt = np.ascontiguousarray(np.asarray(n_tokens, dtype=np.int32))
        dg = np.ascontiguousarray(np.frombuffer(digests, dtype=np.uint8) if isinstance(
            digests, (bytes, bytearray)) else np.asarray(digests, dtype=np.uint8))
        _need(nt.shape == (n,), "n_tokens must have one entry a request")
        _need(dg.size >= 32 * int((np.maximum(nt, 0) // self.block_size).sum()),
              "digests must hold 32 bytes for every full block of every request")
        if out is None:
            cached = np.zeros(n, dtype=np.int32)
            slots = np.zeros(int(nt.sum()), dtype=np.int64)
            tables = np.zeros((n, table_width), dtype=np.int32)
        else:
            cached, slots, tables = out
            _host_out(cached, np.int32, n, "cached")
            _host_out(slots, np.int64, int(nt.sum()), "slots")
            _host_out(tables, np.int32, n * int(table_width), "tables")
        done = ctypes.c_int(0)
        _check(lib().pa_pool_allocate_hashed_batch(
            self._h, n, ids.ctypes.data, nt.ctypes.data, dg.ctypes.data if dg.size else None,
            cached.ctypes.data, slots.ctypes.data, tables.ctypes.data, int(table_width),
            ctypes.byref(done)), "allocate_hashed_batch")
        used = int((nt - cached).sum())
        return cached, slots[:used], tables

    def free_batch(self, seq_ids):
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        _check(lib().pa_pool_free_batch(self._h, ids.ctypes.data, ids.size), "free_batch")
