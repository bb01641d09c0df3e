"""FP8 (E4M3) KV blocks: the format, the quantising cache write and paged decode over it.

Test infrastructure only.  Paging does not cut the bytes a KV cache needs; quantising the
cached K/V does (daiw.org "Paged Attention", section 量化, the callout: GQA, a quantised
KV cache or a shorter context reduce the bytes), and serving engines store KV blocks in
FP8 or INT4 (horeb.top "vLLM PagedAttention：大模型推理的显存管理革命", section 生态现状).
The pages fix no format; the readings here:

* element format E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
  bits; exponent field 0 holds the subnormals m * 2^-9; no infinities; S.1111.111 is NaN,
  so the largest finite magnitude is 1.75 * 2^8 = 448;
* one float32 scale per cache (k_scale for K, v_scale for V): a stored code c means the
  value decode(c) * scale;
* the cache write quantises each 16-bit input value x as follows: x / scale in float32
  (exact decode of x, one IEEE division), then round to nearest E4M3, ties to even, with
  magnitudes above 448 (and infinities) clamped to 448 and NaN kept NaN (0x7F, sign
  kept).  The decision is taken in float32 on both sides;
* decode is ordinary attention over the dequantised values decode(c) * scale, in float64
  (the same definition as the 16-bit cache, with different stored rows).
"""
import numpy as np

from .attention import attend, validate_item
from .formats import decode_bits, encode_bits

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def decode_e4m3(codes):
    """Exact float64 value of each E4M3 code (uint8)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    out = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


def encode_e4m3(x):
    """E4M3 codes of float values: clamp to [-448, 448], round to nearest, ties to even;
    NaN -> 0x7F with the sign bit of the input."""
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    sign = np.signbit(x)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), E4M3_MAX)
    # quantum of the binade of a: 2^(max(e, -6) - 3), e = exponent of the leading bit
    _, e2 = np.frexp(a)
    e = np.maximum(e2 - 1, -6)
    q = np.ldexp(1.0, e - 3)
    r = np.rint(a / q) * q                 # exact scaling; rint is half-to-even
    r = np.minimum(r, E4M3_MAX)            # (a <= 448 already; rounding cannot pass it)
    # code of the magnitude r
    _, re2 = np.frexp(r)
    re = re2 - 1
    normal = r >= 2.0 ** -6
    exp_field = np.where(normal, re + 7, 0)
    mant = np.where(normal, np.rint((r / np.ldexp(1.0, re) - 1.0) * 8.0), np.rint(r * 2.0 ** 9))
    code = (exp_field.astype(np.int64) << 3) | mant.astype(np.int64)
    code = np.where(r == 0, 0, code)
    code = code | np.where(sign, 0x80, 0)
    code = np.where(nan, E4M3_NAN | np.where(sign, 0x80, 0), code)
    return code.astype(np.uint8)


def quantize(bits16, dtype, scale):
    """Cache-write quantisation of 16-bit values: float32(x) / float32(scale), then E4M3."""
    x32 = decode_bits(bits16, dtype).astype(np.float32)   # exact
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        y = x32 / np.float32(scale)                        # one IEEE float32 division
    return encode_e4m3(y.astype(np.float64))


def reshape_and_cache(k_cache8, v_cache8, key_bits, value_bits, slot_mapping, k_scale,
                      v_scale, dtype):
    """Copies of the FP8 caches [NB, Hkv, B, d] (uint8) with the quantised rows of key/value
    [n_tok, Hkv, d] (16-bit patterns) written at their slots; slot < 0 is skipped."""
    nb, hkv, b, d = k_cache8.shape
    k_out, v_out = k_cache8.copy(), v_cache8.copy()
    seen = set()
    for i, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        slot = int(slot)
        if slot < 0:
            continue
        if slot >= nb * b:
            raise IndexError(f"slot {slot} outside the pool of {nb * b} slots")
        if slot in seen:
            raise ValueError(f"slot {slot} written twice in one call")
        seen.add(slot)
        k_out[slot // b, :, slot % b, :] = quantize(key_bits[i], dtype, k_scale)
        v_out[slot // b, :, slot % b, :] = quantize(value_bits[i], dtype, v_scale)
    return k_out, v_out


def logical_rows(cache8, table_row, ctx, block_size, scale):
    """Row t = decode(cache[table_row[t // B], :, t % B, :]) * scale, float64 [ctx, Hkv, d]."""
    out = np.empty((ctx,) + cache8.shape[1:2] + cache8.shape[3:], dtype=np.float64)
    for t in range(ctx):
        blk = int(table_row[t // block_size])
        out[t] = decode_e4m3(cache8[blk, :, t % block_size, :]) * float(np.float32(scale))
    return out


def paged_decode(q_bits, k_cache8, v_cache8, block_tables, context_lens, scale, k_scale,
                 v_scale, block_size, dtype, seqs=None):
    """Paged decode over FP8 K/V blocks; q and out are 16-bit (dtype).  Returns (out float64
    [n_sel, Hq, d], error bits) with the same invalid-item convention as the 16-bit path."""
    n = q_bits.shape[0]
    seqs = range(n) if seqs is None else seqs
    nb = k_cache8.shape[0]
    outs, errs = [], []
    for s in seqs:
        ctx = int(context_lens[s])
        err = validate_item(block_tables[s], ctx, block_size, nb)
        errs.append(err)
        if err:
            outs.append(np.zeros(q_bits.shape[1:], dtype=np.float64))
            continue
        k = logical_rows(k_cache8, block_tables[s], ctx, block_size, k_scale)
        v = logical_rows(v_cache8, block_tables[s], ctx, block_size, v_scale)
        outs.append(attend(decode_bits(q_bits[s], dtype), k, v, scale))
    return np.stack(outs), np.array(errs, dtype=np.int64)


def paged_decode_bits(*args, **kw):
    """``paged_decode`` rounded to the 16-bit output format (RNE); also the error bits."""
    dtype = args[9] if len(args) > 9 else kw["dtype"]
    out, err = paged_decode(*args, **kw)
    return encode_bits(out, dtype), err
