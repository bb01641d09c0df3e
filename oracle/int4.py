"""INT4 KV blocks: the format, the quantising cache write and paged decode over it.

Test infrastructure only.  Quantising the cached K/V cuts the bytes a KV cache needs
(daiw.org "Paged Attention", section 量化, the callout), and serving engines store KV
blocks in FP8 or INT4 (horeb.top "vLLM PagedAttention：大模型推理的显存管理革命", section
生态现状).  The pages fix no INT4 format; the readings here (the plainest symmetric
integer quantisation, with one scale per cached row because four bits cannot share one
scale over a whole cache):

* a row is one token of one kv head (d values); it is stored as d 4-bit codes c in
  [-7, 7] plus one float32 scale s, and means the values c * s;
* s = max_i |x_i| / 7, one IEEE float32 division of the exact float32 maximum (s = 0 for
  an all-zero row, whose codes are then all 0);
* c_i = x_i / s in float32 (one IEEE division), rounded to nearest, ties to even, and
  clamped to [-7, 7];
* storage: the code c is kept as the nibble u = c + 8 (1..15); element 2i is the low
  nibble of byte i and element 2i + 1 the high nibble; the scales of a block are a
  separate float32 array [NB, Hkv, B] beside the codes [NB, Hkv, B, d/2];
* decode is ordinary attention over the dequantised rows c * s, in float64 (the same
  definition as for 16-bit and FP8 blocks, with different stored rows).

Inputs are finite; a row holding an infinity or NaN has unspecified codes.
"""
import numpy as np

from .attention import attend, validate_item
from .formats import decode_bits, encode_bits

CODE_MAX = 7
OFFSET = 8


def quantize_rows(bits16, dtype):
    """Rows [..., d] of 16-bit patterns -> (packed codes uint8 [..., d/2], scales float32 [...])."""
    x = decode_bits(bits16, dtype).astype(np.float32)            # exact
    amax = np.max(np.abs(x), axis=-1)                            # exact
    scale = (amax / np.float32(CODE_MAX)).astype(np.float32)     # one float32 division
    with np.errstate(divide="ignore", invalid="ignore"):
        y = x / scale[..., None]                                 # one float32 division each
    c = np.where(scale[..., None] == 0, 0.0, np.rint(y))        # rint: half to even
    c = np.clip(c, -CODE_MAX, CODE_MAX).astype(np.int64)
    u = (c + OFFSET).astype(np.uint8)
    packed = (u[..., 0::2] | (u[..., 1::2] << 4)).astype(np.uint8)
    return packed, scale


def unpack_codes(packed):
    """Packed bytes [..., d/2] -> signed codes int64 [..., d] (low nibble first)."""
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int64)
    out[..., 0::2] = (p & 0xF) - OFFSET
    out[..., 1::2] = (p >> 4) - OFFSET
    return out


def dequantize(packed, scales):
    """c * s in float64: packed [..., d/2], scales [...] -> [..., d]."""
    return unpack_codes(packed).astype(np.float64) * np.asarray(scales, np.float32).astype(np.float64)[..., None]


def reshape_and_cache(k_codes, v_codes, k_scales, v_scales, key_bits, value_bits, slot_mapping,
                      dtype):
    """Copies of the INT4 caches (codes [NB, Hkv, B, d/2] uint8, scales [NB, Hkv, B] float32)
    with the quantised rows of key/value [n_tok, Hkv, d] (16-bit patterns) written at their
    slots; slot < 0 is skipped."""
    nb, hkv, b, _ = k_codes.shape
    kc, vc = k_codes.copy(), v_codes.copy()
    ks, vs = k_scales.copy(), v_scales.copy()
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
        pk, sk = quantize_rows(key_bits[i], dtype)
        pv, sv = quantize_rows(value_bits[i], dtype)
        kc[slot // b, :, slot % b, :] = pk
        vc[slot // b, :, slot % b, :] = pv
        ks[slot // b, :, slot % b] = sk
        vs[slot // b, :, slot % b] = sv
    return kc, vc, ks, vs


def logical_rows(codes, scales, table_row, ctx, block_size):
    """Row t = dequantize(codes[table_row[t // B], :, t % B], scales[...]): float64 [ctx, Hkv, d]."""
    hkv, d2 = codes.shape[1], codes.shape[3]
    out = np.empty((ctx, hkv, 2 * d2), dtype=np.float64)
    for t in range(ctx):
        blk = int(table_row[t // block_size])
        out[t] = dequantize(codes[blk, :, t % block_size, :], scales[blk, :, t % block_size])
    return out


def paged_decode(q_bits, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, scale,
                 block_size, dtype, seqs=None):
    """Paged decode over INT4 K/V blocks; q and out are 16-bit (dtype).  Returns (out float64
    [n_sel, Hq, d], error bits) with the same invalid-item convention as the 16-bit path."""
    n = q_bits.shape[0]
    seqs = range(n) if seqs is None else seqs
    nb = k_codes.shape[0]
    outs, errs = [], []
    for s in seqs:
        ctx = int(context_lens[s])
        err = validate_item(block_tables[s], ctx, block_size, nb)
        errs.append(err)
        if err:
            outs.append(np.zeros(q_bits.shape[1:], dtype=np.float64))
            continue
        k = logical_rows(k_codes, k_scales, block_tables[s], ctx, block_size)
        v = logical_rows(v_codes, v_scales, block_tables[s], ctx, block_size)
        outs.append(attend(decode_bits(q_bits[s], dtype), k, v, scale))
    return np.stack(outs), np.array(errs, dtype=np.int64)


def paged_decode_bits(*args, **kw):
    """``paged_decode`` rounded to the 16-bit output format (RNE); also the error bits."""
    dtype = args[9] if len(args) > 9 else kw["dtype"]
    out, err = paged_decode(*args, **kw)
    return encode_bits(out, dtype), err
