"""ctypes front-end of the C oracle (``kvq_oracle.c``); numpy arrays in, numpy arrays out.

Test infrastructure only.  bf16 / fp16 values cross this interface as their uint16 bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build_oracle

FP8_E4M3 = 1
Q8_0 = 2
FP8_E4M3_UNSCALED = 3
FP8_E5M2_UNSCALED = 4
KIND_BY_NAME = {"fp8_e4m3": FP8_E4M3, "q8_0": Q8_0, "fp8_e4m3_unscaled": FP8_E4M3_UNSCALED,
                "fp8_e5m2_unscaled": FP8_E5M2_UNSCALED}
UNSCALED = (FP8_E4M3_UNSCALED, FP8_E5M2_UNSCALED)

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        sig = {
            "kvo_f16_value": (dbl, [ctypes.c_uint16]),
            "kvo_bf16_value": (dbl, [ctypes.c_uint16]),
            "kvo_e4m3_value": (dbl, [ctypes.c_uint8]),
            "kvo_f16_rne": (ctypes.c_uint16, [dbl]),
            "kvo_bf16_rne": (ctypes.c_uint16, [dbl]),
            "kvo_e4m3_rne": (ctypes.c_uint8, [dbl]),
            "kvo_e4m3_sat_rne": (ctypes.c_uint8, [ctypes.c_float]),
            "kvo_e4m3_double_round": (ctypes.c_uint8, [ctypes.c_float]),
            "kvo_q8_rhaz": (ctypes.c_int8, [ctypes.c_float]),
            "kvo_dequant": (dbl, [i32, ctypes.c_uint8, ctypes.c_uint16]),
            "kvo_block_scale": (ctypes.c_uint16, [i32, P, i32]),
            "kvo_quantize_block": (None, [i32, P, i32, P, P]),
            "kvo_bytes_per_token": (dbl, [i32, i32, i32]),
            "kvo_store": (i32, [P, P, P, P, P, i64, i32, i32, i32, i32, i32, i64]),
            "kvo_scatter_bf16": (i32, [P, P, P, P, i64, i32, i32, i32, i32, i64]),
            "kvo_decode": (i32, [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, i32, dbl, i32]),
            "kvo_decode_bf16": (i32, [P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, dbl, i32]),
            "kvo_decode_sparse": (i32, [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                        dbl, i32]),
            "kvo_extend": (i32, [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32, i32, dbl, i32]),
            "kvo_f16_rne_f32_batch": (None, [P, P, i64]),
            "kvo_bf16_rne_f64_batch": (None, [P, P, i64]),
            "kvo_e4m3_sat_rne_batch": (None, [P, P, i64]),
            "kvo_e4m3_double_round_batch": (None, [P, P, i64]),
            "kvo_q8_rhaz_batch": (None, [P, P, i64]),
            "kvo_dequant_batch": (None, [i32, P, P, P, i64]),
            "kvo_e5m2_value": (dbl, [ctypes.c_uint8]),
            "kvo_e5m2_rne": (ctypes.c_uint8, [dbl]),
            "kvo_e5m2_sat_rne_batch": (None, [P, P, i64]),
            "kvo_bytes_per_element": (dbl, [i32]),
            "kvo_act_quant64": (None, [P, i64, P]),
            "kvo_store_act_quant": (i32, [P, P, P, P, i64, i32, i32, i32, i32, i64]),
            "kvo_has_openmp": (i32, []),
            "kvo_code_of": (ctypes.c_uint8, [i32, ctypes.c_uint16, ctypes.c_uint16]),
            "kvo_code_table": (None, [i32, P, i64, P, i64, P, i32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _kind(kind):
    return KIND_BY_NAME[kind] if isinstance(kind, str) else int(kind)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _c_opt(a, dtype):
    """As _c, or (None, NULL) for None (the scales of an unscaled pool)."""
    return (None, None) if a is None else _c(a, dtype)


# ----------------------------------------------------------------------------- scalar formats
def f16_value(bits):
    return lib().kvo_f16_value(int(bits))


def bf16_value(bits):
    return lib().kvo_bf16_value(int(bits))


def e4m3_value(code):
    return lib().kvo_e4m3_value(int(code))


def e4m3_rne(y):
    """Nearest-even E4M3 code of a double with |y| <= 448."""
    return lib().kvo_e4m3_rne(float(y))


def e5m2_value(code):
    return lib().kvo_e5m2_value(int(code))


def e5m2_rne(y):
    """Nearest-even E5M2 code of a double with |y| <= 57344."""
    return lib().kvo_e5m2_rne(float(y))


def e5m2_sat_rne(y):
    """Codes of fp32 values clamped to +-57344, then rounded to nearest-even E5M2."""
    y = np.ascontiguousarray(y, np.float32)
    out = np.empty(y.shape, np.uint8)
    lib().kvo_e5m2_sat_rne_batch(y.ctypes.data_as(ctypes.c_void_p), out.ctypes.data_as(ctypes.c_void_p), y.size)
    return out


def bytes_per_element(kind):
    return lib().kvo_bytes_per_element(_kind(kind))


def code_value(kind, code):
    k = _kind(kind)
    if k in (FP8_E4M3, FP8_E4M3_UNSCALED):
        return e4m3_value(code)
    if k == FP8_E5M2_UNSCALED:
        return e5m2_value(code)
    return float(np.int8(np.uint8(code)))


# ----------------------------------------------------------------------------- batch maps
def f16_rne(x_f32):
    x, px = _c(x_f32, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().kvo_f16_rne_f32_batch(px, out.ctypes.data_as(ctypes.c_void_p), x.size)
    return out


def bf16_rne(x_f64):
    x, px = _c(x_f64, np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().kvo_bf16_rne_f64_batch(px, out.ctypes.data_as(ctypes.c_void_p), x.size)
    return out


def e4m3_sat_rne(y_f32):
    y, py = _c(y_f32, np.float32)
    out = np.empty(y.shape, np.uint8)
    lib().kvo_e4m3_sat_rne_batch(py, out.ctypes.data_as(ctypes.c_void_p), y.size)
    return out


def e4m3_double_round(y_f32):
    y, py = _c(y_f32, np.float32)
    out = np.empty(y.shape, np.uint8)
    lib().kvo_e4m3_double_round_batch(py, out.ctypes.data_as(ctypes.c_void_p), y.size)
    return out


def q8_rhaz(y_f32):
    y, py = _c(y_f32, np.float32)
    out = np.empty(y.shape, np.int8)
    lib().kvo_q8_rhaz_batch(py, out.ctypes.data_as(ctypes.c_void_p), y.size)
    return out


def dequant(kind, codes, s16):
    """RNE_bf16(value(code) * fp16 scale) as float64, elementwise (codes and s16 broadcast)."""
    c, s = np.broadcast_arrays(np.asarray(codes, np.uint8), np.asarray(s16, np.uint16))
    c, pc = _c(c, np.uint8)
    s, ps = _c(s, np.uint16)
    out = np.empty(c.shape, np.float64)
    lib().kvo_dequant_batch(_kind(kind), pc, ps, out.ctypes.data_as(ctypes.c_void_p), c.size)
    return out


# ----------------------------------------------------------------------------- blocks
def block_scale(kind, x_bits):
    x, px = _c(x_bits, np.uint16)
    return lib().kvo_block_scale(_kind(kind), px, x.size)


def quantize_block(kind, x_bits):
    """Return (codes uint8[32], fp16 scale bits) of one block given as bf16 bit patterns."""
    x, px = _c(x_bits, np.uint16)
    codes = np.empty(x.size, np.uint8)
    s = np.zeros(1, np.uint16)
    lib().kvo_quantize_block(_kind(kind), px, x.size, codes.ctypes.data_as(ctypes.c_void_p),
                             s.ctypes.data_as(ctypes.c_void_p))
    return codes, int(s[0])


def code_table(kind, x_bits, s_bits, nthreads=0):
    """codes[i, j] = code of bf16 x[j] against nonzero fp16 scale s[i] (IEEE fp32 division, then rounding)."""
    x, px = _c(x_bits, np.uint16)
    s, ps = _c(s_bits, np.uint16)
    out = np.empty((s.size, x.size), np.uint8)
    lib().kvo_code_table(_kind(kind), px, x.size, ps, s.size, out.ctypes.data_as(ctypes.c_void_p), int(nthreads))
    return out


def bytes_per_token(n_kv, num_kv_heads, head_dim):
    return lib().kvo_bytes_per_token(n_kv, num_kv_heads, head_dim)


# ----------------------------------------------------------------------------- pool
def pool_shapes(num_pages, page_size, num_kv_heads, head_dim, mla):
    n_kv = 1 if mla else 2
    codes = (num_pages, n_kv, num_kv_heads, page_size, head_dim)
    scales = (num_pages, n_kv, num_kv_heads, page_size, head_dim // 32)
    return codes, scales


def store(codes, scales, k_bits, v_bits, slot_mapping, *, num_kv_heads, head_dim, page_size, mla, kind):
    """Quantize-and-scatter into ``codes`` (uint8) / ``scales`` (uint16) in place (the unscaled kinds have no
    scales: pass None)."""
    assert codes.dtype == np.uint8 and codes.flags.c_contiguous
    if scales is None:
        assert _kind(kind) in UNSCALED, "the block-scaled kinds need a scale array"
    else:
        assert scales.dtype == np.uint16 and scales.flags.c_contiguous
    k, pk = _c(k_bits, np.uint16)
    if mla:
        v, pv = None, None
    else:
        v, pv = _c(v_bits, np.uint16)
    sm, psm = _c(slot_mapping, np.int64)
    num_pages = codes.shape[0]
    rc = lib().kvo_store(codes.ctypes.data_as(ctypes.c_void_p),
                         None if scales is None else scales.ctypes.data_as(ctypes.c_void_p),
                         pk, pv, psm, sm.size, num_kv_heads, head_dim, page_size, int(bool(mla)),
                         _kind(kind), num_pages)
    if rc != 0:
        raise ValueError("oracle store rejected its arguments")


def scatter_bf16(pool16, k_bits, v_bits, slot_mapping, *, num_kv_heads, head_dim, page_size, mla):
    k, pk = _c(k_bits, np.uint16)
    v, pv = (None, None) if mla else _c(v_bits, np.uint16)
    sm, psm = _c(slot_mapping, np.int64)
    rc = lib().kvo_scatter_bf16(pool16.ctypes.data_as(ctypes.c_void_p), pk, pv, psm, sm.size, num_kv_heads,
                                head_dim, page_size, int(bool(mla)), pool16.shape[0])
    if rc != 0:
        raise ValueError("oracle scatter rejected its arguments")


def act_quant64(x_bits):
    """The model's rounding of an MLA latent onto the E4M3 grid, one fp32 scale (amax / 448) per 64 elements
    along the last axis; returns bf16 bit patterns of the same shape."""
    x, px = _c(x_bits, np.uint16)
    assert x.shape[-1] % 64 == 0
    out = np.empty_like(x)
    rows = x.reshape(-1, x.shape[-1])
    o = out.reshape(-1, x.shape[-1])
    for i in range(rows.shape[0]):  # blocks never straddle rows
        r = np.ascontiguousarray(rows[i])
        lib().kvo_act_quant64(r.ctypes.data_as(ctypes.c_void_p), r.size, o[i].ctypes.data_as(ctypes.c_void_p))
    return out


def store_act_quant(codes, scales, k_bits, slot_mapping, *, head_dim, rope_dim, page_size, kind):
    """The MLA store fused with its producer: act_quant64 over each row's latent part, then the store."""
    k, pk = _c(k_bits, np.uint16)
    sm, psm = _c(slot_mapping, np.int64)
    rc = lib().kvo_store_act_quant(codes.ctypes.data_as(ctypes.c_void_p), scales.ctypes.data_as(ctypes.c_void_p), pk,
                                   psm, sm.size, head_dim, rope_dim, page_size, _kind(kind), codes.shape[0])
    if rc != 0:
        raise ValueError("oracle fused store rejected its arguments")


def decode(q_bits, codes, scales, block_table, seq_lens, *, num_q_heads, num_kv_heads, head_dim, v_dim,
           page_size, mla, kind, sm_scale, nthreads=1):
    """fp64 attention over the dequantized pool; returns out[B, Hq, Dv] float64."""
    q, pq = _c(q_bits, np.uint16)
    c, pc = _c(codes, np.uint8)
    s, ps = _c_opt(scales, np.uint16)
    bt, pbt = _c(block_table, np.int32)
    sl, psl = _c(seq_lens, np.int32)
    B = sl.size
    out = np.zeros((B, num_q_heads, v_dim), np.float64)
    rc = lib().kvo_decode(out.ctypes.data_as(ctypes.c_void_p), pq, pc, ps, pbt, bt.shape[1], psl, B,
                          num_q_heads, num_kv_heads, head_dim, v_dim, page_size, int(bool(mla)),
                          _kind(kind), float(sm_scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle decode rejected its arguments")
    return out


def decode_sparse(q_bits, codes, scales, block_table, seq_lens, indices, *, num_q_heads, num_kv_heads, head_dim,
                  v_dim, page_size, mla, kind, sm_scale, nthreads=1):
    """fp64 attention of each sequence's query over the tokens its index list selects ([B, topk] int32
    positions; -1, positions at or past seq_len and positions on masked pages are skipped; a repeated
    position counts once per listing); returns out[B, Hq, Dv] float64 (zeros without a valid column)."""
    q, pq = _c(q_bits, np.uint16)
    c, pc = _c(codes, np.uint8)
    s, ps = _c_opt(scales, np.uint16)
    bt, pbt = _c(block_table, np.int32)
    sl, psl = _c(seq_lens, np.int32)
    ix, pix = _c(indices, np.int32)
    B = sl.size
    topk = ix.shape[1] if ix.ndim == 2 else 0
    out = np.zeros((B, num_q_heads, v_dim), np.float64)
    rc = lib().kvo_decode_sparse(out.ctypes.data_as(ctypes.c_void_p), pq, pc, ps, pbt, bt.shape[1], psl, pix, topk,
                                 B, num_q_heads, num_kv_heads, head_dim, v_dim, page_size, int(bool(mla)),
                                 _kind(kind), float(sm_scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle sparse decode rejected its arguments")
    return out


def extend(q_bits, codes, scales, block_table, seq_lens, q_start, *, num_q_heads, num_kv_heads, head_dim, v_dim,
           page_size, mla, kind, sm_scale, nthreads=1):
    """fp64 causal attention of the new tokens of every sequence ("feat(kvcache): 8-bit KV cache (q8_0 /
    fp8_e4m3) behind --kv-cache-dtype", section "What": dequant inside the prefill kernel too).  q_bits is
    [total_q, Hq, D]; q_start[B + 1] (q_start[0] = 0) gives each sequence's rows; the n_b = q_start[b+1] -
    q_start[b] new tokens are the last n_b of its seq_lens[b] stored tokens, so new token i sits at position
    seq_lens[b] - n_b + i and attends to the unmasked positions up to and including its own.  Returns
    out[total_q, Hq, Dv] float64 (zeros where no position is valid)."""
    q, pq = _c(q_bits, np.uint16)
    c, pc = _c(codes, np.uint8)
    s, ps = _c_opt(scales, np.uint16)
    bt, pbt = _c(block_table, np.int32)
    sl, psl = _c(seq_lens, np.int32)
    qs, pqs = _c(q_start, np.int32)
    B = sl.size
    if qs.size != B + 1:
        raise ValueError("q_start needs batch + 1 entries")
    total = int(qs[-1])
    out = np.zeros((total, num_q_heads, v_dim), np.float64)
    rc = lib().kvo_extend(out.ctypes.data_as(ctypes.c_void_p), pq, pc, ps, pbt, bt.shape[1], psl, pqs, B,
                          num_q_heads, num_kv_heads, head_dim, v_dim, page_size, int(bool(mla)), _kind(kind),
                          float(sm_scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle extend rejected its arguments")
    return out


def decode_bf16(q_bits, pool16, block_table, seq_lens, *, num_q_heads, num_kv_heads, head_dim, v_dim,
                page_size, mla, sm_scale, nthreads=1):
    """fp64 attention over an unquantized bf16 pool (reported error only)."""
    q, pq = _c(q_bits, np.uint16)
    p16, pp = _c(pool16, np.uint16)
    bt, pbt = _c(block_table, np.int32)
    sl, psl = _c(seq_lens, np.int32)
    B = sl.size
    out = np.zeros((B, num_q_heads, v_dim), np.float64)
    rc = lib().kvo_decode_bf16(out.ctypes.data_as(ctypes.c_void_p), pq, pp, pbt, bt.shape[1], psl, B,
                               num_q_heads, num_kv_heads, head_dim, v_dim, page_size, int(bool(mla)),
                               float(sm_scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle decode rejected its arguments")
    return out


def openmp_threads():
    return lib().kvo_has_openmp()
