"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against an independent implementation (numpy's float16 cast, torch's
float8_e4m3fn / bfloat16 casts, Python's decimal rounding, scipy's softmax), a number the pages
print (tests/golden/page_facts.json), a closed form, or an invariant.  The pages are the four pull
requests on the 8-bit KV cache; sections are named in each docstring.
"""
import decimal
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))
FP8, Q8 = "fp8_e4m3", "q8_0"


def f32_patterns(stride, offset=0):
    """Every ``stride``-th fp32 bit pattern, NaNs removed, as float32."""
    bits = np.arange(offset, 1 << 32, stride, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    return x[~np.isnan(x)]


def torch_e4m3_bits(y_f32):
    return torch.from_numpy(np.ascontiguousarray(y_f32, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def bf16_bits(x_f32):
    return torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def rhaz_decimal(y):
    """Round half away from zero with Python's decimal module (exact on the float's value)."""
    r = int(decimal.Decimal(float(y)).to_integral_value(rounding=decimal.ROUND_HALF_UP))
    return max(-127, min(127, r))


# ============================================================================ number formats
def test_e4m3_decode_matches_torch_for_all_256_codes():
    """OCP E4M3 'fn' decode of every code equals torch's float8_e4m3fn decode."""
    ours = np.array([O.e4m3_value(c) for c in range(256)])
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert O.e4m3_value(0x7E) == 448.0 and O.e4m3_value(0x01) == 2.0 ** -9 and O.e4m3_value(0x08) == 2.0 ** -6


def test_e4m3_enumeration_reencodes_every_finite_code():
    """Decode-then-encode is the identity on the 254 finite codes; NaN codes are never produced."""
    for c in range(256):
        v = O.e4m3_value(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(v)
            continue
        assert O.e4m3_rne(v) == c, hex(c)
    y = np.linspace(-500, 500, 200001, dtype=np.float32)
    codes = O.e4m3_sat_rne(y)
    assert not np.any((codes == 0x7F) | (codes == 0xFF))


def test_e4m3_midpoints_tie_to_even_and_neighbours_round_to_nearer():
    """Every midpoint between adjacent E4M3 values goes to the even code; +-1 fp32 ulp goes to the nearer.

    The fp8 store must be a single round-to-nearest-even (review comment 'A bug on sm_89', the fix).
    """
    pos = sorted({O.e4m3_value(c) for c in range(0x7F)})           # 0 .. 448, 127 values
    assert len(pos) == 127 and pos[-1] == 448.0
    for a, b in zip(pos[:-1], pos[1:]):
        mid = (a + b) / 2.0
        ca, cb = O.e4m3_rne(a), O.e4m3_rne(b)
        even = ca if ca % 2 == 0 else cb
        m32 = np.float32(mid)
        assert float(m32) == mid
        assert O.e4m3_sat_rne(np.array([mid], np.float32))[0] == even
        up = np.nextafter(m32, np.float32(np.inf))
        dn = np.nextafter(m32, np.float32(-np.inf))
        assert O.e4m3_sat_rne(np.array([up], np.float32))[0] == cb
        assert O.e4m3_sat_rne(np.array([dn], np.float32))[0] == ca
        got = torch_e4m3_bits(np.array([mid, up, dn], np.float32))
        assert list(got) == [even, cb, ca]


def test_e4m3_saturating_encoder_matches_torch_on_dense_fp32_sample():
    """Clamp to +-448, then torch's RNE float8 cast, over ~4M fp32 bit patterns of every binade."""
    y = f32_patterns(1021)
    ours = O.e4m3_sat_rne(y)
    ref = torch_e4m3_bits(np.clip(y, -448.0, 448.0))
    assert np.array_equal(ours, ref)


def test_e4m3_special_values():
    """Subnormal ties (2^-10 -> 0, 3*2^-10 -> 2*2^-9), sign of zero kept, out-of-range saturates."""
    y = np.array([2.0 ** -10, 3 * 2.0 ** -10, -0.0, -1e-9, 448.0, 463.9, 1e30, -1e30, np.inf, -np.inf], np.float32)
    assert list(O.e4m3_sat_rne(y)) == [0x00, 0x02, 0x80, 0x80, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]


def test_fp16_encoder_matches_numpy_on_dense_fp32_sample():
    """IEEE binary16 nearest-even with overflow to inf, against numpy's float32 -> float16 cast."""
    x = f32_patterns(251)
    ours = O.f16_rne(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_fp16_decode_matches_numpy_for_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    ours = np.array([O.f16_value(int(b)) for b in bits[::7]])
    r = ref[::7]
    fin = ~np.isnan(r)
    assert np.array_equal(ours[fin], r[fin]) and np.all(np.isnan(ours[~fin]))


def test_bf16_encoder_matches_torch_on_dense_fp32_sample():
    x = f32_patterns(1009, offset=3)
    ours = O.bf16_rne(x.astype(np.float64))
    ref = bf16_bits(x)
    fin = np.isfinite(x)
    assert np.array_equal(ours[fin], ref[fin])


def test_dequant_matches_torch_product_then_bf16():
    """Dequant = bf16 RNE of code value x fp16 scale ('What': K/V dequantize to bf16 before the dot).

    Checked for every code against torch: the fp32 product is exact (<= 18 significant bits) and
    torch's float -> bfloat16 cast rounds to nearest-even.
    """
    rng = np.random.default_rng(5)
    s16 = np.concatenate([np.array([0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF], np.uint16),
                          rng.integers(1, 0x7C00, 400).astype(np.uint16)])
    s_f32 = s16.view(np.float16).astype(np.float32)
    for kind in (FP8, Q8):
        codes = np.arange(256, dtype=np.uint8)
        if kind == FP8:
            codes = codes[(codes != 0x7F) & (codes != 0xFF)]
            cval = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
        else:
            cval = codes.view(np.int8).astype(np.float32)
        C, S = np.meshgrid(codes, s16, indexing="ij")
        CV, SF = np.meshgrid(cval, s_f32, indexing="ij")
        prod = CV * SF
        ref = bf16_to_f32(bf16_bits(prod)).astype(np.float64)
        ours = O.dequant(kind, C, S)
        assert np.array_equal(ours, ref), kind


# ============================================================================ scales and codes
def _random_blocks(n, rng, scale_spread=True):
    x = rng.standard_normal((n, 32)).astype(np.float32)
    if scale_spread:
        x *= np.exp(rng.uniform(-12, 12, (n, 1))).astype(np.float32)
    return bf16_bits(x)


@pytest.mark.parametrize("kind,Q", [(FP8, 448), (Q8, 127)])
def test_block_scale_is_fp16_of_fp32_amax_over_q(kind, Q):
    """s = fp16(amax / Q) with amax/Q in fp32 (section 'What': s = max/448 or max/127, fp16 scale)."""
    assert Q == GOLDEN["fp8_scale_divisor" if kind == FP8 else "q8_scale_divisor"]["value"]
    rng = np.random.default_rng(11)
    blocks = _random_blocks(3000, rng)
    for blk in blocks:
        amax = np.abs(bf16_to_f32(blk)).max()
        with np.errstate(over="ignore"):
            ref = (np.float32(amax) / np.float32(Q)).astype(np.float16).view(np.uint16)
        assert O.block_scale(kind, blk) == int(ref)


def test_block_scale_saturates_at_fp16_max():
    big = bf16_bits(np.full(32, 3.0e38, np.float32))
    assert O.block_scale(FP8, big) == 0x7BFF and O.block_scale(Q8, big) == 0x7BFF


@pytest.mark.parametrize("kind", [FP8, Q8])
def test_block_codes_match_independent_rounding(kind):
    """Codes = round(x / s16) in fp32 division; fp8 via torch's RNE cast after clamping, int8 via decimal."""
    rng = np.random.default_rng(12)
    blocks = _random_blocks(1500, rng)
    for blk in blocks:
        codes, s16 = O.quantize_block(kind, blk)
        s = np.float32(np.uint16(s16).view(np.float16))
        if s16 == 0:
            assert not codes.any()
            continue
        y = bf16_to_f32(blk) / s
        if kind == FP8:
            ref = torch_e4m3_bits(np.clip(y, -448, 448))
        else:
            ref = np.array([rhaz_decimal(v) for v in y], np.int8).view(np.uint8)
        assert np.array_equal(codes, ref)


def test_q8_round_half_away_from_zero_special_values():
    """Review comment 'A bug on sm_89': int8 rounds half away from zero, then clamps to +-127."""
    y = np.array([0.5, -0.5, 1.5, 2.5, -2.5, 0.49999997, -0.49999997, 126.5, 127.49, 127.5, 1000.0, -1000.0, -0.0],
                 np.float32)
    assert list(O.q8_rhaz(y)) == [1, -1, 2, 3, -3, 0, 0, 127, 127, 127, 127, -127, 0]
    assert [rhaz_decimal(v) for v in y] == list(O.q8_rhaz(y))


def test_q8_roundtrip_error_at_most_half_scale():
    """|x - q * s| <= s/2 for every element, the block maximum included (amax/s16 < 127.5).

    This holds whenever the fp16 scale is a normal number (relative rounding <= 2^-11).  A block
    with amax < 127 * 2^-14 gets a subnormal scale whose relative error can be large; there the
    elements with |x / s| <= 127 keep the bound and the rest clamp to +-127.
    """
    rng = np.random.default_rng(13)
    blocks = _random_blocks(4000, rng)
    n_normal = n_sub = 0
    for blk in blocks:
        codes, s16 = O.quantize_block(Q8, blk)
        s = float(np.uint16(s16).view(np.float16))
        x = bf16_to_f32(blk).astype(np.float64)
        q = codes.view(np.int8).astype(np.float64)
        err = np.abs(x - q * s)
        if s16 >= 0x0400:
            n_normal += 1
            assert np.all(err <= s / 2)
        elif s16 != 0:
            n_sub += 1
            inside = np.abs(x) <= 127 * s
            assert np.all(err[inside] <= s / 2)
            assert np.all(np.abs(q[~inside]) == 127)
    assert n_normal > 1000 and n_sub > 50


@pytest.mark.parametrize("kind", [FP8, Q8])
def test_zero_and_underflowing_blocks_store_zero(kind):
    codes, s16 = O.quantize_block(kind, np.zeros(32, np.uint16))
    assert s16 == 0 and not codes.any()
    tiny = bf16_bits(np.full(32, 1e-30, np.float32))   # amax / Q underflows fp16
    codes, s16 = O.quantize_block(kind, tiny)
    assert s16 == 0 and not codes.any()


def test_fp8_saturation_block_clamps_to_448_without_nan():
    """A block whose fp16 scale rounds below amax/448 pushes its maximum past 448; it must clamp."""
    rng = np.random.default_rng(3)
    found = 0
    for _ in range(2000):
        amax = np.float32(rng.uniform(1, 2000))
        blk = np.zeros(32, np.float32)
        blk[0] = amax
        blk[1] = -amax
        b = bf16_bits(blk)
        a = bf16_to_f32(b)[0]
        s16 = O.block_scale(FP8, b)
        s = np.float32(np.uint16(s16).view(np.float16))
        if a / s > 448.0:
            codes, _ = O.quantize_block(FP8, b)
            assert codes[0] == 0x7E and codes[1] == 0xFE
            found += 1
    assert found > 50
    blk = np.zeros(32, np.float32)
    blk[8], blk[19] = 1000.0, -1000.0
    codes, _ = O.quantize_block(FP8, bf16_bits(blk))
    assert codes[8] == 0x7E and codes[19] == 0xFE and not np.any((codes == 0x7F) | (codes == 0xFF))


def test_double_round_negative_control_differs_downward_at_the_quoted_rate():
    """Review comment 'A bug on sm_89': truncating through fp16 then RNE disagrees on ~0.4% of elements.

    Pins that the oracle's fp8 rounding is the single RNE (a value just above a midpoint goes up),
    and that the double round it is contrasted with only ever moves codes down by one step.
    """
    y = np.array([1.0625 + 2.0 ** -20, 1.1875 + 2.0 ** -18], np.float32)
    assert list(O.e4m3_sat_rne(y)) == [0x39, 0x3A + 0]  # 1.125 ; 1.25 (1.1875+ rounds up to even 1.25)
    assert list(O.e4m3_double_round(y)) == [0x38, 0x3A]  # first collapses onto the tie and goes down
    rng = np.random.default_rng(21)
    x = rng.standard_normal((1 << 15, 32)).astype(np.float32)
    xb = bf16_bits(x)
    ys = []
    for blk in xb:
        s16 = O.block_scale(FP8, blk)
        ys.append(bf16_to_f32(blk) / np.float32(np.uint16(s16).view(np.float16)))
    ys = np.concatenate(ys)
    a, b = O.e4m3_sat_rne(ys), O.e4m3_double_round(ys)
    diff = a != b
    rate = diff.mean()
    approx = GOLDEN["double_round_disagreement"]["approx_fraction"]
    assert 0.5 * approx < rate < 2.0 * approx, rate
    assert np.all((a[diff] & 0x7F).astype(int) - (b[diff] & 0x7F).astype(int) == 1)


# ============================================================================ cost model
@pytest.mark.parametrize("n_kv,hkv,d", [(2, 8, 128), (2, 2, 256), (1, 1, 576), (2, 4, 64)])
def test_bytes_per_token_is_1_0625_per_element(n_kv, hkv, d):
    per_elem = GOLDEN["bytes_per_element_8bit"]["value"]
    bq = O.bytes_per_token(n_kv, hkv, d)
    bb = GOLDEN["bytes_per_element_bf16"]["value"] * n_kv * hkv * d
    assert bq == per_elem * n_kv * hkv * d
    assert bq * 32 == bb * 17


def test_pool_growth_matches_the_quoted_token_counts():
    """Review comment 'End-to-end numbers': 305,730 bf16 tokens become 575,493 at the same budget."""
    pool = GOLDEN["kv_pool_tokens"]
    for layers, hkv, d in [(40, 2, 256), (40, 4, 256), (1, 1, 128)]:
        cb = 2.0 * 2 * hkv * d * layers
        cq = O.bytes_per_token(2, hkv, d) * layers
        lo = max(pool["bf16"] * cb, pool["fp8_e4m3"] * cq)
        hi = min((pool["bf16"] + 1) * cb, (pool["fp8_e4m3"] + 1) * cq)
        assert lo < hi                                   # a budget with both floors exists
        budget = (lo + hi) / 2
        assert math.floor(budget / cb) == pool["bf16"] and math.floor(budget / cq) == pool["q8_0"]
    assert abs(pool["fp8_e4m3"] / pool["bf16"] - 2 / 1.0625) < 1e-5


# ============================================================================ store
def _store_case(kind, mla=False, T=40, Hkv=2, D=64, P=16, num_pages=6, seed=0):
    rng = np.random.default_rng(seed)
    k = bf16_bits(rng.standard_normal((T, Hkv, D)).astype(np.float32) * 3)
    v = None if mla else bf16_bits(rng.standard_normal((T, Hkv, D)).astype(np.float32))
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    slots[::7] = -1
    cshape, sshape = O.pool_shapes(num_pages, P, Hkv, D, mla)
    codes = np.full(cshape, 0xA5, np.uint8)
    scales = np.full(sshape, 0xA5A5, np.uint16)
    O.store(codes, scales, k, v, slots, num_kv_heads=Hkv, head_dim=D, page_size=P, mla=mla, kind=kind)
    return k, v, slots, codes, scales


@pytest.mark.parametrize("kind", [FP8, Q8])
@pytest.mark.parametrize("mla", [False, True])
def test_store_scatters_rows_and_leaves_skipped_slots_untouched(kind, mla):
    P, D, Hkv = 16, 64, 2
    k, v, slots, codes, scales = _store_case(kind, mla=mla, Hkv=Hkv, D=D, P=P)
    written = np.zeros(codes.shape[:4], bool)  # [page, kv, h, off]
    for t, s in enumerate(slots):
        if s < 0:
            continue
        page, off = divmod(int(s), P)
        for kv, src in enumerate([k] if mla else [k, v]):
            for h in range(Hkv):
                for j in range(D // 32):
                    c, s16 = O.quantize_block(kind, src[t, h, 32 * j:32 * j + 32])
                    assert np.array_equal(codes[page, kv, h, off, 32 * j:32 * j + 32], c)
                    assert scales[page, kv, h, off, j] == s16
                written[page, kv, h, off] = True
    assert np.all(codes[~written] == 0xA5) and np.all(scales[~written] == 0xA5A5)


def test_store_is_independent_of_row_order():
    k, v, slots, codes, scales = _store_case(FP8, seed=4)
    perm = np.random.default_rng(9).permutation(len(slots))
    codes2 = np.full_like(codes, 0xA5)
    scales2 = np.full_like(scales, 0xA5A5)
    O.store(codes2, scales2, k[perm], v[perm], slots[perm], num_kv_heads=2, head_dim=64, page_size=16,
            mla=False, kind=FP8)
    assert np.array_equal(codes, codes2) and np.array_equal(scales, scales2)


# ============================================================================ decode
def _gather_dequant(codes, scales, kind, slots, kv, h, D):
    """Dequantized rows at the given slots, read by plain indexing of the pool arrays."""
    P = codes.shape[3]
    unscaled = O.KIND_BY_NAME.get(kind, kind) in O.UNSCALED  # the cast value (no scale), pinned code table
    table = np.array([O.code_value(kind, c) for c in range(256)]) if unscaled else None
    rows = []
    for s in slots:
        page, off = divmod(int(s), P)
        c = codes[page, kv, h, off]
        if unscaled:
            rows.append(table[c])
        else:
            sc = np.repeat(scales[page, kv, h, off], 32)
            rows.append(O.dequant(kind, c, sc))
    return np.array(rows).reshape(len(slots), D)


def _decode_setup(kind, *, B=2, Hq=8, Hkv=2, D=64, Dv=None, mla=False, lens=(37, 70), seed=0, P=16,
                  kfun=None, qfun=None, mask=()):
    rng = np.random.default_rng(seed)
    Dv = Dv or D
    npages = [(L + P - 1) // P for L in lens]
    num_pages = sum(npages) + 1
    perm = rng.permutation(num_pages)
    maxp = max(npages)
    bt = np.full((B, maxp), -1, np.int32)
    off = 0
    for b, n in enumerate(npages):
        bt[b, :n] = perm[off:off + n]
        off += n
    for (b, j) in mask:
        bt[b, j] = -1
    T = sum(lens)
    kf = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    if kfun is not None:
        kf = kfun(kf)
    k = bf16_bits(kf)
    v = None if mla else bf16_bits(rng.standard_normal((T, Hkv, D)).astype(np.float32))
    qf = (rng.standard_normal((B, Hq, D)) / math.sqrt(D)).astype(np.float32)
    if qfun is not None:
        qf = qfun(qf)
    q = bf16_bits(qf)
    slots = []
    for b, L in enumerate(lens):
        for t in range(L):
            p = bt[b, t // P]
            slots.append(-1 if p < 0 else p * P + t % P)
    slots = np.array(slots, np.int64)
    cshape, sshape = O.pool_shapes(num_pages, P, Hkv, D, mla)
    codes = np.zeros(cshape, np.uint8)
    scales = np.zeros(sshape, np.uint16)
    O.store(codes, scales, k, v, slots, num_kv_heads=Hkv, head_dim=D, page_size=P, mla=mla, kind=kind)
    return dict(q=q, codes=codes, scales=scales, bt=bt, lens=np.array(lens, np.int32), slots=slots,
                Hq=Hq, Hkv=Hkv, D=D, Dv=Dv, P=P, mla=mla, kind=kind, k=k, v=v)


def _run(s, sm_scale=1.0, lens=None):
    return O.decode(s["q"], s["codes"], s["scales"], s["bt"], s["lens"] if lens is None else lens,
                    num_q_heads=s["Hq"], num_kv_heads=s["Hkv"], head_dim=s["D"], v_dim=s["Dv"],
                    page_size=s["P"], mla=s["mla"], kind=s["kind"], sm_scale=sm_scale)


def _expected_scipy(s, sm_scale):
    """Attention through scipy.special.softmax over rows gathered from the pool by slot."""
    B, Hq, Hkv, D, Dv, P = len(s["lens"]), s["Hq"], s["Hkv"], s["D"], s["Dv"], s["P"]
    out = np.zeros((B, Hq, Dv))
    start = 0
    for b, L in enumerate(s["lens"]):
        sl = s["slots"][start:start + L]
        start += L
        sl = sl[sl >= 0]
        for h in range(Hq):
            g = h // (Hq // Hkv)
            if len(sl) == 0:
                continue
            K = _gather_dequant(s["codes"], s["scales"], s["kind"], sl, 0, g, D)
            V = K[:, :Dv] if s["mla"] else _gather_dequant(s["codes"], s["scales"], s["kind"], sl, 1, g, D)
            qv = bf16_to_f32(s["q"][b, h]).astype(np.float64)
            p = scipy.special.softmax(sm_scale * (K @ qv))
            out[b, h] = p @ V[:, :Dv]
    return out


@pytest.mark.parametrize("kind", [FP8, Q8])
@pytest.mark.parametrize("mla", [False, True])
def test_decode_matches_scipy_softmax_attention(kind, mla):
    D, Dv = (96, 64) if mla else (64, 64)
    s = _decode_setup(kind, mla=mla, D=D, Dv=Dv, Hkv=1 if mla else 2, mask=[(1, 2)])
    for sm_scale in (1.0, 0.37):
        np.testing.assert_allclose(_run(s, sm_scale), _expected_scipy(s, sm_scale), rtol=1e-12, atol=1e-13)


def test_decode_single_token_returns_its_value_row():
    s = _decode_setup(FP8, lens=(1, 1))
    out = _run(s)
    for b in range(2):
        for h in range(8):
            g = h // 4
            v = _gather_dequant(s["codes"], s["scales"], FP8, [s["slots"][b]], 1, g, 64)[0]
            assert np.array_equal(out[b, h], v)


def test_decode_identical_keys_or_zero_query_give_the_mean_value():
    s = _decode_setup(Q8, kfun=lambda k: np.broadcast_to(k[:1], k.shape).copy())
    s0 = _decode_setup(Q8, qfun=lambda q: q * 0)
    for st in (s, s0):
        out = _run(st, 2.0)
        start = 0
        for b, L in enumerate(st["lens"]):
            sl = st["slots"][start:start + L]
            start += L
            for h in range(8):
                V = _gather_dequant(st["codes"], st["scales"], Q8, sl, 1, h // 4, 64)
                np.testing.assert_allclose(out[b, h], V.mean(0), rtol=1e-12, atol=1e-14)


def test_decode_dominant_logit_returns_that_value_and_survives_huge_scores():
    def kfun(k):
        k = k * 0.01
        k[5] = 30.0          # token 5 (sequence 0) dominates every head
        return k
    s = _decode_setup(FP8, kfun=kfun, qfun=lambda q: np.abs(q) + 1.0, lens=(20, 3))
    out = _run(s, 50.0)      # scores ~ 1e5: plain exp() without max subtraction would overflow
    assert np.all(np.isfinite(out))
    for h in range(8):
        v = _gather_dequant(s["codes"], s["scales"], FP8, [s["slots"][5]], 1, h // 4, 64)[0]
        np.testing.assert_allclose(out[0, h], v, rtol=0, atol=1e-12)


def test_decode_masked_page_equals_removing_its_tokens():
    s = _decode_setup(FP8, lens=(70, 37), mask=[(0, 1), (0, 4)])
    out = _run(s)
    ref = _expected_scipy(s, 1.0)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    # all pages masked, or no tokens: zeros
    s2 = _decode_setup(FP8, lens=(20, 5), mask=[(1, 0)])
    out2 = _run(s2, lens=np.array([0, 5], np.int32))
    assert not out2[0].any() and not out2[1].any()


def test_decode_gqa_heads_read_their_own_kv_head():
    """q head h reads kv head h // (Hq/Hkv): permuting kv heads permutes the output head groups."""
    s = _decode_setup(FP8, Hq=8, Hkv=2)
    out = _run(s)
    swapped = dict(s)
    swapped["codes"] = s["codes"][:, :, ::-1].copy()
    swapped["scales"] = s["scales"][:, :, ::-1].copy()
    q2 = np.concatenate([s["q"][:, 4:], s["q"][:, :4]], axis=1)
    swapped["q"] = q2
    out2 = _run(swapped)
    np.testing.assert_array_equal(out2[:, 4:], out[:, :4])
    np.testing.assert_array_equal(out2[:, :4], out[:, 4:])


def _expected_bf16_scipy(s, sm_scale):
    """Unquantized attention by scipy over the input bf16 rows themselves, taken by token index (not through
    any pool): row t of sequence b is visible when its slot is not -1 (its page is not masked)."""
    B, Hq, Hkv, D, Dv = len(s["lens"]), s["Hq"], s["Hkv"], s["D"], s["Dv"]
    kf = bf16_to_f32(s["k"]).astype(np.float64)
    vf = kf if s["mla"] else bf16_to_f32(s["v"]).astype(np.float64)
    out = np.zeros((B, Hq, Dv))
    start = 0
    for b, L in enumerate(s["lens"]):
        rows = np.arange(start, start + L)[s["slots"][start:start + L] >= 0]
        start += L
        for h in range(Hq):
            g = h // (Hq // Hkv)
            if len(rows) == 0:
                continue
            qv = bf16_to_f32(s["q"][b, h]).astype(np.float64)
            p = scipy.special.softmax(sm_scale * (kf[rows, g] @ qv))
            out[b, h] = p @ vf[rows, g, :Dv]
    return out


def _run_bf16(s, sm_scale=1.0, lens=None):
    pool16 = np.zeros(s["codes"].shape, np.uint16)
    O.scatter_bf16(pool16, s["k"], s["v"], s["slots"], num_kv_heads=s["Hkv"], head_dim=s["D"], page_size=s["P"],
                   mla=s["mla"])
    return O.decode_bf16(s["q"], pool16, s["bt"], s["lens"] if lens is None else lens, num_q_heads=s["Hq"],
                         num_kv_heads=s["Hkv"], head_dim=s["D"], v_dim=s["Dv"], page_size=s["P"], mla=s["mla"],
                         sm_scale=sm_scale)


@pytest.mark.parametrize("mla", [False, True])
def test_unquantized_decode_matches_scipy_attention_over_the_input_rows(mla):
    """The unquantized reference (bf16 K/V scattered to a 2-byte pool, then exact attention) equals scipy
    attention over the input rows taken by token index, so a wrong pool index, head or V row in either the
    scatter or the decode fails it; masked pages, GQA grouping and MLA's shared row included."""
    D, Dv = (96, 64) if mla else (64, 64)
    s = _decode_setup(FP8, mla=mla, D=D, Dv=Dv, Hkv=1 if mla else 2, mask=[(1, 2), (0, 0)])
    for sm_scale in (1.0, 0.37):
        np.testing.assert_allclose(_run_bf16(s, sm_scale), _expected_bf16_scipy(s, sm_scale), rtol=1e-12,
                                   atol=1e-13)
    # no valid token gives zeros, as in the quantized decode
    out0 = _run_bf16(s, lens=np.array([0, 5], np.int32))
    assert not out0[0].any()


def test_unquantized_decode_of_exactly_representable_rows_equals_the_quantized_decode():
    """Rows whose values are code * scale exactly (one fp16 power-of-two scale per block, values on the E4M3
    grid) dequantize to themselves, so the quantized and unquantized references must agree to the last bit."""
    rng = np.random.default_rng(5)

    def on_grid(x):
        # E4M3 grid values times 2^-3 (max |x| per block 448 * 2^-3): the block scale amax/448 is 2^-3 exactly
        # when every block holds a +-448 * 2^-3 element
        c = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float32).numpy()
        c = c.reshape(*c.shape[:-1], -1, 32)
        c[..., 0] = 448.0
        return (c * 0.125).reshape(x.shape)

    s = _decode_setup(FP8, kfun=lambda k: on_grid(k * 40), lens=(23, 41))
    s["v"] = bf16_bits(on_grid(rng.standard_normal((sum(s["lens"]), 2, 64)) * 40).astype(np.float32))
    O.store(s["codes"], s["scales"], s["k"], s["v"], s["slots"], num_kv_heads=2, head_dim=64, page_size=16, mla=False,
            kind=FP8)
    assert np.array_equal(_run_bf16(s, 0.05), _run(s, 0.05))


# ===================================================================== sparse (top-K) decode
def _sparse_indices(s, topk, rng, *, junk=True):
    """[B, topk] positions: a random selection of each sequence's positions (a few listed twice), with
    -1 entries and positions past the sequence end mixed in when `junk`."""
    B = len(s["lens"])
    ix = np.full((B, topk), -1, np.int32)
    for b, L in enumerate(s["lens"]):
        pos = rng.permutation(int(L))[: max(1, topk // 2)]
        sel = list(pos) + list(pos[:3])                        # three positions listed twice
        if junk:
            sel += [-1, int(L), int(L) + 5]                     # masked and out-of-range columns
        sel = np.array(sel[:topk], np.int32)
        rng.shuffle(sel)
        ix[b, :len(sel)] = sel
    return ix


def _run_sparse(s, ix, sm_scale=1.0):
    return O.decode_sparse(s["q"], s["codes"], s["scales"], s["bt"], s["lens"], ix, num_q_heads=s["Hq"],
                           num_kv_heads=s["Hkv"], head_dim=s["D"], v_dim=s["Dv"], page_size=s["P"],
                           mla=s["mla"], kind=s["kind"], sm_scale=sm_scale)


def _expected_sparse_scipy(s, ix, sm_scale):
    """scipy softmax attention over the listed columns, each valid column gathered by its slot."""
    B, Hq, Hkv, D, Dv, P = len(s["lens"]), s["Hq"], s["Hkv"], s["D"], s["Dv"], s["P"]
    out = np.zeros((B, Hq, Dv))
    for b, L in enumerate(s["lens"]):
        slots = []
        for p in ix[b]:
            if 0 <= p < L and s["bt"][b, p // P] >= 0:
                slots.append(int(s["bt"][b, p // P]) * P + int(p) % P)
        if not slots:
            continue
        for h in range(Hq):
            g = h // (Hq // Hkv)
            K = _gather_dequant(s["codes"], s["scales"], s["kind"], slots, 0, g, D)
            V = K[:, :Dv] if s["mla"] else _gather_dequant(s["codes"], s["scales"], s["kind"], slots, 1, g, D)
            qv = bf16_to_f32(s["q"][b, h]).astype(np.float64)
            out[b, h] = scipy.special.softmax(sm_scale * (K @ qv)) @ V[:, :Dv]
    return out


@pytest.mark.parametrize("kind", [FP8, Q8])
@pytest.mark.parametrize("mla", [False, True])
def test_sparse_decode_matches_scipy_attention_over_the_listed_columns(kind, mla):
    """Random selections with repeated positions, -1 columns, positions past the end and a masked page."""
    D, Dv = (96, 64) if mla else (64, 64)
    s = _decode_setup(kind, mla=mla, D=D, Dv=Dv, Hkv=1 if mla else 2, mask=[(1, 2)])
    ix = _sparse_indices(s, 40, np.random.default_rng(5))
    for sm_scale in (1.0, 0.37):
        np.testing.assert_allclose(_run_sparse(s, ix, sm_scale), _expected_sparse_scipy(s, ix, sm_scale),
                                   rtol=1e-12, atol=1e-13)


def test_sparse_decode_listing_every_position_equals_the_dense_decode():
    s = _decode_setup(FP8, mask=[(0, 1)])
    topk = int(max(s["lens"]))
    ix = np.full((len(s["lens"]), topk), -1, np.int32)
    for b, L in enumerate(s["lens"]):
        ix[b, :L] = np.random.default_rng(b).permutation(int(L))   # order does not matter
    np.testing.assert_allclose(_run_sparse(s, ix), _run(s), rtol=1e-12, atol=1e-13)


def test_sparse_decode_closed_forms():
    s = _decode_setup(Q8, mla=True, D=96, Dv=64, Hkv=1)
    B = len(s["lens"])
    # one listed column: the output is that token's value row
    ix = np.full((B, 8), -1, np.int32)
    ix[:, 3] = 5
    got = _run_sparse(s, ix)
    for b in range(B):
        slot = int(s["bt"][b, 0]) * s["P"] + 5
        row = _gather_dequant(s["codes"], s["scales"], Q8, [slot], 0, 0, 96)[0, :64]
        for h in range(s["Hq"]):
            np.testing.assert_allclose(got[b, h], row, rtol=0, atol=1e-15)
    # no valid column (all -1, or all past the end): zeros
    none = np.full((B, 8), -1, np.int32)
    assert not np.any(_run_sparse(s, none))
    past = np.tile(np.array([[1000, 2000]], np.int32), (B, 1))
    assert not np.any(_run_sparse(s, past))
    # listing a position twice equals listing it once with twice the weight: two columns, one doubled
    two = np.full((B, 3), -1, np.int32)
    two[:, 0], two[:, 1], two[:, 2] = 2, 9, 9
    ref = _expected_sparse_scipy(s, two, 1.0)
    np.testing.assert_allclose(_run_sparse(s, two), ref, rtol=1e-12, atol=1e-13)


# ===================================================================== extend (prefill) attention
def _extend_q(s, n_new, seed=9):
    """Query rows [sum(n_new), Hq, D] and q_start for n_new new tokens per sequence."""
    rng = np.random.default_rng(seed)
    total = int(sum(n_new))
    qf = (rng.standard_normal((total, s["Hq"], s["D"])) / math.sqrt(s["D"])).astype(np.float32)
    q_start = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    return bf16_bits(qf), q_start


def _run_extend(s, q, q_start, sm_scale=1.0, lens=None):
    return O.extend(q, s["codes"], s["scales"], s["bt"], s["lens"] if lens is None else lens, q_start,
                    num_q_heads=s["Hq"], num_kv_heads=s["Hkv"], head_dim=s["D"], v_dim=s["Dv"], page_size=s["P"],
                    mla=s["mla"], kind=s["kind"], sm_scale=sm_scale)


def _expected_extend_scipy(s, q, q_start, sm_scale):
    """scipy softmax attention of each new token over the positions 0..pos of its sequence, every valid
    position gathered from the pool by its slot (pos = seq_len - n_new + i)."""
    Hq, Hkv, D, Dv, P = s["Hq"], s["Hkv"], s["D"], s["Dv"], s["P"]
    out = np.zeros((q.shape[0], Hq, Dv))
    for b, L in enumerate(s["lens"]):
        n = int(q_start[b + 1] - q_start[b])
        for i in range(n):
            pos = int(L) - n + i
            slots = [int(s["bt"][b, t // P]) * P + t % P for t in range(pos + 1) if s["bt"][b, t // P] >= 0]
            if not slots:
                continue
            row = int(q_start[b]) + i
            for h in range(Hq):
                g = h // (Hq // Hkv)
                K = _gather_dequant(s["codes"], s["scales"], s["kind"], slots, 0, g, D)
                V = K[:, :Dv] if s["mla"] else _gather_dequant(s["codes"], s["scales"], s["kind"], slots, 1, g, D)
                qv = bf16_to_f32(q[row, h]).astype(np.float64)
                out[row, h] = scipy.special.softmax(sm_scale * (K @ qv)) @ V[:, :Dv]
    return out


@pytest.mark.parametrize("kind", [FP8, Q8])
@pytest.mark.parametrize("mla", [False, True])
def test_extend_matches_scipy_causal_attention(kind, mla):
    """Every new token against scipy softmax over its causal prefix: a masked page, one sequence wholly new
    (a first prefill: its token 0 sees only itself), one with a few new tokens after its context."""
    D, Dv = (96, 64) if mla else (64, 64)
    s = _decode_setup(kind, mla=mla, D=D, Dv=Dv, Hkv=1 if mla else 2, mask=[(1, 2)])
    q, q_start = _extend_q(s, [37, 21])
    for sm_scale in (1.0, 0.37):
        np.testing.assert_allclose(_run_extend(s, q, q_start, sm_scale), _expected_extend_scipy(s, q, q_start, sm_scale),
                                   rtol=1e-12, atol=1e-13)


def test_extend_one_new_token_per_sequence_equals_the_decode():
    s = _decode_setup(FP8, mask=[(0, 1)])
    q_start = np.arange(len(s["lens"]) + 1, dtype=np.int32)
    q = s["q"].reshape(len(s["lens"]), s["Hq"], s["D"])
    np.testing.assert_array_equal(_run_extend(s, q, q_start), _run(s))


def test_extend_each_new_token_equals_the_decode_of_its_prefix():
    """Causality: new token i of sequence b gives what a decode of the same query over a sequence cut to
    pos + 1 tokens gives; no later position contributes."""
    s = _decode_setup(Q8, mask=[(1, 3)])
    n_new = [9, 30]
    q, q_start = _extend_q(s, n_new)
    got = _run_extend(s, q, q_start)
    for b, L in enumerate(s["lens"]):
        for i in range(n_new[b]):
            pos = int(L) - n_new[b] + i
            lens = np.array(s["lens"])
            lens[b] = pos + 1
            row = int(q_start[b]) + i
            sd = dict(s, q=np.repeat(q[row][None], len(lens), axis=0))
            np.testing.assert_array_equal(got[row], _run(sd, lens=lens)[b])


def test_extend_closed_forms():
    """Identical keys: new token i gives the plain mean of the value rows at the unmasked positions 0..pos,
    so an off-by-one in the causal bound changes the mean; a first-prefill token 0 returns value row 0;
    a masked page drops out; a sequence with no new token adds no row."""
    s = _decode_setup(Q8, kfun=lambda k: np.broadcast_to(k[:1], k.shape).copy(), mask=[(1, 1)])
    n_new = [37, 5]
    q, q_start = _extend_q(s, n_new)
    got = _run_extend(s, q, q_start, 3.0)
    P = s["P"]
    for b, L in enumerate(s["lens"]):
        for i in range(n_new[b]):
            pos = int(L) - n_new[b] + i
            slots = [int(s["bt"][b, t // P]) * P + t % P for t in range(pos + 1) if s["bt"][b, t // P] >= 0]
            for h in range(s["Hq"]):
                g = h // (s["Hq"] // s["Hkv"])
                V = _gather_dequant(s["codes"], s["scales"], Q8, slots, 1, g, s["D"])
                np.testing.assert_allclose(got[int(q_start[b]) + i, h], V.mean(axis=0), rtol=1e-12, atol=1e-14)
    v0 = _gather_dequant(s["codes"], s["scales"], Q8, [int(s["bt"][0, 0]) * P], 1, 0, s["D"])[0]
    np.testing.assert_array_equal(got[0, 0], v0)
    # no new token for sequence 0: only sequence 1's rows, unchanged
    q1, qs1 = q[37:], np.array([0, 0, 5], np.int32)
    np.testing.assert_array_equal(_run_extend(s, q1, qs1, 3.0), got[37:])


def test_extend_rejects_more_new_tokens_than_stored_and_a_bad_q_start():
    s = _decode_setup(FP8)
    q, q_start = _extend_q(s, [38, 2])  # sequence 0 holds 37 tokens
    with pytest.raises(ValueError):
        _run_extend(s, q, q_start)
    q, q_start = _extend_q(s, [3, 2])
    with pytest.raises(ValueError):
        _run_extend(s, q, q_start + 1)


@pytest.mark.parametrize("kind", [FP8, Q8])
def test_absolute_value_pool_gives_the_weighted_mean_of_abs_v(kind):
    """The parity tests' error scale sum_t p_t |V_t|: over the pool with absolute V codes the decode is at
    least |decode| everywhere (triangle inequality), and equals the decode when every V is already >= 0."""
    from parity import abs_value_pool
    s = _decode_setup(kind, mask=[(1, 2)])
    out = _run(s)
    sa = dict(s, codes=abs_value_pool(s["codes"], kind))
    scale = _run(sa)
    assert np.all(scale >= np.abs(out) - 1e-12) and np.any(scale > np.abs(out) + 1e-3)
    pos = _decode_setup(kind, seed=3)
    pos["codes"] = abs_value_pool(pos["codes"], kind)
    np.testing.assert_array_equal(_run(dict(pos, codes=abs_value_pool(pos["codes"], kind))), _run(pos))


# ===================================================================== unscaled fp8 (e4m3 / e5m2 casts)
def test_e5m2_value_of_every_code_matches_torch():
    """The E5M2 decoding written from the format's definition against torch's float8_e5m2 (library routine)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    got = np.array([O.e5m2_value(c) for c in codes])
    np.testing.assert_array_equal(got, ref)
    assert O.e5m2_value(0x3C) == 1.0 and O.e5m2_value(0x7B) == 57344.0 and O.e5m2_value(0x01) == 2.0 ** -16


def test_e5m2_nearest_even_matches_torch_cast_on_every_bf16_in_range():
    """Every finite bf16 value with |x| <= 57344: one nearest-even rounding, as torch's float8_e5m2 cast; beyond
    the largest finite value the cache's cast saturates instead of producing infinity."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    xf = x.float().numpy()
    ok = np.isfinite(xf) & (np.abs(xf) <= 57344.0)
    got = O.e5m2_sat_rne(xf[ok])
    ref = x[torch.from_numpy(ok)].to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(got, ref), int((got != ref).sum())
    big = xf[np.isfinite(xf) & (np.abs(xf) > 57344.0)]
    sat = O.e5m2_sat_rne(big)
    assert np.all(sat == np.where(big > 0, 0x7B, 0xFB))


def test_unscaled_store_is_the_plain_cast_and_costs_one_byte_per_element():
    """The unscaled kinds cast each bf16 value to fp8 with no scale (1 byte per element, twice the bf16
    token budget: the pages' 27,142 -> 54,284 tokens at equal bytes)."""
    g = GOLDEN["unscaled_fp8_kv_budget_tokens"]
    for kind in ("fp8_e4m3_unscaled", "fp8_e5m2_unscaled"):
        assert O.bytes_per_element(kind) == 1.0
        assert round(GOLDEN["bytes_per_element_bf16"]["value"] / O.bytes_per_element(kind), 2) == g["ratio"]
        assert abs(g["fp8_e4m3"] / g["bf16"] - 2.0) < 1e-3
        s = _decode_setup(kind, mask=[(1, 1)])
        P = s["P"]
        for t, slot in enumerate(s["slots"]):
            if slot < 0:
                continue
            page, off = divmod(int(slot), P)
            for kv, src in ((0, s["k"]), (1, s["v"])):
                xf = bf16_to_f32(src[t]).reshape(-1)
                want = (O.e4m3_sat_rne(xf) if kind == "fp8_e4m3_unscaled" else O.e5m2_sat_rne(xf))
                assert np.array_equal(s["codes"][page, kv, :, off].reshape(-1), want)


@pytest.mark.parametrize("kind", ["fp8_e4m3_unscaled", "fp8_e5m2_unscaled"])
def test_unscaled_decode_and_extend_match_scipy_over_the_cast_values(kind):
    s = _decode_setup(kind, mask=[(1, 2)])
    for sm_scale in (1.0, 0.37):
        np.testing.assert_allclose(_run(s, sm_scale), _expected_scipy(s, sm_scale), rtol=1e-12, atol=1e-13)
    q, q_start = _extend_q(s, [37, 21])
    np.testing.assert_allclose(_run_extend(s, q, q_start), _expected_extend_scipy(s, q, q_start, 1.0),
                               rtol=1e-12, atol=1e-13)


# ===================================================================== the store fused with its producer
def test_act_quant64_matches_torch_float8_rounding():
    """One fp32 scale (amax / 448) per 64 elements, torch's float8_e4m3fn cast of x / s, times s in fp32, to
    bf16: the same numbers through a library routine (the mla workload generator does the same)."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn(32, 512, generator=g) * torch.exp(torch.randn(32, 8, 1, generator=g)).repeat(1, 1, 64).reshape(32, 512)
    x[3, 64:128] = 0.0                                   # an all-zero block stays zero
    x[4, 0] = 3.0e38                                     # a huge block: its scale is still finite
    xb = x.to(torch.bfloat16)
    blocks = xb.float().reshape(32, 8, 64)
    s = blocks.abs().amax(-1, keepdim=True) / 448.0
    s = torch.where(s > 0, s, torch.ones_like(s))
    ref = ((blocks / s).to(torch.float8_e4m3fn).float() * s).reshape(32, 512).to(torch.bfloat16)
    got = O.act_quant64(xb.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(got, ref.view(torch.int16).numpy().view(np.uint16))


def test_fused_mla_store_rounds_the_latent_and_keeps_the_rope_tail():
    """The fused store's codes: latent = the store of the act_quant64 rows; rope tail = the plain store of the
    same bf16 values (those dims are rounded for the first time by the store itself)."""
    g = torch.Generator().manual_seed(6)
    T, D, rope, P = 40, 576, 64, 16
    k = (torch.randn(T, 1, D, generator=g) * 2).to(torch.bfloat16)
    kb = k.view(torch.int16).numpy().view(np.uint16)
    slots = np.arange(T, dtype=np.int64)
    cs, ss = O.pool_shapes(3, P, 1, D, True)
    fused_c, fused_s = np.zeros(cs, np.uint8), np.zeros(ss, np.uint16)
    O.store_act_quant(fused_c, fused_s, kb.reshape(T, D), slots, head_dim=D, rope_dim=rope, page_size=P, kind=FP8)
    lat = O.act_quant64(kb[:, 0, :D - rope])
    pre = np.concatenate([lat, kb[:, 0, D - rope:]], axis=1)[:, None, :]
    plain_c, plain_s = np.zeros(cs, np.uint8), np.zeros(ss, np.uint16)
    O.store(plain_c, plain_s, pre, None, slots, num_kv_heads=1, head_dim=D, page_size=P, mla=True, kind=FP8)
    assert np.array_equal(fused_c, plain_c) and np.array_equal(fused_s, plain_s)
    raw_c, raw_s = np.zeros(cs, np.uint8), np.zeros(ss, np.uint16)
    O.store(raw_c, raw_s, kb, None, slots, num_kv_heads=1, head_dim=D, page_size=P, mla=True, kind=FP8)
    assert np.array_equal(fused_c[..., D - rope:], raw_c[..., D - rope:])      # rope tail untouched by act_quant
    assert not np.array_equal(fused_c[..., :D - rope], raw_c[..., :D - rope])  # the latent is not
    with pytest.raises(ValueError):
        O.store_act_quant(fused_c, fused_s, kb.reshape(T, D), slots, head_dim=D, rope_dim=32, page_size=P, kind=FP8)
