"""GPU store parity: the CUDA store is bit-exact against the oracle (every code byte, every scale bit),
and its rounding primitives agree with the oracle exhaustively on their domains."""
import numpy as np
import pytest
import torch

import oracle as O
from block_quantized_bit_gb300 import kvq, workloads

from parity import bits, gpu_pool, gpu_store, oracle_pool, oracle_store

pytestmark = pytest.mark.gpu
KINDS = ["fp8_e4m3", "q8_0"]

# reduced sizes of every workload family: several warps' worth of blocks and a ragged tail
CASES = {
    "tiny": dict(),
    "qwen3_1p7b": dict(batch=3, ctx_lo=100, ctx_hi=900, new_rows_per_seq=97),
    "long_gqa": dict(batch=2, ctx=2100, mask_frac=0.02),
    "mla": dict(ctx=1037),
    "serving": dict(batch=6, median=300, lo=40, hi=2000),
}


def _case(name, kind, **kw):
    return workloads.make(name, kind=kind, device="cpu", **{**CASES[name], **kw})


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("name", list(CASES))
def test_store_bit_exact(name, kind):
    case = _case(name, kind)
    L, codes, scales = gpu_pool(case)
    oc, osc = oracle_pool(case)
    gpu_store(case, codes, scales)
    oracle_store(case, oc, osc)
    if case.new_k is not None:
        gpu_store(case, codes, scales, rows="new")
        oracle_store(case, oc, osc, rows="new")
    torch.cuda.synchronize()
    gc = codes.cpu().numpy()
    gs = scales.cpu().numpy().view(np.uint16)
    assert np.array_equal(gc, oc), "code bytes differ at %d places" % int((gc != oc).sum())
    assert np.array_equal(gs, osc), "scale bits differ at %d places" % int((gs != osc).sum())
    # never a NaN code
    if kind == "fp8_e4m3":
        written = gs != 0xA5A5
        assert not np.any((gc[np.repeat(written, 32, axis=-1)] & 0x7F) == 0x7F)


@pytest.mark.parametrize("kind", KINDS)
def test_store_edge_cases(kind):
    case = workloads.tiny(kind=kind, ctx=37)
    L, codes, scales = gpu_pool(case)
    dev = "cuda"
    # zero rows: nothing happens
    kvq.kvq_store(codes, scales, case.k[:0].to(dev), case.v[:0].to(dev), case.slot_mapping[:0].to(dev), L, kind)
    # every slot skipped: the poisoned pool stays as it was
    skip = torch.full_like(case.slot_mapping, -1)
    kvq.kvq_store(codes, scales, case.k.to(dev), case.v.to(dev), skip.to(dev), L, kind)
    torch.cuda.synchronize()
    assert bool((codes == 0xA5).all()) and bool((scales.view(torch.int16) == np.int16(np.uint16(0xA5A5))).all())
    # a single row, then the rest in reverse order
    one = slice(5, 6)
    kvq.kvq_store(codes, scales, case.k[one].to(dev), case.v[one].to(dev), case.slot_mapping[one].to(dev), L, kind)
    idx = torch.arange(case.k.shape[0] - 1, -1, -1)
    kvq.kvq_store(codes, scales, case.k[idx].to(dev), case.v[idx].to(dev), case.slot_mapping[idx].to(dev), L, kind)
    oc, osc = oracle_pool(case)
    oracle_store(case, oc, osc)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), osc)


def test_store_special_blocks_of_the_tiny_workload():
    """All-zero block -> zero scale and codes; +-1000 block saturates to 0x7E/0xFE (fp8) or +-127 (q8_0)."""
    for kind in KINDS:
        case = workloads.tiny(kind=kind)
        L, codes, scales = gpu_pool(case)
        gpu_store(case, codes, scales)
        torch.cuda.synchronize()
        c = codes.cpu().numpy()
        s = scales.cpu().numpy().view(np.uint16)
        assert s[0, 0, 0, 0, 0] == 0 and not c[0, 0, 0, 0, 0:32].any()     # token 0, K, head 0, block 0
        blk = c[0, 1, 1, 1, 32:64]                                          # token 1, V, head 1, block 1
        if kind == "fp8_e4m3":
            assert blk[8] == 0x7E and blk[19] == 0xFE
        else:
            assert blk.view(np.int8)[8] == 127 and blk.view(np.int8)[19] == -127


def _fp32_sweep():
    """fp32 values covering every E4M3 binade: a strided sweep of all bit patterns plus every
    midpoint between adjacent E4M3 values with its 64 neighbours on each side."""
    pats = np.arange(0, 1 << 32, 257, dtype=np.uint64).astype(np.uint32).view(np.float32)
    pats = pats[np.isfinite(pats)]
    vals = sorted({O.e4m3_value(c) for c in range(0x7F)})
    mids = np.array([(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])] + [448.0, 464.0], np.float32)
    near = [mids]
    for d in range(1, 65):
        near.append(np.nextafter(mids, np.float32(np.inf)) if d == 1 else
                    (mids.view(np.uint32) + d).view(np.float32))
        near.append((mids.view(np.uint32) - d).view(np.float32))
    near = np.concatenate(near)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 0.49999997, 0.5, 126.5, 127.5, -127.5, 1e30],
                       np.float32)
    # every integer tie k + 0.5 of the int8 range and its four fp32 neighbours on each side
    ties = np.arange(-130, 131, dtype=np.float32) + np.float32(0.5)
    tie_near = [ties] + [(ties.view(np.uint32) + d).view(np.float32) for d in range(1, 5)] + \
        [(ties.view(np.uint32) - d).view(np.float32) for d in range(1, 5)]
    tie_near = np.concatenate(tie_near)
    y = np.concatenate([pats, near, -near, special, np.linspace(-130, 130, 1 << 20, dtype=np.float32), tie_near,
                        -tie_near])
    return y


@pytest.mark.parametrize("kind", KINDS)
def test_encode_probe_matches_oracle_on_fp32_sweep(kind):
    """The store's code step (hardware satfinite RNE for fp8; the truncated half-offset sum and saturating pack for
    q8_0) vs the oracle."""
    y = _fp32_sweep()
    yd = torch.from_numpy(y).cuda()
    codes = torch.empty(y.size, dtype=torch.uint8, device="cuda")
    kvq.kvq_encode_probe(kind, yd, codes)
    torch.cuda.synchronize()
    got = codes.cpu().numpy()
    ref = O.e4m3_sat_rne(y) if kind == "fp8_e4m3" else O.q8_rhaz(y).view(np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(y[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


@pytest.mark.parametrize("kind", KINDS)
def test_dequant_probe_matches_oracle_for_every_code_and_scale(kind):
    """The decode's dequant routine vs RNE_bf16(code * scale) for all codes x all finite positive fp16 scales."""
    codes = np.arange(256, dtype=np.uint8)
    if kind == "fp8_e4m3":
        codes = codes[(codes != 0x7F) & (codes != 0xFF)]
    codes = np.concatenate([codes, np.zeros((-codes.size) % 16, np.uint8)])  # whole 16-code chunks
    s16 = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    chunk_codes = np.tile(codes, s16.size)
    chunk_scales = np.repeat(s16, codes.size // 16)
    got = torch.empty(chunk_codes.size, dtype=torch.int16, device="cuda")
    kvq.kvq_dequant_probe(kind, torch.from_numpy(chunk_codes).cuda(),
                          torch.from_numpy(chunk_scales.view(np.int16)).cuda(), got)
    torch.cuda.synchronize()
    g = got.cpu().numpy().view(np.uint16)
    ref = O.dequant(kind, chunk_codes, np.repeat(s16, codes.size))
    ref_bits = O.bf16_rne(ref)
    if kind == "q8_0":
        # A zero scale only ever comes with zero codes (zero block).  For a negative int8 code the exact
        # product is -0; the offset form of the routine returns +0 there: the same number.
        zero = np.repeat(s16, codes.size) == 0
        assert np.all(g[zero] & 0x7FFF == 0) and np.all(ref_bits[zero] & 0x7FFF == 0)
        g, ref_bits = g[~zero], ref_bits[~zero]
    assert np.array_equal(g, ref_bits), int((g != ref_bits).sum())


@pytest.mark.parametrize("kind", KINDS)
def test_store_quotient_gives_ieee_codes_for_every_bf16_and_fp16_scale(kind):
    """The store's division (reciprocal + FMA-remainder correction) yields, for every finite bf16 x and
    every nonzero finite fp16 scale s with |x / s| <= 2^64, the same code as the oracle's IEEE fp32 x / s.

    Larger quotients cannot occur in a block: |x| <= amax, and the scale s = fp16(amax / Q) is at
    least amax / (1.5 Q) even when it is subnormal, so |x / s| <= 1.5 * 448."""
    xb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    xb = xb[((xb >> 7) & 0xFF) != 0xFF]                          # finite bf16 only
    sb = np.arange(1, 0x7C00, dtype=np.uint32).astype(np.uint16)  # every nonzero finite fp16 scale
    x_d = torch.from_numpy(xb.view(np.int16)).cuda()
    chunk = 2048
    for i0 in range(0, sb.size, chunk):
        s = sb[i0:i0 + chunk]
        out = torch.empty(s.size * xb.size, dtype=torch.uint8, device="cuda")
        kvq.kvq_quantize_probe(kind, x_d, torch.from_numpy(s.view(np.int16)).cuda(), out)
        got = out.cpu().numpy().reshape(s.size, xb.size)
        ref = O.code_table(kind, xb, s)
        xf = np.abs((xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
        sf = s.view(np.float16).astype(np.float64)
        reachable = xf[None, :] <= (2.0 ** 64) * sf[:, None]
        bad = np.argwhere((got != ref) & reachable)
        assert bad.size == 0, [(hex(int(s[i])), hex(int(xb[j])), int(got[i, j]), int(ref[i, j])) for i, j in bad[:8]]


@pytest.mark.parametrize("kind", KINDS)
def test_store_quotient_at_the_saturated_scale_for_every_bf16(kind):
    """A block whose amax / Q exceeds the largest fp16 gets the scale 65504 (0x7BFF) and its quotients reach
    |x / s| ~ 2^112, beyond the 2^64 the general sweep covers: the store's division still gives the oracle's
    code for every finite bf16 x at that scale (the large quotients saturate on both sides)."""
    xb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    xb = xb[((xb >> 7) & 0xFF) != 0xFF]
    s = np.array([0x7BFF], np.uint16)
    out = torch.empty(xb.size, dtype=torch.uint8, device="cuda")
    kvq.kvq_quantize_probe(kind, torch.from_numpy(xb.view(np.int16)).cuda(), torch.from_numpy(s.view(np.int16)).cuda(),
                           out)
    got = out.cpu().numpy()
    ref = O.code_table(kind, xb, s).reshape(-1)
    assert np.array_equal(got, ref), int((got != ref).sum())


@pytest.mark.parametrize("kind", KINDS)
def test_store_blocks_beyond_the_largest_scale_are_bit_exact(kind):
    """Rows whose blocks hold magnitudes up to 3e38 (amax far above 65504 * Q): the scale saturates at 0x7BFF
    and the codes at +-448 / +-127, identically on the GPU and in the oracle."""
    g = torch.Generator().manual_seed(12)
    T, Hkv, D, P = 40, 2, 128, 16
    k = torch.randn(T, Hkv, D, generator=g) * torch.exp(torch.rand(T, Hkv, 1, generator=g) * 80.0)  # up to ~1e34
    k[0, 0, :32] = torch.linspace(-1.0, 1.0, 32) * 3.0e38    # (a linspace over +-3e38 overflows its fp32 step)
    k[1, 1, 32:64] = 3.0e7                                   # just above 65504 * 448
    v = torch.randn(T, Hkv, D, generator=g) * 1e9
    kb, vb = k.to(torch.bfloat16), v.to(torch.bfloat16)
    assert torch.isfinite(kb.float()).all() and torch.isfinite(vb.float()).all()
    slots = torch.randperm(4 * P, generator=g)[:T].to(torch.int64)
    L = kvq.Layout(4, P, Hkv, D, D)
    codes, scales = kvq.alloc_pool(L, "cuda")
    codes.fill_(0x33)
    scales.fill_(0x1111)
    kvq.kvq_store(codes, scales, kb.cuda(), vb.cuda(), slots.cuda(), L, kind)
    torch.cuda.synchronize()
    oc = np.full(L.codes_shape(), 0x33, np.uint8)
    osc = np.full(L.scales_shape(), 0x1111, np.uint16)
    O.store(oc, osc, bits(kb), bits(vb), slots.numpy(), num_kv_heads=Hkv, head_dim=D, page_size=P, mla=False, kind=kind)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), osc)
    assert (osc == 0x7BFF).any()                             # the saturated scale occurs
