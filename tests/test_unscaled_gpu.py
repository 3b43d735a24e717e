"""GPU parity of attention over unscaled fp8 pools ("Add fp8 KV-cache quantization (--kv-dtype)", section
"How it works": the store casts bf16 K/V to the pool's fp8 type with scale 1.0 and attention reads the fp8
values back).  Pools written by kvq_store_unscaled (e4m3 and e5m2) are read by the decode on both kernels and
every family, the sparse decode and the extend, against the oracle's fp64 attention over the same codes,
within the decode tolerance.  The dequant routine is checked on every code."""
import numpy as np
import pytest
import torch

import oracle as O
from block_quantized_bit_gb300 import kvq, workloads

from parity import abs_value_pool, assert_decode_close, bits, gpu_decode, layout_of, oracle_decode

pytestmark = pytest.mark.gpu
KINDS = ["fp8_e4m3_unscaled", "fp8_e5m2_unscaled"]
CASES = {
    "tiny": dict(),
    "qwen3_1p7b": dict(batch=3, ctx_lo=100, ctx_hi=1500, new_rows_per_seq=16),
    "long_gqa": dict(batch=2, ctx=9000),
    "mla": dict(ctx=2085, num_q_heads=16),
    "serving": dict(batch=6, median=400, lo=40, hi=3000),
}


def _stored(name, kind, poison=0xA5, **kw):
    """The family's context (and its new rows) cast into an unscaled pool, on the GPU and in the oracle."""
    case = workloads.make(name, kind=kind, device="cpu", **{**CASES.get(name, {}), **kw})
    L = layout_of(case)
    codes = torch.full(L.codes_shape(), poison, dtype=torch.uint8, device="cuda")
    oc = np.full(L.codes_shape(), poison, np.uint8)
    rows = [(case.k, case.v, case.slot_mapping)]
    if case.new_k is not None:
        rows.append((case.new_k, case.new_v, case.new_slots))
    for k, v, sm in rows:
        kvq.kvq_store_unscaled(codes, k.cuda(), None if v is None else v.cuda(), sm.cuda(), L, kind)
        O.store(oc, None, bits(k), None if v is None else bits(v), sm.numpy(), num_kv_heads=case.num_kv_heads,
                head_dim=case.head_dim, page_size=case.page_size, mla=case.mla, kind=kind)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), oc)
    return case, codes, oc


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("name", list(CASES))
def test_unscaled_decode_matches_oracle(name, kind, path):
    case, codes, oc = _stored(name, kind)
    ref = oracle_decode(case, oc, None)
    got = gpu_decode(case, codes, None, path=path)
    if path == 2 and name == "serving":
        # bf16 P on the tensor cores against the spiked values: the bound of the block-scaled decode test
        assert_decode_close(got, ref, rel=2.0 ** -8, scale=oracle_decode(case, abs_value_pool(oc, kind), None))
    else:
        assert_decode_close(got, ref)


@pytest.mark.parametrize("kind", KINDS)
def test_unscaled_decode_wide_groups_on_the_tensor_cores(kind):
    """G = 16 at head_dim 128 and MLA with 128 heads, the shapes the automatic choice sends to tcgen05."""
    for name, kw in (("long_gqa", dict(batch=3, ctx=2500, num_q_heads=32, num_kv_heads=2, head_dim=128)),
                     ("mla", dict(batch=1, ctx=1037, num_q_heads=128))):
        case, codes, oc = _stored(name, kind, **kw)
        assert_decode_close(gpu_decode(case, codes, None, path=2), oracle_decode(case, oc, None))


@pytest.mark.parametrize("kind", KINDS)
def test_unscaled_sparse_decode_matches_oracle(kind):
    case, codes, oc = _stored("mla", kind, batch=2, ctx=3000, num_q_heads=128)
    ix = workloads.sparse_indices(case, 300)
    L = layout_of(case)
    out = torch.full((case.batch, case.num_q_heads, case.v_dim), float("nan"), device="cuda")
    ws = kvq.alloc_sparse_workspace(L, case.batch, case.num_q_heads, 300, "cuda")
    kvq.kvq_decode_sparse(case.q.cuda(), codes, None, case.block_table.cuda(), case.seq_lens.cuda(), ix.cuda(), out,
                          ws, L, kind, case.sm_scale)
    torch.cuda.synchronize()
    assert kvq.kvq_workspace_status(ws) == 0
    ref = O.decode_sparse(bits(case.q), oc, None, case.block_table.numpy(), case.seq_lens.numpy(), ix.numpy(),
                          num_q_heads=case.num_q_heads, num_kv_heads=1, head_dim=case.head_dim, v_dim=case.v_dim,
                          page_size=16, mla=True, kind=kind, sm_scale=case.sm_scale)
    assert_decode_close(out.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("precise", [False, True])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("D", [128, 256])
def test_unscaled_extend_matches_oracle(kind, D, precise):
    case, codes, oc = _stored("long_gqa", kind, batch=2, ctx=700, head_dim=D, mask_frac=0.02)
    q, q_start, _ = workloads.extend_inputs(case, [300, 129])
    L = layout_of(case)
    out = torch.full((q.shape[0], case.num_q_heads, case.v_dim), float("nan"), device="cuda")
    ws = kvq.alloc_extend_workspace("cuda", L, q.shape[0], case.num_q_heads, case.max_pages, precise_p=precise)
    kvq.kvq_extend(q.cuda(), codes, None, case.block_table.cuda(), case.seq_lens.cuda(), q_start.cuda(), out, ws, L,
                   kind, case.sm_scale, precise_p=precise)
    torch.cuda.synchronize()
    assert kvq.kvq_workspace_status(ws) == 0
    ref = O.extend(bits(q), oc, None, case.block_table.numpy(), case.seq_lens.numpy(), q_start.numpy(),
                   num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads, head_dim=D, v_dim=D, page_size=16,
                   mla=False, kind=kind, sm_scale=case.sm_scale)
    assert_decode_close(out.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("kind", KINDS)
def test_unscaled_dequant_gives_the_value_of_every_finite_code(kind):
    """The decode kernels' own dequant routine on all 256 codes: the bf16 bits of each code's value (exact),
    for every code the cast can write (e5m2's infinity and NaN codes are never stored)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).repeat(4).cuda()
    out = torch.empty(codes.numel(), dtype=torch.int16, device="cuda")
    kvq.kvq_dequant_probe(kind, codes, None, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)[:256]
    want_f = np.array([O.code_value(kind, c) for c in range(256)])
    finite = np.isfinite(want_f)
    assert finite.sum() == (254 if kind == "fp8_e4m3_unscaled" else 248)
    want = O.bf16_rne(want_f[finite])
    assert np.array_equal(got[finite], want)
