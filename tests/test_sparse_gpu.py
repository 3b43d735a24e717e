"""GPU parity of the sparse (top-K) decode through the C ABI against the oracle's fp64 attention over
the listed columns (max abs <= 1.5e-2, mean abs <= 2e-3): MLA and GQA pools, repeated positions, -1,
past-the-end and masked-page columns, lists shorter than a page, the maximum list length, empty lists,
bf16 output, and an out-of-range block-table entry reported in the status word."""
import numpy as np
import pytest
import torch

import oracle as O
from block_quantized_bit_gb300 import kvq, workloads

from parity import assert_decode_close, bits, gpu_pool, gpu_store, layout_of, oracle_pool, oracle_store

pytestmark = pytest.mark.gpu
KINDS = ["fp8_e4m3", "q8_0"]


def _stored(name, kind, **kw):
    case = workloads.make(name, kind=kind, device="cpu", **kw)
    L, codes, scales = gpu_pool(case)
    oc, osc = oracle_pool(case)
    gpu_store(case, codes, scales)
    oracle_store(case, oc, osc)
    return case, codes, scales, oc, osc


def _gpu_sparse(case, codes, scales, ix, out_dtype=torch.float32, bt=None):
    L = layout_of(case)
    topk = ix.shape[1]
    out = torch.full((case.batch, case.num_q_heads, case.v_dim), float("nan"), dtype=out_dtype, device="cuda")
    ws = kvq.alloc_sparse_workspace(L, case.batch, case.num_q_heads, topk)
    bt = case.block_table if bt is None else bt
    kvq.kvq_decode_sparse(case.q.cuda(), codes, scales, bt.cuda(), case.seq_lens.cuda(), ix.cuda(), out, ws, L,
                          case.kind, case.sm_scale)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), kvq.kvq_workspace_status(ws)


def _oracle_sparse(case, oc, osc, ix, bt=None):
    bt = case.block_table if bt is None else bt
    return O.decode_sparse(bits(case.q), oc, osc, bt.cpu().numpy(), case.seq_lens.cpu().numpy(), ix.cpu().numpy(),
                           num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
                           v_dim=case.v_dim, page_size=case.page_size, mla=case.mla, kind=case.kind,
                           sm_scale=case.sm_scale, nthreads=0)


def _messy(case, topk, seed):
    """Random positions plus repeated positions, -1 and past-the-end columns."""
    ix = workloads.sparse_indices(case, topk, seed=seed, masked_frac=0.05).cpu()
    rng = np.random.default_rng(seed)
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        if topk >= 4:
            ix[b, 0] = ix[b, 1]                       # a position listed twice
            ix[b, 2] = L + int(rng.integers(1, 50))   # past the end
            ix[b, 3] = -1
    return ix


CASES = [("mla", dict(ctx=3000, num_q_heads=128), 256),
         ("mla", dict(ctx=700, num_q_heads=16, batch=3), 37),
         ("long_gqa", dict(batch=2, ctx=9000), 512),
         ("qwen3_1p7b", dict(batch=3, ctx_lo=100, ctx_hi=1500, new_rows_per_seq=16), 200)]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("ci", range(len(CASES)))
def test_sparse_decode_matches_oracle(ci, kind):
    name, kw, topk = CASES[ci]
    case, codes, scales, oc, osc = _stored(name, kind, **kw)
    ix = _messy(case, topk, seed=ci)
    ref = _oracle_sparse(case, oc, osc, ix)
    got, st = _gpu_sparse(case, codes, scales, ix)
    assert st == 0
    assert_decode_close(got, ref)
    got16, _ = _gpu_sparse(case, codes, scales, ix, out_dtype=torch.bfloat16)
    assert_decode_close(got16, ref, rel=2.0 ** -8)


def test_sparse_decode_empty_and_fully_invalid_lists_give_zeros():
    case, codes, scales, oc, osc = _stored("mla", "fp8_e4m3", ctx=500, num_q_heads=16, batch=2)
    empty = torch.zeros((case.batch, 0), dtype=torch.int32)
    got, st = _gpu_sparse(case, codes, scales, empty)
    assert st == 0 and not np.any(got)
    junk = torch.tensor([[-1, 10000, -1], [600, -5, 501]], dtype=torch.int32)   # none valid
    got, st = _gpu_sparse(case, codes, scales, junk)
    assert st == 0 and not np.any(got)


def test_sparse_decode_longest_list_and_masked_pages():
    case, codes, scales, oc, osc = _stored("long_gqa", "q8_0", batch=1, ctx=9000, mask_frac=0.05)
    ix = workloads.sparse_indices(case, 8192, seed=3, masked_frac=0.0).cpu()   # the maximum list length
    ref = _oracle_sparse(case, oc, osc, ix)
    got, st = _gpu_sparse(case, codes, scales, ix)
    assert st == 0
    assert_decode_close(got, ref)


def test_sparse_decode_reports_an_out_of_range_page():
    case, codes, scales, oc, osc = _stored("mla", "fp8_e4m3", ctx=500, num_q_heads=16, batch=1)
    bt = case.block_table.clone()
    bt[0, 3] = case.num_pages + 7                     # pages 48..63 point past the pool
    ix = torch.tensor([[1, 50, 60, 100]], dtype=torch.int32)
    got, st = _gpu_sparse(case, codes, scales, ix, bt=bt)
    assert st == -1                                   # KVQ_EINVAL
    ok = torch.tensor([[1, 100]], dtype=torch.int32)  # the same query without the bad columns
    ref = _oracle_sparse(case, oc, osc, ok)
    assert_decode_close(got, ref)
