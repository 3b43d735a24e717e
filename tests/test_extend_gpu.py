"""GPU parity of the extend (prefill) attention, through the C ABI, against the oracle's fp64 causal attention.

Each case stores every row of its sequences (kvq_store on the GPU, the oracle's store on the host, checked
bit-exact by the store tests) and declares the last n_b stored tokens of sequence b new; the kernel's output
for every (new token, query head) must meet the decode bound (max abs <= 1.5e-2, mean abs <= 2e-3).  The
cases span several key tiles and query blocks with ragged tails, D = 128 and 256, 1 to 16 query heads per kv
head, masked pages, a first prefill (every token new), single new tokens and sequences without new tokens.
The MLA latent row runs through the decode kernels, one causal prefix per new token, with the same bound.
The same prefix path serves GQA shapes the flash kernel does not (head_dim 64, group sizes not dividing
128), and, forced onto the CUDA-core decode, keeps P in fp32 and meets the plain bound on spiked V too."""
import numpy as np
import pytest
import torch

import oracle as O
from block_quantized_bit_gb300 import kvq, workloads

from parity import (abs_value_pool, assert_decode_close, bits, gpu_pool, gpu_store, layout_of, oracle_pool,
                    oracle_store)

pytestmark = pytest.mark.gpu

KVQ_EINVAL, KVQ_EUNSUPPORTED = -1, -8


def _case(name, kind, **kw):
    return workloads.make(name, kind=kind, device="cuda", **kw)


CASES = {
    # D = 128, 2 query heads per kv head: 64 new tokens per query block, 128-key tiles
    "qwen3_small": (lambda kind: _case("qwen3_1p7b", kind, batch=3, ctx_lo=150, ctx_hi=700), [None, 37, 1]),
    # D = 256, 8 heads per kv head (16 tokens per block), 64-key tiles, masked pages
    "long_gqa_small": (lambda kind: _case("long_gqa", kind, batch=2, ctx=900, mask_frac=0.05), [300, 900]),
    # D = 128, 4 heads per kv head, randomly permuted pages, 1% of K/V values x100 (outputs reach ~130)
    "serving_small": (lambda kind: _case("serving", kind, batch=4, median=300, lo=40, hi=600), [40, 0, 17, 129]),
    # 1 head per kv head (128 new tokens per block) and 16 heads per kv head (8 per block)
    "mha": (lambda kind: _case("long_gqa", kind, batch=2, ctx=333, mask_frac=0.0, num_q_heads=8,
                               num_kv_heads=8, head_dim=128), [333, 130]),
    "g16": (lambda kind: _case("long_gqa", kind, batch=1, ctx=520, mask_frac=0.02, num_q_heads=32,
                               num_kv_heads=2, head_dim=128), [200]),
}


def _stored(key, kind):
    make, n_new = CASES[key]
    case = make(kind)
    lens = case.seq_lens.cpu().tolist()
    n_new = [L if x is None else x for x, L in zip(n_new, lens)]
    L, codes, scales = gpu_pool(case)
    gpu_store(case, codes, scales)
    oc, osc = oracle_pool(case)
    oracle_store(case, oc, osc)
    q, q_start, _ = workloads.extend_inputs(case, n_new)
    return case, L, codes, scales, oc, osc, q, q_start


def _gpu_extend(case, L, codes, scales, q, q_start, out_dtype=torch.float32, path=None, precise_p=False):
    out = torch.full((q.shape[0], case.num_q_heads, case.v_dim), float("nan"), dtype=out_dtype, device="cuda")
    if path is None and not precise_p:
        ws = kvq.alloc_extend_workspace()
    else:
        ws = kvq.alloc_extend_workspace("cuda", L, q.shape[0], case.num_q_heads, case.max_pages, path=path,
                                        precise_p=precise_p)
    ws.fill_(0x5A)
    kvq.kvq_extend(q, codes, scales, case.block_table, case.seq_lens, q_start, out, ws, L, case.kind, case.sm_scale,
                   path=path, precise_p=precise_p)
    torch.cuda.synchronize()
    return out, ws


def _oracle_extend(case, oc, osc, q, q_start):
    return O.extend(bits(q), oc, osc, case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(),
                    q_start.cpu().numpy(), num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads,
                    head_dim=case.head_dim, v_dim=case.v_dim, page_size=case.page_size, mla=case.mla,
                    kind=case.kind, sm_scale=case.sm_scale, nthreads=0)


# P enters the MMA as bf16 (relative error 2^-9 per probability), so the output error scales with
# sum_t p_t |V_t|, which the oracle gives over the pool with absolute V codes.  With the x100 spikes of the
# serving family that sum reaches hundreds while outputs cancel to a few units, so there the bound gains
# 2^-8 (twice the rounding) times that sum.
SPIKED = {"serving_small"}


@pytest.mark.parametrize("kind", ["fp8_e4m3", "q8_0"])
@pytest.mark.parametrize("key", list(CASES))
def test_extend_matches_the_oracle(key, kind):
    case, L, codes, scales, oc, osc, q, q_start = _stored(key, kind)
    out, ws = _gpu_extend(case, L, codes, scales, q, q_start)
    assert kvq.kvq_workspace_status(ws) == 0
    ref = _oracle_extend(case, oc, osc, q, q_start)
    got = out.cpu().numpy().astype(np.float64)
    if key in SPIKED:
        scale = _oracle_extend(case, abs_value_pool(oc, kind), osc, q, q_start)
        assert_decode_close(got, ref, rel=2.0 ** -8, scale=scale)
    else:
        assert_decode_close(got, ref)


@pytest.mark.parametrize("kind", ["fp8_e4m3", "q8_0"])
@pytest.mark.parametrize("key", list(CASES))
def test_extend_on_the_cuda_core_decode_meets_the_plain_bound(key, kind):
    """Path 1: every new token's causal prefix on the CUDA-core decode, P in fp32.  The x100 spikes of the
    serving family get no widened bound here."""
    case, L, codes, scales, oc, osc, q, q_start = _stored(key, kind)
    assert kvq.kvq_extend_path(L, q.shape[0], case.num_q_heads, case.max_pages, path=1) == 1
    out, ws = _gpu_extend(case, L, codes, scales, q, q_start, path=1)
    assert kvq.kvq_workspace_status(ws) == 0
    assert_decode_close(out.cpu().numpy().astype(np.float64), _oracle_extend(case, oc, osc, q, q_start))


@pytest.mark.parametrize("kind", ["fp8_e4m3", "q8_0"])
@pytest.mark.parametrize("key", list(CASES))
def test_extend_with_p_as_two_bf16_terms_meets_the_plain_bound(key, kind):
    """precise_p on the flash kernel: P = hi + lo through two PVs (lo in S's own columns at D = 128, in
    columns of its own at D = 256), so the serving family's x100 spikes need no widened bound."""
    case, L, codes, scales, oc, osc, q, q_start = _stored(key, kind)
    assert kvq.kvq_extend_path(L, q.shape[0], case.num_q_heads, case.max_pages, precise_p=True) == 4
    out, ws = _gpu_extend(case, L, codes, scales, q, q_start, precise_p=True)
    assert kvq.kvq_workspace_status(ws) == 0
    ref = _oracle_extend(case, oc, osc, q, q_start)
    got = out.cpu().numpy().astype(np.float64)
    assert_decode_close(got, ref)
    if key in SPIKED:
        # and it is closer to the oracle than the bf16-P kernel where the spikes dominate
        plain, _ = _gpu_extend(case, L, codes, scales, q, q_start)
        assert np.abs(got - ref).max() < np.abs(plain.cpu().numpy().astype(np.float64) - ref).max()


def test_extend_bf16_output_is_the_rounded_f32_output():
    case, L, codes, scales, oc, osc, q, q_start = _stored("qwen3_small", "fp8_e4m3")
    out32, _ = _gpu_extend(case, L, codes, scales, q, q_start)
    out16, ws = _gpu_extend(case, L, codes, scales, q, q_start, torch.bfloat16)
    assert kvq.kvq_workspace_status(ws) == 0
    assert torch.equal(out16, out32.to(torch.bfloat16))


def test_extend_is_deterministic_and_leaves_the_pool_alone():
    case, L, codes, scales, oc, osc, q, q_start = _stored("long_gqa_small", "q8_0")
    c0, s0 = codes.clone(), scales.clone()
    a, _ = _gpu_extend(case, L, codes, scales, q, q_start)
    b, _ = _gpu_extend(case, L, codes, scales, q, q_start)
    assert torch.equal(a, b)
    assert torch.equal(codes, c0) and torch.equal(scales, s0)


def test_extend_with_no_new_token_is_a_no_op_and_a_bad_q_start_is_reported():
    case, L, codes, scales, oc, osc, q, q_start = _stored("qwen3_small", "fp8_e4m3")
    # no new token anywhere: nothing is written
    empty_q = q[:0]
    zeros = torch.zeros_like(q_start)
    out, ws = _gpu_extend(case, L, codes, scales, empty_q, zeros)
    assert out.numel() == 0 and kvq.kvq_workspace_status(ws) == 0
    # sequence 1 claims more new tokens than it stores: it is skipped and reported; the others are exact
    lens = case.seq_lens.cpu().tolist()
    bad = torch.tensor([0, 3, 3 + lens[1] + 1, 3 + lens[1] + 2], dtype=torch.int32, device="cuda")
    qb = torch.randn((int(bad[-1]), case.num_q_heads, case.head_dim), device="cuda").to(torch.bfloat16) / 12
    out, ws = _gpu_extend(case, L, codes, scales, qb, bad)
    assert kvq.kvq_workspace_status(ws) == KVQ_EINVAL
    good = np.r_[0:3, int(bad[2]):int(bad[3])]
    ok_start = torch.tensor([0, 3, 3, 4], dtype=torch.int32)
    ref = O.extend(bits(qb[good]), oc, osc, case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(),
                   ok_start.numpy(), num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads,
                   head_dim=case.head_dim, v_dim=case.v_dim, page_size=case.page_size, mla=False, kind=case.kind,
                   sm_scale=case.sm_scale, nthreads=0)
    assert_decode_close(out[good].cpu().numpy().astype(np.float64), ref)
    assert torch.isnan(out[3:int(bad[2])]).all()  # the skipped sequence's rows are untouched


def _mla_stored(kind, n_new, mask=(), **kw):
    case = _case("mla", kind, **kw)
    L, codes, scales = gpu_pool(case)
    gpu_store(case, codes, scales)
    oc, osc = oracle_pool(case)
    oracle_store(case, oc, osc)
    bt = case.block_table.clone()
    for b, j in mask:          # pages masked after the store: their rows are hidden from the attention
        bt[b, j] = -1
    case.block_table = bt
    lens = case.seq_lens.cpu().tolist()
    n_new = [L_ if x is None else x for x, L_ in zip(n_new, lens)]
    q, q_start, _ = workloads.extend_inputs(case, n_new)
    return case, L, codes, scales, oc, osc, q, q_start


def _gpu_extend_mla(case, L, codes, scales, q, q_start, out_dtype=torch.float32):
    out = torch.full((q.shape[0], case.num_q_heads, case.v_dim), float("nan"), dtype=out_dtype, device="cuda")
    ws = kvq.alloc_extend_workspace("cuda", L, q.shape[0], case.num_q_heads, case.max_pages)
    ws.fill_(0x5A)
    kvq.kvq_extend(q, codes, scales, case.block_table, case.seq_lens, q_start, out, ws, L, case.kind, case.sm_scale)
    torch.cuda.synchronize()
    return out, ws


MLA_CASES = [
    # 16 heads (one padded group of 64 on the tensor cores), a first prefill and a partial one, masked pages
    (dict(batch=2, ctx=200, num_q_heads=16), [None, 30], [(0, 3), (1, 10)]),
    # 128 heads (two groups of 64), one sequence
    (dict(batch=1, ctx=130, num_q_heads=128), [20], []),
    # more new tokens than one chunk of 1024 prefixes (one head, the oracle's cost kept small)
    (dict(batch=2, ctx=560, num_q_heads=1), [None, 480], [(1, 2)]),
]


@pytest.mark.parametrize("kind", ["fp8_e4m3", "q8_0"])
@pytest.mark.parametrize("ci", range(len(MLA_CASES)))
def test_mla_extend_matches_the_oracle(ci, kind):
    """The MLA latent row (576 / 512): each new token decoded over its causal prefix by the decode kernels."""
    kw, n_new, mask = MLA_CASES[ci]
    case, L, codes, scales, oc, osc, q, q_start = _mla_stored(kind, n_new, mask, **kw)
    out, ws = _gpu_extend_mla(case, L, codes, scales, q, q_start)
    assert kvq.kvq_workspace_status(ws) == 0
    assert_decode_close(out.cpu().numpy().astype(np.float64), _oracle_extend(case, oc, osc, q, q_start))


def test_mla_extend_skips_a_bad_sequence_with_zeros_and_reports_it():
    case, L, codes, scales, oc, osc, q, q_start = _mla_stored("fp8_e4m3", [None, 40], [], batch=2, ctx=200,
                                                              num_q_heads=16)
    lens = case.seq_lens.cpu().tolist()
    bad = torch.tensor([0, 5, 5 + lens[1] + 1], dtype=torch.int32, device="cuda")  # sequence 1: too many
    qb = q[:1].repeat(int(bad[-1]), 1, 1)
    out, ws = _gpu_extend_mla(case, L, codes, scales, qb, bad)
    assert kvq.kvq_workspace_status(ws) == KVQ_EINVAL
    assert not out[5:].any()
    ref = O.extend(bits(qb[:5]), oc, osc, case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy()[:1],
                   np.array([0, 5], np.int32), num_q_heads=case.num_q_heads, num_kv_heads=1, head_dim=case.head_dim,
                   v_dim=case.v_dim, page_size=16, mla=True, kind=case.kind, sm_scale=case.sm_scale, nthreads=0)
    assert_decode_close(out[:5].cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("kind", ["fp8_e4m3", "q8_0"])
@pytest.mark.parametrize("shape", ["d64", "g3", "g12"])
def test_extend_shapes_without_a_flash_kernel_run_on_the_prefixes(shape, kind):
    """head_dim 64, 3 and 12 query heads per kv head: the automatic choice runs each new token's prefix on
    the decode (CUDA cores for the first two, tensor cores for 12 heads per kv head); asking for the flash
    kernel is KVQ_EUNSUPPORTED."""
    kw = {"d64": dict(head_dim=64, num_q_heads=8, num_kv_heads=2),
          "g3": dict(head_dim=128, num_q_heads=6, num_kv_heads=2),
          "g12": dict(head_dim=128, num_q_heads=24, num_kv_heads=2)}[shape]
    case = _case("long_gqa", kind, batch=2, ctx=400, mask_frac=0.03, **kw)
    L, codes, scales = gpu_pool(case)
    gpu_store(case, codes, scales)
    oc, osc = oracle_pool(case)
    oracle_store(case, oc, osc)
    q, q_start, _ = workloads.extend_inputs(case, [400, 77])
    want = 2 if shape == "g12" else 1
    assert kvq.kvq_extend_path(L, q.shape[0], case.num_q_heads, case.max_pages) == want
    out, ws = _gpu_extend(case, L, codes, scales, q, q_start, path=0)
    assert kvq.kvq_workspace_status(ws) == 0
    assert_decode_close(out.cpu().numpy().astype(np.float64), _oracle_extend(case, oc, osc, q, q_start))
    assert kvq.kvq_extend_path(L, q.shape[0], case.num_q_heads, case.max_pages, path=2) == KVQ_EUNSUPPORTED
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_extend(q, codes, scales, case.block_table, case.seq_lens, q_start, out, kvq.alloc_extend_workspace(),
                       L, case.kind, case.sm_scale, path=2)
    assert e.value.status == KVQ_EUNSUPPORTED


@pytest.mark.parametrize("path", [1, 2])
def test_mla_extend_on_either_decode_kernel(path):
    """The MLA prefixes forced onto the CUDA-core (fp32 P) or the tensor-core decode."""
    kw, n_new, mask = MLA_CASES[0]
    case, L, codes, scales, oc, osc, q, q_start = _mla_stored("q8_0", n_new, mask, **kw)
    assert kvq.kvq_extend_path(L, q.shape[0], case.num_q_heads, case.max_pages, path=path) == path
    out, ws = _gpu_extend(case, L, codes, scales, q, q_start, path=path)
    assert kvq.kvq_workspace_status(ws) == 0
    assert_decode_close(out.cpu().numpy().astype(np.float64), _oracle_extend(case, oc, osc, q, q_start))


def test_gqa_extend_on_the_prefixes_zeroes_a_bad_sequence_and_reports_it():
    case, L, codes, scales, oc, osc, q, q_start = _stored("qwen3_small", "fp8_e4m3")
    lens = case.seq_lens.cpu().tolist()
    bad = torch.tensor([0, 3, 3 + lens[1] + 1, 3 + lens[1] + 2], dtype=torch.int32, device="cuda")
    qb = torch.randn((int(bad[-1]), case.num_q_heads, case.head_dim), device="cuda").to(torch.bfloat16) / 12
    out, ws = _gpu_extend(case, L, codes, scales, qb, bad, path=1)
    assert kvq.kvq_workspace_status(ws) == KVQ_EINVAL
    good = np.r_[0:3, int(bad[2]):int(bad[3])]
    ok_start = torch.tensor([0, 3, 3, 4], dtype=torch.int32)
    ref = O.extend(bits(qb[good]), oc, osc, case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(),
                   ok_start.numpy(), num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads,
                   head_dim=case.head_dim, v_dim=case.v_dim, page_size=case.page_size, mla=False, kind=case.kind,
                   sm_scale=case.sm_scale, nthreads=0)
    assert_decode_close(out[good].cpu().numpy().astype(np.float64), ref)
    assert not out[3:int(bad[2])].any()  # the skipped sequence's rows are zeros on this path


@pytest.mark.parametrize("precise", [False, True])
@pytest.mark.parametrize("path", [None, 1, 2])
def test_extend_with_no_new_token_is_a_no_op_on_every_kernel_choice(path, precise):
    """total_q = 0 (every q_start entry 0): nothing is written and the status word is clear, on the flash
    kernel, the prefixes and the two-term P instances alike."""
    case, L, codes, scales, oc, osc, q, q_start = _stored("qwen3_small", "fp8_e4m3")
    empty_q = q[:0]
    zeros = torch.zeros_like(q_start)
    out, ws = _gpu_extend(case, L, codes, scales, empty_q, zeros, path=path, precise_p=precise)
    assert out.numel() == 0 and kvq.kvq_workspace_status(ws) == 0
