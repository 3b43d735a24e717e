"""GPU decode parity: split-K decode through the C ABI against the oracle's fp64 attention over the
same dequantized pool (max abs <= 1.5e-2, mean abs <= 2e-3), on every workload family at reduced
sizes, plus split-count invariance, masked pages, ragged tails, empty sequences and NaN-poisoned
pool bytes beyond each sequence's end."""
import numpy as np
import pytest
import torch

from block_quantized_bit_gb300 import workloads

from parity import (abs_value_pool, assert_decode_close, gpu_decode, gpu_pool, gpu_store, oracle_decode, oracle_pool,
                    oracle_store)

pytestmark = pytest.mark.gpu
KINDS = ["fp8_e4m3", "q8_0"]
CASES = {
    "tiny": dict(),
    "qwen3_1p7b": dict(batch=3, ctx_lo=100, ctx_hi=1500, new_rows_per_seq=16),
    "long_gqa": dict(batch=2, ctx=9000),
    "mla": dict(ctx=2085, num_q_heads=16),
    "serving": dict(batch=6, median=400, lo=40, hi=3000),
}


def _stored(name, kind, poison=0xA5, **kw):
    case = workloads.make(name, kind=kind, device="cpu", **{**CASES[name], **kw})
    L, codes, scales = gpu_pool(case, poison_codes=poison)
    oc, osc = oracle_pool(case, poison_codes=poison)
    gpu_store(case, codes, scales)
    oracle_store(case, oc, osc)
    if case.new_k is not None:
        gpu_store(case, codes, scales, rows="new")
        oracle_store(case, oc, osc, rows="new")
    return case, codes, scales, oc, osc


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("name", list(CASES))
def test_decode_matches_oracle(name, kind, path):
    """Every family on the automatic choice, the CUDA-core kernel (1) and the tensor-core kernel (2)."""
    case, codes, scales, oc, osc = _stored(name, kind)
    ref = oracle_decode(case, oc, osc)
    got = gpu_decode(case, codes, scales, path=path)
    if path == 2 and name == "serving":
        # 1% of the values are scaled by 100.  The tensor-core kernel feeds P to the MMA as bf16 (relative
        # error 2^-9 each), so its error scales with sum_t p_t |V_t| (the oracle over the pool with absolute
        # V codes), which the spikes make ~100: the bound gains 2^-8 times that sum.  The automatic choice
        # keeps this group size (4) on the CUDA-core kernel, whose P stays fp32.
        assert_decode_close(got, ref, rel=2.0 ** -8, scale=oracle_decode(case, abs_value_pool(oc, kind), osc))
    else:
        assert_decode_close(got, ref)
    got16 = gpu_decode(case, codes, scales, out_dtype=torch.bfloat16)
    assert_decode_close(got16, ref, rel=2.0 ** -8)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("pps", [1, 3, 16])
def test_decode_is_invariant_to_the_split_size(pps, path):
    """Any split size gives the oracle's answer.  The CUDA-core path keeps fp32 probabilities, so its
    splits agree to fp32 rounding; the tensor-core path rounds P to bf16 against a split-dependent
    running max, so its splits agree to that rounding."""
    case, codes, scales, oc, osc = _stored("long_gqa", "fp8_e4m3")
    ref = oracle_decode(case, oc, osc)
    auto = gpu_decode(case, codes, scales, path=path)
    forced = gpu_decode(case, codes, scales, pages_per_split=pps, path=path)
    assert_decode_close(forced, ref)
    np.testing.assert_allclose(forced, auto, rtol=0, atol=2e-5 if path == 1 else 5e-3)


def test_decode_never_reads_nan_bytes_past_a_sequence_end():
    """Pool poisoned with 0xFF (an E4M3 NaN code) except where rows were stored."""
    case, codes, scales, oc, osc = _stored("long_gqa", "fp8_e4m3", poison=0xFF, ctx=1000 + 7)
    ref = oracle_decode(case, oc, osc)
    got = gpu_decode(case, codes, scales)
    assert_decode_close(got, ref)


@pytest.mark.parametrize("path", [1, 2])
def test_decode_empty_and_fully_masked_sequences_give_zeros(path):
    """Both kernels: the CUDA-core one merges in-kernel, so an empty sequence still needs a (trivial)
    work item to write its zeros; the tensor-core one leaves that to the merge kernel."""
    case = workloads.long_gqa(kind="q8_0", batch=3, ctx=300, mask_frac=0.0)
    case.block_table[1, :] = -1                      # every page of sequence 1 masked
    case.seq_lens[2] = 0                             # sequence 2 empty
    L, codes, scales = gpu_pool(case)
    gpu_store(case, codes, scales)
    got = gpu_decode(case, codes, scales, path=path)
    oc, osc = oracle_pool(case)
    oracle_store(case, oc, osc)
    ref = oracle_decode(case, oc, osc)
    assert not got[1].any() and not got[2].any()
    assert_decode_close(got, ref)


def test_decode_masked_pages_and_ragged_lengths():
    case = workloads.serving(kind="fp8_e4m3", batch=9, median=150, lo=1, hi=700)
    bt = case.block_table
    for b in range(0, 9, 2):                          # mask a page in every other sequence
        n = int((case.seq_lens[b] + 15) // 16)
        if n > 1:
            bt[b, n // 2] = -1
    L, codes, scales = gpu_pool(case)
    oc, osc = oracle_pool(case)
    gpu_store(case, codes, scales)
    gpu_store(case, codes, scales, rows="new")
    oracle_store(case, oc, osc)
    oracle_store(case, oc, osc, rows="new")
    assert_decode_close(gpu_decode(case, codes, scales), oracle_decode(case, oc, osc))


def test_decode_sm_scale_is_applied():
    case, codes, scales, oc, osc = _stored("tiny", "fp8_e4m3")
    case.sm_scale = 0.3
    assert_decode_close(gpu_decode(case, codes, scales), oracle_decode(case, oc, osc))


# ------------------------------------------------------------------ tensor-core (tcgen05) path
TC_CASES = [
    dict(batch=2, ctx=9000),                                              # G = 8, D = 256
    dict(batch=3, ctx=2500, num_q_heads=32, num_kv_heads=2, head_dim=128),  # G = 16, D = 128
    dict(batch=2, ctx=3001, num_q_heads=16, num_kv_heads=2, head_dim=128, mask_frac=0.03),
    dict(batch=3, ctx=2100, num_q_heads=16, num_kv_heads=8, head_dim=128),  # G = 2 (padded to 16)
    dict(batch=2, ctx=1500, num_q_heads=12, num_kv_heads=4, head_dim=256),  # G = 3
    dict(batch=2, ctx=2000, num_q_heads=8, num_kv_heads=8, head_dim=128),   # G = 1
    dict(batch=2, ctx=1800, num_q_heads=24, num_kv_heads=2, head_dim=128),  # G = 12
]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("ci", range(len(TC_CASES)))
def test_tensor_core_decode_matches_oracle(ci, kind):
    case, codes, scales, oc, osc = _stored("long_gqa", kind, **TC_CASES[ci])
    ref = oracle_decode(case, oc, osc)
    got = gpu_decode(case, codes, scales, path=2)
    assert_decode_close(got, ref)


@pytest.mark.parametrize("pps", [8, 12, 40])
def test_tensor_core_decode_split_sizes_and_many_items_per_cta(pps):
    """Split sizes that are not whole 128-token tiles (ragged last tile) and enough items that every
    persistent CTA runs several of them, against the oracle and the CUDA-core path."""
    case, codes, scales, oc, osc = _stored("long_gqa", "fp8_e4m3", batch=3, ctx=9000, mask_frac=0.01)
    ref = oracle_decode(case, oc, osc)
    tc = gpu_decode(case, codes, scales, path=2, pages_per_split=pps)
    assert_decode_close(tc, ref)
    cc = gpu_decode(case, codes, scales, path=1, pages_per_split=pps)
    np.testing.assert_allclose(tc, cc, rtol=0, atol=5e-3)


def test_tensor_core_decode_nan_poisoned_tails_and_empty_sequences():
    case = workloads.long_gqa(kind="q8_0", batch=4, ctx=1000 + 9, mask_frac=0.0)
    case.block_table[1, :] = -1
    case.seq_lens[2] = 0
    L, codes, scales = gpu_pool(case, poison_codes=0xFF)
    gpu_store(case, codes, scales)
    oc, osc = oracle_pool(case, poison_codes=0xFF)
    oracle_store(case, oc, osc)
    got = gpu_decode(case, codes, scales, path=2)
    ref = oracle_decode(case, oc, osc)
    assert not got[1].any() and not got[2].any()
    assert_decode_close(got, ref)


# ------------------------------------------------------------------ MLA on the tensor cores
MLA_TC_CASES = [
    dict(batch=1, ctx=1037, num_q_heads=128),   # two head groups of 64, ragged last tile
    dict(batch=3, ctx=2300),                    # 16 heads: one padded head group; several splits
    dict(batch=2, ctx=700, num_q_heads=64),     # a single full head group
    dict(batch=1, ctx=1500, num_q_heads=192),   # three head groups
]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("ci", range(len(MLA_TC_CASES)))
def test_mla_tensor_core_decode_matches_oracle(ci, kind):
    case, codes, scales, oc, osc = _stored("mla", kind, **MLA_TC_CASES[ci])
    ref = oracle_decode(case, oc, osc)
    got = gpu_decode(case, codes, scales, path=2)
    assert_decode_close(got, ref)


@pytest.mark.parametrize("pps", [8, 12, 40])
def test_mla_tensor_core_masked_pages_ragged_lengths_and_split_sizes(pps):
    """Masked (-1) pages, sequences shorter than their stored rows (ragged tails, one shorter than a
    tile) and split sizes that are not whole tiles, against the oracle and the CUDA-core kernel."""
    case, codes, scales, oc, osc = _stored("mla", "fp8_e4m3", batch=3, ctx=2300, num_q_heads=128)
    sl = case.seq_lens.clone()
    sl[1], sl[2] = 1507, 129
    case.seq_lens = sl
    bt = case.block_table.clone()
    g = torch.Generator().manual_seed(7)
    bt[torch.rand(bt.shape, generator=g) < 0.03] = -1
    case.block_table = bt
    ref = oracle_decode(case, oc, osc)
    tc = gpu_decode(case, codes, scales, path=2, pages_per_split=pps)
    assert_decode_close(tc, ref)
    cc = gpu_decode(case, codes, scales, path=1, pages_per_split=pps)
    np.testing.assert_allclose(tc, cc, rtol=0, atol=5e-3)
