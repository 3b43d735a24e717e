"""kvq_decode_noalloc: the decode for callers that cannot allocate device memory.

Such callers (a serving loop whose memory is all reserved up front, a plugin under another
framework's allocator, code without an allocator) cannot hand kvq_decode a workspace; this entry
point uses the library's fixed device scratch instead.  Its output must match the oracle within the
decode tolerance, and equal kvq_decode's output, on two calls in a row after a larger call of another
shape has left its split partials and counters in the shared scratch.  kvq_noalloc_status reads the
status word that only that scratch holds.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_quantized_bit_gb300 import build_lib, kvq, workloads

from parity import (MAX_ABS, MEAN_ABS, assert_decode_close, gpu_pool, gpu_store, layout_of, oracle_decode,
                    oracle_pool, oracle_store)

pytestmark = pytest.mark.gpu


def _noalloc_call(case, codes, scales, out, block_table=None):
    lib = kvq.lib()
    L = layout_of(case)
    dev = out.device
    q, sl = case.q.to(dev), case.seq_lens.to(dev)
    bt = (case.block_table if block_table is None else block_table).to(dev)
    st = lib.kvq_decode_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(codes.data_ptr()),
                                ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(bt.data_ptr()), bt.shape[1],
                                ctypes.c_void_p(sl.data_ptr()), case.batch, case.num_q_heads, case.sm_scale,
                                ctypes.c_void_p(out.data_ptr()), kvq.KVQ_OUT_F32, ctypes.byref(L.c()),
                                kvq.KIND[case.kind], ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st


def _stored(name, kw, kind="fp8_e4m3"):
    case = workloads.make(name, kind=kind, device="cpu", **kw)
    L, codes, scales = gpu_pool(case)
    gpu_store(case, codes, scales)
    oc, osc = oracle_pool(case)
    oracle_store(case, oc, osc)
    return case, codes, scales, oc, osc


@pytest.mark.parametrize("name,kw", [("long_gqa", dict(batch=2, ctx=3000)),
                                     ("qwen3_1p7b", dict(batch=4, ctx_lo=200, ctx_hi=2000, new_rows_per_seq=16))])
def test_noalloc_decode_matches_the_oracle_twice_after_another_shape(name, kw):
    build_lib.build()
    case, codes, scales, oc, osc = _stored(name, kw)
    ref = oracle_decode(case, oc, osc)
    # larger decodes of other shapes on both kernels first, so that the shared scratch holds their partials
    # and split counters when the calls under test start
    for pname, pkw in (("serving", dict(batch=4, median=2000, lo=500, hi=4000)),
                       ("long_gqa", dict(batch=2, ctx=10000))):
        big, bcodes, bscales, _, _ = _stored(pname, pkw, kind="q8_0")
        bout = torch.empty(big.batch, big.num_q_heads, big.v_dim, dtype=torch.float32, device=codes.device)
        assert _noalloc_call(big, bcodes, bscales, bout) == 0
        assert kvq.kvq_noalloc_status() == 0
        del bcodes, bscales
    dev = codes.device
    wsref = torch.empty(case.batch, case.num_q_heads, case.v_dim, dtype=torch.float32, device=dev)
    ws = kvq.alloc_workspace(layout_of(case), case.batch, case.num_q_heads, case.max_pages, dev)
    kvq.kvq_decode(case.q.to(dev), codes, scales, case.block_table.to(dev), case.seq_lens.to(dev), wsref, ws,
                   layout_of(case), case.kind, case.sm_scale)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(wsref, float("nan"))
        assert _noalloc_call(case, codes, scales, out) == 0, call
        assert kvq.kvq_noalloc_status() == 0, call
        got = out.cpu().numpy().astype(np.float64)
        assert_decode_close(got, ref, MAX_ABS, MEAN_ABS)
        # the same kernels on the same inputs: the scratch's history changes nothing
        assert torch.equal(out, wsref), call


def test_noalloc_status_reports_a_page_past_the_pool_and_clears_on_the_next_call():
    """A block-table entry >= num_pages is treated as masked (never dereferenced) and flagged in the status
    word, which lives in the library's scratch; the next good call clears it."""
    build_lib.build()
    case, codes, scales, oc, osc = _stored("qwen3_1p7b", dict(batch=2, ctx_lo=100, ctx_hi=400, new_rows_per_seq=16))
    bad = case.block_table.clone()
    bad[0, 1] = case.num_pages + 7
    out = torch.empty(case.batch, case.num_q_heads, case.v_dim, dtype=torch.float32, device=codes.device)
    assert _noalloc_call(case, codes, scales, out, block_table=bad) == 0
    assert kvq.kvq_noalloc_status() == -1   # KVQ_EINVAL
    assert _noalloc_call(case, codes, scales, out) == 0
    assert kvq.kvq_noalloc_status() == 0
    assert_decode_close(out.cpu().numpy().astype(np.float64), oracle_decode(case, oc, osc))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    build_lib.build()
    L = kvq.Layout(num_pages=1 << 20, page_size=16, num_kv_heads=8, head_dim=128, v_dim=128)
    need = kvq.kvq_decode_workspace_bytes(L, 4096, 64, 8192)
    assert need > (8 << 20)
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = kvq.lib().kvq_decode_noalloc(p, p, p, p, 8192, p, 4096, 64, 1.0, p, kvq.KVQ_OUT_F32, ctypes.byref(L.c()),
                                      kvq.KVQ_FP8_E4M3, None)
    assert st == -5   # KVQ_EWORKSPACE: nothing launched
