"""kvq_decode_noalloc: the decode for callers that cannot allocate device memory.

Such callers (a serving loop whose memory is all reserved up front, a plugin under another
framework's allocator, code without an allocator) cannot hand kvq_decode a workspace; this entry
point uses the library's fixed device scratch instead.  Its output must match kvq_decode's, within
the decode tolerance, on two calls in a row (the second call reuses the scratch the first one
left behind).  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_quantized_bit_gb300 import build_lib, kvq, workloads

from parity import MAX_ABS, MEAN_ABS, gpu_pool, gpu_store, layout_of

pytestmark = pytest.mark.gpu


def _noalloc_call(case, codes, scales, out):
    lib = kvq.lib()
    L = layout_of(case)
    dev = out.device
    q, bt, sl = case.q.to(dev), case.block_table.to(dev), case.seq_lens.to(dev)
    st = lib.kvq_decode_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(codes.data_ptr()),
                                ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(bt.data_ptr()), bt.shape[1],
                                ctypes.c_void_p(sl.data_ptr()), case.batch, case.num_q_heads, case.sm_scale,
                                ctypes.c_void_p(out.data_ptr()), kvq.KVQ_OUT_F32, ctypes.byref(L.c()),
                                kvq.KIND[case.kind], ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("name,kw", [("long_gqa", dict(batch=2, ctx=3000)),
                                     ("qwen3_1p7b", dict(batch=4, ctx_lo=200, ctx_hi=2000, new_rows_per_seq=16))])
def test_noalloc_decode_matches_workspace_decode_twice(name, kw):
    build_lib.build()
    case = workloads.make(name, kind="fp8_e4m3", device="cpu", **kw)
    L, codes, scales = gpu_pool(case)
    gpu_store(case, codes, scales)
    dev = codes.device
    ref = torch.empty(case.batch, case.num_q_heads, case.v_dim, dtype=torch.float32, device=dev)
    ws = kvq.alloc_workspace(L, case.batch, case.num_q_heads, case.max_pages, dev)
    kvq.kvq_decode(case.q.to(dev), codes, scales, case.block_table.to(dev), case.seq_lens.to(dev), ref, ws, L,
                   case.kind, case.sm_scale)
    torch.cuda.synchronize()
    r = ref.cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_call(case, codes, scales, out) == 0, call
        got = out.cpu().numpy().astype(np.float64)
        err = np.abs(got - r)
        assert np.all(np.isfinite(got)), call
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (call, err.max(), err.mean())


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
