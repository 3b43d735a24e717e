"""Shared helpers for the GPU parity tests: run a workload through the C ABI and through the oracle."""
import numpy as np
import torch

import oracle as O
from block_quantized_bit_gb300 import kvq

MAX_ABS = 1.5e-2   # decode tolerance against the fp64 oracle (max abs error)
MEAN_ABS = 2e-3    # decode tolerance (mean abs error)


def bits(t):
    """uint16 bit patterns of a bf16 tensor, on the host."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def layout_of(case):
    return kvq.Layout(case.num_pages, case.page_size, case.num_kv_heads, case.head_dim, case.v_dim, case.mla)


def gpu_pool(case, poison_codes=0xA5, poison_scales=0xA5A5, device="cuda"):
    L = layout_of(case)
    codes, scales = kvq.alloc_pool(L, device)
    codes.fill_(poison_codes)
    scales.fill_(int(np.uint16(poison_scales).view(np.int16)))
    return L, codes, scales


def gpu_store(case, codes, scales, rows="context", device="cuda"):
    L = layout_of(case)
    if rows == "context":
        k, v, sm = case.k, case.v, case.slot_mapping
    else:
        k, v, sm = case.new_k, case.new_v, case.new_slots
    kvq.kvq_store(codes, scales, k.to(device), None if v is None else v.to(device), sm.to(device), L, case.kind)


def oracle_pool(case, poison_codes=0xA5, poison_scales=0xA5A5):
    L = layout_of(case)
    oc = np.full(L.codes_shape(), poison_codes, np.uint8)
    osc = np.full(L.scales_shape(), poison_scales, np.uint16)
    return oc, osc


def oracle_store(case, oc, osc, rows="context"):
    if rows == "context":
        k, v, sm = case.k, case.v, case.slot_mapping
    else:
        k, v, sm = case.new_k, case.new_v, case.new_slots
    O.store(oc, osc, bits(k), None if v is None else bits(v), sm.cpu().numpy(), num_kv_heads=case.num_kv_heads,
            head_dim=case.head_dim, page_size=case.page_size, mla=case.mla, kind=case.kind)


def gpu_decode(case, codes, scales, out_dtype=torch.float32, pages_per_split=0, path=0, device="cuda"):
    L = layout_of(case)
    out = torch.full((case.batch, case.num_q_heads, case.v_dim), float("nan"), dtype=out_dtype, device=device)
    ws = kvq.alloc_workspace(L, case.batch, case.num_q_heads, case.max_pages, device,
                             pages_per_split=pages_per_split, path=path)
    ws.fill_(0x5A)
    kvq.kvq_decode(case.q.to(device), codes, scales, case.block_table.to(device), case.seq_lens.to(device), out, ws,
                   L, case.kind, case.sm_scale, pages_per_split=pages_per_split, path=path)
    torch.cuda.synchronize()
    assert kvq.kvq_workspace_status(ws) == 0
    return out.float().cpu().numpy().astype(np.float64)


def oracle_decode(case, oc, osc, nthreads=0):
    return O.decode(bits(case.q), oc, osc, case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(),
                    num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
                    v_dim=case.v_dim, page_size=case.page_size, mla=case.mla, kind=case.kind,
                    sm_scale=case.sm_scale, nthreads=nthreads)


def abs_value_pool(oc, kind):
    """The pool with every V code replaced by the code of its absolute value (fp8 of every kind: sign bit
    cleared; q8_0: |int8|, the store never writes -128) and K unchanged.  Attention over it gives, for each output row,
    sum_t softmax_t * |V_t|: the scale of the error that rounding the probabilities to bf16 (relative
    2^-9 each, as the tensor-core kernels feed them to the MMA) can cause."""
    a = oc.copy()
    if kind != "q8_0":
        a[:, 1] &= 0x7F
    else:
        a[:, 1] = np.abs(a[:, 1].view(np.int8)).astype(np.uint8)
    return a


def assert_decode_close(got, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, rel=0.0, scale=None):
    """Elementwise |got - ref| <= max_abs + rel * scale and mean |got - ref| <= mean_abs + rel * mean(scale);
    scale defaults to |ref|."""
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), "non-finite decode output"
    sc = np.abs(ref) if scale is None else scale
    err = np.abs(got - ref)
    bound = max_abs + rel * sc
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), ("max abs error", float(err.max()), worst, float(got[worst]), float(ref[worst]))
    assert err.mean() <= mean_abs + rel * sc.mean(), ("mean abs error", float(err.mean()))
    return float(err.max()), float(err.mean())
