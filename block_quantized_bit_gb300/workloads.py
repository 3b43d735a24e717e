"""Seeded synthetic workloads shaped like the pages' KV-cache workloads.

This module holds no arithmetic of the method (no scale, no code, no attention).  It draws bf16
K/V rows, queries, slot mappings, block tables and sequence lengths with torch's seeded
generators, on whichever device is asked for; the same tensors feed the CUDA library and (after a
copy to the host) the CPU oracle.

Five families, named for what they are:

* ``tiny``   -- 1 sequence, Hq=8, Hkv=2, D=128, 512 cached tokens.  K ~ N(0,1) times a per-(head,
               channel) lognormal(0, 0.5) multiplier, V ~ N(0,1), q ~ N(0,1)/sqrt(128).  Token 0 /
               head 0 has an all-zero first K block; token 1 / head 1 has a +1000 and a -1000 element in
               its second V block (saturation).
* ``qwen3_1p7b`` -- Hq=16, Hkv=8, D=128.  Decode over batch 8 with contexts uniform in [1024, 16384];
               a store step of 8 x 2048 new rows into fresh pages.  K has per-channel lognormal(0, 0.5)
               multipliers and two outlier channels (x20) per kv head.
* ``long_gqa`` -- Hq=16, Hkv=2, D=256 (8 query heads per kv head); one context length for every
               sequence of the batch; 0.5% of block-table entries are -1 (masked pages).
* ``mla``    -- one 576-wide latent row per token (512 latent + 64 rope) serving as K and V; Hq=128,
               Dv=512.  The latent dims are pre-rounded onto the E4M3 grid with one fp32 scale per 64
               elements (as the model's own activation quantizer does before the cache store; here
               through torch's float8 cast); the rope tail is bf16 N(0,1); q ~ N(0,1)/sqrt(576).
* ``serving`` -- Hq=32, Hkv=8, D=128, batch 64, contexts lognormal (median 4096, sigma 1) clipped to
               [256, 131072], pages randomly permuted, 1% of K/V values scaled by 100; each step stores
               one new row per sequence and decodes it.

``sparse_indices`` draws the per-sequence index lists of the sparse (top-K) decode for any family;
``extend_inputs`` the queries of an extend (prefill) step whose new tokens are the last ones stored.

Page size is 16 everywhere.  The softmax scale is 1.0 because q is drawn already divided by
sqrt(head_dim).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

PAGE_SIZE = 16


@dataclass
class Case:
    name: str
    kind: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    v_dim: int
    page_size: int
    mla: bool
    num_pages: int
    # rows that fill the cached context (stored before decode)
    k: torch.Tensor                 # bf16 [T, Hkv, D]
    v: Optional[torch.Tensor]       # bf16 [T, Hkv, D] (None for MLA)
    slot_mapping: torch.Tensor      # int64 [T], -1 = not stored
    # decode inputs
    q: torch.Tensor                 # bf16 [B, Hq, D]
    block_table: torch.Tensor       # int32 [B, max_pages], -1 = masked / unused
    seq_lens: torch.Tensor          # int32 [B]
    sm_scale: float = 1.0
    # rows stored by each serving step (may be None)
    new_k: Optional[torch.Tensor] = None
    new_v: Optional[torch.Tensor] = None
    new_slots: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device, dtype=torch.float32):
    return torch.randn(shape, generator=g, device=device, dtype=dtype)


def _k_rows(T, Hkv, D, g, device, *, outlier_channels=0, spike_frac=0.0):
    """K ~ N(0,1) * lognormal(0, 0.5) per (kv head, channel); optional outlier channels and spikes."""
    mult = torch.exp(0.5 * _randn((Hkv, D), g, device))
    if outlier_channels:
        for h in range(Hkv):
            ch = torch.randperm(D, generator=g, device=device)[:outlier_channels]
            mult[h, ch] *= 20.0
    k = _randn((T, Hkv, D), g, device) * mult
    if spike_frac:
        k = _spike(k, spike_frac, g, device)
    return k


def _spike(x, frac, g, device):
    hit = torch.rand(x.shape, generator=g, device=device) < frac
    return torch.where(hit, x * 100.0, x)


def _layout_context(seq_lens, seed, *, permute_pages, mask_frac, extra_pages=0):
    """Allocate pages for each sequence; return block_table, slot_mapping (context rows), num_pages.

    Runs on the host (block tables are small); the caller moves the results to its device.
    """
    P = PAGE_SIZE
    g = _gen("cpu", seed + 17)
    lens = [int(x) for x in seq_lens]
    npages = [(L + P - 1) // P for L in lens]
    total = sum(npages)
    num_pages = total + extra_pages
    if permute_pages:
        phys = torch.randperm(total, generator=g)
    else:
        phys = torch.arange(total)
    max_pages = max(max(npages), 1)
    bt = torch.full((len(lens), max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(npages):
        bt[b, :n] = phys[off:off + n].to(torch.int32)
        off += n
    if mask_frac > 0:
        valid = torch.nonzero(bt >= 0)
        nmask = int(round(mask_frac * valid.shape[0]))
        if nmask:
            pick = torch.randperm(valid.shape[0], generator=g)[:nmask]
            rows, cols = valid[pick, 0], valid[pick, 1]
            bt[rows, cols] = -1
    # context slot mapping, sequence by sequence
    slots = []
    for b, L in enumerate(lens):
        t = torch.arange(L, dtype=torch.int64)
        page = bt[b, (t // P)].to(torch.int64)
        s = torch.where(page >= 0, page * P + t % P, torch.full_like(t, -1))
        slots.append(s)
    slot_mapping = torch.cat(slots) if slots else torch.zeros(0, dtype=torch.int64)
    return bt, slot_mapping, num_pages


def _bf16(x):
    return x.to(torch.bfloat16)


def tiny(kind="fp8_e4m3", seed=1001, device="cpu", ctx=512):
    g = _gen(device, seed)
    Hq, Hkv, D = 8, 2, 128
    seq_lens = torch.tensor([ctx], dtype=torch.int32)
    bt, sm, num_pages = _layout_context(seq_lens, seed, permute_pages=False, mask_frac=0.0)
    T = ctx
    k = _k_rows(T, Hkv, D, g, device)
    v = _randn((T, Hkv, D), g, device)
    if T > 0:
        k[0, 0, 0:32] = 0.0                      # all-zero block
    if T > 1:
        v[1, 1, 32:64] = _randn((32,), g, device)
        v[1, 1, 40] = 1000.0                     # saturating outliers
        v[1, 1, 51] = -1000.0
    q = _randn((1, Hq, D), g, device) / math.sqrt(D)
    return Case("tiny", kind, Hq, Hkv, D, D, PAGE_SIZE, False, num_pages, _bf16(k), _bf16(v),
                sm.to(device), _bf16(q), bt.to(device), seq_lens.to(device))


def qwen3_1p7b(kind="fp8_e4m3", seed=1002, device="cpu", batch=8, ctx_lo=1024, ctx_hi=16384,
               new_rows_per_seq=2048):
    g = _gen(device, seed)
    Hq, Hkv, D = 16, 8, 128
    gl = _gen("cpu", seed)
    seq_lens = torch.randint(ctx_lo, ctx_hi + 1, (batch,), generator=gl, dtype=torch.int64).to(torch.int32)
    new_total = batch * new_rows_per_seq
    new_pages = (new_total + PAGE_SIZE - 1) // PAGE_SIZE
    bt, sm, num_pages = _layout_context(seq_lens, seed, permute_pages=False, mask_frac=0.0,
                                        extra_pages=new_pages)
    T = int(seq_lens.sum())
    k = _k_rows(T, Hkv, D, g, device, outlier_channels=2)
    v = _randn((T, Hkv, D), g, device)
    q = _randn((batch, Hq, D), g, device) / math.sqrt(D)
    first_new = num_pages - new_pages
    new_slots = torch.arange(new_total, dtype=torch.int64) + first_new * PAGE_SIZE
    nk = _k_rows(new_total, Hkv, D, g, device, outlier_channels=2)
    nv = _randn((new_total, Hkv, D), g, device)
    return Case("qwen3_1p7b", kind, Hq, Hkv, D, D, PAGE_SIZE, False, num_pages, _bf16(k), _bf16(v),
                sm.to(device), _bf16(q), bt.to(device), seq_lens.to(device),
                new_k=_bf16(nk), new_v=_bf16(nv), new_slots=new_slots.to(device))


def long_gqa(kind="fp8_e4m3", seed=1003, device="cpu", batch=1, ctx=9000, mask_frac=0.005, num_q_heads=16,
             num_kv_heads=2, head_dim=256):
    g = _gen(device, seed)
    Hq, Hkv, D = num_q_heads, num_kv_heads, head_dim
    seq_lens = torch.full((batch,), ctx, dtype=torch.int32)
    bt, sm, num_pages = _layout_context(seq_lens, seed, permute_pages=True, mask_frac=mask_frac)
    T = int(seq_lens.sum())
    k = _k_rows(T, Hkv, D, g, device)
    v = _randn((T, Hkv, D), g, device)
    q = _randn((batch, Hq, D), g, device) / math.sqrt(D)
    return Case("long_gqa", kind, Hq, Hkv, D, D, PAGE_SIZE, False, num_pages, _bf16(k), _bf16(v),
                sm.to(device), _bf16(q), bt.to(device), seq_lens.to(device))


def mla(kind="fp8_e4m3", seed=1004, device="cpu", batch=1, ctx=163840, num_q_heads=128):
    g = _gen(device, seed)
    D, Dv, rope = 576, 512, 64
    seq_lens = torch.full((batch,), ctx, dtype=torch.int32)
    bt, sm, num_pages = _layout_context(seq_lens, seed, permute_pages=True, mask_frac=0.0)
    T = int(seq_lens.sum())
    lat = _randn((T, Dv // 64, 64), g, device)
    s64 = lat.abs().amax(dim=-1, keepdim=True) / 448.0
    s64 = torch.where(s64 > 0, s64, torch.ones_like(s64))
    lat = (lat / s64).to(torch.float8_e4m3fn).to(torch.float32) * s64   # already on the e4m3 grid
    rows = torch.cat([lat.reshape(T, Dv), _randn((T, rope), g, device)], dim=1)
    k = rows.reshape(T, 1, D)
    q = _randn((batch, num_q_heads, D), g, device) / math.sqrt(D)
    return Case("mla", kind, num_q_heads, 1, D, Dv, PAGE_SIZE, True, num_pages, _bf16(k), None,
                sm.to(device), _bf16(q), bt.to(device), seq_lens.to(device))


def serving(kind="fp8_e4m3", seed=1005, device="cpu", batch=64, median=4096, sigma=1.0,
            lo=256, hi=131072):
    """Contexts of ``seq_lens - 1`` tokens are filled; each step stores token ``seq_lens - 1``."""
    g = _gen(device, seed)
    gl = _gen("cpu", seed)
    Hq, Hkv, D = 32, 8, 128
    ctx = torch.exp(math.log(median) + sigma * torch.randn((batch,), generator=gl, dtype=torch.float64))
    ctx = ctx.round().clamp(lo, hi).to(torch.int32)
    seq_lens = ctx + 1                                   # the stepped token included
    bt, sm_all, num_pages = _layout_context(seq_lens, seed, permute_pages=True, mask_frac=0.0)
    ends = torch.cumsum(seq_lens.to(torch.int64), 0) - 1   # index of each sequence's last token
    is_new = torch.zeros(sm_all.shape[0], dtype=torch.bool)
    is_new[ends] = True
    T = int(seq_lens.sum())
    k = _k_rows(T, Hkv, D, g, device, spike_frac=0.01)
    v = _spike(_randn((T, Hkv, D), g, device), 0.01, g, device)
    q = _randn((batch, Hq, D), g, device) / math.sqrt(D)
    is_new_d = is_new.to(device)
    sm_ctx = torch.where(is_new, torch.full_like(sm_all, -1), sm_all)
    return Case("serving", kind, Hq, Hkv, D, D, PAGE_SIZE, False, num_pages, _bf16(k), _bf16(v),
                sm_ctx.to(device), _bf16(q), bt.to(device), seq_lens.to(device),
                new_k=_bf16(k[is_new_d]), new_v=_bf16(v[is_new_d]), new_slots=sm_all[is_new].to(device))


def sparse_indices(case, topk, seed=1006, masked_frac=0.01, device=None):
    """[B, topk] int32 index lists for the sparse (top-K) decode: for each sequence, topk distinct token
    positions drawn uniformly from [0, seq_len) in random order (all positions, then -1 padding, when the
    sequence is shorter), with a fraction ``masked_frac`` of the columns set to -1 (masked columns)."""
    g = _gen("cpu", seed)
    lens = [int(x) for x in case.seq_lens.cpu()]
    ix = torch.full((len(lens), topk), -1, dtype=torch.int32)
    for b, L in enumerate(lens):
        n = min(topk, L)
        if n:
            ix[b, :n] = torch.randperm(L, generator=g)[:n].to(torch.int32)
        if masked_frac > 0 and topk:
            drop = torch.rand((topk,), generator=g) < masked_frac
            ix[b][drop] = -1
    return ix.to(device if device is not None else case.seq_lens.device)


def extend_inputs(case, n_new, seed=1007, device=None):
    """Inputs of one extend (prefill) step over a GQA case: the last n_b of each sequence's stored tokens are
    the step's new tokens (n_new: one count for every sequence, capped at its length, or a list).  Returns
    (q [total, Hq, D] bf16 ~ N(0,1)/sqrt(D), q_start [B + 1] int32, rows) where rows (int64) indexes the
    new tokens' K/V rows in case.k / case.v and case.slot_mapping, sequence by sequence."""
    dev = device if device is not None else case.seq_lens.device
    lens = [int(x) for x in case.seq_lens.cpu()]
    if isinstance(n_new, int):
        n = [min(n_new, L) for L in lens]
    else:
        n = [int(x) for x in n_new]
    if any(x < 0 or x > L for x, L in zip(n, lens)):
        raise ValueError("0 <= new tokens <= seq_len")
    q_start = torch.zeros(len(lens) + 1, dtype=torch.int32)
    q_start[1:] = torch.cumsum(torch.tensor(n, dtype=torch.int64), 0).to(torch.int32)
    total = int(q_start[-1])
    g = _gen("cpu", seed)
    q = _randn((total, case.num_q_heads, case.head_dim), g, "cpu") / math.sqrt(case.head_dim)
    rows, off = [], 0
    for L, x in zip(lens, n):
        rows.append(torch.arange(off + L - x, off + L, dtype=torch.int64))
        off += L
    rows = torch.cat(rows) if rows else torch.zeros(0, dtype=torch.int64)
    return _bf16(q).to(dev), q_start.to(dev), rows.to(dev)


FAMILIES = {"tiny": tiny, "qwen3_1p7b": qwen3_1p7b, "long_gqa": long_gqa, "mla": mla, "serving": serving}


def make(name, **kw) -> Case:
    return FAMILIES[name](**kw)
