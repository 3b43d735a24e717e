"""GPU parity at the benchmark's full sizes, in the launch configuration bench.py times (automatic
kernel choice, automatic split size): the whole workload is stored and decoded on the GPU through the
C ABI, and the oracle checks samples it can afford one by one.

* Store: bit-exact codes and fp16 scales for a random sample of rows, which the oracle quantizes into
  a compact pool of its own.
* Decode: for sampled (sequence, kv head) pairs the oracle stores that sequence's rows of that kv head
  into a compact pool (the same masked pages, identity page order) and runs its fp64 attention for the
  query heads of that kv head (a sample of them for the 128-head MLA row); the GPU rows must meet the
  decode bound (max abs <= 1.5e-2, mean abs <= 2e-3).

* Extend: the bench's extend step (the last 2048 stored tokens of each qwen3_1p7b sequence attend causally);
  for sampled (sequence, new token, kv head) the oracle attends over a compact pool of that sequence's rows
  of that kv head, cut at the token's position.

Sizes: qwen3_1p7b (batch 8, 1k-16k), long_gqa batch 8 x 262144 and batch 1 x 262144, mla (163840
tokens, 128 heads), serving (batch 64, lognormal contexts).  The oracle's share is a few million rows,
so the file runs in a few minutes on the GPU machine's host cores."""
import numpy as np
import pytest
import torch

import oracle as O
from block_quantized_bit_gb300 import kvq, workloads

from parity import assert_decode_close, bits, gpu_decode, gpu_pool, gpu_store

pytestmark = pytest.mark.gpu

FULL = {
    "qwen3_1p7b": dict(),
    "long_gqa_b8": dict(batch=8, ctx=262144),
    "long_gqa_b1": dict(batch=1, ctx=262144),
    "mla": dict(),
    "serving": dict(),
}
STORE_SAMPLE_ROWS = 512
MLA_SAMPLE_HEADS = 8


def _make(key, kind):
    name = "long_gqa" if key.startswith("long_gqa") else key
    return workloads.make(name, kind=kind, device="cuda", **FULL[key])


def _rows_of_sequence(case, b):
    lens = case.seq_lens.cpu().numpy().astype(np.int64)
    off = int(lens[:b].sum())
    return off, int(lens[b])


def _oracle_subcase(case, b, g, heads):
    """Oracle output of query heads `heads` (all reading kv head g) of sequence b, from a compact pool
    holding only that sequence's rows of kv head g (masked pages stay masked)."""
    P = case.page_size
    off, L = _rows_of_sequence(case, b)
    npg = max((L + P - 1) // P, 1)
    bt_full = case.block_table[b, :npg].cpu().numpy()
    sbt = np.where(bt_full >= 0, np.arange(npg, dtype=np.int32), -1).astype(np.int32)[None, :]
    t = np.arange(L)
    slots = np.where(sbt[0, t // P] >= 0, t, -1).astype(np.int64)
    k = bits(case.k[off:off + L, g:g + 1, :])
    v = None if case.mla else bits(case.v[off:off + L, g:g + 1, :])
    cs, ss = O.pool_shapes(npg, P, 1, case.head_dim, case.mla)
    oc, osc = np.zeros(cs, np.uint8), np.zeros(ss, np.uint16)
    O.store(oc, osc, k, v, slots, num_kv_heads=1, head_dim=case.head_dim, page_size=P, mla=case.mla,
            kind=case.kind)
    q = bits(case.q[b:b + 1, heads, :])
    return O.decode(q, oc, osc, sbt, np.array([L], np.int32), num_q_heads=len(heads), num_kv_heads=1,
                    head_dim=case.head_dim, v_dim=case.v_dim, page_size=P, mla=case.mla, kind=case.kind,
                    sm_scale=case.sm_scale, nthreads=0)[0]


def _check_store_sample(case, codes, scales, rng):
    """Bit-exact codes and scales at a random sample of the stored context rows."""
    sm = case.slot_mapping.cpu().numpy()
    stored = np.nonzero(sm >= 0)[0]
    pick = np.sort(rng.choice(stored, size=min(STORE_SAMPLE_ROWS, stored.size), replace=False))
    P, Hkv, D = case.page_size, case.num_kv_heads, case.head_dim
    n = pick.size
    cs, ss = O.pool_shapes((n + P - 1) // P, P, Hkv, D, case.mla)
    oc, osc = np.zeros(cs, np.uint8), np.zeros(ss, np.uint16)
    O.store(oc, osc, bits(case.k[pick]), None if case.mla else bits(case.v[pick]), np.arange(n, dtype=np.int64),
            num_kv_heads=Hkv, head_dim=D, page_size=P, mla=case.mla, kind=case.kind)
    slots = torch.as_tensor(sm[pick], device=codes.device)
    gc = codes[slots // P, :, :, slots % P, :].cpu().numpy()          # [n, n_kv, Hkv, D]
    gs = scales[slots // P, :, :, slots % P, :].cpu().numpy()         # [n, n_kv, Hkv, D/32]
    j = np.arange(n)
    rc = oc[j // P, :, :, j % P, :]
    rs = osc[j // P, :, :, j % P, :]
    assert np.array_equal(gc, rc), ("codes differ", int((gc != rc).sum()))
    assert np.array_equal(gs.view(np.uint16), rs), ("scales differ", int((gs.view(np.uint16) != rs).sum()))


def _decode_samples(case):
    """(sequence, kv head, query heads) pairs to check: the longest sequence and one more."""
    rng = np.random.default_rng(7)
    lens = case.seq_lens.cpu().numpy()
    bs = [int(np.argmax(lens))]
    if case.batch > 1:
        other = int(rng.integers(case.batch))
        bs.append(other if other != bs[0] else (bs[0] + 1) % case.batch)
    G = case.num_q_heads // case.num_kv_heads
    out = []
    for i, b in enumerate(bs):
        g = int(rng.integers(case.num_kv_heads))
        heads = list(range(g * G, (g + 1) * G))
        if case.mla:
            heads = sorted(rng.choice(heads, size=MLA_SAMPLE_HEADS, replace=False).tolist())
        out.append((b, g, heads))
    return out


@pytest.mark.parametrize("kind", ["fp8_e4m3", "q8_0"])
@pytest.mark.parametrize("key", list(FULL))
def test_full_size_store_and_decode_match_the_oracle_on_samples(key, kind):
    case = _make(key, kind)
    L, codes, scales = gpu_pool(case)
    gpu_store(case, codes, scales)
    _check_store_sample(case, codes, scales, np.random.default_rng(11))
    if case.new_k is not None:  # the step's rows (serving: each sequence's last token), as the bench stores them
        gpu_store(case, codes, scales, rows="new")
    got = gpu_decode(case, codes, scales)  # automatic kernel and split size, as the benchmark runs it
    samples = _decode_samples(case)
    if key == "long_gqa_b8":
        # four (sequence, kv head) pairs of 262144 tokens, two query heads of each: the oracle's share stays
        # at about one pair's worth of all eight heads, spread over sequences and both kv heads
        rng = np.random.default_rng(17)
        G = case.num_q_heads // case.num_kv_heads
        bs = rng.choice(case.batch, size=4, replace=False)
        samples = [(int(b), i % 2, sorted(rng.choice(range((i % 2) * G, (i % 2 + 1) * G), size=2,
                                                     replace=False).tolist())) for i, b in enumerate(bs)]
    for b, g, heads in samples:
        ref = _oracle_subcase(case, b, g, heads)
        assert_decode_close(got[b, heads, :], ref)
    del codes, scales, case
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kind", ["fp8_e4m3", "q8_0"])
def test_full_size_sparse_mla_decode_matches_the_oracle(kind):
    """The pages' sparse configuration: 163840-token latent pool, 128 heads, 256 selected columns (1%
    masked).  The oracle quantizes only the selected rows, in list order, into a compact pool and
    attends over all of them (attention does not depend on the order of its columns)."""
    case = workloads.make("mla", kind=kind, device="cuda")
    L, codes, scales = gpu_pool(case)
    gpu_store(case, codes, scales)
    ix = workloads.sparse_indices(case, 256)
    out = torch.empty(case.batch, case.num_q_heads, case.v_dim, dtype=torch.float32, device="cuda")
    ws = kvq.alloc_sparse_workspace(L, case.batch, case.num_q_heads, ix.shape[1])
    kvq.kvq_decode_sparse(case.q, codes, scales, case.block_table, case.seq_lens, ix, out, ws, L, case.kind,
                          case.sm_scale)
    torch.cuda.synchronize()
    assert kvq.kvq_workspace_status(ws) == 0
    got = out.cpu().numpy().astype(np.float64)
    P = case.page_size
    for b in range(case.batch):
        off, Lb = _rows_of_sequence(case, b)
        bt = case.block_table[b].cpu().numpy()
        cols = [int(p) for p in ix[b].cpu().numpy() if 0 <= p < Lb and bt[p // P] >= 0]
        n = len(cols)
        npg = max((n + P - 1) // P, 1)
        cs, ss = O.pool_shapes(npg, P, 1, case.head_dim, case.mla)
        oc, osc = np.zeros(cs, np.uint8), np.zeros(ss, np.uint16)
        O.store(oc, osc, bits(case.k[[off + p for p in cols]]), None, np.arange(n, dtype=np.int64), num_kv_heads=1,
                head_dim=case.head_dim, page_size=P, mla=True, kind=case.kind)
        ref = O.decode_sparse(bits(case.q[b:b + 1]), oc, osc, np.arange(npg, dtype=np.int32)[None, :],
                              np.array([n], np.int32), np.arange(n, dtype=np.int32)[None, :],
                              num_q_heads=case.num_q_heads, num_kv_heads=1, head_dim=case.head_dim,
                              v_dim=case.v_dim, page_size=P, mla=True, kind=case.kind, sm_scale=case.sm_scale,
                              nthreads=0)[0]
        assert_decode_close(got[b], ref)


@pytest.mark.parametrize("kind", ["fp8_e4m3", "q8_0"])
def test_full_size_extend_matches_the_oracle_on_samples(kind):
    case = workloads.make("qwen3_1p7b", kind=kind, device="cuda")
    L, codes, scales = gpu_pool(case)
    gpu_store(case, codes, scales)
    q, q_start, _ = workloads.extend_inputs(case, 2048)
    out = torch.empty(q.shape[0], case.num_q_heads, case.v_dim, dtype=torch.float32, device="cuda")
    ws = kvq.alloc_extend_workspace()
    kvq.kvq_extend(q, codes, scales, case.block_table, case.seq_lens, q_start, out, ws, L, case.kind, case.sm_scale)
    torch.cuda.synchronize()
    assert kvq.kvq_workspace_status(ws) == 0
    got = out.cpu().numpy().astype(np.float64)
    qs = q_start.cpu().numpy()
    lens = case.seq_lens.cpu().numpy()
    rng = np.random.default_rng(13)
    G = case.num_q_heads // case.num_kv_heads
    for b in rng.choice(case.batch, size=3, replace=False):
        n = int(qs[b + 1] - qs[b])
        for i in (0, int(rng.integers(n)), n - 1):          # first, a random and the last new token
            g = int(rng.integers(case.num_kv_heads))
            heads = list(range(g * G, (g + 1) * G))
            pos = int(lens[b]) - n + i
            # the oracle's extend of that one token over the sequence cut at its position, compact pool
            sub = type(case)(**{**case.__dict__, "seq_lens": case.seq_lens.clone()})
            sub.seq_lens[b] = pos + 1
            row = int(qs[b]) + i
            sub.q = case.q.clone()
            sub.q[b] = q[row]
            ref = _oracle_subcase(sub, int(b), g, heads)
            assert_decode_close(got[row, heads, :], ref)
