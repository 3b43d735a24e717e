"""Benchmark of the 8-bit paged KV cache hot path on GB300: one step = kvq_store + kvq_decode.

Default workload (``long_gqa``, batch 8 x 262144 tokens): a long-context GQA layer -- Hq=16, Hkv=2,
head_dim=256, page 16, 0.5% of the block-table entries masked -- whose step re-stores the whole cached
context (8 x 262144 rows) and decodes batch 8 over it, fp8_e4m3.  ``--workload qwen3_1p7b`` (Hq=16,
Hkv=8, head_dim=128; 8 x 2048 new rows stored, batch 8 decoded over contexts uniform in [1024, 16384]),
``mla``, ``serving`` and ``tiny`` select the other shapes.  Inputs are seeded synthetic tensors
(workloads.py).  Prints one JSON line.

Metric: algorithmic HBM bytes moved by the step per second (GB/s), i.e. store bytes (bf16 in, codes
and fp16 scales out, slot mapping) plus decode bytes (codes and scales of every valid token, q,
block table, output), divided by the device time of the step.  L2 is flushed between steps.

``--extend N`` measures the extend (prefill) step instead: the store of each sequence's last N rows (the
step's new tokens) plus the causal attention of those tokens over the pool (kvq_extend, tensor cores),
reported in TFLOP/s (4 * head_dim * query heads * the keys each new token sees) against the measured bf16
tensor peak.

``--impl reference`` times the CPU oracle (the plain C reference of the same computation) on the
host cores, on a bounded sample of the same workload, and prints the same line with
``"impl": "reference"``.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402


# Code bytes per element of each kind: the block-scaled kinds add an fp16 scale per 32 elements; the unscaled
# fp8 casts have none.
KINDS = {"fp8_e4m3": 17 / 16, "q8_0": 17 / 16, "fp8_e4m3_unscaled": 1.0, "fp8_e5m2_unscaled": 1.0}


def unscaled(kind):
    return KINDS[kind] == 1.0


def store_rows_into(kvq, codes, scales, k, v, slots, L, kind):
    """The step's store: kvq_store (block-scaled) or kvq_store_unscaled (the plain fp8 cast)."""
    if unscaled(kind):
        kvq.kvq_store_unscaled(codes, k, v, slots, L, kind)
    else:
        kvq.kvq_store(codes, scales, k, v, slots, L, kind)


def alloc_pool(kvq, L, kind, dev):
    codes, scales = kvq.alloc_pool(L, dev)
    codes.zero_()
    if unscaled(kind):
        return codes, None
    scales.zero_()
    return codes, scales


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_gqa",
                    choices=["qwen3_1p7b", "long_gqa", "mla", "serving", "tiny"])
    ap.add_argument("--kind", default="fp8_e4m3", choices=list(KINDS))
    ap.add_argument("--batch", type=int, default=None, help="long_gqa (default 8) / serving batch override")
    ap.add_argument("--ctx", type=int, default=None, help="long_gqa / mla context override")
    ap.add_argument("--path", type=int, default=0, help="decode path: 0 auto, 1 CUDA cores, 2 tcgen05")
    ap.add_argument("--topk", type=int, default=0,
                    help="sparse (top-K) decode: this many index-list columns per sequence (0: dense decode)")
    ap.add_argument("--extend", type=int, default=0,
                    help="extend (prefill) step: this many new tokens per sequence (0: the decode step)")
    ap.add_argument("--precise-p", action="store_true",
                    help="extend with P carried to 16+ bits (two bf16 terms on the flash kernel; fp32 on the "
                         "CUDA-core decode)")
    ap.add_argument("--extend-path", type=int, default=None, choices=[0, 1, 2],
                    help="extend kernel: 0 automatic (the default), 1 each new token's prefix on the CUDA-core "
                         "decode (fp32 P), 2 the flash kernel (GQA) / the tensor-core decode (MLA)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=None)
    return ap.parse_args()


# ------------------------------------------------------------------------------------------ setup
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def make_case(args, device):
    from block_quantized_bit_gb300 import workloads
    kw = {}
    if args.seed is not None:
        kw["seed"] = args.seed
    if args.workload == "long_gqa":
        kw.update(batch=args.batch or 8, ctx=args.ctx or 262144)
    elif args.workload == "mla":
        kw.update(ctx=args.ctx or 163840)
    elif args.workload == "serving" and args.batch:
        kw.update(batch=args.batch)
    return workloads.make(args.workload, kind=args.kind, device=device, **kw)


def valid_tokens(case):
    """Tokens the decode reads: t < seq_len whose page is not masked."""
    bt = case.block_table.cpu()
    lens = case.seq_lens.cpu().tolist()
    P = case.page_size
    total = 0
    for b, L in enumerate(lens):
        n = (L + P - 1) // P
        pages = bt[b, :n]
        full = int((pages >= 0).sum())
        last_masked = n > 0 and int(pages[n - 1]) < 0
        tail = L - (n - 1) * P if n > 0 else 0
        total += full * P - ((P - tail) if (n > 0 and not last_masked) else 0)
    return total


def valid_columns(case, ix):
    """Columns a sparse decode reads: listed positions p < seq_len whose page is not masked."""
    bt = case.block_table.cpu()
    lens = case.seq_lens.cpu().tolist()
    P = case.page_size
    total = 0
    for b, L in enumerate(lens):
        for p in ix[b].cpu().tolist():
            if 0 <= p < L and int(bt[b, p // P]) >= 0:
                total += 1
    return total


def algorithmic_bytes(case, ix=None):
    """(store_bytes, decode_bytes) of one step -- the method's own traffic."""
    n_kv = 1 if case.mla else 2
    row_elems = n_kv * case.num_kv_heads * case.head_dim
    if case.new_k is not None:
        store_rows = int(case.new_k.shape[0])
    else:
        store_rows = int(case.k.shape[0])
    bpe = KINDS[case.kind]
    store = store_rows * (row_elems * (2 + bpe) + 8)
    out_bytes = case.q.numel() * 2 + case.batch * case.num_q_heads * case.v_dim * 2 + case.batch * 4
    if ix is not None:  # sparse: the selected rows, the index lists and their block-table lookups
        toks = valid_columns(case, ix)
        decode = toks * row_elems * bpe + out_bytes + ix.numel() * 8
        return store, decode, store_rows, toks
    toks = valid_tokens(case)
    pages = sum((int(L) + case.page_size - 1) // case.page_size for L in case.seq_lens.cpu().tolist())
    decode = toks * row_elems * bpe + out_bytes + pages * 4
    return store, decode, store_rows, toks


# ------------------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------ ours
def run_ours(args, world, rank):
    from block_quantized_bit_gb300 import kvq
    dev = torch.device("cuda", torch.cuda.current_device())
    case = make_case(args, "cuda")
    L = kvq.Layout(case.num_pages, case.page_size, case.num_kv_heads, case.head_dim, case.v_dim, case.mla)
    codes, scales = alloc_pool(kvq, L, case.kind, dev)
    # fill the cached context (untimed)
    store_rows_into(kvq, codes, scales, case.k, case.v, case.slot_mapping, L, case.kind)
    if case.new_k is not None:
        sk, sv, ss = case.new_k, case.new_v, case.new_slots
    else:  # the store step re-stores the context rows
        sk, sv, ss = case.k, case.v, case.slot_mapping
    out = torch.empty(case.batch, case.num_q_heads, case.v_dim, dtype=torch.bfloat16, device=dev)
    ix = None
    if args.topk > 0:
        from block_quantized_bit_gb300 import workloads
        ix = workloads.sparse_indices(case, args.topk, device=dev)
        ws = kvq.alloc_sparse_workspace(L, case.batch, case.num_q_heads, args.topk, dev)
    else:
        ws = kvq.alloc_workspace(L, case.batch, case.num_q_heads, case.max_pages, dev, path=args.path)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)  # 4x L2
    stream = torch.cuda.current_stream()

    def decode(q, bt, sl, ix_, o):
        if ix_ is not None:
            kvq.kvq_decode_sparse(q, codes, scales, bt, sl, ix_, o, ws, L, case.kind, case.sm_scale)
        else:
            kvq.kvq_decode(q, codes, scales, bt, sl, o, ws, L, case.kind, case.sm_scale, path=args.path)

    def step():
        store_rows_into(kvq, codes, scales, sk, sv, ss, L, case.kind)
        decode(case.q, case.block_table, case.seq_lens, ix, out)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    st = kvq.kvq_workspace_status(ws)
    if st != 0:
        raise RuntimeError("decode reported status %d" % st)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        store_rows_into(kvq, codes, scales, sk, sv, ss, L, case.kind)
        ev[i][1].record(stream)
        decode(case.q, case.block_table, case.seq_lens, ix, out)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    store_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    step_ms = [a + b for a, b in zip(store_ms, dec_ms)]
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / K

    store_b, dec_b, store_rows, toks = algorithmic_bytes(case, ix)
    value = world * (store_b + dec_b) * K / (total_ms / 1e3) / 1e9
    peaks = load_peaks()
    hbm = peaks.get("hbm_gbs")
    dec_avg_s = statistics.mean(dec_ms) / 1e3
    store_avg_s = statistics.mean(store_ms) / 1e3
    dec_gbs = dec_b / dec_avg_s / 1e9
    store_gbs = store_b / store_avg_s / 1e9

    # end to end through the public API: host inputs (pinned) in, host output back, every step
    e2e = run_e2e(args, case, L, codes, scales, sk, sv, ss, ix, decode, flush, world)
    e2e["value"] = world * (store_b + dec_b) / e2e.pop("step_s") / 1e9
    e2e["unit"] = "GB/s"

    # store kernel + decode kernel (+ merge kernel on the tensor-core path; + the gather when sparse, whose
    # dense decode runs over topk tokens per sequence)
    if ix is not None:
        Lc = kvq.Layout(case.batch * max(1, (args.topk + 15) // 16), case.page_size, case.num_kv_heads,
                        case.head_dim, case.v_dim, case.mla)
        cpages = max(1, (args.topk + 15) // 16)
        launches_per_step = 2 + (2 if kvq.kvq_decode_path(Lc, case.batch, case.num_q_heads, cpages) == 2 else 1)
    else:
        launches_per_step = 1 + (2 if kvq.kvq_decode_path(L, case.batch, case.num_q_heads, case.max_pages,
                                                          path=args.path) == 2 else 1)
    res = {
        "metric": "quantized-KV decode attention HBM GB/s (% of GB300 peak); kvq_store GB/s",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",  # K and V dequantized to bf16 before the dot; fp32 accumulation
        "data": "synthetic (seeded; workloads.py)",
        "config": workload_config(args, case, store_rows, toks, world),
        "store_gbs": round(store_gbs, 1),
        "store_frac_hbm": round(store_gbs / hbm, 4) if hbm else None,
        "decode_gbs": round(dec_gbs, 1),
        "decode_frac_hbm": round(dec_gbs / hbm, 4) if hbm else None,
        "decode_us": round(dec_avg_s * 1e6, 2),
        "decode_us_per_token": round(dec_avg_s * 1e6 / case.batch, 3),
        "store_us": round(store_avg_s * 1e6, 2),
        "roofline": {"bound": "hbm", "kernel": "kvq_decode_sparse (gather + decode)" if ix is not None
                     else "kvq_decode (split kernel + merge)",
                     "achieved": round(dec_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(dec_gbs / hbm, 4) if hbm else None,
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if hbm else "fallback 6800",
                     "traffic": recorded_traffic(args)},
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(case, args)
    return res


def workload_config(args, case, store_rows, toks, world):
    """The workload a bench line measures (both arms report the same one)."""
    return {"workload": args.workload, "kind": args.kind, "batch": case.batch,
            "num_q_heads": case.num_q_heads, "num_kv_heads": case.num_kv_heads,
            "head_dim": case.head_dim, "v_dim": case.v_dim, "page_size": case.page_size,
            "store_rows": store_rows, "decode_tokens": toks, **({"topk": args.topk} if args.topk else {}),
            "seq_lens": [int(x) for x in case.seq_lens.cpu().tolist()][:16],
            "l2": "flushed between steps (512 MB write)", "parallelism": "replicas" if world > 1 else "1 gpu"}


def run_e2e(args, case, L, codes, scales, sk, sv, ss, ix, decode, flush, world):
    from block_quantized_bit_gb300 import kvq
    dev = codes.device
    hk = sk.cpu().pin_memory()
    hv = None if sv is None else sv.cpu().pin_memory()
    hs = ss.cpu().pin_memory()
    hq = case.q.cpu().pin_memory()
    hbt = case.block_table.cpu().pin_memory()
    hsl = case.seq_lens.cpu().pin_memory()
    hix = None if ix is None else ix.cpu().pin_memory()
    dix = None if ix is None else torch.empty_like(ix)
    hout = torch.empty((case.batch, case.num_q_heads, case.v_dim), dtype=torch.bfloat16).pin_memory()
    dk, dv, ds = torch.empty_like(sk), None if sv is None else torch.empty_like(sv), torch.empty_like(ss)
    dq, dbt, dsl = torch.empty_like(case.q), torch.empty_like(case.block_table), torch.empty_like(case.seq_lens)
    dout = torch.empty((case.batch, case.num_q_heads, case.v_dim), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def one():
        dk.copy_(hk, non_blocking=True)
        if dv is not None:
            dv.copy_(hv, non_blocking=True)
        ds.copy_(hs, non_blocking=True)
        dq.copy_(hq, non_blocking=True)
        dbt.copy_(hbt, non_blocking=True)
        dsl.copy_(hsl, non_blocking=True)
        if dix is not None:
            dix.copy_(hix, non_blocking=True)
        store_rows_into(kvq, codes, scales, dk, dv, ds, L, case.kind)
        decode(dq, dbt, dsl, dix, dout)
        hout.copy_(dout, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        one()
    torch.cuda.synchronize()
    K = args.steps
    tot = 0.0
    for _ in range(K):
        flush.fill_(3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        one()
        e1.record(stream)
        torch.cuda.synchronize()
        tot += e0.elapsed_time(e1)
    tot = max_over_ranks(tot, world)
    h2d = sum(t.numel() * t.element_size() for t in (hk, hs, hq, hbt, hsl) + (() if hix is None else (hix,))) + \
        (0 if hv is None else hv.numel() * hv.element_size())
    d2h = hout.numel() * hout.element_size()
    return {"step_s": tot / K / 1e3, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# The sources the decode call is built from (host planning, kernels, shared device code): the traffic record
# stays valid while these are unchanged, whatever else changes in the library.
DECODE_SOURCES = ("kvq_api.cu", "kvq_decode.cu", "kvq_decode_mla.cu", "kvq_decode_tc.cu", "kvq_device.cuh",
                  "kvq_internal.h", "kvq_plan.cuh", "kvq_tc.cuh")


def sources_sha256(files):
    """sha256 over the named library sources, each preceded by its name, in the given order."""
    h = hashlib.sha256()
    d = os.path.join(os.path.dirname(os.path.abspath(__file__)), "block_quantized_bit_gb300", "csrc")
    for f in files:
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(args):
    """DRAM bytes per decode call (split kernel + merge) from the committed ncu record, or None when
    there is no record for this workload or the sources it names changed since it was taken."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "dram_traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    for e in rec.get("entries", []):
        files = e.get("sources")
        if not files or e.get("sources_sha256") != sources_sha256(files):
            continue
        if (e.get("workload") == args.workload and e.get("kind") == args.kind and e.get("path", 0) == args.path
                and args.batch is None and args.ctx is None):
            return int(e["dram_read_bytes"]) + int(e["dram_write_bytes"])
    return None


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "_fallback": True}


# ------------------------------------------------------------------------------------------ oracle
def oracle_sample(case, budget_rows=None, max_seqs=None):
    """A bounded sample of the workload for the CPU oracle: the store rows and the sequences decoded."""
    n_rows = int((case.new_k if case.new_k is not None else case.k).shape[0])
    if budget_rows is not None:
        n_rows = min(n_rows, budget_rows)
    seqs = list(range(case.batch if max_seqs is None else min(case.batch, max_seqs)))
    return n_rows, seqs


def sample_text(n_rows, seqs, batch, tok_cap):
    cap = "" if tok_cap is None else ", each cut to its first %d tokens" % tok_cap
    return "store of %d rows + fp64 decode of %d of %d sequences (all heads%s)" % (n_rows, len(seqs), batch, cap)


def oracle_step(case, codes, scales, n_rows, seqs, threads, ix=None, tok_cap=None):
    """One oracle step over the sample: store n_rows rows, decode the chosen sequences (each cut to its first
    tok_cap tokens when given: a prefix of a sequence is a shorter sequence of the same workload).  Returns
    bytes."""
    import oracle as O
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    if case.new_k is not None:
        k, v, s = case.new_k[:n_rows], None if case.new_v is None else case.new_v[:n_rows], case.new_slots[:n_rows]
    else:
        k, v, s = case.k[:n_rows], None if case.v is None else case.v[:n_rows], case.slot_mapping[:n_rows]
    O.store(codes, scales, bits(k), None if v is None else bits(v), s.numpy(), num_kv_heads=case.num_kv_heads,
            head_dim=case.head_dim, page_size=case.page_size, mla=case.mla, kind=case.kind)
    idx = torch.tensor(seqs, dtype=torch.long)
    lens = case.seq_lens[idx] if tok_cap is None else case.seq_lens[idx].clamp(max=tok_cap)
    dims = dict(num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
                v_dim=case.v_dim, page_size=case.page_size, mla=case.mla, kind=case.kind, sm_scale=case.sm_scale,
                nthreads=threads)
    if ix is not None:
        O.decode_sparse(bits(case.q[idx]), codes, scales, case.block_table[idx].numpy(), lens.numpy(),
                        ix[idx].numpy(), **dims)
    else:
        O.decode(bits(case.q[idx]), codes, scales, case.block_table[idx].numpy(), lens.numpy(), **dims)
    n_kv = 1 if case.mla else 2
    row = n_kv * case.num_kv_heads * case.head_dim
    sub = type(case)(**{**case.__dict__, "seq_lens": lens, "block_table": case.block_table[idx],
                        "q": case.q[idx]})
    toks = valid_tokens(sub) if ix is None else valid_columns(sub, ix[idx])
    bpe = KINDS[case.kind]
    return n_rows * (row * (2 + bpe) + 8) + toks * row * bpe


def sparse_lists(case, args):
    """The sparse decode's index lists (host), or None for the dense decode."""
    if args.topk <= 0:
        return None
    from block_quantized_bit_gb300 import workloads
    return workloads.sparse_indices(case, args.topk, device="cpu")


def prepare_oracle(case):
    import oracle as O
    from oracle import build_oracle
    build_oracle.build()
    cpu = type(case)(**{k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in case.__dict__.items()})
    codes = np.zeros((cpu.num_pages, 1 if cpu.mla else 2, cpu.num_kv_heads, cpu.page_size, cpu.head_dim), np.uint8)
    scales = None if unscaled(cpu.kind) else np.zeros(codes.shape[:-1] + (cpu.head_dim // 32,), np.uint16)
    return O, cpu, codes, scales


def cpu_baseline(case, args):
    """The oracle, as it stands, on a bounded sample of the same workload (~10-30 s of CPU work)."""
    O, cpu, codes, scales = prepare_oracle(case)
    threads = max(1, O.openmp_threads())
    ix = sparse_lists(cpu, args)
    # whole workload steps while they fit ~10 s, else a sub-sample (fewer store rows and sequences, and
    # sequences cut to a prefix); a first pass on a small sample sizes it, so that no pass runs for minutes
    n_rows, seqs = oracle_sample(cpu)
    tok_cap = None
    big = n_rows * cpu.head_dim * cpu.num_kv_heads > (64 << 20) or valid_tokens(cpu) * cpu.num_q_heads > (1 << 26)
    if big:
        n_rows, seqs = oracle_sample(cpu, budget_rows=4096, max_seqs=1)
        tok_cap = 16384
        t0 = time.perf_counter()
        oracle_step(cpu, codes, scales, n_rows, seqs, threads, ix, tok_cap)
        one = time.perf_counter() - t0
        seqs = list(range(max(1, min(cpu.batch, int(5.0 / max(one, 1e-3))))))
    t0 = time.perf_counter()
    nbytes = oracle_step(cpu, codes, scales, n_rows, seqs, threads, ix, tok_cap)
    passes = 1
    while time.perf_counter() - t0 < 10.0 and passes < 200:
        nbytes += oracle_step(cpu, codes, scales, n_rows, seqs, threads, ix, tok_cap)
        passes += 1
    dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "%d passes of: %s; %.1f s" % (passes, sample_text(n_rows, seqs, cpu.batch, tok_cap), dt)}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle on the host cores, same workload/metric, bounded sample per step."""
    if rank != 0:
        return None
    case = make_case(args, "cpu")
    O, cpu, codes, scales = prepare_oracle(case)
    threads = max(1, O.openmp_threads())
    ix = sparse_lists(cpu, args)
    n_rows, seqs = oracle_sample(cpu, budget_rows=512, max_seqs=1)
    tok_cap = 8192 if int(cpu.seq_lens[0]) > 8192 else None   # about 0.1-0.5 s per step on 16 cores
    for _ in range(args.warmup):
        oracle_step(cpu, codes, scales, n_rows, seqs, threads, ix, tok_cap)
    t0 = time.perf_counter()
    nb = 0.0
    for _ in range(args.steps):
        nb += oracle_step(cpu, codes, scales, n_rows, seqs, threads, ix, tok_cap)
    dt = time.perf_counter() - t0
    value = nb / dt / 1e9
    sample = sample_text(n_rows, seqs, cpu.batch, tok_cap) + " per step"
    return {
        "impl": "reference",
        "metric": "quantized-KV decode attention HBM GB/s (% of GB300 peak); kvq_store GB/s",
        "value": round(value, 5), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; workloads.py)",
        "config": dict(workload_config(args, case, *algorithmic_bytes(case, ix)[2:], world), sample=sample),
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------------------------------ extend
EXTEND_METRIC = "quantized-KV extend (prefill) attention TFLOP/s (% of GB300 bf16 peak); kvq_store of the new rows"


def extend_choice(kvq, case, L, total_q, path, precise=False):
    """The extend kernel the library picks: 3 (flash kernel), 4 (flash, P as two bf16 terms), 1 or 2 (prefixes
    on the CUDA-core / tensor-core decode)."""
    p = kvq.kvq_extend_path(L, total_q, case.num_q_heads, case.max_pages, path, precise)
    if p < 0:
        raise RuntimeError("no extend kernel for this shape and path (status %d)" % p)
    return p


def extend_kernel_name(choice):
    if choice == 3:
        return "kvq_extend (extend_tc_kernel)"
    if choice == 4:
        return "kvq_extend (extend_tc_kernel, P as two bf16 terms)"
    if choice == 1:
        return "kvq_extend (CUDA-core decode over each new token's causal prefix)"
    return "kvq_extend (tensor-core decode over each new token's causal prefix, + merge)"


def extend_launches(choice, total_q):
    """Kernels one extend step launches: the store, then the flash kernel; or the prefix expansion and, per
    chunk of 1024 new tokens, the decode (with the merge on the tensor-core path)."""
    if choice >= 3:
        return 2
    chunk = min(total_q, 1024)
    per = 2 if choice == 2 else 1
    return 2 + per * ((total_q + chunk - 1) // chunk)


def extend_flops_per_key(case):
    """FLOPs of one (new token, visible key) pair over all query heads: QK over the K width plus PV over the V
    width (4 * D * Hq for GQA; 2 * Hq * (576 + 512) for the MLA latent row)."""
    return 2.0 * case.num_q_heads * (case.head_dim + case.v_dim)


def extend_keys(case, q_start):
    """Keys the extend reads, summed over new tokens: the unmasked positions up to each token's own."""
    bt = case.block_table.cpu().numpy()
    lens = case.seq_lens.cpu().numpy()
    qs = q_start.cpu().numpy()
    P = case.page_size
    total = 0
    for b, L in enumerate(lens):
        n = int(qs[b + 1] - qs[b])
        if n == 0:
            continue
        seen = np.cumsum(bt[b, np.arange(L) // P] >= 0)
        total += int(seen[L - n + np.arange(n)].sum())
    return total


def extend_inputs(case, args):
    from block_quantized_bit_gb300 import workloads
    return workloads.extend_inputs(case, args.extend)


def run_extend(args, world, rank):
    from block_quantized_bit_gb300 import kvq
    dev = torch.device("cuda", torch.cuda.current_device())
    case = make_case(args, "cuda")
    L = kvq.Layout(case.num_pages, case.page_size, case.num_kv_heads, case.head_dim, case.v_dim, case.mla)
    codes, scales = alloc_pool(kvq, L, case.kind, dev)
    store_rows_into(kvq, codes, scales, case.k, case.v, case.slot_mapping, L, case.kind)  # the context (untimed)
    q, q_start, rows = extend_inputs(case, args)
    sk, ss = case.k[rows], case.slot_mapping[rows]  # the step re-stores its new rows
    sv = None if case.mla else case.v[rows]
    out = torch.empty(q.shape[0], case.num_q_heads, case.v_dim, dtype=torch.bfloat16, device=dev)
    path, precise = args.extend_path, args.precise_p
    choice = extend_choice(kvq, case, L, int(q.shape[0]), path, precise)
    ws = kvq.alloc_extend_workspace(dev, L, q.shape[0], case.num_q_heads, case.max_pages, path=path,
                                    precise_p=precise)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)  # 4x L2
    stream = torch.cuda.current_stream()

    def extend(q_, qs_, bt_, sl_, o):
        kvq.kvq_extend(q_, codes, scales, bt_, sl_, qs_, o, ws, L, case.kind, case.sm_scale, path=path,
                       precise_p=precise)

    for _ in range(args.warmup):
        flush.fill_(1)
        store_rows_into(kvq, codes, scales, sk, sv, ss, L, case.kind)
        extend(q, q_start, case.block_table, case.seq_lens, out)
    torch.cuda.synchronize()
    st = kvq.kvq_workspace_status(ws)
    if st != 0:
        raise RuntimeError("extend reported status %d" % st)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        store_rows_into(kvq, codes, scales, sk, sv, ss, L, case.kind)
        ev[i][1].record(stream)
        extend(q, q_start, case.block_table, case.seq_lens, out)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    store_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    ext_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    total_ms = max_over_ranks(sum(store_ms) + sum(ext_ms), world)
    keys = extend_keys(case, q_start)
    flops = extend_flops_per_key(case) * keys
    ext_s = statistics.mean(ext_ms) / 1e3
    achieved = flops / ext_s / 1e12
    peaks = load_peaks()
    peak = peaks.get("bf16_tflops")
    store_rows = int(rows.numel())
    row_elems = (1 if case.mla else 2) * case.num_kv_heads * case.head_dim
    store_b = store_rows * (row_elems * (2 + KINDS[case.kind]) + 8)

    # end to end through the public API: the step's inputs from pinned host memory, its output back
    hq, hqs = q.cpu().pin_memory(), q_start.cpu().pin_memory()
    hk, hs = sk.cpu().pin_memory(), ss.cpu().pin_memory()
    hv = None if sv is None else sv.cpu().pin_memory()
    hbt, hsl = case.block_table.cpu().pin_memory(), case.seq_lens.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dq, dqs, dk, ds = (torch.empty_like(t) for t in (q, q_start, sk, ss))
    dv = None if sv is None else torch.empty_like(sv)
    dbt, dsl = torch.empty_like(case.block_table), torch.empty_like(case.seq_lens)
    dout = torch.empty_like(out)
    pairs = [(dq, hq), (dqs, hqs), (dk, hk), (ds, hs), (dbt, hbt), (dsl, hsl)] + ([] if dv is None else [(dv, hv)])

    def one():
        for d, h in pairs:
            d.copy_(h, non_blocking=True)
        store_rows_into(kvq, codes, scales, dk, dv, ds, L, case.kind)
        extend(dq, dqs, dbt, dsl, dout)
        hout.copy_(dout, non_blocking=True)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(K):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world) / K
    h2d = sum(h.numel() * h.element_size() for _, h in pairs)
    res = {
        "metric": EXTEND_METRIC,
        "value": round(world * flops * K / (total_ms / 1e3) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16",  # K and V dequantized to bf16, fp32 accumulation (P bf16 on the tensor cores)
        "data": "synthetic (seeded; workloads.py)",
        "config": dict(workload_config(args, case, store_rows, keys, world), new_tokens_per_seq=args.extend,
                       total_new_tokens=int(q.shape[0]), keys_read=keys, extend_path=path or 0,
                       precise_p=bool(precise)),
        "extend_us": round(ext_s * 1e6, 2),
        "extend_tflops": round(achieved, 1),
        "store_us": round(statistics.mean(store_ms) * 1e3, 2),
        "store_gbs": round(store_b / (statistics.mean(store_ms) / 1e3) / 1e9, 1),
        "roofline": {"bound": "tensor", "kernel": extend_kernel_name(choice), "achieved": round(achieved, 1),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4) if peak else None,
                     "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst; of measured)", "traffic": None},
        "clocks": clk,
        "e2e": {"value": round(world * flops / e2e_s / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": hout.numel() * hout.element_size()},
        "gpu_launches": extend_launches(choice, int(q.shape[0])) * K,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = extend_cpu_baseline(case, args)
    return res


def extend_oracle_pass(O, cpu, codes, scales, q, q_start, m, threads):
    """The oracle on the first m new tokens of sequence 0 (their rows stored, their causal attention):
    returns the FLOPs of that attention."""
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    n0 = int(q_start[1] - q_start[0])
    L0 = int(cpu.seq_lens[0])
    lens = cpu.seq_lens.clone()
    lens[0] = L0 - n0 + m                          # the sample's last new token is token m - 1
    qs = torch.zeros_like(q_start)
    qs[1:] = m
    rows = torch.arange(L0 - n0, L0 - n0 + m)      # sequence 0's rows come first in the context order
    O.store(codes, scales, bits(cpu.k[rows]), None if cpu.mla else bits(cpu.v[rows]), cpu.slot_mapping[rows].numpy(),
            num_kv_heads=cpu.num_kv_heads, head_dim=cpu.head_dim, page_size=cpu.page_size, mla=cpu.mla,
            kind=cpu.kind)
    O.extend(bits(q[:m]), codes, scales, cpu.block_table.numpy(), lens.numpy(), qs.numpy(),
             num_q_heads=cpu.num_q_heads, num_kv_heads=cpu.num_kv_heads, head_dim=cpu.head_dim, v_dim=cpu.v_dim,
             page_size=cpu.page_size, mla=cpu.mla, kind=cpu.kind, sm_scale=cpu.sm_scale, nthreads=threads)
    sub = type(cpu)(**{**cpu.__dict__, "seq_lens": lens})
    return extend_flops_per_key(cpu) * extend_keys(sub, qs)


def extend_oracle_setup(case, args):
    O, cpu, codes, scales = prepare_oracle(case)
    ctx = cpu.slot_mapping
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    O.store(codes, scales, bits(cpu.k), None if cpu.mla else bits(cpu.v), ctx.numpy(), num_kv_heads=cpu.num_kv_heads,
            head_dim=cpu.head_dim, page_size=cpu.page_size, mla=cpu.mla, kind=cpu.kind)  # the context, untimed
    q, q_start, _ = extend_inputs(cpu, args)
    return O, cpu, codes, scales, q.cpu(), q_start.cpu(), max(1, O.openmp_threads())


def extend_cpu_baseline(case, args):
    """The oracle on a bounded sample of the extend: the first m new tokens of sequence 0 (~10 s)."""
    O, cpu, codes, scales, q, q_start, threads = extend_oracle_setup(case, args)
    n0 = int(q_start[1] - q_start[0])
    m = min(4, n0)
    t0 = time.perf_counter()
    extend_oracle_pass(O, cpu, codes, scales, q, q_start, m, threads)
    one = time.perf_counter() - t0
    m = max(1, min(n0, int(m * 10.0 / max(one, 1e-3))))
    t0 = time.perf_counter()
    fl = extend_oracle_pass(O, cpu, codes, scales, q, q_start, m, threads)
    dt = time.perf_counter() - t0
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "store + fp64 causal attention of the first %d of %d new tokens of sequence 0 (all heads); "
                      "%.1f s" % (m, n0, dt)}


def run_extend_reference(args, world, rank):
    if rank != 0:
        return None
    case = make_case(args, "cpu")
    O, cpu, codes, scales, q, q_start, threads = extend_oracle_setup(case, args)
    m = min(1 if cpu.mla else 8, int(q_start[1] - q_start[0]))   # a 128-head latent row costs ~16x a GQA one
    for _ in range(args.warmup):
        extend_oracle_pass(O, cpu, codes, scales, q, q_start, m, threads)
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += extend_oracle_pass(O, cpu, codes, scales, q, q_start, m, threads)
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    sample = "store + fp64 causal attention of the first %d new tokens of sequence 0 (all heads) per step" % m
    return {
        "impl": "reference", "metric": EXTEND_METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; workloads.py)",
        "config": dict(workload_config(args, case, int(q.shape[0]), extend_keys(case, q_start), world),
                       new_tokens_per_seq=args.extend, sample=sample),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world, rank = dist_setup(args)
    if args.impl == "reference":
        res = run_extend_reference(args, world, rank) if args.extend > 0 else run_reference(args, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
        from __graft_entry__ import build
        build()
        res = run_extend(args, world, rank) if args.extend > 0 else run_ours(args, world, rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
