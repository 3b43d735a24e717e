"""Error of the 8-bit cache against unquantized bf16 K/V, by the oracle alone.

"feat(kvcache): 8-bit DSV4 window/compressed KV", section "Why the precision cost is small", and the review
comment "q8_0 vs fp8" of "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype" argue
that the block-scaled 8-bit cache costs little precision.  This module measures that cost on the seeded
workloads: the same rows are stored once through the 8-bit store and once as plain bf16 into a 2-byte pool of
the same layout, both are decoded by the oracle in fp64, and the outputs are compared.  It is a report, not
a parity bound: the GPU path is checked against the quantized oracle; this is what quantizing costs.

``python -m tests.error_vs_bf16`` prints the table for every workload family at its benchmark shapes
(sequences sampled where the family is large); ``measure`` is used by the CPU test at small sizes.
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from block_quantized_bit_gb300 import workloads  # noqa: E402


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def measure(case, seqs=None, nthreads=0):
    """Quantized and unquantized oracle decodes of `case` (a CPU workload) over the sequences `seqs`.

    Returns a dict: max and mean |quantized - bf16| over every output element, the largest |output|, the
    output arrays themselves (float64 [len(seqs), Hq, Dv]), and the 8-bit pool with the input rows and slots
    it was filled from."""
    seqs = list(range(case.batch)) if seqs is None else list(seqs)
    P, Hkv, D = case.page_size, case.num_kv_heads, case.head_dim
    n_kv = 1 if case.mla else 2
    nth = nthreads or max(1, os.cpu_count() or 1)
    codes = np.zeros((case.num_pages, n_kv, Hkv, P, D), np.uint8)
    unscaled = case.kind.endswith("_unscaled")   # the plain fp8 casts keep no scales
    scales = None if unscaled else np.zeros((case.num_pages, n_kv, Hkv, P, D // 32), np.uint16)
    pool16 = np.zeros((case.num_pages, n_kv, Hkv, P, D), np.uint16)
    # only the rows of the chosen sequences are needed
    lens = [int(x) for x in case.seq_lens.cpu()]
    starts = np.concatenate([[0], np.cumsum(lens)])
    rows = np.concatenate([np.arange(starts[b], starts[b + 1]) for b in seqs]) if seqs else np.zeros(0, np.int64)
    rows_t = torch.from_numpy(rows.astype(np.int64))
    k = bits(case.k[rows_t])
    v = None if case.mla else bits(case.v[rows_t])
    sm = case.slot_mapping.cpu().numpy()[rows]
    dims = dict(num_kv_heads=Hkv, head_dim=D, page_size=P, mla=case.mla)
    O.store(codes, scales, k, v, sm, kind=case.kind, **dims)
    O.scatter_bf16(pool16, k, v, sm, **dims)
    idx = torch.tensor(seqs, dtype=torch.long)
    q = bits(case.q[idx])
    bt = case.block_table.cpu()[idx].numpy()
    sl = case.seq_lens.cpu()[idx].numpy()
    common = dict(num_q_heads=case.num_q_heads, num_kv_heads=Hkv, head_dim=D, v_dim=case.v_dim, page_size=P,
                  mla=case.mla, sm_scale=case.sm_scale, nthreads=nth)
    out_q = O.decode(q, codes, scales, bt, sl, kind=case.kind, **common)
    out_16 = O.decode_bf16(q, pool16, bt, sl, **common)
    d = np.abs(out_q - out_16)
    return {"max_abs": float(d.max()) if d.size else 0.0, "mean_abs": float(d.mean()) if d.size else 0.0,
            "max_out": float(np.abs(out_16).max()) if d.size else 0.0, "out_q": out_q, "out_bf16": out_16,
            "codes": codes, "scales": scales, "rows": rows, "slots": sm}


# The families at the shapes bench.py measures; where the oracle would take minutes, a declared sample of the
# sequences (every head of each) stands for the whole batch -- the distributions are the same per sequence.
REPORT = [
    ("tiny (512 tokens)", "tiny", {}, None),
    ("qwen3_1p7b (B=8, 1k-16k)", "qwen3_1p7b", {}, None),
    ("long_gqa (262144 tokens, 0.5% pages masked)", "long_gqa", {"batch": 1, "ctx": 262144}, None),
    ("mla (Hq=128, 163840 tokens)", "mla", {}, None),
    ("serving (B=64; 8 sequences sampled)", "serving", {}, range(0, 64, 8)),
]


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--families", nargs="*", default=None)
    ap.add_argument("--kinds", nargs="*", default=["fp8_e4m3", "q8_0", "fp8_e4m3_unscaled", "fp8_e5m2_unscaled"])
    a = ap.parse_args()
    print("| Workload | Kind | max abs vs bf16 | mean abs vs bf16 | max abs output | oracle s |")
    print("|---|---|---|---|---|---|")
    for label, fam, kw, seqs in REPORT:
        if a.families and fam not in a.families:
            continue
        for kind in a.kinds:
            t0 = time.time()
            case = workloads.make(fam, kind=kind, device="cpu", **kw)
            r = measure(case, seqs)
            print("| %s | %s | %.3e | %.3e | %.3g | %.0f |" % (label, kind, r["max_abs"], r["mean_abs"], r["max_out"],
                                                            time.time() - t0), flush=True)


if __name__ == "__main__":
    main()
