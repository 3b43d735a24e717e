"""The 8-bit cache against unquantized bf16 K/V, by the oracle (a report, checked against a bound it must obey).

"feat(kvcache): 8-bit DSV4 window/compressed KV", section "Why the precision cost is small": quantizing the
cache perturbs attention only a little.  Softmax perturbation gives a bound that the quantized decode must
satisfy against the unquantized one for every output element (b, h, d):

    |out_q - out_bf16| <= max_t |V'_t[d] - V_t[d]| + (exp(2 delta) - 1) * max_t |V_t[d]|,
    delta = max_t |sm_scale * q_h . (K'_t - K_t)|,

over the visible tokens t, with K', V' the dequantized rows: the logits move by at most delta, so each
probability moves by a factor within exp(+-2 delta).  The measured error is printed for the small cases; the
full table comes from ``python -m tests.error_vs_bf16``.
"""
import numpy as np
import pytest
import torch

import oracle as O
from block_quantized_bit_gb300 import workloads
from tests.error_vs_bf16 import bits, measure


def _f64(bits_u16):
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).view(torch.bfloat16).double().numpy()


def _bound(case, r, seqs):
    codes, scales, rows, slots = r["codes"], r["scales"], r["rows"], r["slots"]
    P, Hkv, D, Dv, Hq = case.page_size, case.num_kv_heads, case.head_dim, case.v_dim, case.num_q_heads
    G = Hq // Hkv
    kf = case.k.double().numpy()
    vf = kf if case.mla else case.v.double().numpy()
    lens = [int(x) for x in case.seq_lens]
    out = np.zeros((len(seqs), Hq, Dv))
    pos = 0
    for i, b in enumerate(seqs):
        n = lens[b]
        sl = slots[pos:pos + n]
        rr = rows[pos:pos + n][sl >= 0]
        sl = sl[sl >= 0]
        pos += n
        if len(sl) == 0:
            continue
        pg, off = sl // P, sl % P
        for g in range(Hkv):
            if scales is None:   # unscaled: the code's own value
                val = np.vectorize(lambda c: O.code_value(case.kind, int(c)))
                kq = val(codes[pg, 0, g, off])
                vq = kq[:, :Dv] if case.mla else val(codes[pg, 1, g, off])
            else:
                kq = O.dequant(case.kind, codes[pg, 0, g, off], np.repeat(scales[pg, 0, g, off], 32, axis=-1))
                vq = kq[:, :Dv] if case.mla else O.dequant(case.kind, codes[pg, 1, g, off],
                                                            np.repeat(scales[pg, 1, g, off], 32, axis=-1))
            k16, v16 = kf[rr, g], (kf[rr, g, :Dv] if case.mla else vf[rr, g])
            dv = np.abs(vq - v16).max(0)
            vmax = np.abs(v16).max(0)
            for h in range(g * G, (g + 1) * G):
                q = _f64(bits(case.q[b, h]))
                delta = np.abs(case.sm_scale * ((kq - k16) @ q)).max()
                out[i, h] = dv + np.expm1(2 * delta) * vmax
    return out


CASES = [
    ("tiny", dict(ctx=200)),
    ("qwen3_1p7b", dict(batch=2, ctx_lo=100, ctx_hi=300, new_rows_per_seq=16)),
    ("long_gqa", dict(batch=2, ctx=333)),
    ("mla", dict(batch=1, ctx=150, num_q_heads=16)),
    ("serving", dict(batch=4, median=200, lo=64, hi=400)),
]


@pytest.mark.parametrize("kind", ["fp8_e4m3", "q8_0", "fp8_e4m3_unscaled", "fp8_e5m2_unscaled"])
@pytest.mark.parametrize("fam,kw", CASES, ids=[c[0] for c in CASES])
def test_quantized_decode_stays_within_the_softmax_perturbation_bound_of_bf16(fam, kw, kind):
    case = workloads.make(fam, kind=kind, device="cpu", **kw)
    seqs = list(range(case.batch))
    r = measure(case, seqs, nthreads=2)
    bound = _bound(case, r, seqs)
    err = np.abs(r["out_q"] - r["out_bf16"])
    assert np.all(err <= bound * (1 + 1e-9) + 1e-12)
    assert r["max_abs"] > 0  # quantization changed something
    print("%s %s: max |q - bf16| %.3e, mean %.3e (bound max %.3e)" % (fam, kind, r["max_abs"], r["mean_abs"],
                                                                       bound.max()))
