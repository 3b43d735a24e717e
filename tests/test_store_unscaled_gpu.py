"""GPU parity of kvq_store_unscaled (the plain e4m3 / e5m2 cast into an unscaled fp8 pool) against the oracle:
every code byte equal, for GQA and MLA rows with outliers beyond the formats' largest finite values (they
saturate), values in the subnormal ranges and signed zeros; slots of -1 leave the pool untouched."""
import numpy as np
import pytest
import torch

import oracle as O
from block_quantized_bit_gb300 import kvq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", ["fp8_e4m3_unscaled", "fp8_e5m2_unscaled"])
@pytest.mark.parametrize("mla", [False, True])
def test_unscaled_store_matches_the_oracle_bit_exactly(kind, mla):
    g = torch.Generator().manual_seed(8)
    T, Hkv, D, P = 200, 1 if mla else 4, 576 if mla else 128, 16
    num_pages = (T + P - 1) // P + 1
    k = torch.randn(T, Hkv, D, generator=g) * torch.exp(3 * torch.randn(T, Hkv, 1, generator=g))
    k[0, 0, :8] = torch.tensor([1e6, -1e6, 500.0, -460.0, 6e4, -7e4, 0.0, -0.0])  # beyond 448 / 57344; zeros
    k[1, 0, :4] = torch.tensor([1e-3, 2e-6, 3e-9, -1e-5])                            # subnormal ranges
    v = None if mla else torch.randn(T, Hkv, D, generator=g) * 10
    slots = torch.randperm(num_pages * P)[:T].to(torch.int64)
    slots[3] = -1
    L = kvq.Layout(num_pages, P, Hkv, D, 512 if mla else D, mla)
    codes = torch.full((kvq.kvq_pool_bytes(L),), 0x5A, dtype=torch.uint8, device="cuda")
    kb = k.to(torch.bfloat16)
    vb = None if v is None else v.to(torch.bfloat16)
    kvq.kvq_store_unscaled(codes, kb.cuda(), None if vb is None else vb.cuda(), slots.cuda(), L, kind)
    torch.cuda.synchronize()
    cs, _ = O.pool_shapes(num_pages, P, Hkv, D, mla)
    oc = np.full(cs, 0x5A, np.uint8)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    O.store(oc, None, bits(kb), None if vb is None else bits(vb), slots.numpy(), num_kv_heads=Hkv, head_dim=D,
            page_size=P, mla=mla, kind=kind)
    got = codes.cpu().numpy().reshape(cs)
    assert np.array_equal(got, oc), int((got != oc).sum())
