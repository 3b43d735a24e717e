"""GPU parity of kvq_store_act_quant (the MLA store fused with the model's per-64 E4M3 rounding of the
latent) against the oracle: every code byte and scale bit equal, for raw bf16 rows as they leave the
producer; slots of -1 leave the pool untouched; a decode over the fused pool reads exactly what a plain
store of the rounded rows would hold."""
import numpy as np
import pytest
import torch

import oracle as O
from block_quantized_bit_gb300 import kvq

pytestmark = pytest.mark.gpu


def _rows(T, D, seed):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(T, D, generator=g) * torch.exp(torch.randn(T, D // 64, 1, generator=g)).repeat(1, 1, 64).reshape(T, D)
    k[1, 64:128] = 0.0       # an all-zero latent unit
    k[2, :64] *= 1e-30       # a tiny one (fp32 subnormal products)
    k[3, 7] = 1.0e4          # an outlier
    return k.to(torch.bfloat16)


@pytest.mark.parametrize("kind", ["fp8_e4m3", "q8_0"])
@pytest.mark.parametrize("rope", [64, 0])
def test_fused_store_matches_the_oracle_bit_exactly(kind, rope):
    T, D, P = 300, 576, 16
    num_pages = (T + P - 1) // P + 2
    k = _rows(T, D, 3)
    slots = torch.randperm(num_pages * P)[:T].to(torch.int64)
    slots[5] = -1
    L = kvq.Layout(num_pages, P, 1, D, 512, True)
    codes, scales = kvq.alloc_pool(L, "cuda")
    codes.fill_(0xA5)
    scales.fill_(0x1234)
    kvq.kvq_store_act_quant(codes, scales, k.cuda(), slots.cuda(), L, kind, rope_dim=rope)
    torch.cuda.synchronize()
    cs, ss = O.pool_shapes(num_pages, P, 1, D, True)
    oc, osc = np.full(cs, 0xA5, np.uint8), np.full(ss, 0x1234, np.uint16)
    O.store_act_quant(oc, osc, k.view(torch.int16).numpy().view(np.uint16), slots.numpy(), head_dim=D, rope_dim=rope,
                      page_size=P, kind=kind)
    assert np.array_equal(codes.cpu().numpy(), oc), int((codes.cpu().numpy() != oc).sum())
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), osc)
