"""Failure detection without a GPU fault: a bounded wait that nothing completes ends, after the library's
2 s limit, in KVQ_ETIMEOUT in the workspace status word, and the context stays usable (a decode right
after it still matches the oracle)."""
import time

import pytest
import torch

from block_quantized_bit_gb300 import kvq, workloads

from parity import assert_decode_close, gpu_decode, gpu_pool, gpu_store, oracle_decode, oracle_pool, oracle_store

pytestmark = pytest.mark.gpu


def test_a_wait_that_never_completes_reports_a_timeout_and_the_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    kvq.kvq_wait_probe(ws)
    st = kvq.kvq_workspace_status(ws)                 # synchronises with the probe kernel
    dt = time.perf_counter() - t0
    assert st == -9, st                                # KVQ_ETIMEOUT
    assert 1.5 < dt < 30.0, dt                         # it waited for the limit, then returned
    # the context is intact: an ordinary store and decode still agree with the oracle
    case = workloads.make("tiny", kind="fp8_e4m3", device="cpu")
    L, codes, scales = gpu_pool(case)
    oc, osc = oracle_pool(case)
    gpu_store(case, codes, scales)
    oracle_store(case, oc, osc)
    assert_decode_close(gpu_decode(case, codes, scales), oracle_decode(case, oc, osc))
