"""Host-side checks of bench.py's contract, with no GPU: the reference arm's JSON line, the multi-process
path under torchrun with the gloo backend (world size 2: rank 0 alone prints; the others exit 0 without
work), the barrier and the max over ranks that bound the timed region, and the extend leg's FLOP count."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

CONTRACT = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config")


def _json_lines(out):
    return [json.loads(line) for line in out.splitlines() if line.startswith("{")]


def _env():
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", CUDA_VISIBLE_DEVICES="")
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    return env


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, env=_env())
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    for k in CONTRACT + ("impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny"


def test_reference_arm_under_torchrun_with_two_gloo_ranks():
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", "29731", os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, env=_env())
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1, r.stdout[-2000:]  # rank 0 only
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def _ranks_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    got = bench.max_over_ranks(1.5 + rank, world)
    bench.barrier(world)
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_and_barrier_with_two_gloo_ranks():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ranks_worker, args=(r, 2, 29741, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 2.5, 1: 2.5}  # every rank times the slowest rank


def test_single_process_helpers_are_identities():
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)


def test_extend_keys_count_the_causal_unmasked_positions():
    """extend_keys against a brute-force count: each new token sees the unmasked positions up to its own."""
    from block_quantized_bit_gb300 import workloads
    case = workloads.make("long_gqa", kind="fp8_e4m3", device="cpu", batch=3, ctx=300, mask_frac=0.1,
                          num_q_heads=8, num_kv_heads=2, head_dim=128)
    n_new = [300, 17, 0]
    q, q_start, rows = workloads.extend_inputs(case, n_new)
    bt = case.block_table.numpy()
    want = 0
    for b, L in enumerate(case.seq_lens.tolist()):
        for i in range(n_new[b]):
            pos = L - n_new[b] + i
            want += sum(1 for t in range(pos + 1) if bt[b, t // 16] >= 0)
    assert bench.extend_keys(case, q_start) == want
    assert q.shape == (317, 8, 128) and q_start.tolist() == [0, 300, 317, 317]
    assert rows.numel() == 317 and int(rows[300]) == 300 + 300 - 17  # sequence 1's first new row
    with pytest.raises(ValueError):
        workloads.extend_inputs(case, [301, 0, 0])
    assert np.array_equal(workloads.extend_inputs(case, 5)[1].numpy(), [0, 5, 10, 15])


def test_oracle_sample_with_a_token_cap_counts_the_prefix_it_decodes():
    """The bounded oracle samples cut each decoded sequence to a prefix: the bytes a step reports are those of
    the stored rows plus the valid (unmasked) tokens of that prefix, and the default workload is the long-context
    batch-8 layer."""
    from block_quantized_bit_gb300 import workloads
    case = workloads.make("long_gqa", kind="fp8_e4m3", device="cpu", batch=2, ctx=3000, mask_frac=0.05)
    O, cpu, codes, scales = bench.prepare_oracle(case)
    nb = bench.oracle_step(cpu, codes, scales, 64, [0, 1], 1, tok_cap=1000)
    bt = case.block_table.numpy()
    toks = sum(1 for b in range(2) for t in range(1000) if bt[b, t // 16] >= 0)
    row = 2 * case.num_kv_heads * case.head_dim
    assert nb == 64 * (row * (2 + 1 + 2 / 32) + 8) + toks * row * 17 / 16
    import sys as _sys
    argv, _sys.argv = _sys.argv, ["bench.py"]
    try:
        a = bench.parse()
    finally:
        _sys.argv = argv
    assert a.workload == "long_gqa" and a.kind == "fp8_e4m3" and a.batch is None and a.ctx is None


def test_extend_launch_count_and_kernel_name_follow_the_kernel_choice():
    """The extend's gpu_launches claim: the store plus the flash kernel (choice 3 or 4), or the store, the
    prefix expansion and per chunk of 1024 new tokens the decode (with its merge on the tensor-core path)."""
    assert bench.extend_launches(3, 16384) == 2
    assert bench.extend_launches(4, 16384) == 2
    assert bench.extend_launches(1, 1000) == 3
    assert bench.extend_launches(1, 2049) == 2 + 3
    assert bench.extend_launches(2, 2048) == 2 + 2 * 2
    assert bench.extend_launches(2, 1) == 4
    assert "two bf16 terms" in bench.extend_kernel_name(4)
    assert "extend_tc_kernel" in bench.extend_kernel_name(3)
    assert "CUDA-core" in bench.extend_kernel_name(1)
    assert "tensor-core" in bench.extend_kernel_name(2)
