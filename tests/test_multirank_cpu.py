"""The N > 1 bench path on CPU: two gloo ranks, each a replica with its own
time; the reported time is the slowest rank's and the value counts both
ranks' work."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [120.0, 180.0][rank]
    mx = bench.max_over_ranks(local_ms)
    val = bench.whole_job_tflops(2.0e12, 10, world, mx)
    dist.barrier()
    q.put((rank, mx, val))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, val in got:
        assert mx == 180.0
        assert val == pytest.approx(2.0e12 * 10 * 2 / 0.18 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(1e12, 1, 1, 1000.0) == pytest.approx(1.0)


@pytest.mark.parametrize("workload,mean_len", [("bf16_8k", 1024), ("bf16_32k_causal", 4096)])
def test_bench_flops_with_documents_match_the_oracle_pair_count(workload, mean_len):
    """bench.py --docs counts 4 * B * Hq * D flops per visible (query, key)
    pair; the pair count is the oracle's for the same seeded documents."""
    import numpy as np
    import bench
    import oracle
    from blockwise_attention_online_gb300 import workloads
    w = workloads.WORKLOADS[workload]
    docs, flops = bench._docs(w, mean_len)
    assert docs[0] == 0 and docs[-1] == w.S and len(docs) >= 2
    pos = np.arange(w.S)
    pairs = oracle.unmasked_pairs(pos, pos, w.causal, docs)
    assert flops == 4.0 * w.B * w.Hq * w.D * pairs
    assert bench._docs(w, 0) == (None, w.flops())
