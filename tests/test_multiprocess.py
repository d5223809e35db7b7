"""Multi-rank host logic on CPU: two gloo ranks exercise bench.py's distributed
plumbing (rank discovery, barrier, max-over-ranks timing) and the partition of
(sequence, head) units across ranks, which needs no collective on the data path."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist

    import bench
    import oracle
    import workloads
    r, w, local = bench.dist_init()
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # Per-rank step times: the job's time is the slowest rank's.
    t = bench.max_over_ranks(1.5 + rank, w)
    # Each rank runs the scan on its own share of the sequences (no collective).
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=[40, 17, 64, 3, 90], h_qk=1,
                                              h_v=2, d_k=16, d_v=8, seed=5, state_std=0.05))
    n_seq, h_v = inp.n_seq, inp.spec.h_v
    mine = [u for u in range(n_seq * h_v) if (u // h_v) % w == r]
    o, s = oracle.scan_inputs(inp, units=mine)
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), t=t, o=o, s=s, units=np.array(mine))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_share_units_and_time(tmp_path):
    pytest.importorskip("torch.distributed")
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r0, r1 = (np.load(tmp_path / f"rank{i}.npz") for i in range(2))
    assert float(r0["t"]) == float(r1["t"]) == 2.5          # max over ranks
    assert not set(r0["units"]) & set(r1["units"])          # disjoint shards
    # The shards put together equal the whole run.
    import oracle
    import workloads
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=[40, 17, 64, 3, 90], h_qk=1,
                                              h_v=2, d_k=16, d_v=8, seed=5, state_std=0.05))
    o_all, s_all = oracle.scan_inputs(inp)
    assert np.array_equal(r0["o"] + r1["o"], o_all)
    assert np.array_equal(r0["s"] + r1["s"], s_all)
