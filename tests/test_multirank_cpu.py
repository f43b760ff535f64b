"""World-size-2 checks of the multi-GPU host logic on CPU (gloo): the step
shards by sequence with no data-path collective, each rank times its own
independent batch, and the slowest rank's time defines the whole-job rate."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + rank * 5.0                        # rank 1 is the slow one
        out[rank] = (bench.replica_ids(rank), bench.max_over_ranks(mine, world))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_rank_sharding_and_timing():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    ids0, t0 = res[0]
    ids1, t1 = res[1]
    assert set(ids0).isdisjoint(ids1)                   # independent batches per rank
    assert len(ids0) == len(ids1) == 4
    assert t0 == t1 == 15.0                             # both see the slowest rank's time
    import bench
    assert bench.whole_job_rate(384, 2, 0.05) == pytest.approx(384 * 2 / 5e-5)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.replica_ids(0) == [0, 1, 2, 3]


def test_metric_names_the_call_variant():
    """Each non-default call is named in the metric; the plain call adds nothing."""
    import argparse
    import bench
    base = dict(lenience=None, eos=None, per_seq_rules=False, early_exit=False)
    assert bench.variant_of(argparse.Namespace(**base)) == ""
    assert bench.variant_of(argparse.Namespace(**{**base, "early_exit": True})) == " (early exit)"
    both = bench.variant_of(argparse.Namespace(**{**base, "lenience": 0.5, "early_exit": True}))
    assert "lenience 0.5" in both and "early exit" in both


def _shard_worker(rank, world, port, out):
    """One rank: a contiguous slice of the batch through the oracle, then gather."""
    import numpy as np
    import torch.distributed as dist
    import oracle
    from speculative_decoding_verification_44_gb300 import workloads
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _small_serving_workload(workloads, oracle, np)
        lo, hi = rank * w.B // world, (rank + 1) * w.B // world
        mine = _oracle_rows(w, lo, hi, oracle, np)
        parts = [None] * world
        dist.all_gather_object(parts, mine)
        if rank == 0:
            out["gathered"] = [s for p in parts for s in p]
    finally:
        dist.barrier()
        dist.destroy_process_group()


def _small_serving_workload(workloads, oracle, np):
    import torch

    def oracle_probs(rows, params):
        p, _ = oracle.transform_rows(rows.float().double().numpy(), float(np.float32(params.temperature)),
                                     int(params.top_k), float(np.float32(params.top_p)))
        return torch.from_numpy(p)
    return workloads.make(3, "cpu", draft_probs=oracle_probs, B=6, V=2048)


def _oracle_rows(w, lo, hi, oracle, np):
    """Per-sequence oracle results of sequences lo..hi-1 (tokens, count, a_i, Z)."""
    tp = (float(np.float32(w.target_params.temperature)), int(w.target_params.top_k),
          float(np.float32(w.target_params.top_p)))
    res = oracle.verify_sample(w.target_logits[lo:hi].float().double().numpy(),
                               w.draft_logits[lo:hi].float().double().numpy(), w.draft_tokens[lo:hi].numpy(),
                               w.u_accept[lo:hi].double().numpy(), w.u_sample[lo:hi].double().numpy(), tp, tp)
    return [(list(map(int, s.tokens)), int(s.num_accepted), [float(x) for x in s.accept_prob],
             float(s.residual_Z)) for s in res.seqs]


def test_batch_shards_reassemble_to_the_single_rank_result():
    """Replicas only: sequences are independent, so two gloo ranks that each verify a
    contiguous half of the batch and gather the results reproduce the one-rank result
    exactly (no data-path exchange is needed).  Runs the oracle on CPU; the GPU path
    shards the same way but is unmeasured on more than one GPU here."""
    import numpy as np
    import oracle
    from speculative_decoding_verification_44_gb300 import workloads
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_shard_worker, args=(world, port, out), nprocs=world, join=True)
        gathered = out["gathered"]
    w = _small_serving_workload(workloads, oracle, np)
    assert gathered == _oracle_rows(w, 0, w.B, oracle, np)
