"""The replica path on several ranks, tested on CPU with gloo (world size 2):
request sharding with rebased cu_rows needs no exchange for verification
(each shard's results equal the whole batch's), and one sum all-reduce of the
prefix-acceptance counters gives the job-wide counters; the bench's job time
is the slowest rank's.  The oracle stands in for the GPU path on each rank.
The adaptive step controller, fed the job-wide counters on every rank, takes
the same batch-uniform step everywhere without exchanging its decision."""
import os
import socket
import tempfile

import numpy as np
import pytest

import workloads as W
from speculative_decoding_verification_ragged_gb300 import shard


def test_request_shard_covers_the_batch_in_contiguous_balanced_blocks():
    rng = np.random.default_rng(3)
    for world in [1, 2, 3, 7]:
        kb = rng.integers(0, 8, size=50)
        cu = np.concatenate([[0], np.cumsum(kb + 1)]).astype(np.int32)
        R = int(cu[-1])
        prev = 0
        for rank in range(world):
            b_lo, b_hi, r_lo, r_hi = shard.request_shard(cu, world, rank)
            assert b_lo == prev and b_hi >= b_lo
            assert (r_lo, r_hi) == (cu[b_lo], cu[b_hi])
            assert r_hi - r_lo <= R // world + int((kb + 1).max()) + 1
            loc = shard.rebase(cu, b_lo, b_hi)
            assert loc[0] == 0 and loc[-1] == r_hi - r_lo
            prev = b_hi
        assert prev == 50
    with pytest.raises(ValueError):
        shard.request_shard(np.array([0, 2], np.int32), 2, 2)


def test_prefix_acceptance_ratio():
    np.testing.assert_allclose(shard.prefix_acceptance([3, 1, 0], [4, 2, 0]), [0.75, 0.5, 0.0])


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vb = W.ragged_batch(seed=11, B=13, k_max=5, V=777, dtype="f32")
    b_lo, b_hi, r_lo, r_hi = shard.request_shard(vb.cu_rows, world, rank)
    cu = shard.rebase(vb.cu_rows, b_lo, b_hi)
    ref = oracle.verify_greedy(vb.logits[r_lo:r_hi], vb.dtype, vb.V, b_hi - b_lo, vb.k_max, cu,
                               vb.draft_ids[r_lo:r_hi])
    acc, ver, hist, _ = oracle.prefix_stats(ref.accepted_len, cu, b_hi - b_lo, vb.k_max)
    acc_t, ver_t, hist_t = (torch.from_numpy(x.copy()) for x in (acc, ver, hist))
    shard.reduce_prefix_stats(acc_t, ver_t, hist_t)
    slow = shard.max_over_ranks(1.0 + rank)
    rows = shard.sum_over_ranks(float(r_hi - r_lo))
    np.savez(os.path.join(out_dir, "rank%d.npz" % rank), b=np.array([b_lo, b_hi]),
             accepted=ref.accepted_len, out=ref.out_tokens, acc=acc_t.numpy(), ver=ver_t.numpy(),
             hist=hist_t.numpy(), slow=np.array([slow]), rows=np.array([rows]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_requests_and_reduce_counters():
    import torch.multiprocessing as mp
    import oracle
    oracle.build()
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(world, _free_port(), d), nprocs=world,
                           start_method="spawn", join=True)
        res = [np.load(os.path.join(d, "rank%d.npz" % r)) for r in range(world)]
    vb = W.ragged_batch(seed=11, B=13, k_max=5, V=777, dtype="f32")
    whole = oracle.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                                 vb.draft_ids)
    acc, ver, hist, _ = oracle.prefix_stats(whole.accepted_len, vb.cu_rows, vb.B, vb.k_max)
    # verification needs no exchange: the shards' results are the batch's
    np.testing.assert_array_equal(np.concatenate([r["accepted"] for r in res]), whole.accepted_len)
    np.testing.assert_array_equal(np.concatenate([r["out"] for r in res]), whole.out_tokens)
    assert res[0]["b"][1] == res[1]["b"][0] and res[0]["b"][0] == 0 and res[1]["b"][1] == vb.B
    for r in res:
        # one sum all-reduce gives the job-wide counters on every rank
        np.testing.assert_array_equal(r["acc"], acc)
        np.testing.assert_array_equal(r["ver"], ver)
        np.testing.assert_array_equal(r["hist"], hist)
        # the job's time is its slowest rank's; units add up over ranks
        assert r["slow"][0] == 2.0
        assert r["rows"][0] == vb.R


def _ctl_rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    import speculative_decoding_verification_ragged_gb300 as sv
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(100 + rank)           # each rank its own requests
    K = 5
    ctl = sv.StepController(1, K, 3)
    k, ks, accs, vers, bs = 3, [], [], [], []
    for t in range(40):
        B_local = 12 + 5 * rank
        alpha = 0.9 if t < 20 else 0.3                # the acceptance collapses halfway
        a = np.minimum(rng.geometric(1 - alpha, size=B_local) - 1, k)
        acc = torch.tensor([(a > j).sum() for j in range(K)], dtype=torch.int64)
        ver = torch.tensor([B_local if j < k else 0 for j in range(K)], dtype=torch.int64)
        shard.reduce_prefix_stats(acc, ver)           # job-wide counters on every rank
        B = int(shard.sum_over_ranks(float(B_local)))
        cost = sv.step_cost_sps(B, K, [64, 128, 192, 256], [90.0, 70.0, 55.0, 45.0])
        k = sv.StepController.update(ctl, acc.numpy(), ver.numpy(), cost, B)
        ks.append(k); accs.append(acc.numpy()); vers.append(ver.numpy()); bs.append(B)
    np.savez(os.path.join(out_dir, "ctl%d.npz" % rank), ks=np.array(ks), acc=np.array(accs),
             ver=np.array(vers), B=np.array(bs))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_same_adaptive_step():
    import torch.multiprocessing as mp
    import speculative_decoding_verification_ragged_gb300 as sv
    from oracle.step_policy import StepController, step_cost_sps
    sv.build()
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_ctl_rank_main, args=(world, _free_port(), d), nprocs=world,
                           start_method="spawn", join=True)
        res = [np.load(os.path.join(d, "ctl%d.npz" % r)) for r in range(world)]
    np.testing.assert_array_equal(res[0]["ks"], res[1]["ks"])
    np.testing.assert_array_equal(res[0]["acc"], res[1]["acc"])
    # the oracle controller on the job-wide counters takes the same steps
    orc = StepController(1, 5, 3)
    ks = [orc.update(a, v, step_cost_sps(int(B), 5, [64, 128, 192, 256],
                                         [90.0, 70.0, 55.0, 45.0]), int(B))
          for a, v, B in zip(res[0]["acc"], res[0]["ver"], res[0]["B"])]
    np.testing.assert_array_equal(res[0]["ks"], np.array(ks))
    # high acceptance lengthens the step, the collapse shortens it again
    assert ks[3] == 3 and ks[19] == 5 and ks[-1] < 5
