"""The multi-rank paths on CPU ranks (gloo, world size 2), with real rank logic and no GPU.

Row replicas (what ``bench.py --gpus N`` runs): every rank draws its own seeded batch of rows
(``bench.rank_rows_seed``) and projects it against its own replica of W; nothing is exchanged
on the data path; the timing is the maximum over ranks and the value counts every rank's rows.

Vocabulary lanes (the record exchange of a vocabulary-sharded head, "SemBridge" Figure 1 and
Section 5.2: each lane ships its per-lane projection instead of its logit slice): rank r holds
the columns [r V/2, (r+1) V/2) of W, computes its shard-local record (max logit, lowest global
column attaining it, sum of exp(z - max)) per row with the oracle, packs it as the 12-byte
payload (float32 m, int32 column, float32 s), all-gathers the payloads over gloo and merges them
in ascending lane order; the merged token and logsumexp must equal the oracle's projection of
the complete vocabulary.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


M, D, V = 6, 64, 512


def _merge(a, b):
    """The record merge in fp64: larger max, lower column on an equal max, rescaled sums."""
    (ma, ia, sa), (mb, ib, sb) = a, b
    m = max(ma, mb)
    i = ia if ma > mb else (ib if mb > ma else min(ia, ib))
    s = (0.0 if ma == -math.inf else sa * math.exp(ma - m)) + \
        (0.0 if mb == -math.inf else sb * math.exp(mb - m))
    return m, i, s


def _payload(rec_m, rec_i, rec_s) -> torch.Tensor:
    """Lane payload: per row (float32 m, int32 global column, float32 s) = 12 bytes."""
    raw = np.empty((len(rec_m), 3), np.uint32)
    raw[:, 0] = np.asarray(rec_m, np.float32).view(np.uint32)
    raw[:, 1] = np.asarray(rec_i, np.int32).view(np.uint32)
    raw[:, 2] = np.asarray(rec_s, np.float32).view(np.uint32)
    return torch.from_numpy(raw.view(np.int32).copy())


def _unpack(t: torch.Tensor):
    raw = t.numpy().view(np.uint32)
    return (raw[:, 0].view(np.float32).astype(np.float64), raw[:, 1].view(np.int32),
            raw[:, 2].view(np.float32).astype(np.float64))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from gemm_epilogue_reduction_gb300 import synth

        # ---- row replicas: the rank's own batch against the shared W
        H0, W = synth.make_hw(M, D, V, seed=0)
        H = H0 if rank == 0 else synth.make_hw(M, D, 1, seed=bench.rank_rows_seed(rank))[0]
        Hb, Wb = synth.bf16_bits(H), synth.bf16_bits(W)
        rep = oracle.project(Hb, Wb, 1)
        toks = [torch.zeros(M, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(toks, torch.from_numpy(rep["token"].copy()))  # results, not data path
        hb = [torch.zeros(M, D, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(hb, torch.from_numpy(Hb.astype(np.int32)))  # bf16 bits, widened
        ms = [0.25, 0.31][rank]
        mx = bench.max_over_ranks(ms, "cpu")

        # ---- vocabulary lanes: this rank's slice of W, its records, the exchange, the merge
        S = V // world
        lane = oracle.project(synth.bf16_bits(H0), Wb[rank * S:(rank + 1) * S], 1)
        rec_m = lane["shard_max"][:, 0]
        rec_i = lane["shard_token"][:, 0] + rank * S
        rec_s = np.exp(lane["shard_lse"][:, 0] - rec_m)
        mine = _payload(rec_m, rec_i, rec_s)
        assert mine.numel() * 4 == 12 * M
        got = [torch.zeros_like(mine) for _ in range(world)]
        dist.all_gather(got, mine)
        lanes = [_unpack(t) for t in got]
        merged = []
        for r in range(M):
            acc = (-math.inf, 2 ** 31 - 1, 0.0)
            for lm, li, ls in lanes:  # ascending lane order
                acc = _merge(acc, (float(lm[r]), int(li[r]), float(ls[r])))
            merged.append((acc[1], acc[0] + math.log(acc[2])))
        q.put((rank, mx, bench.job_rows_per_s(world, M, mx), bench.rank_rows_seed(rank),
               [t.numpy() for t in toks], [t.numpy() for t in hb], merged))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas_and_vocabulary_lanes():
    import oracle
    from gemm_epilogue_reduction_gb300 import synth
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in range(2)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0

    # replicas: slowest rank's time, all rows counted, distinct batches, each rank's tokens
    # those of the oracle on that rank's rows
    assert [r[1] for r in res] == [0.31, 0.31]
    assert res[0][2] == pytest.approx(2 * M / 0.31e-3)
    assert res[0][3] != res[1][3]
    hb0, hb1 = res[0][5]
    assert not np.array_equal(hb0, hb1)
    H, W = synth.make_hw(M, D, V, seed=0)
    Wb = synth.bf16_bits(W)
    for rank in range(2):
        Hr = res[0][5][rank].astype(np.uint16)
        ref = oracle.project(Hr, Wb, 1)
        assert np.array_equal(res[0][4][rank], ref["token"])

    # vocabulary lanes: the merged payloads give the complete vocabulary's token and lse on
    # every rank
    full = oracle.project(synth.bf16_bits(H), Wb, 2)
    for rank in range(2):
        for r, (tok, lse) in enumerate(res[rank][6]):
            gap = full["key_top1"][r] - full["key_top2"][r]
            if gap > 1e-6:  # fp32 packing of the maxima cannot reorder a wider gap
                assert tok == full["token"][r]
            assert abs(lse - full["lse"][r]) < 1e-5
    assert res[0][6] == res[1][6]  # every rank merges to the same result


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(1.5, "cpu") == 1.5
    assert bench.job_rows_per_s(1, 16, 0.25) == pytest.approx(64000.0)
