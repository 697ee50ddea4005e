"""GPU parity of the top-K log-probability surface against the fp64 oracle.

Rule: position q of a row's list must hold a column whose oracle logit is within 1e-2 of the
oracle's q-th largest logit (exactly the oracle's column where that value is more than 1e-2
away from its neighbours in the sorted order); the K columns are distinct; each log-prob is
within 5e-3 of the oracle's z - lse for the column returned."""
import numpy as np
import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
import oracle
from gemm_epilogue_reduction_gb300 import synth
from gpu_helpers import GAP, TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def check_topk(res, H, W, K, rows=None):
    M = H.shape[0]
    rows = list(range(M)) if rows is None else list(rows)
    Hb, Wb = synth.bf16_bits(H)[rows], synth.bf16_bits(W)
    ref = oracle.topk(Hb, Wb, K)
    z = oracle.logits(Hb, Wb)
    ids = res["topk_ids"].cpu().numpy()[rows]
    lp = res["topk_logprob"].cpu().numpy()[rows].astype(np.float64)
    tok = res["token"].cpu().numpy()[rows]
    V = W.shape[0]
    for i in range(len(rows)):
        zr = z[i]
        srt = np.sort(zr)[::-1]
        assert len(set(ids[i].tolist())) == K
        assert ids[i].min() >= 0 and ids[i].max() < V
        for q in range(K):
            want = zr[ref["ids"][i, q]]
            assert abs(zr[ids[i, q]] - want) <= GAP, (rows[i], q)
            lo = srt[q + 1] if q + 1 < V else -np.inf
            hi = srt[q - 1] if q > 0 else np.inf
            if want - lo > GAP and hi - want > GAP:
                assert ids[i, q] == ref["ids"][i, q], (rows[i], q)
            assert abs(lp[i, q] - (zr[ids[i, q]] - ref["lse"][i])) <= TOL, (rows[i], q)
        assert tok[i] == ids[i, 0]
        assert abs(float(res["lse"][rows[i]]) - ref["lse"][i]) <= TOL


@pytest.mark.parametrize("M,d,V,k,K", [
    (16, 256, 4096, 4, 5),     # vocab mode
    (3, 64, 1000, 1, 16),
    (100, 128, 3000, 3, 8),
    (5, 64, 21, 7, 3),         # S = 3: shard lists shorter than useful
    (300, 64, 2000, 2, 16),    # rows mode, 2-CTA clusters
    (129, 64, 1024, 4, 1),
    (257, 72, 1500, 3, 7),
])
def test_topk_parity(M, d, V, k, K):
    H, W = synth.make_hw(M, d, V, seed=M + K)
    H, W = H.cuda(), W.cuda()
    res = sb.project(H, W, k, sb.SB_TOPK_LOGPROB, topk=K)
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(res["_outputs"]) == sb.SB_OK
    check_topk(res, H, W, K)


@pytest.mark.parametrize("M", [4, 300])
def test_topk_ties_list_lower_columns_first(M):
    """Duplicated W rows give bit-identical logits in different tiles and shards: the list
    holds them in ascending column order."""
    d, V, k, K = 64, 2048, 4, 4
    H, W = synth.make_hw(M, d, V, seed=3)
    W = W.clone()
    W[1500] = (H[0].float() * 6.0 / d).to(torch.bfloat16)
    W = synth.duplicate_rows(W, [(1500, 700), (1500, 701), (1500, 1999)])
    res = sb.project(H.cuda(), W.cuda(), k, sb.SB_TOPK_LOGPROB, topk=K)
    torch.cuda.synchronize()
    assert res["topk_ids"][0].tolist() == [700, 701, 1500, 1999]
    lp = res["topk_logprob"][0]
    assert bool((lp == lp[0]).all())


@pytest.mark.parametrize("M,k", [(4, 4), (300, 2)])
def test_topk_more_ties_than_k_keep_the_lowest_columns(M, k):
    """Six bit-identical maxima in five records and up to four shards, K = 4: the list is the
    four lowest columns (the combine ranks records by maximum, then by record number, which
    is column order)."""
    d, V, K = 64, 2048, 4
    H, W = synth.make_hw(M, d, V, seed=4)
    W = W.clone()
    W[1500] = (H[0].float() * 6.0 / d).to(torch.bfloat16)
    W = synth.duplicate_rows(W, [(1500, c) for c in (1999, 701, 700, 300, 100)])
    res = sb.project(H.cuda(), W.cuda(), k, sb.SB_TOPK_LOGPROB, topk=K)
    torch.cuda.synchronize()
    assert res["topk_ids"][0].tolist() == [100, 300, 700, 701]
    assert int(res["token"][0]) == 100


def test_topk_decode_shape():
    """The decode token-only shape (M=16, d=5120, V=151936, k=4) with K = 8."""
    M, d, V, k, K = 16, 5120, 151936, 4, 8
    H, W = synth.make_hw(M, d, V, seed=0, device="cuda")
    res = sb.project(H, W, k, sb.SB_TOPK_LOGPROB, topk=K)
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(res["_outputs"]) == sb.SB_OK
    check_topk(res, H, W, K)


def test_topk_sampling_batch_shape():
    """The 256-row batch shape (rows mode, CTA pairs, 8-entry lists) with K = 8; rows from
    both M tiles of the pair, checked against the oracle."""
    M, d, V, k, K = 256, 5120, 151936, 4, 8
    H, W = synth.make_hw(M, d, V, seed=0, device="cuda")
    res = sb.project(H, W, k, sb.SB_TOPK_LOGPROB, topk=K)
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(res["_outputs"]) == sb.SB_OK
    check_topk(res, H, W, K, rows=[0, 77, 128, 255])


@pytest.mark.parametrize("M,d,V,k", [(16, 256, 4096, 4), (300, 64, 2000, 2)])
def test_topk_surface_token_and_lse_bits_equal_the_token_surface(M, d, V, k):
    """The top-K combine completes lse and the token with the same fixed tree as the token
    surface, so those outputs agree bit for bit."""
    H, W = synth.make_hw(M, d, V, seed=31)
    H, W = H.cuda(), W.cuda()
    a = sb.project(H, W, k, sb.SB_TOPK_LOGPROB, topk=6)
    b = sb.project(H, W, k, sb.SB_TOKEN_LOGPROB)
    torch.cuda.synchronize()
    for key in ("token", "token_logprob", "lse"):
        assert torch.equal(a[key], b[key]), key
