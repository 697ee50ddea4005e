"""A seeded sweep of random problem shapes through every surface, against the fp64 oracle.

The shapes are drawn once from a fixed generator (so the list is the same on every run) over
the ranges the validation accepts: 1 to 400 rows (both tilings and the boundary at 128),
d a multiple of 8 from 8 to 776, 1 to 9 lane shards of 1 to 3000 columns (ragged last
tiles, shards narrower than a tile), with and without scoring targets.  Each shape runs one
surface; the checks are those of the other parity tests (tokens by the candidate rule,
log-probs and lse within 5e-3, bf16 logits within 5e-3 plus half an ulp, top-K lists by
rank)."""
import numpy as np
import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
from gemm_epilogue_reduction_gb300 import synth
from gpu_helpers import run_and_check

pytestmark = pytest.mark.gpu

SURFACES = [sb.SB_TOKEN, sb.SB_TOKEN_LOGPROB, sb.SB_FULL_LOGITS, sb.SB_GUMBEL_TOKEN,
            sb.SB_TOPK_LOGPROB]


def _draw(n=30, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        M = int(rng.choice([int(rng.integers(1, 129)), int(rng.integers(129, 401))]))
        d = 8 * int(rng.integers(1, 98))
        k = int(rng.integers(1, 10))
        S = int(rng.integers(1, 3001))
        surface = SURFACES[i % len(SURFACES)]
        targets = bool(rng.integers(0, 2))
        cases.append((M, d, k * S, k, surface, targets, int(rng.integers(0, 2 ** 31))))
    return cases


CASES = _draw()


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("M,d,V,k,surface,targets,seed", CASES)
def test_random_shape(M, d, V, k, surface, targets, seed):
    if surface == sb.SB_TOPK_LOGPROB:
        from test_topk import check_topk
        K = min(1 + seed % 16, V)
        H, W = synth.make_hw(M, d, V, seed=seed % 1000)
        H, W = H.cuda(), W.cuda()
        res = sb.project(H, W, k, sb.SB_TOPK_LOGPROB, topk=K)
        torch.cuda.synchronize()
        assert sb.sb_last_device_status(res["_outputs"]) == sb.SB_OK
        rows = sorted({0, M - 1, M // 2})
        check_topk(res, H, W, K, rows=rows)
        return
    T = 0.5 + (seed % 100) / 50.0 if surface == sb.SB_GUMBEL_TOKEN else 1.0
    run_and_check(M, d, V, k, surface, seed=seed % 1000, T=T, gseed=seed, targets=targets)
