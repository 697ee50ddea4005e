"""GPU parity of the row-parallel partial completion against the fp64 oracle (Section 6.4 of
the SemBridge pages: lane partials of a split reduction, completed by a sum)."""
import os

import numpy as np
import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
import oracle
from gemm_epilogue_reduction_gb300 import synth
from gpu_helpers import TOL, bf16_half_ulp

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(M, N, K, seed, device="cpu"):
    # X ~ N(0, 1), W ~ N(0, 1/K): outputs on an N(0, 1) scale
    X, W = synth.make_hw(M, K, N, seed=seed, device=device)
    return X.cuda(), W.cuda()


@pytest.mark.parametrize("M,N,K,lanes", [
    (1, 384, 1024, 2), (8, 1000, 2048, 2), (17, 300, 512, 4), (64, 640, 1280, 5),
    (200, 130, 640, 1), (256, 257, 768, 3),
    # several segments per CTA, and tiles summed in two row groups
    (32, 2048, 8192, 16),
    # one-block lanes: a tile of 512 slabs, summed in two batches through a running sum
    (4, 128, 32768, 512),
    # a single feature tile split over every CTA (152 slabs per tile on a 152-SM part)
    (64, 128, 17408, 2),
])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_partial_completion_parity(M, N, K, lanes, bf16_out):
    X, W = _inputs(M, N, K, seed=M + N)
    Y, ws = sb.partial_completion(X, W, lanes, out_bf16=bf16_out)
    torch.cuda.synchronize()
    ref = oracle.partial_completion(synth.bf16_bits(X), synth.bf16_bits(W), lanes)["Y"]
    got = Y.float().cpu().numpy().astype(np.float64)
    bound = TOL + (bf16_half_ulp(ref) if bf16_out else 0.0)
    assert np.all(np.abs(got - ref) <= bound), float(np.abs(got - ref).max())


def test_partial_completion_is_deterministic():
    """Same bits from a fresh workspace and from a reused one (whose per-tile arrival
    counters still hold the previous call's counts)."""
    X, W = _inputs(64, 512, 2048, seed=3)
    a, ws = sb.partial_completion(X, W, 2, out_bf16=False)
    b, _ = sb.partial_completion(X, W, 2, out_bf16=False)
    c, _ = sb.partial_completion(X, W, 2, out_bf16=False, workspace=ws)
    X2, W2 = _inputs(64, 5120, 17408, seed=4)
    d, ws2 = sb.partial_completion(X2, W2, 2, out_bf16=False)
    e, _ = sb.partial_completion(X2, W2, 2, out_bf16=False, workspace=ws2)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)
    assert torch.equal(d, e)


def _table3():
    rows = {}
    with open(os.path.join(GOLDEN, "mlp_slice_table3.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                t, l2, mx = line.split()
                rows[int(t)] = (float(l2), float(mx))
    return rows


@pytest.mark.parametrize("tokens", [1, 8, 64])
def test_mlp_down_projection_error_within_the_pages_table3(tokens):
    """Qwen3-14B-sized down projection (hidden 5120, intermediate 17408 split over 2 lanes)
    with bf16 output: relative L2 error against the fp64 oracle stays below the value the
    pages report for the same token count (Table 3)."""
    N, K, lanes = 5120, 17408, 2
    X, W = _inputs(tokens, N, K, seed=tokens, device="cuda")
    Y, ws = sb.partial_completion(X, W, lanes, out_bf16=True)
    torch.cuda.synchronize()
    ref = oracle.partial_completion(synth.bf16_bits(X), synth.bf16_bits(W), lanes)["Y"]
    got = Y.float().cpu().numpy().astype(np.float64)
    rel_l2 = 100.0 * np.linalg.norm(got - ref) / np.linalg.norm(ref)
    pages_l2, _ = _table3()[tokens]
    assert rel_l2 <= pages_l2, (rel_l2, pages_l2)
    assert np.all(np.abs(got - ref) <= TOL + bf16_half_ulp(ref))
