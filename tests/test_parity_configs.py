"""GPU parity at the five workload sizes, in the launch configuration the benchmark times.

Each workload draws its inputs on the GPU (seed 0; targets seed 1) and runs the projection
once through the C ABI.  Rows the fp64 oracle can afford are compared element by element
(every row of the two decode shapes and of the 256-row sampling batch; a fixed sample spread
over the M tiles for prefill scoring); every row is also checked against torch's fp32 matmul
+ logsumexp (a library routine, used here as a second reference that scales to every row),
including the target log-prob of each of the 4096 prefill rows.
"""
import numpy as np
import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
import oracle
from gemm_epilogue_reduction_gb300 import synth
from gpu_helpers import GAP, TOL, bf16_half_ulp, check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _library_reference_check(H, W, res, *, T=1.0, lse_only=False, targets=None):
    """All rows: tokens, logsumexp and (given targets) the target log-prob against torch
    fp32 (tf32 off) on the GPU."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        Wf = W.float()
        for r0 in range(0, H.shape[0], 512):
            z = H[r0:r0 + 512].float() @ Wf.T
            y = z / T
            lse = torch.logsumexp(y, dim=1)
            assert float((res["lse"][r0:r0 + 512] - lse).abs().max()) <= TOL
            if targets is not None:
                tl = z.gather(1, targets[r0:r0 + 512].long()[:, None])[:, 0] - lse
                assert float((res["target_logprob"][r0:r0 + 512] - tl).abs().max()) <= TOL
            if lse_only:
                continue
            top2 = torch.topk(z, 2, dim=1).values
            tok = res["token"][r0:r0 + 512].long()
            zt = z.gather(1, tok[:, None])[:, 0]
            # within the tie band the token must be a near-maximum; outside it, the maximum
            assert bool((zt >= top2[:, 0] - GAP).all())
            safe = (top2[:, 0] - top2[:, 1]) > 2 * GAP
            assert bool((zt[safe] == top2[safe, 0]).all())
            del z, y
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def _oracle(H, W, k, rows, **kw):
    return oracle.project(synth.bf16_bits(H)[rows], synth.bf16_bits(W), k, row_ids=rows,
                          keep_z=True, **kw)


def test_decode16_token_logprob():
    """M=16, d=5120, V=151936, k=4 (S=37984): TOKEN + chosen log-prob, every row."""
    M, d, V, k = 16, 5120, 151936, 4
    H, W = synth.make_hw(M, d, V, seed=0, device="cuda")
    res = sb.project(H, W, k, sb.SB_TOKEN_LOGPROB)
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(res["_outputs"]) == sb.SB_OK
    rows = list(range(M))
    check_rows(res, _oracle(H, W, k, rows), rows)
    _library_reference_check(H, W, res)


def test_decode64_full_logits_vs_token():
    """M=64, d=4096, V=151936, k=2: FULL_LOGITS and TOKEN on the same inputs give the same
    tokens; the bf16 logits, lse and log-probs match the oracle on every row."""
    M, d, V, k = 64, 4096, 151936, 2
    H, W = synth.make_hw(M, d, V, seed=0, device="cuda")
    full = sb.project(H, W, k, sb.SB_FULL_LOGITS)
    tok = sb.project(H, W, k, sb.SB_TOKEN)
    torch.cuda.synchronize()
    assert torch.equal(full["token"], tok["token"])
    rows = list(range(M))
    ref = _oracle(H, W, k, rows)
    check_rows(full, ref, rows)
    lg = full["logits"].float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref["z"]) <= TOL + bf16_half_ulp(ref["z"]))
    _library_reference_check(H, W, full)


def test_prefill_scoring_lse_and_target_logprob():
    """M=4096, d=6144, V=200064, k=4 (S=50016): lse + target log-prob, no logits written.
    Oracle on 12 rows spread over the M tiles (first, last, tile edges); torch on all rows,
    target log-probs included."""
    M, d, V, k = 4096, 6144, 200064, 4
    H, W = synth.make_hw(M, d, V, seed=0, device="cuda")
    tg = synth.make_targets(M, V, seed=1, device="cuda")
    res = sb.project(H, W, k, sb.SB_TOKEN_LOGPROB, targets=tg)
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(res["_outputs"]) == sb.SB_OK
    rows = [0, 1, 127, 128, 255, 1000, 2047, 2048, 3001, 3967, 4094, 4095]
    ref = _oracle(H, W, k, rows, targets=tg.cpu().numpy()[rows])
    check_rows(res, ref, rows, check_targets=True)
    _library_reference_check(H, W, res, targets=tg)


def test_sampling_gumbel_token():
    """M=256, d=5120, V=151936, k=4: GUMBEL_TOKEN at T=0.7 with seed 1234; the oracle on
    every row (tokens by the candidate rule on the Gumbel key, tempered lse and log-prob)."""
    M, d, V, k, T, seed = 256, 5120, 151936, 4, 0.7, 1234
    H, W = synth.make_hw(M, d, V, seed=0, device="cuda")
    res = sb.project(H, W, k, sb.SB_GUMBEL_TOKEN, temperature=T, seed=seed)
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(res["_outputs"]) == sb.SB_OK
    rows = list(range(M))
    ref = _oracle(H, W, k, rows, gumbel=True, temperature=np.float32(T).item(), seed=seed)
    check_rows(res, ref, rows, gumbel=True, T=np.float32(T).item(), seed=seed)
    _library_reference_check(H, W, res, T=np.float32(T).item(), lse_only=True)


def test_rows_mode_full_logits_at_the_sampling_shape():
    """M=256, d=5120, V=151936, k=4, FULL_LOGITS (rows mode: CTA pairs, each thread storing
    whole 32-byte sectors of its row): every bf16 logit within the tolerance plus half a bf16
    ulp of torch's fp32 product, the tokens those of TOKEN on the same inputs, and 32 rows
    spread over the batch against the oracle element by element."""
    M, d, V, k = 256, 5120, 151936, 4
    H, W = synth.make_hw(M, d, V, seed=0, device="cuda")
    full = sb.project(H, W, k, sb.SB_FULL_LOGITS)
    tok = sb.project(H, W, k, sb.SB_TOKEN)
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(full["_outputs"]) == sb.SB_OK
    assert torch.equal(full["token"], tok["token"])
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        z = H.float() @ W.float().T
        lg = full["logits"].float()
        half_ulp = torch.exp2(torch.floor(torch.log2(z.abs().clamp_min(2.0 ** -126))) - 8)
        assert bool(((lg - z).abs() <= TOL + half_ulp).all())
        del z, lg
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    rows = list(range(0, M, 8))
    ref = _oracle(H, W, k, rows)
    check_rows(full, ref, rows)
    lg = full["logits"][rows].float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref["z"]) <= TOL + bf16_half_ulp(ref["z"]))
    _library_reference_check(H, W, full)
