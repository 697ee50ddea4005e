"""Shared checks for the GPU parity tests: the CUDA path against the fp64 oracle.

Tolerances (numbers on the N(0, 1) logit scale of the synthetic inputs):
  * logsumexp, chosen and target log-probs: |gpu - oracle| <= 5e-3;
  * token: equal to the oracle's where the oracle's top-1 minus top-2 selection key exceeds
    1e-2, else a column whose oracle key lies within 1e-2 of the maximum;
  * bf16 logits: |gpu - z| <= 5e-3 + half a bf16 ulp of z (round-to-nearest of an fp32
    value within 5e-3 of z).
"""

import numpy as np
import torch

import gemm_epilogue_reduction_gb300 as sb
import oracle
from gemm_epilogue_reduction_gb300 import synth

TOL = 5e-3
GAP = 1e-2


def bf16_half_ulp(z: np.ndarray) -> np.ndarray:
    a = np.abs(z)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


def check_rows(res: dict, ref: dict, rows, *, gumbel=False, T=1.0, seed=0, V=None,
               check_targets=False):
    """Compare GPU outputs at `rows` with an oracle result computed for exactly those rows
    (ref must hold z, i.e. keep_z=True)."""
    tok = res["token"].cpu().numpy()[rows]
    z = ref["z"]
    V = z.shape[1] if V is None else V
    mism = 0
    for i, r in enumerate(rows):
        gap = ref["key_top1"][i] - ref["key_top2"][i]
        t = int(tok[i])
        assert 0 <= t < V, (r, t)
        if gap > GAP:
            assert t == ref["token"][i], (r, t, int(ref["token"][i]), gap)
        else:
            key = oracle.selection_key(z[i, t], r, t, V, gumbel, T, seed)
            assert key >= ref["key_top1"][i] - GAP, (r, t, key, ref["key_top1"][i])
            mism += int(t != ref["token"][i])
        if "lse" in res:
            assert abs(float(res["lse"][r]) - ref["lse"][i]) <= TOL, (r, "lse")
        if "token_logprob" in res:
            y_t = z[i, t] / T if gumbel else z[i, t]
            want = y_t - ref["lse"][i]
            assert abs(float(res["token_logprob"][r]) - want) <= TOL, (r, "logprob")
        if check_targets:
            assert abs(float(res["target_logprob"][r]) - ref["target_logprob"][i]) <= TOL, \
                (r, "target_logprob")
    return mism


def run_and_check(M, d, V, k, surface, *, seed=0, T=1.0, gseed=0, targets=False, rows=None,
                  device_inputs=False, HW=None):
    """Draw inputs, run the CUDA path through the C ABI, compare with the oracle."""
    if HW is None:
        dev = "cuda" if device_inputs else "cpu"
        H, W = synth.make_hw(M, d, V, seed=seed, device=dev)
        H, W = H.cuda(), W.cuda()
    else:
        H, W = HW
    tg = synth.make_targets(M, V, seed=1, device="cuda") if targets else None
    res = sb.project(H, W, k, surface, temperature=T, seed=gseed, targets=tg)
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(res["_outputs"]) == sb.SB_OK
    rows = list(range(M)) if rows is None else list(rows)
    Hb = synth.bf16_bits(H)[rows]
    Wb = synth.bf16_bits(W)
    ref = oracle.project(Hb, Wb, k, gumbel=surface == sb.SB_GUMBEL_TOKEN, temperature=T,
                         seed=gseed, targets=None if tg is None else tg.cpu().numpy()[rows],
                         row_ids=rows, keep_z=True)
    check_rows(res, ref, rows, gumbel=surface == sb.SB_GUMBEL_TOKEN, T=T, seed=gseed,
               check_targets=targets)
    if surface == sb.SB_FULL_LOGITS:
        lg = res["logits"].float().cpu().numpy()[rows].astype(np.float64)
        err = np.abs(lg - ref["z"])
        assert np.all(err <= TOL + bf16_half_ulp(ref["z"])), float(err.max())
    return res, ref, (H, W)
