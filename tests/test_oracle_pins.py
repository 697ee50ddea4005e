"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test checks the oracle against exact arithmetic, a closed form, a library routine, a
value printed by the SemBridge pages or a published generator, or an invariant the pages
state. The plausible mistakes each one catches are listed in its docstring. These tests
run on the CPU only.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from gemm_epilogue_reduction_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GAMMA = 0x9E3779B97F4A7C15


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _exact(bits: int) -> Fraction:
    """Exact value of a bf16 bit pattern, decoded by hand (sign, exponent, mantissa)."""
    s = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    assert e != 0xFF
    if e == 0:
        return s * Fraction(m, 128) * Fraction(2) ** -126
    return s * (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)


def _tiny(M, d, V, seed):
    H, W = synth.make_hw(M, d, V, seed=seed)
    return synth.bf16_bits(H), synth.bf16_bits(W)


def _exact_logits(Hb, Wb):
    M, d = Hb.shape
    V = Wb.shape[0]
    He = [[_exact(int(x)) for x in row] for row in Hb]
    We = [[_exact(int(x)) for x in row] for row in Wb]
    return [[sum(He[r][i] * We[j][i] for i in range(d)) for j in range(V)] for r in range(M)]


def test_bf16_widening_exact():
    """Widening must be exact: catches a truncation or a wrong shift in the bit decoding."""
    for bits in [0x0000, 0x3F80, 0xBF80, 0xC000, 0x0001, 0x0080, 0x7F7F, 0x3E20, 0x4049]:
        assert Fraction(oracle.bf16_to_double(bits)) == _exact(bits)


def test_logits_exact_bruteforce():
    """fp64 z equals the exact rational sum to within the fp64 summation bound.

    Catches a dropped term, a wrong index, a transposed operand or a sign error in the
    contraction (Section 5.2: the output head materialises full logits)."""
    Hb, Wb = _tiny(3, 24, 37, seed=11)
    Z = oracle.logits(Hb, Wb)
    Ze = _exact_logits(Hb, Wb)
    d = Hb.shape[1]
    for r in range(3):
        for j in range(37):
            absum = sum(abs(_exact(int(Hb[r, i])) * _exact(int(Wb[j, i]))) for i in range(d))
            bound = float(absum) * d * 2.0 ** -52 + 1e-300
            assert abs(Fraction(Z[r, j]) - Ze[r][j]) <= Fraction(bound)


def _softmax_stats(y):
    m = max(y)
    s = math.fsum(math.exp(v - m) for v in y)
    return m + math.log(s)


@pytest.mark.parametrize("k", [1, 2, 3])
def test_projection_bruteforce(k):
    """Token, logsumexp, chosen and target log-probs and per-shard outputs against a
    brute-force evaluation on exact logits (Section 2.2 surfaces; Section 3.1 tie rule).

    Catches a wrong shard boundary, a wrong tie direction, a log-prob taken at the wrong
    index or a logsumexp that drops the max shift."""
    M, d, V = 5, 16, 48
    Hb, Wb = _tiny(M, d, V, seed=3)
    targets = np.array([0, 47, 13, 24, 5], dtype=np.int32)
    out = oracle.project(Hb, Wb, k, targets=targets)
    Ze = _exact_logits(Hb, Wb)
    S = V // k
    for r in range(M):
        z = Ze[r]
        zmax = max(z)
        tok = min(j for j in range(V) if z[j] == zmax)
        zf = [float(v) for v in z]
        lse = _softmax_stats(zf)
        assert out["token"][r] == tok
        assert abs(out["lse"][r] - lse) < 1e-12
        assert abs(out["logprob"][r] - (zf[tok] - lse)) < 1e-12
        assert abs(out["target_logprob"][r] - (zf[targets[r]] - lse)) < 1e-12
        others = sorted(zf[:tok] + zf[tok + 1:])
        assert abs(out["key_top1"][r] - zf[tok]) < 1e-15
        assert abs(out["key_top2"][r] - others[-1]) < 1e-15
        for s in range(k):
            seg = z[s * S:(s + 1) * S]
            smax = max(seg)
            stok = s * S + min(j for j in range(S) if seg[j] == smax)
            assert out["shard_token"][r, s] == stok
            assert abs(out["shard_max"][r, s] - float(smax)) < 1e-15
            assert abs(out["shard_lse"][r, s] - _softmax_stats([float(v) for v in seg])) < 1e-12


def test_ties_resolve_to_lowest_global_index():
    """Exact duplicate maxima within a shard and across shards pick the lowest index
    (the deterministic tie-breaking the registered projection carries, Section 3.1).

    Catches '>=' in place of '>' and a tie broken toward the later shard."""
    M, d, V, k = 2, 32, 64, 4
    H, W = synth.make_hw(M, d, V, seed=5)
    # make a strong maximum in row 0 at columns 40 and 9 (different shards: S = 16),
    # and in row 1 at columns 21 and 22 (same shard)
    W = W.clone()
    W[40] = (H[0].float() * 4.0 / d).to(torch.bfloat16)
    W = synth.duplicate_rows(W, [(40, 9), (40, 57)])
    W[22] = (H[1].float() * 4.0 / d).to(torch.bfloat16)
    W = synth.duplicate_rows(W, [(22, 21)])
    out = oracle.project(synth.bf16_bits(H), synth.bf16_bits(W), k, keep_z=True)
    assert out["z"][0, 9] == out["z"][0, 40] == out["z"][0, 57] == out["z"][0].max()
    assert out["token"][0] == 9
    assert out["key_top1"][0] == out["key_top2"][0]
    assert list(out["shard_token"][0]) == [9, int(np.argmax(out["z"][0, 16:32])) + 16,
                                          40, 57]
    assert out["token"][1] == 21


def test_zero_hidden_state_closed_form():
    """H = 0 gives z = 0 everywhere: token 0, lse = log V, logprob = -log V, shard lse =
    log S. Catches an off-by-one in the normaliser or a shard size taken as V."""
    V, k, d = 96, 3, 16
    Hb = np.zeros((2, d), np.uint16)
    _, Wb = _tiny(1, d, V, seed=2)
    out = oracle.project(Hb, Wb, k)
    assert list(out["token"]) == [0, 0]
    assert np.allclose(out["lse"], math.log(V), atol=1e-14, rtol=0)
    assert np.allclose(out["logprob"], -math.log(V), atol=1e-14, rtol=0)
    assert np.allclose(out["shard_lse"], math.log(V // k), atol=1e-14, rtol=0)
    assert [list(r) for r in out["shard_token"]] == [[0, 32, 64]] * 2


def test_unit_hidden_vector_selects_a_weight_column():
    """H = e_i gives z_j = W[j, i]: the token is numpy's first argmax of that column.
    Catches a transposed operand (H Wᵀ vs W Hᵀ or indexing W by column)."""
    d, V = 24, 200
    _, Wb = _tiny(1, d, V, seed=8)
    Hb = np.zeros((3, d), np.uint16)
    cols = [0, 7, 23]
    for r, i in enumerate(cols):
        Hb[r, i] = 0x3F80  # bf16 1.0
    out = oracle.project(Hb, Wb, 1, keep_z=True)
    Wf = np.array([[oracle.bf16_to_double(int(x)) for x in row] for row in Wb])
    for r, i in enumerate(cols):
        assert np.array_equal(out["z"][r], Wf[:, i])
        assert out["token"][r] == int(np.argmax(Wf[:, i]))


def test_two_column_vocabulary_closed_form():
    """V = 2: lse = log(e^a + e^b) and the chosen log-prob is -log(1 + e^-|a-b|)."""
    d = 8
    Hb, Wb = _tiny(4, d, 2, seed=21)
    out = oracle.project(Hb, Wb, 2, keep_z=True)
    for r in range(4):
        a, b = out["z"][r]
        assert abs(out["lse"][r] - math.log(math.exp(a) + math.exp(b))) < 1e-12
        assert abs(out["logprob"][r] + math.log1p(math.exp(-abs(a - b)))) < 1e-12
        assert out["token"][r] == (0 if a >= b else 1)


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_shard_merge_identities(k):
    """Figure 1 (R0 and P0 expose the same token) and the logsumexp split identity:
    argmax over the row = merge of the k shard argmaxes (lowest index on ties);
    lse(row) = log sum_s exp(lse_s). Catches a shard range that skips or repeats columns."""
    M, d, V = 6, 64, 3000
    Hb, Wb = _tiny(M, d, V, seed=4)
    out = oracle.project(Hb, Wb, k)
    for r in range(M):
        best = 0
        for s in range(1, k):
            if out["shard_max"][r, s] > out["shard_max"][r, best]:
                best = s
        assert out["token"][r] == out["shard_token"][r, best]
        ls = out["shard_lse"][r]
        m = ls.max()
        assert abs(out["lse"][r] - (m + math.log(np.exp(ls - m).sum()))) < 1e-12


def test_normalisation_and_bounds():
    """sum_j exp(z_j - lse) = 1 and -log V <= logprob(argmax) <= 0."""
    M, d, V = 4, 32, 1000
    Hb, Wb = _tiny(M, d, V, seed=6)
    out = oracle.project(Hb, Wb, 2, keep_z=True)
    for r in range(M):
        assert abs(math.fsum(np.exp(out["z"][r] - out["lse"][r])) - 1.0) < 1e-12
        assert -math.log(V) - 1e-12 <= out["logprob"][r] <= 0.0


def test_logits_match_numpy_matmul():
    """The contraction against numpy's fp64 matmul (a library routine) on a mid-size case."""
    Hb, Wb = _tiny(9, 136, 517, seed=9)
    Z = oracle.logits(Hb, Wb)
    Hf = np.array([[oracle.bf16_to_double(int(x)) for x in row] for row in Hb])
    Wf = (Wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = Hf @ Wf.T
    scale = np.abs(Hf) @ np.abs(Wf).T
    assert np.all(np.abs(Z - ref) <= 1e-13 * scale + 1e-300)


def test_splitmix64_published_outputs():
    """The counter form reproduces the published SplitMix64 stream for seed 0, and the
    seed enters additively in units of the golden-ratio increment (seed = GAMMA shifts the
    stream by one draw). Catches a wrong constant, a wrong shift or an n vs n+1 offset."""
    for n, hx in _read_golden("splitmix64_seed0.txt"):
        assert oracle.splitmix64(0, int(n)) == int(hx, 16)
    assert oracle.splitmix64(GAMMA, 0) == oracle.splitmix64(0, 1)
    assert oracle.splitmix64(2 * GAMMA % 2**64, 0) == oracle.splitmix64(0, 2)


def test_uniform24_grid_and_uniformity():
    """u is the top 24 bits scaled by 2^-24 and is uniform on [0, 1) (chi-square over 64
    bins of 2^16 draws)."""
    seed = 1234
    for n in [0, 1, 5, 2**40 + 3]:
        u = oracle.uniform24(seed, n)
        assert u == (oracle.splitmix64(seed, n) >> 40) / 2.0**24
        assert 0.0 <= u < 1.0
    N, B = 1 << 16, 64
    counts = np.zeros(B)
    for n in range(N):
        counts[int(oracle.uniform24(seed, n) * B)] += 1
    chi2 = ((counts - N / B) ** 2 / (N / B)).sum()
    assert chi2 < 130.0  # 63 degrees of freedom: p < 1e-6 above this


def test_gumbel_noise_moments():
    """-log(-log u) is standard Gumbel: mean = Euler-Mascheroni constant, variance = pi^2/6.
    Catches a sign error or log(-log u) in place of -log(-log u)."""
    N = 200000
    g = np.array([oracle.gumbel(77, n) for n in range(N)])
    assert abs(g.mean() - 0.5772156649) < 0.02
    assert abs(g.var() - math.pi ** 2 / 6) < 0.05
    u0 = (0xE220A8397B1DCDAF >> 40) / 2.0 ** 24  # published first output for seed 0
    assert oracle.gumbel(0, 0) == -math.log(-math.log(u0))


def test_gumbel_max_samples_softmax_of_tempered_logits():
    """Textbook Gumbel-max identity: argmax(z/T + g) is distributed as softmax(z/T).
    20000 rows share one hidden state, so each row is an independent draw (the stream index
    depends on the row). Catches z*T in place of z/T or noise drawn per row instead of per
    (row, column)."""
    d, V, T = 8, 6, 0.7
    zvals = [0.0, 0.5, 1.0, 1.5, -1.0, 2.0]  # exactly representable in bf16
    Wb = np.zeros((V, d), np.uint16)
    for j, v in enumerate(zvals):
        Wb[j, 0] = synth.bf16_bits(torch.tensor([v], dtype=torch.bfloat16))[0]
    N = 20000
    Hb = np.zeros((N, d), np.uint16)
    Hb[:, 0] = 0x3F80
    out = oracle.project(Hb, Wb, 2, gumbel=True, temperature=T, seed=1234)
    counts = np.bincount(out["token"], minlength=V).astype(float)
    p = np.exp(np.array(zvals) / T)
    p /= p.sum()
    chi2 = ((counts - N * p) ** 2 / (N * p)).sum()
    assert chi2 < 30.0  # 5 degrees of freedom: p < 2e-5 above this
    # the chosen log-prob is under the tempered distribution
    lse_T = math.log(np.exp(np.array(zvals) / T).sum())
    assert np.allclose(out["lse"], lse_T, atol=1e-12)
    assert np.allclose(out["logprob"], np.array(zvals)[out["token"]] / T - lse_T, atol=1e-12)


def test_gumbel_key_uses_global_row_and_column():
    """The draw for (row, col) sits at stream index row * V + col, with the row's global
    index (a subset of rows passed with row_ids gets the same keys)."""
    M, d, V = 4, 16, 40
    Hb, Wb = _tiny(M, d, V, seed=12)
    full = oracle.project(Hb, Wb, 2, gumbel=True, temperature=0.7, seed=99, keep_z=True)
    sub = oracle.project(Hb[2:3], Wb, 2, gumbel=True, temperature=0.7, seed=99,
                         row_ids=[2])
    assert sub["token"][0] == full["token"][2]
    r, j = 2, int(full["token"][2])
    key = oracle.selection_key(full["z"][r, j], r, j, V, True, 0.7, 99)
    assert key == full["key_top1"][r]
    u = (oracle.splitmix64(99, r * V + j) >> 40) / 2.0 ** 24
    assert abs(key - (full["z"][r, j] / 0.7 - math.log(-math.log(u)))) < 1e-12


def test_payload_closed_form_against_pages():
    """Token surface: 4 B per row instead of 2 V B of bf16 logits, so the reduction is
    1 - 2/V, which must exceed the pages' 'more than 99.97%' at both vocabularies used here;
    the pages' own R0/P0 byte counts give their printed 12,506x ratio."""
    g = {r[0]: float(r[1]) for r in _read_golden("payload_pages.txt")}
    for V in (151936, 200064):
        red = 1.0 - oracle.payload_bytes_per_row(0, V) / oracle.payload_bytes_per_row(2, V)
        assert abs(red - (1.0 - 2.0 / V)) < 1e-15
        assert red > g["min_traffic_reduction"]
    assert round(g["r0_bytes_per_step"] / g["p0_bytes_per_step"]) == g["p0_ratio"]


def test_payload_token_and_token_logprob_sizes():
    """Token surface: Figure 2(b)'s 256 B per decode step are four lane frames of 16 rows
    (concurrency 16), one int32 token per row in each, so 4 B per row.  Token + chosen
    log-prob adds one fp32 per row: int32 + float32 = 8 B, a reduction of 1 - 4/V against
    bf16 logits, still above the pages' 'more than 99.97%' at both vocabularies."""
    g = {r[0]: float(r[1]) for r in _read_golden("payload_pages.txt")}
    assert oracle.payload_bytes_per_row(0, 151936) == g["p0_bytes_per_step"] / (4 * 16)
    want = np.dtype(np.int32).itemsize + np.dtype(np.float32).itemsize
    for V in (4096, 151936, 200064):
        assert oracle.payload_bytes_per_row(1, V) == want == 8
        red = 1.0 - oracle.payload_bytes_per_row(1, V) / oracle.payload_bytes_per_row(2, V)
        assert abs(red - (1.0 - 4.0 / V)) < 1e-15
        if V > 4096:
            assert red > g["min_traffic_reduction"]
    assert np.isnan(oracle.payload_bytes_per_row(3, 151936))


# ---------------------------------------------------------------- top-K log-prob surface
@pytest.mark.parametrize("K", [1, 3, 7])
def test_topk_bruteforce_on_exact_logits(K):
    """Top-K ids and log-probs against a brute-force sort of exact rational logits by
    (value descending, column ascending). Catches a wrong tie direction, an off-by-one in
    the selection or a log-prob relative to the wrong normaliser."""
    M, d, V = 4, 16, 40
    Hb, Wb = _tiny(M, d, V, seed=17)
    out = oracle.topk(Hb, Wb, K)
    Ze = _exact_logits(Hb, Wb)
    for r in range(M):
        order = sorted(range(V), key=lambda j: (-Ze[r][j], j))[:K]
        assert list(out["ids"][r]) == order
        lse = _softmax_stats([float(v) for v in Ze[r]])
        assert abs(out["lse"][r] - lse) < 1e-12
        for q, j in enumerate(order):
            assert abs(out["logprob"][r, q] - (float(Ze[r][j]) - lse)) < 1e-12


def test_topk_ties_and_equal_logits():
    """All-equal logits (H = 0) give ids 0..K-1 and log-prob -log V each; duplicated W rows
    give equal logits listed by ascending column."""
    V, d, K = 50, 8, 5
    Hb = np.zeros((1, d), np.uint16)
    _, Wb = _tiny(1, d, V, seed=1)
    out = oracle.topk(Hb, Wb, K)
    assert list(out["ids"][0]) == [0, 1, 2, 3, 4]
    assert np.allclose(out["logprob"][0], -math.log(V), atol=1e-14)
    H, W = synth.make_hw(1, 32, 64, seed=2)
    W = W.clone()
    W[30] = (H[0].float() * 5.0 / 32).to(torch.bfloat16)
    W = synth.duplicate_rows(W, [(30, 3), (30, 63)])
    out = oracle.topk(synth.bf16_bits(H), synth.bf16_bits(W), 4)
    assert list(out["ids"][0][:3]) == [3, 30, 63]


def test_topk_matches_numpy_stable_argsort():
    """Against numpy's stable argsort of -z (a library routine) on a mid-size case, and the
    K = 1 entry against the deterministic token surface."""
    M, d, V, K = 6, 64, 3000, 16
    Hb, Wb = _tiny(M, d, V, seed=23)
    out = oracle.topk(Hb, Wb, K)
    Z = oracle.logits(Hb, Wb)
    ref = np.argsort(-Z, axis=1, kind="stable")[:, :K]
    assert np.array_equal(out["ids"], ref)
    proj = oracle.project(Hb, Wb, 3)
    assert np.array_equal(out["ids"][:, 0], proj["token"])
    assert np.allclose(out["logprob"][:, 0], proj["logprob"], atol=1e-13)
    with pytest.raises(ValueError):
        oracle.topk(Hb, Wb, V + 1)


# ---------------------------------------------------------------- partial completion
@pytest.mark.parametrize("lanes", [1, 2, 4])
def test_partial_completion_bruteforce(lanes):
    """Lane partials and their sum against exact rational products (Section 6.4: each lane
    sums its own slice of the reduction dimension; the completion adds the lanes).
    Catches a lane slice that overlaps or skips columns and a dropped lane."""
    M, N, K = 3, 5, 16
    Xb, Wb = _tiny(M, K, N, seed=44)
    out = oracle.partial_completion(Xb, Wb, lanes, keep_partials=True)
    Kl = K // lanes
    for m in range(M):
        for n in range(N):
            parts = [sum(_exact(int(Xb[m, i])) * _exact(int(Wb[n, i]))
                         for i in range(l * Kl, (l + 1) * Kl)) for l in range(lanes)]
            for l in range(lanes):
                assert abs(Fraction(out["P"][l, m, n]) - parts[l]) <= Fraction(1, 2 ** 45)
            assert abs(Fraction(out["Y"][m, n]) - sum(parts)) <= Fraction(1, 2 ** 44)


def test_partial_completion_equals_the_complete_product():
    """Completing the partials gives the complete product (numpy fp64 matmul, a library
    routine), and one lane is exactly the complete product's own summation."""
    M, N, K = 7, 33, 256
    Xb, Wb = _tiny(M, K, N, seed=45)
    Xf = (Xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Wf = (Wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = Xf @ Wf.T
    scale = np.abs(Xf) @ np.abs(Wf).T
    for lanes in (1, 2, 8):
        Y = oracle.partial_completion(Xb, Wb, lanes)["Y"]
        assert np.all(np.abs(Y - ref) <= 1e-13 * scale + 1e-300)
    assert np.array_equal(oracle.partial_completion(Xb, Wb, 1)["Y"], oracle.logits(Xb, Wb))
    with pytest.raises(ValueError):
        oracle.partial_completion(Xb, Wb, 3)


# ---------------------------------------------------------------- Eq. (7) selection
def _fig2():
    return {r[0]: float(r[1]) for r in _read_golden("fig2_result_path.txt")}


def test_selection_reproduces_the_pages_choice_on_their_testbed():
    """With Figure 2's bytes and frames, the 1-GbE link of Section 6.1 and the 0.189 ms
    projection cost, Equation (7) picks source projection, as the deployment did; the saving
    is the logit bytes' wire time (~25.6 ms)."""
    g = _fig2()
    beta = g["link_bits_per_s"] / 8.0
    d, margin = oracle.select_source_projection(g["r0_bytes"], g["p0_bytes"], g["r0_frames"],
                                                g["p0_frames"], beta, g["rtt"],
                                                g["projection_cost"], 0.0)
    assert d == g["chosen_plan"]
    assert abs(margin - ((3201544 - 256) / beta - 0.189e-3)) < 1e-12


def test_selection_flips_when_the_local_cost_exceeds_the_transfer_saved():
    """A link fast enough that the bytes saved take less time than the projection costs
    (closed form: threshold bandwidth = (B_r - B_s) / (L_s - L_r)), and the frame term."""
    g = _fig2()
    dB = g["r0_bytes"] - g["p0_bytes"]
    L = g["projection_cost"]
    thr = dB / L
    assert oracle.select_source_projection(dB + 256, 256, 4, 4, thr * 0.99, 0.0, L, 0.0)[0] == 1
    assert oracle.select_source_projection(dB + 256, 256, 4, 4, thr * 1.01, 0.0, L, 0.0)[0] == 0
    # fewer frames on the projected plan add alpha per frame saved
    d, m = oracle.select_source_projection(1000, 1000, 5, 1, 1e9, 1e-3, 3.5e-3, 0.0)
    assert d == 1 and abs(m - 0.5e-3) < 1e-15
    assert oracle.select_source_projection(1, 0, 1, 1, 0.0, 0.0, 0.0, 0.0)[0] == -1
