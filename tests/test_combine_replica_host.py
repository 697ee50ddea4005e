"""The host restatement of the combine's merge order (tests/combine_replica.py), checked on the
CPU with numpy's exp and log standing in for the device's: whatever the order, the merged
record must be the plain definition -- max over all tiles, the lowest column attaining it,
lse = log sum over tiles of s * e^m -- up to fp32 rounding."""
import numpy as np

import combine_replica as cr


def _np_exp(x):
    return np.exp(x.astype(np.float64)).astype(np.float32)


def _np_log(x):
    with np.errstate(divide="ignore"):
        return np.log(x.astype(np.float64)).astype(np.float32)


def test_replica_reduces_to_the_definition():
    rng = np.random.default_rng(0)
    for (M, k, T) in ((3, 1, 1), (4, 3, 37), (2, 2, 1100), (2, 64, 3)):
        m = rng.normal(0, 2, (M, k, T)).astype(np.float32)
        m[rng.random((M, k, T)) < 0.1] = -np.inf
        m[0, 0, 0] = 5.0  # a live tile in every case
        idx = np.stack([rng.permutation(k * T).reshape(k, T) for _ in range(M)]).astype(np.int32)
        idx[m == -np.inf] = cr.INT_MAX
        s = rng.uniform(1, 100, (M, k, T)).astype(np.float32)
        s[m == -np.inf] = 0
        out = cr.combine(m, idx, s, _np_exp, _np_log, tz=np.zeros(M, np.float32))
        for r in range(M):
            mm = m[r].max()
            assert out["token"][r] == idx[r][m[r] == mm].min()
            live = m[r] != -np.inf
            lse = mm + np.log(np.sum(s[r][live].astype(np.float64) *
                                     np.exp(m[r][live].astype(np.float64) - mm)))
            assert abs(out["lse"][r] - lse) < 1e-5 * max(1.0, abs(lse))
            assert abs(out["token_logprob"][r] - (mm - lse)) < 1e-5 * max(1.0, abs(lse))
            assert abs(out["target_logprob"][r] + lse) < 1e-5 * max(1.0, abs(lse))


def test_replica_gumbel_picks_the_best_key_lowest_column():
    rng = np.random.default_rng(1)
    M, k, T = 3, 4, 600
    m = rng.normal(0, 1, (M, k, T)).astype(np.float32)
    idx = np.stack([rng.permutation(k * T).reshape(k, T) for _ in range(M)]).astype(np.int32)
    s = rng.uniform(1, 10, (M, k, T)).astype(np.float32)
    gk = rng.choice(np.float32([0.5, 1.0, 2.0]), (M, k, T))
    gz = rng.normal(0, 1, (M, k, T)).astype(np.float32)
    out = cr.combine(m, idx, s, _np_exp, _np_log, gk=gk, gi=idx, gz=gz, inv_t=np.float32(1 / 0.7))
    for r in range(M):
        best = gk[r] == gk[r].max()
        col = idx[r][best].min()
        assert out["token"][r] == col
        zc = gz[r][idx[r] == col][0]
        assert abs(out["token_logprob"][r] - (zc / 0.7 - out["lse"][r])) < 1e-5 * 10
