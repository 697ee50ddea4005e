"""Host restatement of the record combine's fixed merge order, in fp32, for bit-exact checks.

A record (m, i, s) of a column set holds the max logit m, the lowest column i attaining it and
s = sum exp(y - m) ("SemBridge: Compiling Consumer Observations into Cross-Stack Communication
Plans", Figure 1: the lanes' projections merge to the token of the complete logits).  The merge
keeps the larger max, the lower column on an equal max, and rescales both sums to the new max.
Its associativity holds only up to rounding, so the combine fixes the order; this module
performs that order on the host:

  per (row, shard): lane l of a 32-lane warp takes tiles l, l + 32, ..., l + 480 of each batch
      of 512 tiles (missing tiles are the empty record (-inf, INT_MAX, 0)) and folds those 16
      as a pairwise tree (adjacent pairs first: strides 1, 2, 4, 8); each batch result is
      merged into the lane's running record in ascending batch order; then an xor butterfly
      over the lanes (16, 8, 4, 2, 1) merges the 32 lane records, lane 0's result being the
      shard record;
  per row: the k shard records merge in ascending shard order into the empty record;
  outputs: lse = m + ln s, token = i, chosen log-prob = -ln s; with Gumbel records the token
      is the best key's column and its log-prob z/T - lse; target log-prob = z_t - lse (z_t/T
      on the Gumbel surface).

Every operation is one IEEE fp32 operation (numpy float32), matching the rounding points the
kernel writes out.  The two transcendental functions are the device's own (e^x of a
non-positive x through the hardware base-2 exponential, and ln): they are passed in as
callables that evaluate a whole float32 array, so the restatement needs no model of them.
The whole warp is simulated, all rows and shards at once, one merge level per array step.
"""
from __future__ import annotations

import numpy as np

INT_MAX = np.int32(2 ** 31 - 1)
NEG_INF = np.float32(-np.inf)
F32 = np.float32


def _merge(a, b, exp_nonpos):
    am, ai, as_ = a
    bm, bi, bs = b
    m = np.maximum(am, bm)
    i = np.where(am > bm, ai, np.where(bm > am, bi, np.minimum(ai, bi))).astype(np.int32)
    a_live = am != NEG_INF
    b_live = bm != NEG_INF
    # the exponent arguments of both sides in one device call (dead sides get a dummy 0)
    with np.errstate(invalid="ignore"):  # -inf - -inf on dead sides, discarded
        xa = np.where(a_live, am - m, F32(0)).astype(np.float32)
        xb = np.where(b_live, bm - m, F32(0)).astype(np.float32)
    e = exp_nonpos(np.concatenate([xa.ravel(), xb.ravel()])).astype(np.float32)
    ea = e[:xa.size].reshape(xa.shape)
    eb = e[xa.size:].reshape(xb.shape)
    sa = np.where(a_live, as_ * ea, F32(0)).astype(np.float32)
    sb = np.where(b_live, bs * eb, F32(0)).astype(np.float32)
    return m.astype(np.float32), i, (sa + sb).astype(np.float32)


def _gmerge(a, b):
    ak, ai, az = a
    bk, bi, bz = b
    take_a = (ak > bk) | ((ak == bk) & (ai < bi))
    return (np.where(take_a, ak, bk).astype(np.float32), np.where(take_a, ai, bi).astype(np.int32),
            np.where(take_a, az, bz).astype(np.float32))


def _empty(shape):
    return (np.full(shape, NEG_INF, np.float32), np.full(shape, INT_MAX, np.int32),
            np.zeros(shape, np.float32))


def _take(rec, sel):
    return tuple(x[sel] for x in rec)


def _where(mask, a, b):
    return tuple(np.where(mask, x, y) for x, y in zip(a, b))


def shard_records(m, idx, s, exp_nonpos, gk=None, gi=None, gz=None):
    """Shard-local completion of records [M, k, T] (float32 m, s; int32 idx) in the combine's
    fixed order; returns the [M, k] shard records (and Gumbel shard records if given)."""
    M, k, T = m.shape
    gumbel = gk is not None
    lanes = np.arange(32)
    r = _empty((M, k, 32))
    g = _empty((M, k, 32))
    nbatch = (T + 511) // 512
    for j in range(nbatch):
        t0 = lanes + 512 * j                      # each lane's first tile of the batch
        active = t0 < T                           # lanes whose loop still runs
        tiles = t0[:, None] + 32 * np.arange(16)[None, :]   # [32, 16]
        valid = tiles < T
        tc = np.minimum(tiles, T - 1)
        x = (np.where(valid, m[:, :, tc], NEG_INF).astype(np.float32),
             np.where(valid, idx[:, :, tc], INT_MAX).astype(np.int32),
             np.where(valid, s[:, :, tc], F32(0)).astype(np.float32))
        if gumbel:
            y = (np.where(valid, gk[:, :, tc], NEG_INF).astype(np.float32),
                 np.where(valid, gi[:, :, tc], INT_MAX).astype(np.int32),
                 np.where(valid, gz[:, :, tc], F32(0)).astype(np.float32))
        w = 1
        while w < 16:                              # pairwise tree over the 16 entries
            lo = np.arange(0, 16 - w, 2 * w)
            new = _merge(_take(x, (..., lo)), _take(x, (..., lo + w)), exp_nonpos)
            for f, nf in zip(x, new):
                f[..., lo] = nf
            if gumbel:
                newg = _gmerge(_take(y, (..., lo)), _take(y, (..., lo + w)))
                for f, nf in zip(y, newg):
                    f[..., lo] = nf
            w *= 2
        rr = _merge(r, _take(x, (..., 0)), exp_nonpos)
        r = _where(active, rr, r)
        if gumbel:
            g = _where(active, _gmerge(g, _take(y, (..., 0))), g)
    for off in (16, 8, 4, 2, 1):                   # xor butterfly over the lanes
        partner = lanes ^ off
        r = _merge(r, _take(r, (..., partner)), exp_nonpos)
        if gumbel:
            g = _gmerge(g, _take(g, (..., partner)))
    r0 = _take(r, (..., 0))
    return (r0, _take(g, (..., 0))) if gumbel else (r0, None)


def combine(m, idx, s, exp_nonpos, log_fn, *, tz=None, gk=None, gi=None, gz=None,
            inv_t=None):
    """The combine's outputs for records [M, k, T]: token, lse, token_logprob (and
    target_logprob if tz [M] is given).  inv_t is the fp32 1/T of the Gumbel surface."""
    M, k, _ = m.shape
    gumbel = gk is not None
    sr, sg = shard_records(m, idx, s, exp_nonpos, gk, gi, gz)
    acc = _empty((M,))
    gacc = _empty((M,))
    for sh in range(k):                            # ascending shard order
        acc = _merge(acc, _take(sr, (..., sh)), exp_nonpos)
        if gumbel:
            gacc = _gmerge(gacc, _take(sg, (..., sh)))
    ln_s = log_fn(acc[2]).astype(np.float32)
    lse = (acc[0] + ln_s).astype(np.float32)
    out = {"lse": lse}
    if gumbel:
        it = F32(inv_t)
        out["token"] = gacc[1]
        out["token_logprob"] = ((gacc[2] * it).astype(np.float32) - lse).astype(np.float32)
    else:
        out["token"] = acc[1]
        out["token_logprob"] = (-ln_s).astype(np.float32)
    if tz is not None:
        tzf = tz.astype(np.float32)
        if gumbel:
            tzf = (tzf * F32(inv_t)).astype(np.float32)
        out["target_logprob"] = (tzf - lse).astype(np.float32)
    out["shard_records"] = sr
    return out
