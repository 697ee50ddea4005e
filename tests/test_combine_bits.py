"""sb_combine_shard_records is bit-exact: given identical fp32 records, its outputs are those of
the fixed merge order performed independently on the host (tests/combine_replica.py), bit for
bit, on crafted records: -inf maxima (empty tiles, empty shards, an empty row), maxima equal
across tiles and shards (the lowest column must win), k = 1 and k = 1024 shards, more than 512
tiles per shard (two batches per lane), and the Gumbel surface.  The replica takes the
device's own e^x and ln through a test hook, so it needs no model of the hardware functions;
everything else is plain fp32 arithmetic in the kernel's order ("SemBridge", Figure 1: the
lanes' projections merge to the complete logits' token)."""
import numpy as np
import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
import combine_replica as cr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _device_fn(op):
    def f(x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        xd = torch.from_numpy(x).cuda()
        yd = torch.empty_like(xd)
        assert sb.sb_debug_combine_math(op, xd, yd, x.size) == sb.SB_OK
        torch.cuda.synchronize()
        return yd.cpu().numpy()
    return f


EXP, LOG = _device_fn(0), _device_fn(1)


def _al(x):
    return (x + 255) // 256 * 256


def _run(m, idx, s, *, tz=None, gk=None, gi=None, gz=None, T_temp=1.0):
    """Write the records into a workspace at the documented layout and run the combine."""
    M, k, T = m.shape
    gumbel = gk is not None
    surface = sb.SB_GUMBEL_TOKEN if gumbel else sb.SB_TOKEN_LOGPROB
    V = k * 128 * T  # so that sb_tiles_per_shard(M, V, k) == T
    assert sb.sb_tiles_per_shard(M, V, k) == T
    nbytes = sb.sb_workspace_bytes(M, V, k, surface)
    ws = torch.zeros(nbytes, dtype=torch.uint8)
    n = M * k * T
    off = 256
    fields = [m.astype(np.float32), idx.astype(np.int32), s.astype(np.float32)]
    if gumbel:
        fields += [gk.astype(np.float32), gi.astype(np.int32), gz.astype(np.float32)]
    for a in fields:
        ws[off:off + 4 * n] = torch.from_numpy(a.reshape(-1).view(np.uint8).copy())
        off += _al(4 * n)
    if tz is not None:
        ws[off:off + 4 * M] = torch.from_numpy(tz.astype(np.float32).view(np.uint8).copy())
    ws = ws.cuda()
    tg = torch.zeros(M, dtype=torch.int32, device="cuda") if tz is not None else None
    out, res = sb.make_outputs(M, V, k, surface, targets=tg, workspace=ws)
    assert sb.sb_combine_shard_records(ws, M, k, T, surface, T_temp, out) == sb.SB_OK
    torch.cuda.synchronize()
    return {key: res[key].cpu().numpy() for key in ("token", "token_logprob", "lse",
                                                   "target_logprob") if key in res}


def _check(m, idx, s, **kw):
    got = _run(m, idx, s, **kw)
    inv_t = np.float32(1.0) / np.float32(kw.get("T_temp", 1.0))
    want = cr.combine(m, idx, s, EXP, LOG, tz=kw.get("tz"), gk=kw.get("gk"), gi=kw.get("gi"),
                      gz=kw.get("gz"), inv_t=inv_t)
    assert np.array_equal(got["token"], want["token"])
    for key in ("lse", "token_logprob", "target_logprob"):
        if key in got:
            a, b = got[key].view(np.uint32), want[key].view(np.uint32)
            bad = np.nonzero(a != b)[0]
            assert bad.size == 0, (key, bad[:5], got[key][bad[:5]], want[key][bad[:5]])
    return want


def _records(rng, M, k, T, *, levels=None, empty_frac=0.0):
    """Random records: maxima N(0, 2) (or drawn from `levels` to force ties), distinct
    columns, exp-sums in [1, 128); a fraction of the tiles empty (-inf, INT_MAX, 0)."""
    if levels is None:
        m = rng.normal(0, 2, (M, k, T)).astype(np.float32)
    else:
        m = rng.choice(np.asarray(levels, np.float32), (M, k, T))
    idx = np.empty((M, k, T), np.int32)
    for r in range(M):
        idx[r] = rng.permutation(k * T).reshape(k, T).astype(np.int32) * 3 + 1
    s = rng.uniform(1.0, 128.0, (M, k, T)).astype(np.float32)
    if empty_frac:
        e = rng.random((M, k, T)) < empty_frac
        m[e] = -np.inf
        idx[e] = cr.INT_MAX
        s[e] = 0.0
    return m, idx, s


def test_random_records_with_a_ragged_tile_count():
    rng = np.random.default_rng(1)
    m, idx, s = _records(rng, 6, 3, 37)
    tz = rng.normal(0, 1, 6).astype(np.float32)
    _check(m, idx, s, tz=tz)


def test_empty_tiles_shards_and_rows():
    rng = np.random.default_rng(2)
    m, idx, s = _records(rng, 5, 4, 50, empty_frac=0.3)
    for arr, v in ((m, -np.inf), (idx, cr.INT_MAX), (s, 0.0)):
        arr[1, 2, :] = v   # one whole shard empty
        arr[3, :, :] = v   # one whole row empty: lse = -inf, token INT_MAX
    want = _check(m, idx, s)
    assert want["token"][3] == cr.INT_MAX and want["lse"][3] == -np.inf


def test_equal_maxima_across_tiles_and_shards_pick_the_lowest_column():
    rng = np.random.default_rng(3)
    m, idx, s = _records(rng, 8, 5, 70, levels=[0.5, 1.25, 1.25, 2.0])
    want = _check(m, idx, s)
    for r in range(8):
        top = m[r] == m[r].max()
        assert want["token"][r] == idx[r][top].min()


def test_one_shard_and_the_largest_shard_count():
    rng = np.random.default_rng(4)
    _check(*_records(rng, 3, 1, 200))
    m, idx, s = _records(rng, 2, 1024, 2, levels=[-1.0, 0.0625, 3.0], empty_frac=0.2)
    _check(m, idx, s)


def test_more_than_512_tiles_per_shard():
    rng = np.random.default_rng(5)
    m, idx, s = _records(rng, 2, 2, 1100, empty_frac=0.05)
    _check(m, idx, s, tz=np.array([0.25, -3.0], np.float32))


@pytest.mark.parametrize("T_temp", [0.7, 1.9])
def test_gumbel_records(T_temp):
    rng = np.random.default_rng(6)
    M, k, T = 4, 3, 600
    m, idx, s = _records(rng, M, k, T, empty_frac=0.1)
    gk = rng.normal(2, 1.5, (M, k, T)).astype(np.float32)
    gk[rng.random((M, k, T)) < 0.2] = np.float32(1.5)  # ties on the key
    gk[m == -np.inf] = -np.inf
    gi = idx.copy()
    gz = rng.normal(0, 1, (M, k, T)).astype(np.float32)
    tz = rng.normal(0, 1, M).astype(np.float32)
    _check(m, idx, s, gk=gk, gi=gi, gz=gz, tz=tz, T_temp=T_temp)
