"""Shard payloads (the per-lane records a vocabulary-sharded deployment would exchange in
place of logit slices): loopback equality with the fused combine, per-shard parity with the
oracle, and a W split into per-device slices merging to the same bits."""
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


def _records(H, W, k, surface, T_=1.0, seed=0, workspace=None):
    M, d = H.shape
    V = W.shape[0]
    out, bufs = sb.make_outputs(M, V, k, surface, workspace=workspace)
    assert sb.sb_lmhead_records(H, W, M, d, V, k, surface, T_, seed, out) == sb.SB_OK
    return out, bufs


def _merge(payload, M, k, surface, T_=1.0):
    out, bufs = sb.make_outputs(M, 1, 1, sb.SB_TOKEN_LOGPROB)
    assert sb.sb_merge_shard_payload(payload, M, k, surface, T_, out) == sb.SB_OK
    return bufs


@pytest.mark.parametrize("surface", [sb.SB_TOKEN_LOGPROB, sb.SB_GUMBEL_TOKEN])
@pytest.mark.parametrize("M,d,V,k", [(16, 256, 4096, 4), (300, 64, 3000, 3)])
def test_pack_then_merge_equals_the_fused_combine(surface, M, d, V, k):
    H, W = synth.make_hw(M, d, V, seed=7)
    H, W = H.cuda(), W.cuda()
    ref = sb.project(H, W, k, surface, temperature=0.7, seed=5)
    out, bufs = _records(H, W, k, surface, 0.7, 5)
    payload = torch.empty(sb.sb_payload_bytes(M, k, surface), dtype=torch.uint8, device="cuda")
    T = sb.sb_tiles_per_shard(M, V, k)
    assert sb.sb_pack_shard_records(bufs["workspace"], M, k, T, surface, 0, payload) == sb.SB_OK
    got = _merge(payload, M, k, surface, 0.7)
    torch.cuda.synchronize()
    for key in ("token", "token_logprob", "lse"):
        assert torch.equal(got[key], ref[key]), key


def test_payload_records_match_the_oracle_per_shard():
    M, d, V, k = 12, 128, 3000, 3
    H, W = synth.make_hw(M, d, V, seed=8)
    H, W = H.cuda(), W.cuda()
    out, bufs = _records(H, W, k, sb.SB_TOKEN)
    payload = torch.empty(sb.sb_payload_bytes(M, k, sb.SB_TOKEN), dtype=torch.uint8, device="cuda")
    T = sb.sb_tiles_per_shard(M, V, k)
    assert sb.sb_pack_shard_records(bufs["workspace"], M, k, T, sb.SB_TOKEN, 0, payload) == sb.SB_OK
    torch.cuda.synchronize()
    rec = payload.cpu().numpy().view(np.dtype([("m", "<f4"), ("i", "<i4"), ("s", "<f4")]))
    rec = rec.reshape(k, M)
    ref = oracle.project(synth.bf16_bits(H), synth.bf16_bits(W), k, keep_z=True)
    S = V // k
    for s in range(k):
        for r in range(M):
            m, i, ssum = float(rec[s, r]["m"]), int(rec[s, r]["i"]), float(rec[s, r]["s"])
            assert s * S <= i < (s + 1) * S
            assert abs(m - ref["shard_max"][r, s]) <= TOL
            assert ref["z"][r, i] >= ref["shard_max"][r, s] - GAP
            assert abs(m + np.log(ssum) - ref["shard_lse"][r, s]) <= TOL


@pytest.mark.parametrize("M,d,V,k", [(16, 256, 4096, 4), (300, 128, 2560, 2)])
def test_w_split_across_devices_merges_to_the_same_bits(M, d, V, k):
    """Each lane's slice of W run on its own (k = 1, column offset s*S) and packed into its
    slot of one payload gives the same token, log-prob and lse bits as one call with k lanes:
    each logit's K-reduction and each tile's columns are the same either way."""
    H, W = synth.make_hw(M, d, V, seed=9)
    H, W = H.cuda(), W.cuda()
    ref = sb.project(H, W, k, sb.SB_TOKEN_LOGPROB)
    S = V // k
    rb = 12
    payload = torch.empty(sb.sb_payload_bytes(M, k, sb.SB_TOKEN_LOGPROB), dtype=torch.uint8,
                          device="cuda")
    keep = []
    for s in range(k):
        Ws = W[s * S:(s + 1) * S].contiguous()
        out, bufs = _records(H, Ws, 1, sb.SB_TOKEN_LOGPROB)
        T = sb.sb_tiles_per_shard(M, S, 1)
        slot = payload.data_ptr() + s * M * rb
        assert sb.sb_pack_shard_records(bufs["workspace"], M, 1, T, sb.SB_TOKEN_LOGPROB, s * S,
                                        slot) == sb.SB_OK
        keep.append((Ws, bufs))
    got = _merge(payload, M, k, sb.SB_TOKEN_LOGPROB)
    torch.cuda.synchronize()
    for key in ("token", "token_logprob", "lse"):
        assert torch.equal(got[key], ref[key]), key


def test_payload_bytes_against_full_logit_transfer():
    """Per decode step at the decode token-only shape: 16 rows x 4 lanes x 12 B of records
    against 16 x 151936 bf16 logits."""
    M, k, V = 16, 4, 151936
    p0 = sb.sb_payload_bytes(M, k, sb.SB_TOKEN)
    assert p0 == M * k * 12
    r0 = M * V * 2
    assert 1 - p0 / r0 > 0.9997
    assert sb.sb_payload_bytes(M, k, sb.SB_TOPK_LOGPROB) == 0
