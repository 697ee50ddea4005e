"""The packed layout of W (sb_pack_weights, SB_W_PACKED): the buffer holds exactly the
documented arrangement, and every call that reads a packed W gives bit for bit the results of
the same call on the row-major W (the same operands reach the same MMAs, so the logits, the
records and everything completed from them are identical)."""
import numpy as np
import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
from gemm_epilogue_reduction_gb300 import synth

pytestmark = pytest.mark.gpu

KEYS = ("token", "token_logprob", "lse", "logits", "target_logprob", "topk_ids",
        "topk_logprob")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _packed_reference(W: torch.Tensor, k: int) -> np.ndarray:
    """The documented packed arrangement, built on the host from the row-major W."""
    V, d = W.shape
    S = V // k
    t128, kbs = -(-S // 128), -(-d // 64)
    w = synth.bf16_bits(W.cpu())  # uint16 [V, d]
    out = np.zeros((k, t128, kbs, 128, 64), np.uint16)
    for s in range(k):
        for t in range(t128):
            rows = w[s * S + t * 128: s * S + min(S, t * 128 + 128)]
            for kb in range(kbs):
                blk = rows[:, kb * 64: kb * 64 + 64]
                out[s, t, kb, :blk.shape[0], :blk.shape[1]] = blk
    return out.reshape(-1)


@pytest.mark.parametrize("V,d,k", [(300, 136, 3), (4096, 64, 4), (21, 8, 7), (1000, 200, 1)])
def test_packed_buffer_is_the_documented_layout(V, d, k):
    _, W = synth.make_hw(1, d, V, seed=V + d)
    W = W.cuda()
    P = sb.pack_weights(W, k)
    torch.cuda.synchronize()
    assert P.buf.numel() == sb.sb_packed_weight_bytes(V, d, k)
    got = P.buf.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, _packed_reference(W, k))


SHAPES = [
    (16, 256, 4096, 4),     # vocab mode, 16 rows: one ring per operand
    (64, 200, 3000, 3),     # vocab mode, joint ring; ragged shards and K
    (5, 64, 21, 7),         # shards of 3 columns
    (300, 136, 3000, 3),    # rows mode, CTA pairs, one atom per stage
    (600, 128, 5000, 2),    # rows mode, several pairs per W tile (two atoms per stage)
]
SURFACES = [sb.SB_TOKEN_LOGPROB, sb.SB_FULL_LOGITS, sb.SB_GUMBEL_TOKEN, sb.SB_TOPK_LOGPROB]


def _call(H, W, k, surface, targets=None):
    return sb.project(H, W, k, surface, temperature=0.8, seed=42, targets=targets,
                      topk=5 if surface == sb.SB_TOPK_LOGPROB else 0)


@pytest.mark.parametrize("M,d,V,k", SHAPES)
@pytest.mark.parametrize("surface", SURFACES)
def test_packed_calls_give_the_bits_of_row_major_calls(M, d, V, k, surface):
    H, W = synth.make_hw(M, d, V, seed=M * 3 + k)
    H, W = H.cuda(), W.cuda()
    tg = None
    if surface in (sb.SB_TOKEN_LOGPROB, sb.SB_GUMBEL_TOKEN):
        tg = synth.make_targets(M, V, seed=2, device="cuda")
    P = sb.pack_weights(W, k)
    a = _call(H, W, k, surface, tg)
    b = _call(H, P, k, surface, tg)
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(b["_outputs"]) == sb.SB_OK
    for key in KEYS:
        if key in a:
            assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("M,surface", [(16, sb.SB_TOKEN_LOGPROB), (256, sb.SB_GUMBEL_TOKEN),
                                       (64, sb.SB_FULL_LOGITS)])
def test_packed_calls_at_the_workload_sizes(M, surface):
    """The decode and sampling shapes (d = 5120, V = 151936, k = 4; 64 rows at d = 4096,
    k = 2) on the packed W: the same bits as on the row-major W."""
    d, V, k = (4096, 151936, 2) if M == 64 else (5120, 151936, 4)
    H, W = synth.make_hw(M, d, V, seed=0, device="cuda")
    P = sb.pack_weights(W, k)
    a = _call(H, W, k, surface)
    b = _call(H, P, k, surface)
    torch.cuda.synchronize()
    for key in KEYS:
        if key in a:
            assert torch.equal(a[key], b[key]), key


def test_records_host_buffer_call_and_host_step_on_a_packed_w():
    M, d, V, k = 16, 512, 20000, 4
    H, W = synth.make_hw(M, d, V, seed=9)
    H, W = H.cuda(), W.cuda()
    P = sb.pack_weights(W, k)
    surf = sb.SB_TOKEN_LOGPROB
    ref = _call(H, W, k, surf)
    # the records alone
    out, bufs = sb.make_outputs(M, V, k, surf)
    assert sb.sb_lmhead_records(H, P, M, d, V, k, surf | sb.SB_W_PACKED, 1.0, 0, out) == sb.SB_OK
    out2, bufs2 = sb.make_outputs(M, V, k, surf)
    assert sb.sb_lmhead_records(H, W, M, d, V, k, surf, 1.0, 0, out2) == sb.SB_OK
    torch.cuda.synchronize()
    T = sb.sb_tiles_per_shard(M, V, k)
    n = M * k * T
    nb = 256 + 3 * ((4 * n + 255) // 256 * 256)
    assert torch.equal(bufs["workspace"][256:nb], bufs2["workspace"][256:nb])
    # the host-buffer call and the captured host step
    H_host = H.cpu().pin_memory()
    res_host = torch.empty(2 * M, dtype=torch.int32).pin_memory()
    tok_host, lp_host = res_host[:M], res_host[M:].view(torch.float32)
    out3, bufs3 = sb.make_outputs(M, V, k, surf)
    H_dev = torch.empty_like(H)
    assert sb.sb_lmhead_project_from_host(H_host, H_dev, P, M, d, V, k, surf | sb.SB_W_PACKED,
                                          1.0, 0, out3, tok_host, lp_host) == sb.SB_OK
    torch.cuda.synchronize()
    assert torch.equal(tok_host, ref["token"].cpu())
    assert torch.equal(lp_host, ref["token_logprob"].cpu())
    step = sb.HostStep(H_host, H_dev, P, M, d, V, k, surf | sb.SB_W_PACKED, 1.0, 0, out3,
                       tok_host, lp_host)
    tok_host.zero_()
    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    step.close()
    assert torch.equal(tok_host, ref["token"].cpu())


def test_pack_weights_rejects_bad_arguments():
    V, d, k = 1000, 64, 2
    W = synth.make_hw(1, d, V, seed=1)[1].cuda()
    need = sb.sb_packed_weight_bytes(V, d, k)
    buf = torch.empty(need + 32, dtype=torch.uint8, device="cuda")
    assert sb.sb_pack_weights(W, V, d, k, buf, need - 1) == sb.SB_ERR_WORKSPACE_TOO_SMALL
    assert sb.sb_pack_weights(W, V, d, k, buf.data_ptr() + 8, need) == sb.SB_ERR_ALIGNMENT
    assert sb.sb_pack_weights(W, V, d, 3, buf, need) == sb.SB_ERR_INVALID_ARG  # V % k != 0
    assert sb.sb_pack_weights(None, V, d, k, buf, need) == sb.SB_ERR_INVALID_ARG
    assert sb.sb_pack_weights(W, V, d, k, buf, need) == sb.SB_OK
    torch.cuda.synchronize()
