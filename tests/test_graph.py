"""The entry points inside a CUDA graph: a decode step captured once and replayed with new
inputs gives the oracle's answer each time (the calls are stream-ordered launches with no
host synchronisation, so they capture; argument checks and tensor-map encoding happen at
capture time)."""
import numpy as np
import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
import oracle
from gemm_epilogue_reduction_gb300 import synth
from gpu_helpers import TOL, bf16_half_ulp, check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _capture(fn):
    """Warm up (per-device opt-ins happen on the first call), then capture fn on a side
    stream; returns the graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        assert fn(s) == sb.SB_OK
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert fn(s) == sb.SB_OK
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("surface,T,gseed", [
    (sb.SB_TOKEN_LOGPROB, 1.0, 0),
    (sb.SB_GUMBEL_TOKEN, 0.7, 77),
    (sb.SB_FULL_LOGITS, 1.0, 0),
])
def test_decode_step_replays_from_a_cuda_graph(surface, T, gseed):
    M, d, V, k = 16, 512, 40000, 4
    H, W = synth.make_hw(M, d, V, seed=11, device="cuda")
    out, bufs = sb.make_outputs(M, V, k, surface)
    g = _capture(lambda s: sb.sb_lmhead_project(H, W, M, d, V, k, surface, T, gseed, out, s))
    gumbel = surface == sb.SB_GUMBEL_TOKEN
    for trial in range(3):
        Hn, _ = synth.make_hw(M, d, 1, seed=100 + trial, device="cuda")
        H.copy_(Hn)                  # new inputs in the captured buffer
        g.replay()
        torch.cuda.synchronize()
        assert sb.sb_last_device_status(out) == sb.SB_OK
        rows = list(range(M))
        ref = oracle.project(synth.bf16_bits(H), synth.bf16_bits(W), k, gumbel=gumbel,
                             temperature=T, seed=gseed, keep_z=True)
        res = {key: bufs[key] for key in ("token", "token_logprob", "lse")}
        check_rows(res, ref, rows, gumbel=gumbel, T=T, seed=gseed)
        if surface == sb.SB_FULL_LOGITS:
            lg = bufs["logits"].float().cpu().numpy().astype(np.float64)
            assert np.all(np.abs(lg - ref["z"]) <= TOL + bf16_half_ulp(ref["z"]))


def test_partial_completion_replays_from_a_cuda_graph():
    M, N, K, lanes = 8, 1024, 4096, 2
    X, W = synth.make_hw(M, K, N, seed=5, device="cuda")
    nbytes = sb.sb_partial_workspace_bytes(M, N, K, lanes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    g = _capture(lambda s: sb.sb_partial_completion(X, W, M, N, K, lanes, Y, False, ws, nbytes,
                                                    s))
    for trial in range(3):
        Xn, _ = synth.make_hw(M, K, 1, seed=200 + trial, device="cuda")
        X.copy_(Xn)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.partial_completion(synth.bf16_bits(X), synth.bf16_bits(W), lanes)["Y"]
        got = Y.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= TOL), float(np.abs(got - ref).max())
    # replaying the same inputs reproduces the same bits
    again = Y.clone()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(again, Y)


def test_host_buffer_decode_step_replays_from_a_cuda_graph():
    """The host-buffer call captured once: each replay reads the current contents of the
    pinned H buffer and leaves the token and log-prob in the pinned result buffers (the
    copy kernel and the combine's host stores are ordinary graph kernel nodes)."""
    M, d, V, k = 16, 512, 40000, 4
    H, W = synth.make_hw(M, d, V, seed=12, device="cuda")
    H_host = H.cpu().pin_memory()
    H_dev = torch.empty_like(H)
    tok = torch.full((M,), -1, dtype=torch.int32).pin_memory()
    lp = torch.full((M,), float("nan"), dtype=torch.float32).pin_memory()
    out, bufs = sb.make_outputs(M, V, k, sb.SB_TOKEN_LOGPROB)
    g = _capture(lambda s: sb.sb_lmhead_project_from_host(H_host, H_dev, W, M, d, V, k,
                                                          sb.SB_TOKEN_LOGPROB, 1.0, 0, out,
                                                          tok, lp, s))
    for trial in range(3):
        Hn, _ = synth.make_hw(M, d, 1, seed=300 + trial)
        H_host.copy_(Hn)             # new inputs in the captured host buffer
        tok.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        ref = sb.project(Hn.cuda(), W, k, sb.SB_TOKEN_LOGPROB)
        torch.cuda.synchronize()
        assert torch.equal(tok, ref["token"].cpu())
        assert torch.equal(lp, ref["token_logprob"].cpu())
