"""Back-to-back calls on one stream with no host synchronisation in between.

Every kernel of the library is a programmatic dependent launch that lets its successor start
early, so consecutive calls overlap on the GPU.  Calls that share one workspace but read
different inputs must still see their own inputs and leave their own results: a record, a
staging buffer or an input read before the previous call has finished with it would show up
here as a result that matches the other input (the values are compared with results computed
one call at a time)."""
import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
from gemm_epilogue_reduction_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("M,d,V,k,surface", [
    (16, 1024, 65536, 4, sb.SB_TOKEN_LOGPROB),   # vocab mode
    (16, 512, 40000, 4, sb.SB_TOPK_LOGPROB),     # vocab mode, top-K lists
    (300, 512, 32768, 2, sb.SB_GUMBEL_TOKEN),    # rows mode, CTA pairs
])
def test_alternating_inputs_sharing_one_workspace(M, d, V, k, surface):
    Hs = [synth.make_hw(M, d, 1, seed=40 + i, device="cuda")[0] for i in range(2)]
    _, W = synth.make_hw(1, d, V, seed=7, device="cuda")
    topk = 8 if surface == sb.SB_TOPK_LOGPROB else 0
    keys = ["token", "token_logprob", "lse"] + (["topk_ids", "topk_logprob"] if topk else [])
    refs = []
    for H in Hs:
        r = sb.project(H, W, k, surface, temperature=0.8, seed=5, topk=topk)
        torch.cuda.synchronize()
        refs.append({key: r[key].clone() for key in keys})
    ws = torch.empty(sb.sb_workspace_bytes(M, V, k, surface), dtype=torch.uint8, device="cuda")
    calls = []
    for i in range(40):
        out, bufs = sb.make_outputs(M, V, k, surface, workspace=ws, topk=topk)
        assert sb.sb_lmhead_project(Hs[i % 2], W, M, d, V, k, surface, 0.8, 5, out) == sb.SB_OK
        calls.append(bufs)
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(out) == sb.SB_OK
    for i, bufs in enumerate(calls):
        for key in keys:
            assert torch.equal(bufs[key], refs[i % 2][key]), (i, key)


def test_host_buffer_calls_back_to_back_with_alternating_inputs():
    """The host-buffer entry point stages H in one device buffer for every call: each call's
    staging waits for the previous call's GEMM to be done with it."""
    M, d, V, k = 16, 1024, 65536, 4
    Hs = [synth.make_hw(M, d, 1, seed=60 + i, device="cuda")[0] for i in range(2)]
    _, W = synth.make_hw(1, d, V, seed=8, device="cuda")
    refs = []
    for H in Hs:
        r = sb.project(H, W, k, sb.SB_TOKEN_LOGPROB)
        torch.cuda.synchronize()
        refs.append((r["token"].cpu(), r["token_logprob"].cpu()))
    H_hosts = [H.cpu().pin_memory() for H in Hs]
    H_dev = torch.empty_like(Hs[0])
    out, bufs = sb.make_outputs(M, V, k, sb.SB_TOKEN_LOGPROB)
    results = []
    for i in range(40):
        tok = torch.full((M,), -1, dtype=torch.int32).pin_memory()
        lp = torch.full((M,), float("nan"), dtype=torch.float32).pin_memory()
        st = sb.sb_lmhead_project_from_host(H_hosts[i % 2], H_dev, W, M, d, V, k,
                                            sb.SB_TOKEN_LOGPROB, 1.0, 0, out, tok, lp)
        assert st == sb.SB_OK
        results.append((tok, lp))
    torch.cuda.synchronize()
    for i, (tok, lp) in enumerate(results):
        assert torch.equal(tok, refs[i % 2][0]), i
        assert torch.equal(lp, refs[i % 2][1]), i


def test_partial_completions_back_to_back_with_alternating_inputs():
    M, N, K, lanes = 64, 2048, 8192, 2
    Xs = [synth.make_hw(M, K, 1, seed=70 + i, device="cuda")[0] for i in range(2)]
    _, W = synth.make_hw(1, K, N, seed=9, device="cuda")
    nbytes = sb.sb_partial_workspace_bytes(M, N, K, lanes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    refs = []
    for X in Xs:
        Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
        assert sb.sb_partial_completion(X, W, M, N, K, lanes, Y, False, ws, nbytes, None) == sb.SB_OK
        torch.cuda.synchronize()
        refs.append(Y)
    Ys = []
    for i in range(40):
        Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
        assert sb.sb_partial_completion(Xs[i % 2], W, M, N, K, lanes, Y, False, ws, nbytes,
                                        None) == sb.SB_OK
        Ys.append(Y)
    torch.cuda.synchronize()
    for i, Y in enumerate(Ys):
        assert torch.equal(Y, refs[i % 2]), i
