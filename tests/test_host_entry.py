"""sb_lmhead_project_from_host: the projection with host-memory hidden states and host-memory
token outputs gives exactly the bits of sb_lmhead_project on the same inputs, for pinned
buffers (moved by the kernels), pageable buffers (copied), and mixtures of the two."""
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
    (16, 512, 40000, 4, sb.SB_TOKEN_LOGPROB),
    (300, 256, 12000, 3, sb.SB_GUMBEL_TOKEN),
    (5, 64, 1000, 1, sb.SB_TOKEN),
])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffer_call_matches_the_device_call(M, d, V, k, surface, pinned):
    H, W = synth.make_hw(M, d, V, seed=M + V, device="cuda")
    T = 0.9 if surface == sb.SB_GUMBEL_TOKEN else 1.0
    ref = sb.project(H, W, k, surface, temperature=T, seed=3)
    H_host = H.cpu()
    tok_host = torch.full((M,), -1, dtype=torch.int32)
    lp_host = torch.full((M,), float("nan"), dtype=torch.float32)
    if pinned:
        H_host, tok_host, lp_host = H_host.pin_memory(), tok_host.pin_memory(), lp_host.pin_memory()
    H_dev = torch.empty_like(H)
    out, bufs = sb.make_outputs(M, V, k, surface)
    want_lp = surface != sb.SB_TOKEN
    st = sb.sb_lmhead_project_from_host(H_host, H_dev, W, M, d, V, k, surface, T, 3, out,
                                        tok_host, lp_host if want_lp else None)
    assert st == sb.SB_OK
    torch.cuda.synchronize()
    assert sb.sb_last_device_status(out) == sb.SB_OK
    assert torch.equal(H_dev, H)
    assert torch.equal(tok_host, ref["token"].cpu())
    if want_lp:
        assert torch.equal(lp_host, ref["token_logprob"].cpu())


def test_host_buffer_call_with_token_and_logprob_back_to_back():
    """Device and host buffers laid out as [token | log-prob]: one copy brings both back."""
    M, d, V, k = 16, 512, 40000, 4
    H, W = synth.make_hw(M, d, V, seed=9, device="cuda")
    ref = sb.project(H, W, k, sb.SB_TOKEN_LOGPROB)
    res_dev = torch.empty(2 * M, dtype=torch.int32, device="cuda")
    res_host = torch.full((2 * M,), -1, dtype=torch.int32).pin_memory()
    out, bufs = sb.make_outputs(M, V, k, sb.SB_TOKEN_LOGPROB)
    out.token, out.token_logprob = res_dev.data_ptr(), res_dev.data_ptr() + 4 * M
    H_dev = torch.empty_like(H)
    st = sb.sb_lmhead_project_from_host(H.cpu().pin_memory(), H_dev, W, M, d, V, k,
                                        sb.SB_TOKEN_LOGPROB, 1.0, 0, out, res_host[:M],
                                        res_host[M:].view(torch.float32))
    assert st == sb.SB_OK
    torch.cuda.synchronize()
    assert torch.equal(res_host[:M], ref["token"].cpu())
    assert torch.equal(res_host[M:].view(torch.float32), ref["token_logprob"].cpu())


@pytest.mark.parametrize("case", ["H_unaligned", "logprob_pageable", "token_pageable"])
def test_host_buffer_call_with_mixed_buffers(case):
    """A pinned H at an address that is not 16-byte aligned is copied; pinned and pageable
    result buffers mixed in one call are copied: the bits stay those of the device call."""
    M, d, V, k = 16, 512, 40000, 4
    H, W = synth.make_hw(M, d, V, seed=21, device="cuda")
    ref = sb.project(H, W, k, sb.SB_TOKEN_LOGPROB)
    n = M * d
    if case == "H_unaligned":
        back = torch.empty(n + 4, dtype=torch.bfloat16).pin_memory()
        H_host = back[4:]  # 8 bytes past a 16-byte boundary
        H_host.copy_(H.cpu().reshape(-1))
        assert H_host.data_ptr() % 16 == 8
    else:
        H_host = H.cpu().pin_memory()
    tok_host = torch.full((M,), -1, dtype=torch.int32)
    lp_host = torch.full((M,), float("nan"), dtype=torch.float32)
    if case != "token_pageable":
        tok_host = tok_host.pin_memory()
    if case != "logprob_pageable":
        lp_host = lp_host.pin_memory()
    H_dev = torch.empty_like(H)
    out, bufs = sb.make_outputs(M, V, k, sb.SB_TOKEN_LOGPROB)
    st = sb.sb_lmhead_project_from_host(H_host, H_dev, W, M, d, V, k, sb.SB_TOKEN_LOGPROB, 1.0,
                                        0, out, tok_host, lp_host)
    assert st == sb.SB_OK
    torch.cuda.synchronize()
    assert torch.equal(H_dev, H)
    assert torch.equal(tok_host, ref["token"].cpu())
    assert torch.equal(lp_host, ref["token_logprob"].cpu())


@pytest.mark.parametrize("surface", [sb.SB_TOKEN_LOGPROB, sb.SB_GUMBEL_TOKEN])
def test_captured_host_step_replays_give_the_device_call_bits(surface):
    """sb_host_step_*: created once, launched several times with new contents of the pinned
    H buffer; every launch leaves the device call's token and log-prob in the host buffers."""
    M, d, V, k = 16, 512, 40000, 4
    _, W = synth.make_hw(1, d, V, seed=31, device="cuda")
    H_host = torch.empty(M, d, dtype=torch.bfloat16).pin_memory()
    H_dev = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    tok = torch.full((M,), -1, dtype=torch.int32).pin_memory()
    lp = torch.full((M,), float("nan"), dtype=torch.float32).pin_memory()
    out, bufs = sb.make_outputs(M, V, k, surface)
    step = sb.HostStep(H_host, H_dev, W, M, d, V, k, surface, 0.8, 17, out, tok, lp)
    try:
        for trial in range(4):
            Hn, _ = synth.make_hw(M, d, 1, seed=500 + trial)
            H_host.copy_(Hn)
            tok.fill_(-1)
            step()
            torch.cuda.synchronize()
            ref = sb.project(Hn.cuda(), W, k, surface, temperature=0.8, seed=17)
            torch.cuda.synchronize()
            assert torch.equal(tok, ref["token"].cpu()), trial
            assert torch.equal(lp, ref["token_logprob"].cpu()), trial
        assert sb.sb_last_device_status(out) == sb.SB_OK
    finally:
        step.close()


def test_captured_host_step_refuses_pageable_buffers():
    M, d, V, k = 16, 512, 40000, 4
    H, W = synth.make_hw(M, d, V, seed=32, device="cuda")
    out, bufs = sb.make_outputs(M, V, k, sb.SB_TOKEN_LOGPROB)
    st, h = sb.sb_host_step_create(H.cpu(), torch.empty_like(H), W, M, d, V, k,
                                   sb.SB_TOKEN_LOGPROB, 1.0, 0, out,
                                   torch.empty(M, dtype=torch.int32), None)
    assert st == sb.SB_ERR_UNSUPPORTED and h == 0
