"""The entry point for callers that cannot allocate device memory.

sb_lmhead_project_static_scratch runs the same projection as sb_lmhead_project but takes its
scratch from an array built into the library, for callers (plug-ins inside an engine that
owns the device memory pool, latency-critical paths that must not trigger cudaMalloc's
device synchronisation, foreign-function callers that link only this library) that cannot
hand it a workspace.  These tests call it through the C ABI twice in a row and compare its
outputs bit for bit with those of sb_lmhead_project on the same inputs (the same kernels on
the same inputs: only where the records live differs), read its device status back, and
check that a call allocates no device memory.  This file sorts last so that a run stopping at
its first failure has already run every other test.
"""
import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
from gemm_epilogue_reduction_gb300 import synth

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _outputs_without_workspace(M, V, k, surface, targets):
    out, bufs = sb.make_outputs(M, V, k, surface, targets=targets,
                                workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
    out.workspace = None
    out.workspace_bytes = 0
    return out, bufs


def _compare_bits(a, b):
    for key in ("token", "token_logprob", "lse", "target_logprob"):
        if key in a:
            assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("M,d,V,k,surface", [
    (16, 512, 8192, 4, sb.SB_TOKEN_LOGPROB),
    (300, 256, 6000, 3, sb.SB_GUMBEL_TOKEN),
])
def test_static_scratch_matches_caller_workspace_two_calls_in_a_row(M, d, V, k, surface):
    assert sb.sb_workspace_bytes(M, V, k, surface) <= SCRATCH_BYTES
    for call in range(2):  # the second call finds the first call's records in the array
        H, W = synth.make_hw(M, d, V, seed=40 + call, device="cuda")
        tg = synth.make_targets(M, V, seed=call, device="cuda")
        ref = sb.project(H, W, k, surface, temperature=0.7, seed=99, targets=tg)
        out, got = _outputs_without_workspace(M, V, k, surface, tg)
        st = sb.sb_lmhead_project_static_scratch(H, W, M, d, V, k, surface, 0.7, 99, out)
        assert st == sb.SB_OK
        torch.cuda.synchronize()
        assert sb.sb_static_scratch_last_status() == sb.SB_OK
        _compare_bits(got, ref)


def test_static_scratch_reports_an_out_of_range_target_and_recovers():
    M, d, V, k = 16, 256, 4096, 2
    H, W = synth.make_hw(M, d, V, seed=7, device="cuda")
    tg = synth.make_targets(M, V, seed=3, device="cuda")
    bad = tg.clone()
    bad[5] = V  # one target past the vocabulary
    out, _ = _outputs_without_workspace(M, V, k, sb.SB_TOKEN_LOGPROB, bad)
    assert sb.sb_lmhead_project_static_scratch(H, W, M, d, V, k, sb.SB_TOKEN_LOGPROB, 1.0, 0,
                                               out) == sb.SB_OK
    torch.cuda.synchronize()
    assert sb.sb_static_scratch_last_status() == sb.SB_ERR_INVALID_ARG
    # the next call with valid targets reports OK again and matches the workspace call
    ref = sb.project(H, W, k, sb.SB_TOKEN_LOGPROB, targets=tg)
    out, got = _outputs_without_workspace(M, V, k, sb.SB_TOKEN_LOGPROB, tg)
    assert sb.sb_lmhead_project_static_scratch(H, W, M, d, V, k, sb.SB_TOKEN_LOGPROB, 1.0, 0,
                                               out) == sb.SB_OK
    torch.cuda.synchronize()
    assert sb.sb_static_scratch_last_status() == sb.SB_OK
    _compare_bits(got, ref)


def test_static_scratch_call_allocates_no_device_memory():
    M, d, V, k = 16, 512, 8192, 4
    H, W = synth.make_hw(M, d, V, seed=11, device="cuda")
    out, got = _outputs_without_workspace(M, V, k, sb.SB_TOKEN_LOGPROB, None)
    # the first call looks up the array's address and loads the kernels
    assert sb.sb_lmhead_project_static_scratch(H, W, M, d, V, k, sb.SB_TOKEN_LOGPROB, 1.0, 0,
                                               out) == sb.SB_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(3):
        assert sb.sb_lmhead_project_static_scratch(H, W, M, d, V, k, sb.SB_TOKEN_LOGPROB, 1.0,
                                                   0, out) == sb.SB_OK
    torch.cuda.synchronize()
    assert sb.sb_static_scratch_last_status() == sb.SB_OK
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == reserved0


def test_static_scratch_rejects_problems_beyond_its_size():
    M, d, V, k = 4096, 64, 200064, 4
    assert sb.sb_workspace_bytes(M, V, k, sb.SB_TOKEN) > SCRATCH_BYTES
    out, _ = _outputs_without_workspace(M, V, k, sb.SB_TOKEN, None)
    H = torch.zeros(M, d, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(V, d, dtype=torch.bfloat16, device="cuda")
    st = sb.sb_lmhead_project_static_scratch(H, W, M, d, V, k, sb.SB_TOKEN, 1.0, 0, out)
    assert st == sb.SB_ERR_WORKSPACE_TOO_SMALL
