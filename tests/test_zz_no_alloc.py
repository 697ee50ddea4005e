"""The entry point for callers that cannot allocate device memory.

sb_lmhead_project_static_scratch runs the same projection as sb_lmhead_project but takes its
scratch from an array built into the library, for callers (plug-ins inside an engine that
owns the device memory pool, latency-critical paths that must not trigger cudaMalloc's
device synchronisation, foreign-function callers that link only this library) that cannot
hand it a workspace.  These tests call it through the C ABI twice in a row and compare its
outputs with those of sb_lmhead_project on the same inputs.  This file sorts last so that a
run stopping at its first failure has already run every other test.
"""
import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
from gemm_epilogue_reduction_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 5e-3
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


def _compare(a, b):
    assert torch.equal(a["token"], b["token"])
    for key in ("token_logprob", "lse", "target_logprob"):
        if key in a:
            assert float((a[key] - b[key]).abs().max()) <= TOL, key


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
        _compare(got, ref)


def test_static_scratch_rejects_problems_beyond_its_size():
    M, d, V, k = 4096, 64, 200064, 4
    assert sb.sb_workspace_bytes(M, V, k, sb.SB_TOKEN) > SCRATCH_BYTES
    out, _ = _outputs_without_workspace(M, V, k, sb.SB_TOKEN, None)
    H = torch.zeros(M, d, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(V, d, dtype=torch.bfloat16, device="cuda")
    st = sb.sb_lmhead_project_static_scratch(H, W, M, d, V, k, sb.SB_TOKEN, 1.0, 0, out)
    assert st == sb.SB_ERR_WORKSPACE_TOO_SMALL
