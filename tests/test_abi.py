"""Host-side checks of the C ABI that need no GPU: the library builds and loads, exports
every entry point the header declares, sizes its workspace as documented, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

import gemm_epilogue_reduction_gb300 as sb
from gemm_epilogue_reduction_gb300 import build as sbbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sb.h")


@pytest.fixture(scope="module", autouse=True)
def _built():
    sbbuild.build()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(sb_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["sb_workspace_bytes", "sb_tiles_per_shard", "sb_lmhead_project", "sb_lmhead_records",
              "sb_combine_shard_records", "sb_last_device_status", "sb_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(sbbuild.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), n


def test_tiles_per_shard_and_workspace_layout():
    # one record per 128 vocabulary columns of a shard, whatever the GEMM tiling
    assert sb.sb_tiles_per_shard(16, 151936, 4) == (37984 + 127) // 128 == 297
    assert sb.sb_tiles_per_shard(4096, 200064, 4) == (50016 + 127) // 128 == 391
    assert sb.sb_tiles_per_shard(256, 151936, 4) == 297
    assert sb.sb_tiles_per_shard(4, 4097, 2) == -1  # V % k != 0
    assert sb.sb_tiles_per_shard(4, 2048, 1025) == -1  # k above 1024

    def al(x):
        return (x + 255) // 256 * 256

    M, V, k = 16, 151936, 4
    n = M * k * 297
    assert sb.sb_workspace_bytes(M, V, k, sb.SB_TOKEN) == 256 + 3 * al(4 * n) + al(4 * M)
    assert sb.sb_workspace_bytes(M, V, k, sb.SB_GUMBEL_TOKEN) == 256 + 6 * al(4 * n) + al(4 * M)
    assert sb.sb_workspace_bytes(0, V, k, sb.SB_TOKEN) == 0
    assert sb.sb_workspace_bytes(M, V, k, 7) == 0
    assert sb.sb_workspace_bytes(M, V, k, sb.SB_TOPK_LOGPROB) == (
        256 + 3 * al(4 * n) + 2 * al(4 * n * sb.SB_MAX_TOPK) + al(4 * M))


def test_packed_weight_bytes_closed_form():
    # k * ceil(S / 128) tiles of ceil(d / 64) K blocks of 128 x 64 bf16 (16 KB each)
    def want(V, d, k):
        return k * (-(-(V // k) // 128)) * (-(-d // 64)) * 16384
    for V, d, k in [(151936, 5120, 4), (151936, 4096, 2), (200064, 6144, 4), (300, 136, 3),
                    (21, 8, 7), (4096, 256, 1)]:
        assert sb.sb_packed_weight_bytes(V, d, k) == want(V, d, k)
    assert sb.sb_packed_weight_bytes(151936, 5120, 4) == 4 * 297 * 80 * 16384
    assert sb.sb_packed_weight_bytes(4097, 256, 2) == 0   # V % k != 0
    assert sb.sb_packed_weight_bytes(4096, 260, 2) == 0   # d % 8 != 0
    assert sb.sb_packed_weight_bytes(4096, 256, 0) == 0
    # the records do not depend on the layout of W
    assert sb.sb_workspace_bytes(16, 151936, 4, sb.SB_TOKEN_LOGPROB | sb.SB_W_PACKED) == \
        sb.sb_workspace_bytes(16, 151936, 4, sb.SB_TOKEN_LOGPROB)


def test_status_strings():
    for code in range(7):
        assert sb.sb_status_string(code)
    assert sb.sb_status_string(99) == "unknown status"


def _outputs(ws_bytes=1 << 20, **kw):
    base = 0x10000000
    fields = dict(token=base, token_logprob=base + 0x1000, lse=base + 0x2000, logits_bf16=None,
                  target_ids=None, target_logprob=None, workspace=base + 0x100000,
                  workspace_bytes=ws_bytes)
    fields.update(kw)
    return sb.sb_outputs(**fields)


@pytest.mark.parametrize("case, expect", [
    (dict(H=None), sb.SB_ERR_INVALID_ARG),
    (dict(M=0), sb.SB_ERR_INVALID_ARG),
    (dict(V=4097), sb.SB_ERR_INVALID_ARG),      # V % k != 0
    (dict(k=0), sb.SB_ERR_INVALID_ARG),
    (dict(d=4), sb.SB_ERR_INVALID_ARG),
    (dict(d=260), sb.SB_ERR_ALIGNMENT),          # d % 8 != 0
    (dict(H=0x10000008), sb.SB_ERR_ALIGNMENT),
    (dict(surface=sb.SB_GUMBEL_TOKEN, T=0.0), sb.SB_ERR_INVALID_ARG),
    (dict(surface=sb.SB_GUMBEL_TOKEN, T=float("inf")), sb.SB_ERR_INVALID_ARG),
    (dict(surface=sb.SB_FULL_LOGITS), sb.SB_ERR_INVALID_ARG),  # logits buffer missing
    (dict(out=dict(token=None)), sb.SB_ERR_INVALID_ARG),
    (dict(out=dict(token_logprob=None), surface=sb.SB_TOKEN_LOGPROB), sb.SB_ERR_INVALID_ARG),
    (dict(out=dict(target_ids=0x20000000)), sb.SB_ERR_INVALID_ARG),  # no target_logprob
    (dict(out=dict(workspace=0x10000010)), sb.SB_ERR_ALIGNMENT),
    (dict(out=dict(workspace_bytes=1024)), sb.SB_ERR_WORKSPACE_TOO_SMALL),
    (dict(surface=sb.SB_TOPK_LOGPROB), sb.SB_ERR_INVALID_ARG),  # no top-K buffers
    (dict(surface=sb.SB_TOPK_LOGPROB,
          out=dict(topk_ids=0x50000000, topk_logprob=0x60000000, topk=17)), sb.SB_ERR_INVALID_ARG),
    (dict(surface=sb.SB_TOPK_LOGPROB, V=8, k=1,
          out=dict(topk_ids=0x50000000, topk_logprob=0x60000000, topk=9)), sb.SB_ERR_INVALID_ARG),
    (dict(surface=sb.SB_TOPK_LOGPROB, V=1024, k=256,
          out=dict(topk_ids=0x50000000, topk_logprob=0x60000000, topk=4)), sb.SB_ERR_INVALID_ARG),
    (dict(surface=5), sb.SB_ERR_INVALID_ARG),
    (dict(surface=sb.SB_TOKEN | 0x200), sb.SB_ERR_INVALID_ARG),  # unknown layout flag
    (dict(surface=sb.SB_W_PACKED | 5), sb.SB_ERR_INVALID_ARG),
])
def test_invalid_arguments_are_rejected_before_any_launch(case, expect):
    args = dict(H=0x30000000, W=0x40000000, M=4, d=256, V=4096, k=2, surface=sb.SB_TOKEN,
                T=1.0)
    args.update({k: v for k, v in case.items() if k != "out"})
    out = _outputs(**case.get("out", {}))
    st = sb.sb_lmhead_project(args["H"], args["W"], args["M"], args["d"], args["V"],
                              args["k"], args["surface"], args["T"], 0, out, 0)
    assert st == expect


def test_valid_arguments_without_a_gpu_report_a_device_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("this machine has a GPU")
    out = _outputs()
    st = sb.sb_lmhead_project(0x30000000, 0x40000000, 4, 256, 4096, 2, sb.SB_TOKEN, 1.0, 0,
                              out, 0)
    assert st in (sb.SB_ERR_CUDA, sb.SB_ERR_UNSUPPORTED)


def test_host_buffer_entry_rejects_missing_host_buffers_before_any_copy():
    out = _outputs()
    for h_host, tok_host in ((0, 0x7000), (0x7000, 0)):
        st = sb.sb_lmhead_project_from_host(h_host, 0x30000000, 0x40000000, 4, 256, 4096, 2,
                                            sb.SB_TOKEN, 1.0, 0, out, tok_host, None, 0)
        assert st == sb.SB_ERR_INVALID_ARG


def test_host_step_rejects_missing_arguments_before_any_capture():
    out = sb.sb_outputs()
    lib = sb.lib()
    h = ctypes.c_void_p(123)
    assert lib.sb_host_step_create(None, None, None, 16, 512, 40000, 4, sb.SB_TOKEN, 1.0, 0,
                                   ctypes.byref(out), None, None, ctypes.byref(h)) == \
        sb.SB_ERR_INVALID_ARG
    assert h.value is None  # the handle is cleared on every error
    assert lib.sb_host_step_create(None, None, None, 16, 512, 40000, 4, sb.SB_TOKEN, 1.0, 0,
                                   ctypes.byref(out), None, None, None) == sb.SB_ERR_INVALID_ARG
    assert lib.sb_host_step_launch(None, None) == sb.SB_ERR_INVALID_ARG
    lib.sb_host_step_destroy(None)  # no-op
