"""GB300-native LM-head contraction fused with the consumer-surface projection.

Thin ctypes binding over the C ABI in ``include/sb.h`` (``libsb.so``, built in-tree by
``gemm_epilogue_reduction_gb300.build``). The functions named ``sb_*`` mirror the C entry
points one to one and only marshal arguments: every step of the path runs in the CUDA
kernels. ``project`` is a convenience wrapper that allocates the outputs and workspace with
torch (the caller-owned memory of the C ABI) and raises on a non-OK status.

There is no CPU fallback: if ``libsb.so`` is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

SB_TOKEN, SB_TOKEN_LOGPROB, SB_FULL_LOGITS, SB_GUMBEL_TOKEN, SB_TOPK_LOGPROB = 0, 1, 2, 3, 4
SB_MAX_TOPK = 16
SB_W_PACKED = 0x100  # layout flag OR'ed into `surface`: W is the packed copy (sb_pack_weights)
SURFACES = {"token": SB_TOKEN, "token_logprob": SB_TOKEN_LOGPROB,
            "full_logits": SB_FULL_LOGITS, "gumbel_token": SB_GUMBEL_TOKEN,
            "topk_logprob": SB_TOPK_LOGPROB}
SB_OK = 0
SB_ERR_INVALID_ARG = 1
SB_ERR_UNSUPPORTED = 2
SB_ERR_ALIGNMENT = 3
SB_ERR_WORKSPACE_TOO_SMALL = 4
SB_ERR_CUDA = 5
SB_ERR_DEVICE_TIMEOUT = 6

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libsb.so")
_lock = threading.Lock()
_lib = None


class SbError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({sb_status_string(status)})")
        self.status = status


class sb_outputs(ctypes.Structure):
    _fields_ = [("token", ctypes.c_void_p), ("token_logprob", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("logits_bf16", ctypes.c_void_p),
                ("target_ids", ctypes.c_void_p), ("target_logprob", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("topk_ids", ctypes.c_void_p), ("topk_logprob", ctypes.c_void_p),
                ("topk", ctypes.c_int32)]


def lib():
    """The loaded libsb.so; raises if it has not been built."""
    global _lib
    L = _lib
    if L is not None:  # the common case: no lock once loaded
        return L
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libsb.so not found at {LIB_PATH}: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
        L.sb_workspace_bytes.argtypes = [i64, i64, i32, i32]
        L.sb_workspace_bytes.restype = ctypes.c_size_t
        L.sb_tiles_per_shard.argtypes = [i64, i64, i32]
        L.sb_tiles_per_shard.restype = i32
        L.sb_packed_weight_bytes.argtypes = [i64, i64, i32]
        L.sb_packed_weight_bytes.restype = ctypes.c_size_t
        L.sb_pack_weights.argtypes = [P, i64, i64, i32, P, ctypes.c_size_t, P]
        L.sb_pack_weights.restype = i32
        L.sb_lmhead_project.argtypes = [P, P, i64, i64, i64, i32, i32, ctypes.c_float, u64,
                                        ctypes.POINTER(sb_outputs), P]
        L.sb_lmhead_project.restype = i32
        L.sb_lmhead_records.argtypes = L.sb_lmhead_project.argtypes
        L.sb_lmhead_records.restype = i32
        L.sb_lmhead_project_static_scratch.argtypes = L.sb_lmhead_project.argtypes
        L.sb_lmhead_project_static_scratch.restype = i32
        L.sb_static_scratch_last_status.argtypes = []
        L.sb_static_scratch_last_status.restype = i32
        L.sb_lmhead_project_from_host.argtypes = [P, P, P, i64, i64, i64, i32, i32,
                                                  ctypes.c_float, u64,
                                                  ctypes.POINTER(sb_outputs), P, P, P]
        L.sb_lmhead_project_from_host.restype = i32
        L.sb_host_step_create.argtypes = [P, P, P, i64, i64, i64, i32, i32, ctypes.c_float,
                                          u64, ctypes.POINTER(sb_outputs), P, P,
                                          ctypes.POINTER(P)]
        L.sb_host_step_create.restype = i32
        L.sb_host_step_launch.argtypes = [P, P]
        L.sb_host_step_launch.restype = i32
        L.sb_host_step_destroy.argtypes = [P]
        L.sb_host_step_destroy.restype = None
        L.sb_combine_shard_records.argtypes = [P, i64, i32, i32, i32, ctypes.c_float,
                                               ctypes.POINTER(sb_outputs), P]
        L.sb_combine_shard_records.restype = i32
        L.sb_payload_bytes.argtypes = [i64, i32, i32]
        L.sb_payload_bytes.restype = ctypes.c_size_t
        L.sb_pack_shard_records.argtypes = [P, i64, i32, i32, i32, i64, P, P]
        L.sb_pack_shard_records.restype = i32
        L.sb_merge_shard_payload.argtypes = [P, i64, i32, i32, ctypes.c_float,
                                             ctypes.POINTER(sb_outputs), P]
        L.sb_merge_shard_payload.restype = i32
        L.sb_partial_workspace_bytes.argtypes = [i64, i64, i64, i32]
        L.sb_partial_workspace_bytes.restype = ctypes.c_size_t
        L.sb_partial_completion.argtypes = [P, P, i64, i64, i64, i32, P, i32, P,
                                            ctypes.c_size_t, P]
        L.sb_partial_completion.restype = i32
        L.sb_select_source_projection.argtypes = [ctypes.c_double] * 8 + [
            ctypes.POINTER(ctypes.c_double)]
        L.sb_select_source_projection.restype = i32
        L.sb_last_device_status.argtypes = [ctypes.POINTER(sb_outputs)]
        L.sb_last_device_status.restype = i32
        L.sb_status_string.argtypes = [i32]
        L.sb_status_string.restype = ctypes.c_char_p
        L.sb_device_info.argtypes = [ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.sb_device_info.restype = i32
        L.sb_debug_combine_math.argtypes = [i32, P, P, i64, P]
        L.sb_debug_combine_math.restype = i32
        L.sb_debug_gumbel_from_bits.argtypes = [P, P, i64, P]
        L.sb_debug_gumbel_from_bits.restype = i32
        L.sb_debug_configure.argtypes = [i32, u64]
        L.sb_debug_configure.restype = i32
        _lib = L
        return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ------------------------------------------------------------------ C entry points
def sb_workspace_bytes(M: int, V: int, k: int, surface: int) -> int:
    return int(lib().sb_workspace_bytes(M, V, k, surface))


def sb_tiles_per_shard(M: int, V: int, k: int) -> int:
    return int(lib().sb_tiles_per_shard(M, V, k))


def sb_packed_weight_bytes(V: int, d: int, k: int) -> int:
    return int(lib().sb_packed_weight_bytes(V, d, k))


def sb_pack_weights(W, V, d, k, W_packed, nbytes, stream=None) -> int:
    return int(lib().sb_pack_weights(_ptr(W), V, d, k, _ptr(W_packed), nbytes,
                                     _stream(stream)))


def sb_lmhead_project(H, W, M, d, V, k, surface, temperature, seed, out: sb_outputs,
                      stream=None) -> int:
    return int(lib().sb_lmhead_project(_ptr(H), _ptr(W), M, d, V, k, surface,
                                       float(temperature), seed & (2**64 - 1),
                                       ctypes.byref(out), _stream(stream)))


def sb_lmhead_project_from_host(H_host, H_dev, W, M, d, V, k, surface, temperature, seed,
                                out: sb_outputs, token_host, token_logprob_host=None,
                                stream=None) -> int:
    """H_host, token_host and token_logprob_host are host tensors (pinned for asynchronous
    copies) or raw host addresses; H_dev and W are device tensors."""
    return int(lib().sb_lmhead_project_from_host(
        _ptr(H_host), _ptr(H_dev), _ptr(W), M, d, V, k, surface, float(temperature),
        seed & (2**64 - 1), ctypes.byref(out), _ptr(token_host), _ptr(token_logprob_host),
        _stream(stream)))


def sb_host_step_create(H_host, H_dev, W, M, d, V, k, surface, temperature, seed,
                        out: sb_outputs, token_host, token_logprob_host=None):
    """Returns (status, handle); the handle is an int (0 on error)."""
    h = ctypes.c_void_p()
    st = int(lib().sb_host_step_create(
        _ptr(H_host), _ptr(H_dev), _ptr(W), M, d, V, k, surface, float(temperature),
        seed & (2**64 - 1), ctypes.byref(out), _ptr(token_host), _ptr(token_logprob_host),
        ctypes.byref(h)))
    return st, (h.value or 0)


def sb_host_step_launch(step: int, stream=None) -> int:
    return int(lib().sb_host_step_launch(step, _stream(stream)))


def sb_host_step_destroy(step: int) -> None:
    lib().sb_host_step_destroy(step)


class HostStep:
    """A host-buffer decode step captured once (sb_host_step_*): call it to enqueue one
    replay; the buffers passed here are read and written by every replay, so the caller
    keeps them alive and pinned."""

    def __init__(self, H_host, H_dev, W, M, d, V, k, surface, temperature, seed,
                 out: sb_outputs, token_host, token_logprob_host=None):
        self._keep = (H_host, H_dev, W, out, token_host, token_logprob_host)
        st, self.handle = sb_host_step_create(H_host, H_dev, W, M, d, V, k, surface,
                                              temperature, seed, out, token_host,
                                              token_logprob_host)
        if st != SB_OK:
            raise SbError(st, "sb_host_step_create")

    def __call__(self, stream=None) -> None:
        st = sb_host_step_launch(self.handle, stream)
        if st != SB_OK:
            raise SbError(st, "sb_host_step_launch")

    def close(self) -> None:
        if self.handle:
            sb_host_step_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def sb_lmhead_records(H, W, M, d, V, k, surface, temperature, seed, out: sb_outputs,
                      stream=None) -> int:
    return int(lib().sb_lmhead_records(_ptr(H), _ptr(W), M, d, V, k, surface,
                                       float(temperature), seed & (2**64 - 1),
                                       ctypes.byref(out), _stream(stream)))


def sb_lmhead_project_static_scratch(H, W, M, d, V, k, surface, temperature, seed,
                                     out: sb_outputs, stream=None) -> int:
    """sb_lmhead_project with the library's built-in 8 MiB scratch instead of
    out.workspace, for callers that cannot allocate device memory."""
    return int(lib().sb_lmhead_project_static_scratch(_ptr(H), _ptr(W), M, d, V, k, surface,
                                                      float(temperature), seed & (2**64 - 1),
                                                      ctypes.byref(out), _stream(stream)))


def sb_static_scratch_last_status() -> int:
    """Device status of the last static-scratch call on the current device (synchronises)."""
    return int(lib().sb_static_scratch_last_status())


def sb_combine_shard_records(workspace, M, k, tiles_per_shard, surface, temperature,
                             out: sb_outputs, stream=None) -> int:
    return int(lib().sb_combine_shard_records(_ptr(workspace), M, k, tiles_per_shard,
                                              surface, float(temperature),
                                              ctypes.byref(out), _stream(stream)))


def sb_payload_bytes(M: int, k: int, surface: int) -> int:
    return int(lib().sb_payload_bytes(M, k, surface))


def sb_pack_shard_records(workspace, M, k, tiles_per_shard, surface, col_offset, payload,
                          stream=None) -> int:
    return int(lib().sb_pack_shard_records(_ptr(workspace), M, k, tiles_per_shard, surface,
                                           int(col_offset), _ptr(payload), _stream(stream)))


def sb_merge_shard_payload(payload, M, k, surface, temperature, out: sb_outputs,
                           stream=None) -> int:
    return int(lib().sb_merge_shard_payload(_ptr(payload), M, k, surface, float(temperature),
                                            ctypes.byref(out), _stream(stream)))


def sb_partial_workspace_bytes(M: int, N: int, K: int, lanes: int) -> int:
    return int(lib().sb_partial_workspace_bytes(M, N, K, lanes))


def sb_partial_completion(X, W, M, N, K, lanes, Y, y_bf16, workspace, workspace_bytes,
                          stream=None) -> int:
    return int(lib().sb_partial_completion(_ptr(X), _ptr(W), M, N, K, lanes, _ptr(Y),
                                           1 if y_bf16 else 0, _ptr(workspace),
                                           int(workspace_bytes), _stream(stream)))


def partial_completion(X, W, lanes: int, *, out_bf16: bool = True, stream=None, workspace=None):
    """Y = sum over lanes of X[:, lane] W[:, lane]^T for torch CUDA bf16 tensors X [M, K] and
    W [N, K]; returns (Y, workspace).  Raises SbError on a bad status."""
    import torch
    M, K = X.shape
    N = W.shape[0]
    nbytes = sb_partial_workspace_bytes(M, N, K, lanes)
    if nbytes == 0:
        raise SbError(SB_ERR_INVALID_ARG, "sb_partial_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=X.device)
    Y = torch.empty(M, N, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=X.device)
    st = sb_partial_completion(X, W, M, N, K, lanes, Y, out_bf16, workspace,
                               workspace.numel(), stream)
    if st != SB_OK:
        raise SbError(st, "sb_partial_completion")
    return Y, workspace


def sb_select_source_projection(bytes_ref, bytes_proj, frames_ref, frames_proj,
                                link_bytes_per_s, frame_startup_s, local_proj_s, local_ref_s):
    """Equation (7) plan choice: returns (decision, margin_s); 1 = project at the source."""
    m = ctypes.c_double(0.0)
    d = lib().sb_select_source_projection(float(bytes_ref), float(bytes_proj),
                                          float(frames_ref), float(frames_proj),
                                          float(link_bytes_per_s), float(frame_startup_s),
                                          float(local_proj_s), float(local_ref_s),
                                          ctypes.byref(m))
    return int(d), float(m.value)


def sb_last_device_status(out: sb_outputs) -> int:
    return int(lib().sb_last_device_status(ctypes.byref(out)))


def sb_status_string(status: int) -> str:
    return lib().sb_status_string(status).decode()


def sb_device_info():
    n, cc = ctypes.c_int32(0), ctypes.c_int32(0)
    if lib().sb_device_info(ctypes.byref(n), ctypes.byref(cc)) != 0:
        return None
    return n.value, cc.value


def sb_debug_gumbel_from_bits(bits, g, count: int, stream=None) -> int:
    return int(lib().sb_debug_gumbel_from_bits(_ptr(bits), _ptr(g), int(count), _stream(stream)))


def sb_debug_combine_math(op: int, x, y, count: int, stream=None) -> int:
    return int(lib().sb_debug_combine_math(int(op), _ptr(x), _ptr(y), int(count),
                                           _stream(stream)))


def sb_debug_configure(stall_epilogue: bool, wait_limit_ns: int) -> int:
    return int(lib().sb_debug_configure(1 if stall_epilogue else 0, int(wait_limit_ns)))


# ------------------------------------------------------------------ convenience wrapper
def make_outputs(M: int, V: int, k: int, surface: int, *, device="cuda", lse=True,
                 logprob=True, targets=None, workspace=None, topk: int = 0):
    """Allocate the caller-owned buffers of one call with torch; returns (sb_outputs, dict)."""
    import torch
    bufs = {"token": torch.empty(M, dtype=torch.int32, device=device)}
    if logprob or surface in (SB_TOKEN_LOGPROB, SB_GUMBEL_TOKEN):
        bufs["token_logprob"] = torch.empty(M, dtype=torch.float32, device=device)
    if lse:
        bufs["lse"] = torch.empty(M, dtype=torch.float32, device=device)
    if surface == SB_FULL_LOGITS:
        bufs["logits"] = torch.empty(M, V, dtype=torch.bfloat16, device=device)
    if targets is not None:
        bufs["target_ids"] = targets
        bufs["target_logprob"] = torch.empty(M, dtype=torch.float32, device=device)
    if surface == SB_TOPK_LOGPROB:
        bufs["topk_ids"] = torch.empty(M, topk, dtype=torch.int32, device=device)
        bufs["topk_logprob"] = torch.empty(M, topk, dtype=torch.float32, device=device)
    nbytes = sb_workspace_bytes(M, V, k, surface)
    if nbytes == 0:
        raise SbError(SB_ERR_INVALID_ARG, "sb_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    bufs["workspace"] = workspace
    out = sb_outputs(_ptr(bufs["token"]), _ptr(bufs.get("token_logprob")), _ptr(bufs.get("lse")),
                     _ptr(bufs.get("logits")), _ptr(bufs.get("target_ids")),
                     _ptr(bufs.get("target_logprob")), _ptr(workspace),
                     workspace.numel() * workspace.element_size(),
                     _ptr(bufs.get("topk_ids")), _ptr(bufs.get("topk_logprob")), int(topk))
    return out, bufs


class PackedWeights:
    """The packed copy of a [V, d] W for k lane shards (``buf``: a uint8 CUDA tensor), as
    written by ``sb_pack_weights``; pass it as ``W`` to ``project``."""

    def __init__(self, buf, V: int, d: int, k: int):
        self.buf, self.V, self.d, self.k = buf, V, d, k

    def data_ptr(self):
        return self.buf.data_ptr()


def pack_weights(W, k: int, stream=None) -> PackedWeights:
    """Pack the row-major bf16 W [V, d] (CUDA tensor) for k lane shards; enqueued on
    ``stream``."""
    import torch
    V, d = W.shape
    nbytes = sb_packed_weight_bytes(V, d, k)
    if nbytes == 0:
        raise SbError(SB_ERR_INVALID_ARG, "sb_packed_weight_bytes")
    buf = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    st = sb_pack_weights(W, V, d, k, buf, nbytes, stream)
    if st != SB_OK:
        raise SbError(st, "sb_pack_weights")
    return PackedWeights(buf, V, d, k)


def project(H, W, k: int, surface: int = SB_TOKEN_LOGPROB, *, temperature: float = 1.0,
            seed: int = 0, targets=None, stream=None, lse=True, logprob=True, workspace=None,
            topk: int = 0):
    """Run one projection call on torch CUDA tensors H [M, d] and W [V, d] (bf16), or W a
    ``PackedWeights`` of the same k (then the call reads the packed layout).

    Returns the dict of output tensors (token, token_logprob, lse, logits, target_logprob,
    workspace, as requested). Asynchronous on ``stream``; raises SbError on a bad status."""
    M, d = H.shape
    if isinstance(W, PackedWeights):
        if W.k != k or W.d != d:
            raise SbError(SB_ERR_INVALID_ARG, "project: packed W of another shape")
        V = W.V
        surface |= SB_W_PACKED
    else:
        V = W.shape[0]
    out, bufs = make_outputs(M, V, k, surface & ~SB_W_PACKED, device=H.device, lse=lse,
                             logprob=logprob, targets=targets, workspace=workspace, topk=topk)
    st = sb_lmhead_project(H, W, M, d, V, k, surface, temperature, seed, out, stream)
    if st != SB_OK:
        raise SbError(st, "sb_lmhead_project")
    bufs["_outputs"] = out
    return bufs
