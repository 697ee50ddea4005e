"""fp64 CPU oracle for the LM-head contraction and its consumer-surface projection.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this package. The product path (the CUDA library and its Python
binding) never imports it, and the two share no code: the only module both sides use is the
seeded input generator, which holds none of the method's arithmetic.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over host cores); this module
only compiles it with the host compiler and marshals numpy arrays through ctypes. Each C
function cites the passage of "SemBridge: Compiling Consumer Observations into Cross-Stack
Communication Plans" that it follows.

Parity pins (see ``tests/test_oracle_pins.py``): exact rational brute force on tiny inputs,
closed forms (zero hidden state, unit hidden vectors, two-column vocabularies), the R0/P0
token-surface identity of Figure 1, the shard logsumexp identity, published SplitMix64
outputs and the Gumbel-max distribution identity.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` with the host C compiler."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, u64, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = f64
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_logits.argtypes = [P, P, i64, i64, i64, P]
        lib.oracle_logits.restype = None
        lib.oracle_splitmix64.argtypes = [u64, u64]
        lib.oracle_splitmix64.restype = u64
        lib.oracle_uniform24.argtypes = [u64, u64]
        lib.oracle_uniform24.restype = f64
        lib.oracle_gumbel.argtypes = [u64, u64]
        lib.oracle_gumbel.restype = f64
        lib.oracle_selection_key.argtypes = [f64, i64, i64, i64, i32, f64, u64]
        lib.oracle_selection_key.restype = f64
        lib.oracle_project.argtypes = [P, P, P, i64, i64, i64, i32, i32, f64, u64, P,
                                       P, P, P, P, P, P, P, P, P, P]
        lib.oracle_project.restype = ctypes.c_int
        lib.oracle_topk.argtypes = [P, P, i64, i64, i64, i32, P, P, P]
        lib.oracle_topk.restype = ctypes.c_int
        lib.oracle_partial_completion.argtypes = [P, P, i64, i64, i64, i32, P, P]
        lib.oracle_partial_completion.restype = ctypes.c_int
        lib.oracle_select_source_projection.argtypes = [f64] * 8 + [P]
        lib.oracle_select_source_projection.restype = ctypes.c_int
        lib.oracle_payload_bytes_per_row.argtypes = [i32, i64]
        lib.oracle_payload_bytes_per_row.restype = f64
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a) -> np.ndarray:
    """bf16 data as a C-contiguous uint16 array of bit patterns."""
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return np.ascontiguousarray(a)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits)))


def logits(H_bits, W_bits) -> np.ndarray:
    """z = H Wᵀ in fp64 (Section 5.2: the output head materialises full logits)."""
    H, W = _bits(H_bits), _bits(W_bits)
    M, d = H.shape
    V, d2 = W.shape
    assert d == d2
    Z = np.empty((M, V), dtype=np.float64)
    _load().oracle_logits(_ptr(H), _ptr(W), M, d, V, _ptr(Z))
    return Z


def splitmix64(seed: int, n: int) -> int:
    return int(_load().oracle_splitmix64(seed & (2**64 - 1), n & (2**64 - 1)))


def uniform24(seed: int, n: int) -> float:
    return float(_load().oracle_uniform24(seed & (2**64 - 1), n & (2**64 - 1)))


def gumbel(seed: int, n: int) -> float:
    return float(_load().oracle_gumbel(seed & (2**64 - 1), n & (2**64 - 1)))


def selection_key(z: float, row: int, col: int, V: int, gumbel: bool = False,
                  temperature: float = 1.0, seed: int = 0) -> float:
    return float(_load().oracle_selection_key(float(z), int(row), int(col), int(V),
                                              1 if gumbel else 0, float(temperature),
                                              seed & (2**64 - 1)))


def payload_bytes_per_row(surface: int, V: int) -> float:
    return float(_load().oracle_payload_bytes_per_row(int(surface), int(V)))


def topk(H_bits, W_bits, K: int) -> dict:
    """Top-K log-probability surface of every row (see ``oracle_topk`` in oracle.c):
    ids [M, K] (logit descending, ties to the lower column), logprob [M, K], lse [M]."""
    H, W = _bits(H_bits), _bits(W_bits)
    M, d = H.shape
    V, d2 = W.shape
    assert d == d2
    out = {"ids": np.empty((M, K), np.int32), "logprob": np.empty((M, K)), "lse": np.empty(M)}
    rc = _load().oracle_topk(_ptr(H), _ptr(W), M, d, V, int(K), _ptr(out["ids"]),
                             _ptr(out["logprob"]), _ptr(out["lse"]))
    if rc != 0:
        raise ValueError("oracle_topk rejected its arguments")
    return out


def select_source_projection(B_r, B_s, F_r, F_s, beta, alpha, L_s, L_r):
    """Equation (7): (decision, margin in seconds); decision 1 = project, 0 = materialise."""
    m = ctypes.c_double(0.0)
    d = _load().oracle_select_source_projection(float(B_r), float(B_s), float(F_r), float(F_s),
                                                float(beta), float(alpha), float(L_s),
                                                float(L_r), ctypes.byref(m))
    return int(d), float(m.value)


def partial_completion(X_bits, W_bits, lanes: int, keep_partials: bool = False) -> dict:
    """Row-parallel partial completion (see ``oracle_partial_completion`` in oracle.c):
    Y [M, N] = sum over lanes of P_l, P_l [M, N] the lane's partial product (fp64)."""
    X, W = _bits(X_bits), _bits(W_bits)
    M, K = X.shape
    N, K2 = W.shape
    assert K == K2
    Y = np.empty((M, N))
    Pp = np.empty((lanes, M, N)) if keep_partials else None
    rc = _load().oracle_partial_completion(_ptr(X), _ptr(W), M, N, K, int(lanes), _ptr(Y),
                                           _ptr(Pp))
    if rc != 0:
        raise ValueError("oracle_partial_completion rejected its arguments")
    out = {"Y": Y}
    if keep_partials:
        out["P"] = Pp
    return out


def project(H_bits, W_bits, k: int, *, gumbel: bool = False, temperature: float = 1.0,
            seed: int = 0, targets=None, row_ids=None, keep_z: bool = False) -> dict:
    """Consumer-surface projection of every row of H (see ``oracle_project`` in oracle.c).

    Returns a dict of numpy arrays: token, lse, logprob, target_logprob, key_top1, key_top2
    (per row), shard_max, shard_token, shard_lse (per row and shard) and, with keep_z, z.
    """
    H, W = _bits(H_bits), _bits(W_bits)
    M, d = H.shape
    V, d2 = W.shape
    assert d == d2
    out = {
        "token": np.empty(M, np.int32), "lse": np.empty(M), "logprob": np.empty(M),
        "target_logprob": np.empty(M), "key_top1": np.empty(M), "key_top2": np.empty(M),
        "shard_max": np.empty((M, k)), "shard_token": np.empty((M, k), np.int32),
        "shard_lse": np.empty((M, k)),
    }
    Z = np.empty((M, V), np.float64) if keep_z else None
    tg = None if targets is None else np.ascontiguousarray(targets, dtype=np.int32)
    rid = None if row_ids is None else np.ascontiguousarray(row_ids, dtype=np.int64)
    rc = _load().oracle_project(
        _ptr(H), _ptr(W), _ptr(rid), M, d, V, int(k), 1 if gumbel else 0,
        float(temperature), seed & (2**64 - 1), _ptr(tg),
        _ptr(out["token"]), _ptr(out["lse"]), _ptr(out["logprob"]),
        _ptr(out["target_logprob"]), _ptr(out["key_top1"]), _ptr(out["key_top2"]),
        _ptr(out["shard_max"]), _ptr(out["shard_token"]), _ptr(out["shard_lse"]), _ptr(Z))
    if rc != 0:
        raise ValueError("oracle_project rejected its arguments")
    if keep_z:
        out["z"] = Z
    return out
