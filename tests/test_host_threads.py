"""Concurrent host threads: the library keeps only small host-side caches (tensor maps, device
properties, launch epochs, cluster occupancy), guarded by a mutex or atomics.  Several Python
threads (ctypes releases the interpreter lock during each call) enqueue projections on their
own streams, on more distinct (H, W) pairs than the tensor-map cache holds, both tilings and
several surfaces; every call must give the same bits as the same call made alone."""
import threading

import pytest
import torch

import gemm_epilogue_reduction_gb300 as sb
from gemm_epilogue_reduction_gb300 import synth

pytestmark = pytest.mark.gpu

# (M, d, V, k, surface): 12 problems, 24 tensor maps (the cache holds 16)
PROBLEMS = [
    (4, 256, 4096, 2, sb.SB_TOKEN_LOGPROB),
    (16, 512, 20000, 4, sb.SB_GUMBEL_TOKEN),
    (64, 256, 30000, 2, sb.SB_FULL_LOGITS),
    (200, 128, 9000, 3, sb.SB_TOKEN_LOGPROB),
    (300, 256, 12000, 4, sb.SB_GUMBEL_TOKEN),
    (8, 128, 5000, 1, sb.SB_TOPK_LOGPROB),
    (33, 64, 7000, 7, sb.SB_TOKEN),
    (129, 96, 6000, 2, sb.SB_FULL_LOGITS),
    (16, 1024, 16384, 8, sb.SB_TOKEN_LOGPROB),
    (256, 192, 8192, 4, sb.SB_TOPK_LOGPROB),
    (1, 8, 300, 3, sb.SB_TOKEN_LOGPROB),
    (77, 320, 10000, 5, sb.SB_GUMBEL_TOKEN),
]
KEYS = ("token", "token_logprob", "lse", "logits", "topk_ids", "topk_logprob")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(i):
    M, d, V, k, surface = PROBLEMS[i]
    H, W = synth.make_hw(M, d, V, seed=100 + i)
    return H.cuda(), W.cuda(), k, surface


def _call(H, W, k, surface, stream, i):
    return sb.project(H, W, k, surface, temperature=0.8, seed=7 + i, stream=stream,
                      topk=5 if surface == sb.SB_TOPK_LOGPROB else 0)


def test_threads_on_their_own_streams_match_the_calls_made_alone():
    inputs = [_inputs(i) for i in range(len(PROBLEMS))]
    alone = []
    for i, (H, W, k, surface) in enumerate(inputs):
        r = _call(H, W, k, surface, torch.cuda.current_stream(), i)
        torch.cuda.synchronize()
        alone.append({key: r[key].clone() for key in KEYS if key in r})

    n_threads, rounds = 4, 6
    got = [[None] * len(PROBLEMS) for _ in range(n_threads)]
    errors = []

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for rnd in range(rounds):
                    for j in range(len(PROBLEMS)):
                        i = (j + 3 * t + rnd) % len(PROBLEMS)  # threads walk in different orders
                        H, W, k, surface = inputs[i]
                        r = _call(H, W, k, surface, stream, i)
                        if rnd == rounds - 1:
                            got[t][i] = r
                stream.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(n_threads)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not errors, errors
    torch.cuda.synchronize()
    for t in range(n_threads):
        for i in range(len(PROBLEMS)):
            r = got[t][i]
            assert r is not None
            assert sb.sb_last_device_status(r["_outputs"]) == sb.SB_OK
            for key, want in alone[i].items():
                assert torch.equal(r[key], want), (t, i, key)
