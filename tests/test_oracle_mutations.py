"""The oracle's pins have teeth: each plausible mistake, planted in a copy of oracle.c on the
CPU, must make tests/test_oracle_pins.py fail."""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "ties_to_highest_index": ("if (key[j] > key[best]) best = j;",
                              "if (key[j] >= key[best]) best = j;"),
    "stream_index_off_by_one": ("(n + 1u) * 0x9E37", "(n) * 0x9E37"),
    "temperature_multiplies": ("y[j] = gumbel ? zr[j] / temperature : zr[j];",
                               "y[j] = gumbel ? zr[j] * temperature : zr[j];"),
    "short_shard_range": ("const int64_t lo = (int64_t)s * S, hi = lo + S;",
                          "const int64_t lo = (int64_t)s * S, hi = lo + S - 1;"),
    "dropped_first_term": ("for (int64_t i = 0; i < d; ++i) a += h[i] * w[i];",
                           "for (int64_t i = 1; i < d; ++i) a += h[i] * w[i];"),
    "wrong_row_operand": ("a3 += h3[i] * w[i];", "a3 += h2[i] * w[i];"),
    "untempered_logprob": ("logprob[r] = y[tok] - l;", "logprob[r] = zr[tok] - l;"),
    "gumbel_sign": ("return -log(-log(u));", "return log(-log(u));"),
    "key_multiplies_temperature": ("return z / temperature + oracle_gumbel",
                                   "return z * temperature + oracle_gumbel"),
    "uniform_wrong_shift": ("(oracle_splitmix64(seed, n) >> 40)",
                            "(oracle_splitmix64(seed, n) >> 41)"),
    "topk_ties_to_highest_index": ("(best < 0 || zr[j] > zr[best])",
                                   "(best < 0 || zr[j] >= zr[best])"),
    "topk_unnormalised_logprob": ("logprob[r * K + q] = zr[best] - l;",
                                  "logprob[r * K + q] = zr[best];"),
    "partial_lane_slice_overlaps": ("for (int64_t i = l * Kl; i < (l + 1) * Kl; ++i)",
                                    "for (int64_t i = l * Kl; i <= (l + 1) * Kl && i < K; ++i)"),
    "selection_local_cost_sign": ("const double rhs = L_s - L_r;", "const double rhs = L_r - L_s;"),
    "selection_frames_ignored": ("+ alpha * (F_r - F_s);", "+ 0.0 * alpha * (F_r - F_s);"),
    "partial_drops_last_lane": ("for (int32_t l = 0; l < lanes; ++l) {",
                                "for (int32_t l = 0; l + 1 < lanes || l == 0; ++l) {"),
}


def _run_pins_on_mutant(name):
    old, new = MUTATIONS[name]
    tmp = tempfile.mkdtemp(prefix=f"mut_{name}_")
    try:
        for sub in ("oracle", "tests", "gemm_epilogue_reduction_gb300"):
            shutil.copytree(os.path.join(ROOT, sub), os.path.join(tmp, sub),
                            ignore=shutil.ignore_patterns("_build", "__pycache__", "*.so"))
        src = os.path.join(tmp, "oracle", "oracle.c")
        text = open(src).read()
        assert text.count(old) == 1, name
        open(src, "w").write(text.replace(old, new))
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            "tests/test_oracle_pins.py"], cwd=tmp, capture_output=True, text=True,
                           timeout=600)
        return r.returncode
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_every_planted_mistake_is_caught():
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        rcs = dict(zip(MUTATIONS, ex.map(_run_pins_on_mutant, MUTATIONS)))
    survivors = [n for n, rc in rcs.items() if rc == 0]
    assert not survivors, f"pins did not catch: {survivors}"
    assert all(rc == 1 for rc in rcs.values()), rcs  # failed tests, not collection errors
