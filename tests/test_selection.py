"""The library's Equation (7) plan selection (host only) against the oracle and the pages'
testbed, plus the choice it makes for the on-device plans of this library."""
import math
import random

import pytest

import gemm_epilogue_reduction_gb300 as sb
import oracle
from gemm_epilogue_reduction_gb300 import build as sbbuild


@pytest.fixture(scope="module", autouse=True)
def _built():
    sbbuild.build()


def test_library_matches_the_oracle_on_random_inputs():
    rng = random.Random(7)
    for _ in range(2000):
        args = (rng.uniform(0, 1e8), rng.uniform(0, 1e6), rng.randint(0, 64), rng.randint(0, 64),
                10 ** rng.uniform(6, 12), rng.uniform(0, 1e-3), rng.uniform(0, 1e-2),
                rng.uniform(0, 1e-2))
        d, m = sb.sb_select_source_projection(*args)
        od, om = oracle.select_source_projection(*args)
        assert d == od and m == om


def test_pages_testbed_picks_source_projection():
    """Figure 2 (MiniMax-M2.7, concurrency 16): 3,201,544 B vs 256 B in four frames each, a
    1-GbE link and 0.189 ms of projection: project."""
    d, m = sb.sb_select_source_projection(3201544, 256, 4, 4, 1e9 / 8, 0.3425e-3, 0.189e-3, 0.0)
    assert d == 1 and m > 25e-3


def test_on_device_plans_of_this_library():
    """Decode shape on one GB300 with the vocabulary split over 2 devices of an NVLink-class
    link: the projected plan ships 12-byte shard records instead of bf16 logits, and its local
    cost is the token path's (234 us measured) against the full-logit path's (which also
    reads W once and writes 19.5 MB more).  Projecting saves transfer and costs no more on
    the device, so Equation (7) projects at any link speed."""
    M, V, k = 64, 151936, 2
    B_r = M * V * 2 * (k - 1) / k          # the remote lanes' logits
    B_s = sb.sb_payload_bytes(M, k, sb.SB_TOKEN) * (k - 1) / k
    for beta in (25e9, 900e9, 1.8e12):
        d, m = sb.sb_select_source_projection(B_r, B_s, 1, 1, beta, 2e-6, 190e-6, 194e-6)
        assert d == 1, beta
    assert sb.sb_select_source_projection(1, 0, 0, 0, -1.0, 0, 0, 0)[0] == -1
    assert sb.sb_select_source_projection(math.nan, 0, 0, 0, 1.0, 0, 0, 0)[0] == -1


def test_bench_plan_selection_on_given_costs():
    """The benchmark's Equation (7) table (host logic, no GPU): payload bytes from the
    library, the oracle's decision on every link, and the threshold link rate where both
    sides meet (none when projecting costs no more on the device)."""
    import bench
    M, V, k = 64, 151936, 2
    cheap = bench.plan_selection(M, V, k, 180e-6, 186e-6)   # projection faster locally
    assert cheap["threshold_bytes_per_s"] is None
    assert cheap["bytes_ref"] == 2 * M * V
    assert cheap["bytes_proj"] == sb.sb_payload_bytes(M, k, sb.SB_TOKEN) == 12 * M * k
    assert all(d["project"] == 1 for d in cheap["decisions"].values())
    costly = bench.plan_selection(M, V, k, 200e-6, 186e-6)  # projection 14 us slower locally
    thr = costly["threshold_bytes_per_s"]
    assert thr == pytest.approx((costly["bytes_ref"] - costly["bytes_proj"]) / 14e-6)
    for name, d in costly["decisions"].items():
        od, om = oracle.select_source_projection(costly["bytes_ref"], costly["bytes_proj"],
                                                 k, k, d["link_bytes_per_s"], 0.0, 200e-6,
                                                 186e-6)
        assert d["project"] == od and d["margin_s"] == om
        assert od == (1 if d["link_bytes_per_s"] < thr else 0), name
