"""Equation (7) of "SemBridge" (Section 8.2) on local costs measured on this GPU: the
complete-logit surface (plan r) and the projected token surface (plan s) are timed at the
64-row decode shape with CUDA events; the library's decision on those measured costs, for the
pages' 1-GbE link and two faster links, must equal the oracle's, and the reported threshold
bandwidth must be the point where the two sides of the inequality meet."""
import math

import pytest

import bench
import gemm_epilogue_reduction_gb300 as sb
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_measured_plan_costs_give_the_oracles_decision():
    peaks, src = bench.load_peaks()
    sel, er, es = bench.measure_plan_costs(0.05, peaks, src, 0)
    L_s, L_r = sel["local_proj_s"], sel["local_ref_s"]
    # both plans stream the same W; the complete-logit plan also writes 2 M V bytes
    assert 50e-6 < L_s < 2e-3 and 50e-6 < L_r < 2e-3
    assert er["surface"] == "full_logits" and es["surface"] == "token_logprob"
    assert sel["bytes_ref"] == 2 * 64 * 151936
    assert sel["bytes_proj"] == sb.sb_payload_bytes(64, 2, sb.SB_TOKEN)
    for name, dcs in sel["decisions"].items():
        od, om = oracle.select_source_projection(
            sel["bytes_ref"], sel["bytes_proj"], sel["frames_ref"], sel["frames_proj"],
            dcs["link_bytes_per_s"], sel["frame_startup_s"], L_s, L_r)
        assert dcs["project"] == od, name
        assert dcs["margin_s"] == om, name
    thr = sel["threshold_bytes_per_s"]
    if L_s <= L_r:
        assert thr is None
        assert all(d["project"] == 1 for d in sel["decisions"].values())
    else:
        # at the threshold the two sides meet; slower links project, faster ones do not
        lhs = (sel["bytes_ref"] - sel["bytes_proj"]) / thr
        assert math.isclose(lhs, L_s - L_r, rel_tol=1e-9)
        assert oracle.select_source_projection(sel["bytes_ref"], sel["bytes_proj"], 2, 2,
                                               thr * 0.5, 0.0, L_s, L_r)[0] == 1
        assert oracle.select_source_projection(sel["bytes_ref"], sel["bytes_proj"], 2, 2,
                                               thr * 2.0, 0.0, L_s, L_r)[0] == 0
