"""AUTO algorithm selection: the library's choice against the oracle's, for
both cost models (CPU only; the choice is host logic).

The link model reproduces the latency-formula page's switch: at N=8 with the
page's NVLink constants the 14.4 MB crossover between Ring and the Double
Binary Tree, with Recursive Halving-Doubling preferred whenever N is a power
of 2 (it has Ring's bandwidth term and DBT's latency term); the HBM model
picks the fused one-pass schedule, which has the fewest steps and bytes.
"""
import pytest

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cost_model as cm
from oracle import selection


@pytest.fixture(autouse=True)
def _restore_model():
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    yield
    vc.vc_set_cost_model("hbm")


COLLS = ["allreduce", "reduce_scatter", "allgather", "broadcast", "scatter", "alltoall"]


@pytest.mark.parametrize("N", [2, 3, 6, 8, 16])
@pytest.mark.parametrize("alpha,beta", [(5e-6, 450e9), (1e-6, 1e12), (2e-5, 100e9)])
def test_link_model_choice_matches_oracle(N, alpha, beta):
    vc.vc_set_cost_model("link", alpha, beta)
    assert vc.vc_get_cost_model() == ("link", alpha, beta)
    for coll in COLLS:
        for count in [16, 1024, 1 << 16, 1 << 20, 5 << 20, 1 << 24]:
            got, t = vc.vc_select_algo(coll, N, count, "f32")
            want, tw = selection.select_link(coll, N, count, "f32", alpha, beta)
            assert got == want, (coll, N, count, got, want)
            assert t == pytest.approx(tw, rel=1e-12)


def test_link_model_reproduces_the_printed_crossover():
    """N=6 has no RHD, so AUTO switches from DBT to Ring at the crossover of
    eq. model-algo-ring-dbt-crossover; at N=8 the printed 14.4 MB is where Ring
    and DBT cost the same."""
    vc.vc_set_cost_model("link", 5e-6, 450e9)
    for N in (6, 12):
        mstar = cm.crossover_ring_dbt(N, 5e-6, 450e9)
        below = int(mstar * 0.98) // 4
        above = int(mstar * 1.02) // 4
        assert vc.vc_select_algo("allreduce", N, below)[0] == "dbt"
        assert vc.vc_select_algo("allreduce", N, above)[0] == "ring"
    assert cm.crossover_ring_dbt(8, 5e-6, 450e9) == pytest.approx(14.4e6)
    assert vc.vc_select_algo("allreduce", 8, 1 << 20)[0] == "rhd"


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 16])
def test_hbm_model_choice_matches_oracle(N):
    vc.vc_set_cost_model("hbm")
    pol, a, b = vc.vc_get_cost_model()
    assert pol == "hbm" and a == pytest.approx(1.9e-6) and b == pytest.approx(6.6e12)
    for coll in COLLS:
        for count in [64, 4096, 1 << 16]:
            for dtype in ("f32", "bf16"):
                got, t = vc.vc_select_algo(coll, N, count, dtype)
                want, tw = selection.select_hbm(coll, N, count, dtype, a, b)
                assert got == want, (coll, N, count, dtype, got, want)
                assert t == pytest.approx(tw, rel=1e-12)
                if N > 1:
                    assert got == "fused"


def test_auto_is_accepted_by_plan_describe():
    vc.vc_set_cost_model("link", 5e-6, 450e9)
    entries, _, nsteps = vc.vc_plan_describe("allreduce", "auto", 8, 1 << 20, "f32")
    assert nsteps == 6  # RHD
    vc.vc_set_cost_model("hbm")
    entries, _, nsteps = vc.vc_plan_describe("allreduce", "auto", 8, 1 << 20, "f32")
    assert nsteps == 1  # fused


def test_cost_model_refuses_non_finite_constants():
    """alpha or beta at or below 0 takes the policy's default; NaN or an
    infinite value is refused and leaves the model as it was."""
    vc.vc_set_cost_model("link", 2e-6, 300e9)
    before = vc.vc_get_cost_model()
    for a, b in ((float("nan"), 1e9), (1e-6, float("nan")), (float("inf"), 1e9), (1e-6, float("-inf"))):
        with pytest.raises(vc.VCError):
            vc.vc_set_cost_model("link", a, b)
        assert vc.vc_get_cost_model() == before
    vc.vc_set_cost_model("link", 0.0, -1.0)
    assert vc.vc_get_cost_model() == ("link", 5e-6, 450e9)
