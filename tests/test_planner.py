"""Host-side launch planner of the linear calls (no GPU): structural limits of
every plan over a grid of shapes, formats and SM counts, and the decisions
that GB300 measurements fixed (the cost of extra tiles in split plans, two
CTAs per SM for single-tile split plans, the headline configuration)."""
import itertools

import pytest

from block_scaled_quantized_gb300 import rs, workloads

SMEM_LIMIT = 232448  # 227 KB opt-in shared memory per block


@pytest.fixture(autouse=True, params=["analytic", "shipped"])
def tactics(request):
    """Structural limits hold for the analytic plans and for the shipped
    measured tactics alike; the cost-rule tests below check the analytic
    planner alone (a measured tactic may override a rule where it measured
    faster)."""
    rs.rs_reset_tactics(request.param == "shipped")
    yield request.param
    rs.rs_reset_tactics(True)

SHAPES = sorted(set(workloads.PROJECTION_SHAPES) | {(4096, 4096), (2048, 2048), (28672, 4096), (4096, 14336),
                                                    (27648, 5120), (8192, 8192), (256, 256), (128, 32)})
MS = [1, 2, 4, 8, 16, 32, 64, 128, 512, 4096]


def _ntl(p):
    tiles = p["n_tiles"] * p["b_tiles"]
    return (tiles + p["grid_x"] - 1) // p["grid_x"]


@pytest.mark.parametrize("sms", [152, 148, 132])
@pytest.mark.parametrize("fmt,comp,x_in_call", list(itertools.product([0, 1], [False, True], [False, True])))
def test_plan_limits(sms, fmt, comp, x_in_call):
    for (N, K), M in itertools.product(SHAPES, MS):
        if K % 32:
            continue
        p = rs.rs_plan_linear(fmt, comp, M, N, K, sms, x_in_call)
        rows = 2 * M if comp else M
        where = (fmt, comp, x_in_call, M, N, K, sms, p)
        assert p["bn"] in (16, 32, 64, 128, 256), where
        assert p["n_tiles"] == (N + 127) // 128 and p["chunks"] == (K + 255) // 256, where
        assert p["b_tiles"] == (rows + p["bn"] - 1) // p["bn"], where
        assert 1 <= p["splits"] <= min(8, p["chunks"]), where
        assert 1 <= p["grid_x"] <= p["n_tiles"] * p["b_tiles"], where
        assert p["grid_x"] * p["splits"] <= sms, where
        assert 1 <= p["stages"] <= 8, where
        assert 0 < p["smem_bytes"] <= SMEM_LIMIT, where
        assert p["tmem_cols"] in (32, 64, 128, 256, 512), where
        assert p["nacc"] in (1, 2) and p["nacc"] * p["bn"] <= p["tmem_cols"], where
        if p["splits"] > 1 and p["smem_bytes"] <= SMEM_LIMIT // 2:
            # CTAs of one cluster may then share an SM and wait on each other:
            # each must get its tensor memory without waiting for the other's
            assert p["tmem_cols"] <= 256, where
        if p["fused"]:
            assert x_in_call and p["b_tiles"] == 1 and p["bn"] <= 32, where
            assert p["slots"] == (p["chunks"] + p["splits"] - 1) // p["splits"] <= 64, where
        else:
            assert p["slots"] == 0, where


def test_headline_plan(tactics):
    """Compensated NVFP4, M = 8, K = N = 4096: one fused launch of 32 tiles x
    4 K splits, 16-column MMAs, small enough for two CTAs per SM (the
    analytic plan, which the shipped table keeps for this shape)."""
    p = rs.rs_plan_linear(0, True, 8, 4096, 4096, 152)
    assert (p["bn"], p["splits"], p["grid_x"], p["fused"]) == (16, 4, 32, 1)
    assert p["smem_bytes"] <= SMEM_LIMIT // 2


@pytest.mark.parametrize("N,K", [(24576, 4096), (34816, 5120), (51200, 5120), (14336, 5120), (10240, 5120)])
def test_split_plans_do_not_stream_many_tiles(N, K, tactics):
    """Measured: a split plan pays each extra tile with a cross-CTA reduction
    that holds the whole cluster (24576 x 4096 with 8 splits x 11 tiles per CTA
    took 64 us; 2 splits x 3 tiles 15 us)."""
    if tactics == "shipped":
        pytest.skip("cost rule of the analytic planner")
    for comp in (False, True):
        p = rs.rs_plan_linear(0, comp, 8, N, K, 152)
        assert p["splits"] * (_ntl(p) - 1) <= 4, p


@pytest.mark.parametrize("N,K", [(2560, 8192), (2560, 9728), (6144, 4096), (4608, 8192)])
def test_single_tile_split_plans_share_sms(N, K, tactics):
    """Measured: with one CTA per SM, 20 clusters of 7 (or 36 of 4) do not all
    fit into the GPCs at once and half the grid ran as a second wave (2x)."""
    if tactics == "shipped":
        pytest.skip("cost rule of the analytic planner")
    for comp in (False, True):
        p = rs.rs_plan_linear(0, comp, 8, N, K, 152)
        if p["splits"] > 1 and _ntl(p) == 1:
            assert p["smem_bytes"] <= SMEM_LIMIT // 2, p


def test_plan_rejects_bad_arguments():
    with pytest.raises(rs.RsError):
        rs.rs_plan_linear(0, True, 0, 4096, 4096, 152)
    with pytest.raises(rs.RsError):
        rs.rs_plan_linear(0, True, 8, 4096, 100, 152)
    with pytest.raises(rs.RsError):
        rs.rs_plan_linear(3, True, 8, 4096, 4096, 152)


def test_multicast_rule(tactics):
    """The activation tile is shared by multicast only by 256-row TMA-fed
    plans without K split, with an even number of channel tiles and at least
    two output tiles per CTA; every other plan loads its own."""
    for sms in (152, 148, 132):
        for fmt, comp, M, N, K in [(0, False, 4096, 8192, 8192), (0, True, 4096, 8192, 8192),
                                   (1, True, 512, 27648, 5120), (0, False, 1024, 4096, 4096),
                                   (1, True, 128, 27648, 5120), (0, True, 64, 4096, 4096),
                                   (0, True, 8, 4096, 4096), (0, False, 4096, 8320, 8192)]:
            p = rs.rs_plan_linear(fmt, comp, M, N, K, sms)
            tiles = p["n_tiles"] * p["b_tiles"]
            want = (p["bn"] == 256 and not p["fused"] and p["splits"] == 1 and p["n_tiles"] % 2 == 0
                    and tiles >= 2 * p["grid_x"])
            assert p["mcast"] == int(want), (fmt, comp, M, N, K, sms, p)
    # the prefill shape shares it; one tile per CTA (W4A4 M = 1024, K = N = 4096:
    # 128 tiles) and an odd channel-tile count (N = 8320) do not
    assert rs.rs_plan_linear(0, False, 4096, 8192, 8192, 152)["mcast"] == 1
    assert rs.rs_plan_linear(0, True, 4096, 8192, 8192, 152)["mcast"] == 1
    assert rs.rs_plan_linear(0, False, 1024, 4096, 4096, 152)["mcast"] == 0
    assert rs.rs_plan_linear(0, False, 4096, 8320, 8192, 152)["mcast"] == 0
