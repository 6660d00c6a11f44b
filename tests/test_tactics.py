"""Host side of layout autotuning (rs_set_tactic / rs_reset_tactics /
rs_plan_linear, ResServe Sec. 5.1 Fig. 3): tactics replace the analytic plan
only for their own shape and SM count, a call of M rows takes the entry with
the smallest tuned row count >= M, tactics whose plans do not fit fall back,
out-of-range fields are refused, and every shipped GB300 entry gives a plan
that fits.  No GPU needed."""
import re

import pytest

from block_scaled_quantized_gb300 import build, rs, tune, workloads

SMS = 152


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    yield
    rs.rs_reset_tactics(True)


@pytest.fixture(autouse=True)
def _clean():
    rs.rs_reset_tactics(False)
    yield
    rs.rs_reset_tactics(True)


def plan(fmt, comp, M, N, K, sms=SMS, x_in_call=True):
    return rs.rs_plan_linear(fmt, comp, M, N, K, sms, x_in_call)


def test_tactic_replaces_the_plan_of_its_shape_only():
    base = plan(0, True, 8, 4096, 4096)
    assert base["tuned"] == 0
    rs.rs_set_tactic(0, True, 8, 4096, 4096, SMS, 8, 1, 32)
    p = plan(0, True, 8, 4096, 4096)
    assert (p["tuned"], p["splits"], p["bn"], p["fused"]) == (1, 8, 32, 1)
    assert plan(0, False, 8, 4096, 4096)["tuned"] == 0      # other mode
    assert plan(1, True, 8, 4096, 4096)["tuned"] == 0       # other format
    assert plan(0, True, 8, 4096, 2048)["tuned"] == 0       # other K
    assert plan(0, True, 8, 4096, 4096, sms=148)["tuned"] == 0  # other GPU
    assert plan(0, True, 9, 4096, 4096)["tuned"] == 0       # above the tuned M
    assert rs.rs_tactic_count() == 1


def test_lookup_takes_the_smallest_tuned_rows_at_least_m():
    rs.rs_set_tactic(0, False, 4, 2048, 2048, SMS, 2, 0, 16)
    rs.rs_set_tactic(0, False, 16, 2048, 2048, SMS, 3, 0, 32)
    for M, splits in ((1, 2), (4, 2), (5, 3), (16, 3)):
        p = plan(0, False, M, 2048, 2048)
        assert p["tuned"] == 1 and p["splits"] == splits, (M, p)
    assert plan(0, False, 17, 2048, 2048)["tuned"] == 0


def test_width_is_raised_to_what_the_rows_need():
    rs.rs_set_tactic(0, True, 32, 1024, 1024, SMS, 1, 0, 16)  # 64 rows need bn 64
    p = plan(0, True, 32, 1024, 1024)
    assert p["tuned"] == 1 and p["bn"] == 64


def test_fused_tactic_without_bf16_input_is_not_fused():
    rs.rs_set_tactic(0, True, 8, 4096, 4096, SMS, 4, 1, 16)
    assert plan(0, True, 8, 4096, 4096, x_in_call=True)["fused"] == 1
    p = plan(0, True, 8, 4096, 4096, x_in_call=False)
    assert p["tuned"] == 1 and p["fused"] == 0 and p["splits"] == 4


def test_tactics_that_do_not_fit_fall_back():
    rs.rs_set_tactic(0, True, 8, 1024, 512, SMS, 3, 0, 16)  # 3 splits of 2 chunks
    assert plan(0, True, 8, 1024, 512) == {**plan(0, True, 8, 1024, 512), "tuned": 0}
    base = dict(plan(0, True, 8, 1024, 512))
    rs.rs_reset_tactics(False)
    assert {k: v for k, v in plan(0, True, 8, 1024, 512).items()} == base


@pytest.mark.parametrize("fields", [(0, 0, 16, 0), (9, 0, 16, 0), (2, 3, 16, 0), (2, -1, 16, 0), (2, 0, 48, 0),
                                    (2, 0, 512, 0), (2, 0, 16, 2), (2, 0, 16, -1)])
def test_out_of_range_tactics_are_refused(fields):
    assert rs.lib().rs_set_tactic(0, 1, 8, 4096, 4096, SMS, *fields) == rs.RS_ERR_INVALID_ARG
    assert rs.rs_tactic_count() == 0


def test_argument_checks():
    lib = rs.lib()
    assert lib.rs_set_tactic(2, 1, 8, 4096, 4096, SMS, 1, 0, 16, 0) == rs.RS_ERR_INVALID_ARG
    assert lib.rs_set_tactic(0, 1, 0, 4096, 4096, SMS, 1, 0, 16, 0) == rs.RS_ERR_INVALID_ARG
    assert lib.rs_set_tactic(0, 1, 8, 4096, 4100, SMS, 1, 0, 16, 0) == rs.RS_ERR_SHAPE
    assert lib.rs_set_tactic(0, 1, 8, 4096, 4096, 0, 1, 0, 16, 0) == rs.RS_ERR_INVALID_ARG


def test_reset_restores_the_shipped_table():
    rs.rs_reset_tactics(True)
    shipped = rs.rs_tactic_count()
    rs.rs_set_tactic(0, True, 3, 333, 4096, SMS, 2, 0, 16)
    assert rs.rs_tactic_count() == shipped + 1
    rs.rs_reset_tactics(True)
    assert rs.rs_tactic_count() == shipped
    rs.rs_reset_tactics(False)
    assert rs.rs_tactic_count() == 0


def shipped_rows():
    path = rs.__file__.replace("rs.py", "csrc/rs_tactics_gb300.inc")
    rows = []
    for line in open(path):
        m = re.match(r"\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)\}", line)
        if m:
            rows.append(tuple(int(t) for t in m.groups()))
    return [r for r in rows if r[2] > 0]


def test_every_shipped_tactic_gives_its_plan():
    rs.rs_reset_tactics(True)
    rows = shipped_rows()
    assert rs.rs_tactic_count() == len(rows)
    keys = set()
    for fmt, comp, M, N, K, sms, splits, fused, bn, deep in rows:
        assert (fmt, comp, M, N, K, sms) not in keys
        keys.add((fmt, comp, M, N, K, sms))
        p = plan(fmt, comp, M, N, K, sms)
        assert p["tuned"] == 1 and p["splits"] == splits and p["bn"] == bn and p["fused"] == fused
        assert p["smem_bytes"] <= 232448 and p["tmem_cols"] <= 512


def test_candidate_set_contains_the_analytic_plan():
    """The tuner's search space holds the analytic plan of every tuned case,
    so a tuned plan is never one the tuner could not compare against it."""
    for fmt, N, K, Ms in tune.tuning_set(False):
        for M in Ms:
            for comp in (False, True):
                p = plan(fmt, comp, M, N, K)
                assert (p["splits"], p["fused"], p["bn"], 0) in set(tune.candidates(M, K, comp)), (fmt, N, K, M, comp)


def test_no_plan_lets_two_ctas_share_more_than_the_tensor_memory():
    for s, f, bn, deep in tune.candidates(8, 4096, True):
        rs.rs_reset_tactics(False)
        rs.rs_set_tactic(0, True, 8, 4096, 4096, SMS, s, f, bn, deep)
        p = plan(0, True, 8, 4096, 4096)
        if p["tmem_cols"] > 256:
            assert p["smem_bytes"] > 232448 // 2


def test_rows_that_kept_the_analytic_plan_reproduce_it():
    """Rows the tuner marked as the analytic plan give exactly that plan, so
    the table only records them to stop a call of M rows from taking the
    tactic of a larger tuned M."""
    path = rs.__file__.replace("rs.py", "csrc/rs_tactics_gb300.inc")
    n = 0
    for line in open(path):
        m = re.match(r"\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)\},.*\(analytic plan\)", line)
        if not m:
            continue
        fmt, comp, M, N, K, sms, splits, fused, bn, deep = (int(v) for v in m.groups())
        rs.rs_reset_tactics(False)
        a = plan(fmt, comp, M, N, K, sms)
        rs.rs_set_tactic(fmt, comp, M, N, K, sms, splits, fused, bn, deep)
        t = plan(fmt, comp, M, N, K, sms)
        assert {**a, "tuned": 1} == t, (fmt, comp, M, N, K)
        n += 1
    assert n > 0 or not shipped_rows()


def test_every_tuned_case_has_its_own_row():
    rows = {(r[0], r[1], r[2], r[3], r[4]) for r in shipped_rows()}
    if not rows:
        pytest.skip("no shipped table")
    for fmt, N, K, Ms in tune.tuning_set(False):
        for M in Ms:
            for comp in (0, 1):
                assert (fmt, comp, M, N, K) in rows, (fmt, comp, M, N, K)


def test_deep_tactic_keeps_the_deep_ring_of_a_split_plan():
    """deep = 1: a split plan whose CTAs take one tile each keeps the deepest
    weight ring that fits (one CTA per SM) instead of the shallow ring that
    lets two CTAs share an SM; plans without that cap are unchanged."""
    rs.rs_set_tactic(0, False, 1, 5120, 25600, SMS, 3, 0, 16, 0)
    shallow = plan(0, False, 1, 5120, 25600)
    rs.rs_set_tactic(0, False, 1, 5120, 25600, SMS, 3, 0, 16, 1)
    deep = plan(0, False, 1, 5120, 25600)
    assert shallow["tuned"] == deep["tuned"] == 1
    assert deep["stages"] > shallow["stages"] and shallow["smem_bytes"] <= 232448 // 2 < deep["smem_bytes"]
    assert deep["smem_bytes"] <= 232448
    same = ("bn", "n_tiles", "b_tiles", "chunks", "splits", "grid_x", "fused", "slots", "nacc")
    assert all(deep[k] == shallow[k] for k in same)
    for t in ((1, 0, 16), (4, 1, 16)):  # one split; a fused ring already past half the SM
        rs.rs_set_tactic(0, False, 1, 4096, 14336, SMS, *t, 0)
        p0 = plan(0, False, 1, 4096, 14336)
        rs.rs_set_tactic(0, False, 1, 4096, 14336, SMS, *t, 1)
        assert plan(0, False, 1, 4096, 14336) == p0 and p0["tuned"] == 1


def test_pair_tactic_pairs_only_where_the_grid_allows():
    """fused = 2: CTA pairs share the quantization of a K slice when the plan
    is fused, its CTAs per split are even and two clusters' worth of splits
    stay within 8 CTAs; otherwise the plan is the unpaired fused one."""
    rs.rs_set_tactic(0, True, 8, 4096, 4096, SMS, 4, 2, 16)
    assert plan(0, True, 8, 4096, 4096)["fused"] == 2          # 32 CTAs per split, 4 splits
    rs.rs_set_tactic(0, True, 8, 4096, 4096, SMS, 8, 2, 16)
    assert plan(0, True, 8, 4096, 4096)["fused"] == 1          # 16-CTA clusters would be needed
    rs.rs_set_tactic(0, True, 8, 384, 4096, SMS, 4, 2, 16)
    assert plan(0, True, 8, 384, 4096)["fused"] == 1           # 3 CTAs per split
    assert plan(0, True, 8, 4096, 4096, x_in_call=False)["fused"] == 0


def test_shipped_table_round_trips_through_the_tuner(tmp_path):
    """tune.py --min-rows reads the shipped table back to keep the rows it does
    not re-measure: parsing and writing it again gives the same file, and the
    rows it would keep for --min-rows 64 are exactly those under 64 rows."""
    import os
    src = os.path.join(os.path.dirname(tune.__file__), "csrc", "rs_tactics_gb300.inc")
    sms, rows = tune.rows_from_table(src)
    assert sms == SMS and len(rows) == sum(1 for line in open(src) if line.startswith("{")) - 1
    out = tmp_path / "table.inc"
    tune.write_table(str(out), sms, rows)
    assert out.read_text() == open(src).read()
    kept = [r for r in rows if (2 * r[2] if r[1] else r[2]) < 64]
    assert kept and all((2 * r[2] if r[1] else r[2]) < 64 for r in kept)
    retuned = sum(1 for _, _, _, Ms in tune.tuning_set(False) for M in Ms for comp in (0, 1)
                  if (2 * M if comp else M) >= 64)
    assert len(kept) + retuned == len(rows)
