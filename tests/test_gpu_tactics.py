"""GPU parity of plans chosen by measured launch tactics (layout autotuning,
ResServe Sec. 5.1 Fig. 3) against the oracle: every K-split count, in-GEMM
quantization on and off, and MMA widths up to four times the one the
activation rows need (zero-padded operand rows), on shapes with several
channel tiles and ragged tails; and the shipped GB300 table's tactics at
full size.  Bar: max|Y_gpu - Y_oracle| <= 1e-3 max|Y_oracle| (fp32 output)."""
import pytest
import torch

from gpu_util import assert_close_f32, gpu_linear, oracle_linear, prepare_weight
from block_scaled_quantized_gb300 import rs, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()
    yield
    rs.rs_reset_tactics(True)


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


# (M, N, K, splits, fused, bn)
FORCED = [(5, 384, 1024, 1, 1, 32), (5, 384, 1024, 3, 1, 32), (5, 384, 1024, 4, 0, 64),
          (8, 640, 2048, 8, 1, 32), (8, 640, 2048, 8, 0, 16), (8, 640, 2048, 2, 0, 128),
          (3, 200, 1280, 5, 1, 16), (16, 256, 2304, 6, 0, 64), (30, 384, 512, 2, 0, 256),
          (64, 256, 1024, 4, 0, 256), (100, 130, 768, 3, 0, 256),
          (4, 384, 16640, 2, 1, 16), (3, 256, 12320, 1, 1, 16)]  # fused slices of 33 and 49 chunks


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("compensated", [False, True])
@pytest.mark.parametrize("M,N,K,splits,fused,bn", FORCED)
def test_forced_tactic_parity(fmt, compensated, M, N, K, splits, fused, bn):
    rs.rs_reset_tactics(False)
    try:
        rs.rs_set_tactic(fmt, compensated, M, N, K, sms(), splits, fused, bn)
        plan = rs.rs_plan_linear(fmt, compensated, M, N, K, sms())
        # W4A4 at width 256 with split-K buffers does not fit: the analytic plan runs
        assert plan["tuned"] == (0 if (not compensated and bn == 256) else 1)
        assert plan["splits"] == splits or not plan["tuned"]
        x = workloads.make_x("gauss_outlier_k2048", M, K=K, seed=M * 3 + K)
        w = workloads.make_w("gauss_outlier_k2048", N=N, K=K, seed=N + 5 * K)
        wp = prepare_weight(fmt, w)
        y, _ = gpu_linear(fmt, compensated, x, wp)
        assert_close_f32(y, oracle_linear(fmt, compensated, x, wp))
    finally:
        rs.rs_reset_tactics(True)


# deep weight rings (M, N, K, splits, fused, bn): some wrap the ring several times
DEEP = [(8, 640, 8192, 4, 1, 16), (3, 384, 6144, 3, 0, 32), (1, 768, 12288, 2, 0, 16),
        (16, 256, 8192, 6, 1, 16), (5, 1024, 4096, 3, 0, 16)]


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("compensated", [False, True])
@pytest.mark.parametrize("M,N,K,splits,fused,bn", DEEP)
def test_deep_tactic_parity(fmt, compensated, M, N, K, splits, fused, bn):
    rs.rs_reset_tactics(False)
    try:
        rs.rs_set_tactic(fmt, compensated, M, N, K, sms(), splits, fused, bn, 0)
        shallow = rs.rs_plan_linear(fmt, compensated, M, N, K, sms())
        rs.rs_set_tactic(fmt, compensated, M, N, K, sms(), splits, fused, bn, 1)
        plan = rs.rs_plan_linear(fmt, compensated, M, N, K, sms())
        assert plan["tuned"] == 1 and plan["splits"] == splits and plan["stages"] >= shallow["stages"]
        x = workloads.make_x("gauss_outlier_k2048", M, K=K, seed=M * 7 + K)
        w = workloads.make_w("gauss_outlier_k2048", N=N, K=K, seed=N + 3 * K)
        wp = prepare_weight(fmt, w)
        y, _ = gpu_linear(fmt, compensated, x, wp)
        assert_close_f32(y, oracle_linear(fmt, compensated, x, wp))
    finally:
        rs.rs_reset_tactics(True)


def shipped_cases(limit):
    """Shipped table entries for this GPU, small enough for the oracle at full
    size, spread over split counts and widths."""
    import re
    path = rs.__file__.replace("rs.py", "csrc/rs_tactics_gb300.inc")
    rows = []
    for line in open(path):
        m = re.match(r"\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)\}", line)
        if m:
            v = [int(t) for t in m.groups()]
            if v[2] > 0 and v[5] == sms() and v[2] <= 16 and v[3] * v[4] <= 40_000_000:
                rows.append(v)
    picked, seen = [], set()
    for v in rows:
        key = (v[6], v[8], v[7])
        if key not in seen:
            seen.add(key)
            picked.append(v)
    return picked[:limit]


def test_shipped_tactics_full_size():
    cases = shipped_cases(6)
    if not cases:
        pytest.skip("no shipped tactics for this GPU's SM count")
    rs.rs_reset_tactics(True)
    for fmt, comp, M, N, K, _, splits, fused, bn, deep in cases:
        plan = rs.rs_plan_linear(fmt, comp, M, N, K, sms())
        assert plan["tuned"] == 1 and plan["splits"] == splits
        x = workloads.make_x("proj_shapes", M, K=K, seed=M + N)
        w = workloads.make_w("proj_shapes", N=N, K=K, seed=K)
        wp = prepare_weight(fmt, w)
        y, _ = gpu_linear(fmt, bool(comp), x, wp)
        assert_close_f32(y, oracle_linear(fmt, bool(comp), x, wp))
