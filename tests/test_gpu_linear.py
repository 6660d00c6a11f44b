"""GPU parity of the W4A4 and residue-compensated linear layers through the
C ABI against the oracle: max|Y_gpu - Y_oracle| <= 1e-3 max|Y_oracle| on the
fp32 output (ResServe Sec. 4.2 Eq. 1, Sec. 4.3 Eq. 2); bf16 output within one
bf16 ulp of the rounded oracle plus the same bound.  Shapes span several
128-channel tiles, ragged channel / token / K tails, split-K and multi-tile
activation operands; the workload configurations are checked at full size
on sampled tokens and channels."""
import numpy as np
import pytest
import torch

from gpu_util import (DEV, assert_close_bf16, assert_close_f32, gpu_linear, gpu_tensor_scale,
                      oracle_linear, prepare_weight)
from block_scaled_quantized_gb300 import rs, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()


SHAPES = [(1, 128, 256), (2, 256, 512), (3, 384, 288), (8, 200, 1024), (8, 1024, 4096), (17, 256, 2048),
          (64, 512, 512), (130, 256, 512), (300, 384, 256)]


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("compensated", [False, True])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_parity_small(fmt, compensated, M, N, K):
    x = workloads.make_x("gauss_outlier_k2048", M, K=K, seed=M + N + K)
    w = workloads.make_w("gauss_outlier_k2048", N=N, K=K, seed=N * 7 + K)
    wp = prepare_weight(fmt, w)
    y, _ = gpu_linear(fmt, compensated, x, wp)
    ref = oracle_linear(fmt, compensated, x, wp)
    assert_close_f32(y, ref)


# More 128-channel tiles than a GB300 has SMs per K split, so that CTAs run
# several tiles (double-buffered accumulators, per-tile split-K exchange):
# fused and TMA-fed activations, ragged channel and K tails, two activation
# row tiles.
SHAPES_MULTI_TILE = [(3, 20416, 512), (8, 40960, 288), (40, 20480, 768), (300, 12800, 256)]


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("compensated", [False, True])
@pytest.mark.parametrize("M,N,K", SHAPES_MULTI_TILE)
def test_linear_parity_multi_tile(fmt, compensated, M, N, K):
    x = workloads.make_x("gauss_outlier_k2048", M, K=K, seed=M + N + K)
    w = workloads.make_w("gauss_outlier_k2048", N=N, K=K, seed=N * 7 + K)
    wp = prepare_weight(fmt, w)
    y, _ = gpu_linear(fmt, compensated, x, wp)
    ref = oracle_linear(fmt, compensated, x, wp)
    assert_close_f32(y, ref)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("compensated", [False, True])
def test_prequantized_input_matches(fmt, compensated):
    M, N, K = 5, 384, 1024
    x = workloads.make_x("attn_proj_k4096", M, K=K, seed=5)
    w = workloads.make_w("attn_proj_k4096", N=N, K=K, seed=6)
    wp = prepare_weight(fmt, w)
    y1, _ = gpu_linear(fmt, compensated, x, wp, prequantized=False)
    y2, _ = gpu_linear(fmt, compensated, x, wp, prequantized=True)
    torch.testing.assert_close(y1, y2, rtol=0, atol=0)
    assert_close_f32(y2, oracle_linear(fmt, compensated, x, wp))


@pytest.mark.parametrize("compensated", [False, True])
def test_bf16_output(compensated):
    M, N, K = 8, 512, 2048
    x = workloads.make_x("attn_proj_k4096", M, K=K, seed=8)
    w = workloads.make_w("attn_proj_k4096", N=N, K=K, seed=9)
    wp = prepare_weight(0, w)
    y, _ = gpu_linear(0, compensated, x, wp, out_dtype=torch.bfloat16)
    assert_close_bf16(y, oracle_linear(0, compensated, x, wp))


def test_deterministic_and_repeatable():
    M, N, K = 8, 4096, 4096
    x = workloads.make_x("attn_proj_k4096", M)
    w = workloads.make_w("attn_proj_k4096")
    wp = prepare_weight(0, w)
    y1, ws = gpu_linear(0, True, x, wp)
    # second call on the same workspace: counters were re-armed
    xg = x.to(DEV)
    ax = gpu_tensor_scale(xg)
    y2 = torch.empty_like(y1)
    rs.rs_linear_compensated(0, M, N, K, x=xg, alpha_x=ax, wq=wp["wq"], alpha_w=wp["aw"], y=y2, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("fmt,recipe", [(0, "gauss_outlier_k2048"), (0, "attn_proj_k4096"), (1, "mx_k5120_n27648")])
def test_compensation_lowers_error_on_gpu(fmt, recipe):
    import oracle
    M, N, K = 8, 1024, 2048
    x = workloads.make_x(recipe, M, K=K, seed=30)
    w = workloads.make_w(recipe, N=N, K=K, seed=31)
    wp = prepare_weight(fmt, w)
    ref = (x.double() @ w.double().T).numpy()
    yp, _ = gpu_linear(fmt, False, x, wp)
    yc, _ = gpu_linear(fmt, True, x, wp)
    assert oracle.nmse(yc.cpu().numpy(), ref) < oracle.nmse(yp.cpu().numpy(), ref)


# ---- workload configurations at full size, sampled tokens / channels ----

def _sampled_parity(fmt, compensated, recipe, M, n_rows=256, n_tok=None, seed=0):
    import oracle
    x = workloads.make_x(recipe, M)
    w = workloads.make_w(recipe)
    N, K = w.shape
    x_gpu, w_gpu = x.to(DEV), w.to(DEV)
    ax = gpu_tensor_scale(x_gpu) if fmt == 0 else None
    aw = gpu_tensor_scale(w_gpu) if fmt == 0 else None
    wq = torch.empty(rs.rs_weight_bytes(fmt, N, K), dtype=torch.uint8, device=DEV)
    rs.rs_quantize_weight(fmt, w_gpu, aw, wq)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    ws = rs.empty_workspace(fmt, M, N, K, compensated)
    fn = rs.rs_linear_compensated if compensated else rs.rs_linear_w4a4
    fn(fmt, M, N, K, x=x_gpu, alpha_x=ax, wq=wq, alpha_w=aw, y=y, workspace=ws)
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    rng = np.random.default_rng(seed)
    cols = np.sort(rng.choice(N, size=min(n_rows, N), replace=False))
    toks = np.arange(M) if n_tok is None else np.sort(rng.choice(M, size=n_tok, replace=False))
    xb, wb = workloads.bf16_bits(x), workloads.bf16_bits(w)
    ax_or = oracle.tensor_scale(xb) if fmt == 0 else np.float32(0)
    aw_or = oracle.tensor_scale(wb) if fmt == 0 else np.float32(0)
    if fmt == 0:
        assert ax.item() == ax_or and aw.item() == aw_or
    cw, sw, _ = oracle.quantize(fmt, np.ascontiguousarray(wb[cols]), aw_or)
    ref = oracle.linear(fmt, compensated, np.ascontiguousarray(xb[toks]), ax_or, cw, sw, aw_or)
    ys = y[torch.from_numpy(toks).to(DEV)][:, torch.from_numpy(cols).to(DEV)]
    assert_close_f32(ys, ref)


@pytest.mark.parametrize("compensated", [False, True])
def test_config_gauss_outlier_m1(compensated):
    _sampled_parity(0, compensated, "gauss_outlier_k2048", 1, n_rows=2048)


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("compensated", [False, True])
def test_config_attn_proj(M, compensated):
    _sampled_parity(0, compensated, "attn_proj_k4096", M, n_rows=4096)


@pytest.mark.parametrize("recipe", ["mlp_gate_up", "mlp_down"])
def test_config_mlp_pair(recipe):
    _sampled_parity(0, True, recipe, 8, n_rows=512)


@pytest.mark.parametrize("M", [1, 8, 64, 128])
@pytest.mark.parametrize("compensated", [False, True])
def test_config_mxfp4(M, compensated):
    _sampled_parity(1, compensated, "mx_k5120_n27648", M, n_rows=384)


@pytest.mark.parametrize("compensated", [False, True])
def test_config_prefill(compensated):
    _sampled_parity(0, compensated, "prefill_k8192", 4096, n_rows=128, n_tok=32)


# The activation tensor scale found by the call itself (alpha_x omitted):
# the same a = fl(amax(X)/2688) as rs_compute_tensor_scale (App. B.2 Eq. 8),
# so Y is bit-identical to the call given that scale, and matches the
# oracle.  Fused plans (one K split and several, one tile per CTA and
# several) and two-kernel plans.
DYN_SHAPES = [(8, 4096, 4096), (1, 2048, 2048), (3, 20416, 512), (8, 1024, 14336), (40, 512, 768),
              (300, 384, 256)]


@pytest.mark.parametrize("compensated", [False, True])
@pytest.mark.parametrize("M,N,K", DYN_SHAPES)
def test_tensor_scale_found_in_call(compensated, M, N, K):
    x = workloads.make_x("attn_proj_k4096", M, K=K, seed=M * 3 + K)
    w = workloads.make_w("attn_proj_k4096", N=N, K=K, seed=N + K)
    wp = prepare_weight(0, w)
    y_given, _ = gpu_linear(0, compensated, x, wp)
    y = torch.full_like(y_given, float("nan"))
    ws = rs.empty_workspace(0, M, N, K, compensated)
    fn = rs.rs_linear_compensated if compensated else rs.rs_linear_w4a4
    fn(0, M, N, K, x=x.to(DEV), alpha_x=None, wq=wp["wq"], alpha_w=wp["aw"], y=y, workspace=ws)
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    assert torch.equal(y, y_given)
    assert_close_f32(y, oracle_linear(0, compensated, x, wp))


def test_tensor_scale_in_call_flags_non_finite_input():
    M, N, K = 4, 256, 512
    x = workloads.make_x("attn_proj_k4096", M, K=K, seed=11)
    x[2, 100] = float("inf")
    wp = prepare_weight(0, workloads.make_w("attn_proj_k4096", N=N, K=K, seed=12))
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    ws = rs.empty_workspace(0, M, N, K, True)
    rs.rs_linear_compensated(0, M, N, K, x=x.to(DEV), alpha_x=None, wq=wp["wq"], alpha_w=wp["aw"], y=y,
                             workspace=ws)
    assert rs.rs_get_device_error() == rs.RS_ERR_INVALID_ARG


@pytest.mark.parametrize("M,N", [(1, 4096), (8, 4096), (5, 387), (64, 1024)])
def test_separate_fold_pipeline(M, N):
    """The unfused alternative the on-chip Fold is measured against (Sec. 5.1,
    Fig. 6b): the paired operand through the plain GEMM as 2M rows with fp32
    output (the expanded Z), then the Fold kernel.  The Fold is the fp32 sum
    of row pairs (bit-exact against torch), and the pipeline matches the
    oracle's compensated layer within the output tolerance."""
    K = 1024
    x = workloads.make_x("attn_proj_k4096", M, K=K, seed=M + 1)
    w = workloads.make_w("attn_proj_k4096", N=N, K=K, seed=N)
    wp = prepare_weight(0, w)
    x_gpu = x.to(DEV)
    ax = gpu_tensor_scale(x_gpu)
    xq = torch.empty(rs.rs_operand_bytes(0, 2 * M, K), dtype=torch.uint8, device=DEV)
    rs.rs_quantize_residue(0, x_gpu, ax, xq)
    z = torch.full((2 * M, N), float("nan"), dtype=torch.float32, device=DEV)
    rs.rs_linear_w4a4(0, 2 * M, N, K, xq=xq, alpha_x=ax, wq=wp["wq"], alpha_w=wp["aw"], y=z)
    y32 = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    y16 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    rs.rs_fold_pairs(M, N, z, y32)
    rs.rs_fold_pairs(M, N, z, y16)
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    want = z[0::2] + z[1::2]
    assert torch.equal(y32, want)
    assert torch.equal(y16, want.to(torch.bfloat16))
    assert_close_f32(y32, oracle_linear(0, True, x, wp))


PAIR_SHAPES = [(0, False, 512, 256, 256), (0, False, 700, 512, 800), (0, True, 256, 256, 512),
               (0, True, 300, 1024, 2048), (1, False, 512, 512, 512), (1, True, 600, 768, 1024),
               (0, False, 1100, 20480, 512)]


@pytest.mark.parametrize("fmt,compensated,M,N,K", PAIR_SHAPES)
def test_paired_cta_gemm_parity(fmt, compensated, M, N, K):
    """The paired-CTA kernel (tcgen05.mma.cta_group::2, 256 x 256 per pair)
    against the oracle: one and several pair tiles per pair, ragged M, N and
    K, both formats, fp32 and bf16 output."""
    x = workloads.make_x("gauss_outlier_k2048", M, K=K, seed=M + N + K)
    w = workloads.make_w("gauss_outlier_k2048", N=N, K=K, seed=N * 7 + K)
    wp = prepare_weight(fmt, w)
    rs.rs_debug_pair_gemm(True)
    try:
        y, _ = gpu_linear(fmt, compensated, x, wp)
        yb, _ = gpu_linear(fmt, compensated, x, wp, out_dtype=torch.bfloat16)
    finally:
        rs.rs_debug_pair_gemm(False)
    ref = oracle_linear(fmt, compensated, x, wp)
    assert_close_f32(y, ref)
    assert_close_bf16(yb, ref)
