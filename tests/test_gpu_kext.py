"""GPU parity of selective prefill compensation (K-Ext, ResServe Sec. 5.3
Eq. 6, App. A Eq. 7, App. B.2 Alg. 1) through the C ABI against the oracle:
the extended activation operand [X^ | R^_S] and the extended weight
[W^ | W^_S] bit-exact (codes and scale bytes, zero scale padding), and the
linear layer within max|dY| <= 1e-3 max|Y| on fp32 output, for both formats,
k in {1, 2, 4, 8}, ragged token counts, the bf16-input, pre-quantized and
own-tensor-scale paths, and sampled rows of the full prefill shape."""
import numpy as np
import pytest
import torch

import layout
from gpu_util import DEV, assert_close_f32, gpu_tensor_scale
from block_scaled_quantized_gb300 import rs, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()


def _mask(x, k, seed):
    """Masks from a calibration score (mean |x| of calibration rows drawn from
    the same recipe) through librs's host selection."""
    rng = np.random.default_rng(seed)
    score = np.abs(x.float().numpy()).mean(axis=0) * rng.uniform(0.5, 1.5, x.shape[1]).astype(np.float32)
    return rs.rs_kext_select(score, k)


def _prep_weight(fmt, w, k, mask):
    import oracle
    N, K = w.shape
    wg = w.to(DEV)
    aw = gpu_tensor_scale(wg) if fmt == 0 else None
    wq = torch.full((rs.rs_kext_weight_bytes(fmt, N, K, k),), 0xCD, dtype=torch.uint8, device=DEV)
    rs.rs_quantize_weight_kext(fmt, wg, k, aw, torch.from_numpy(mask).to(DEV), wq)
    torch.cuda.synchronize()
    wb = workloads.bf16_bits(w)
    aw_or = oracle.tensor_scale(wb) if fmt == 0 else np.float32(0)
    cw, sw = oracle.quantize_weight_kext(fmt, wb, k, mask, aw_or)
    return dict(wq=wq, aw=aw, aw_or=aw_or, cw=cw, sw=sw)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("k", [1, 2, 4, 8])
@pytest.mark.parametrize("rows,K", [(37, 256), (130, 512), (8, 1024)])
def test_extended_operand_bit_exact(fmt, k, rows, K):
    import oracle
    x = workloads.make_x("gauss_outlier_k2048", rows, K=K, seed=rows + K + k)
    mask = _mask(x, k, rows)
    xb = workloads.bf16_bits(x)
    a_or = oracle.tensor_scale(xb) if fmt == 0 else np.float32(0)
    a_gpu = torch.tensor([a_or], dtype=torch.float32, device=DEV) if fmt == 0 else None
    Ke = K + rs.rs_kext_width(K, k)
    buf = torch.full((rs.rs_kext_act_bytes(fmt, rows, K, k),), 0xAB, dtype=torch.uint8, device=DEV)
    rs.rs_quantize_kext(fmt, x.to(DEV), k, a_gpu, torch.from_numpy(mask).to(DEV), buf)
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    host = buf.cpu().numpy()
    codes, sf = layout.unpack_operand(host, fmt, rows, Ke)
    cx, sx = oracle.quantize_kext(fmt, xb, k, mask, a_or)
    np.testing.assert_array_equal(codes, cx)
    np.testing.assert_array_equal(sf, sx)
    assert not np.any(layout.padding_sf_bytes(host, fmt, rows, Ke))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("k", [1, 4])
def test_extended_weight_bit_exact(fmt, k):
    N, K = 300, 512
    w = workloads.make_w("gauss_outlier_k2048", N=N, K=K, seed=k + 40)
    mask = _mask(workloads.make_x("gauss_outlier_k2048", 16, K=K, seed=k), k, k)
    wp = _prep_weight(fmt, w, k, mask)
    codes, sf, pad_ok = layout.unpack_weight(wp["wq"].cpu().numpy(), fmt, N, K + rs.rs_kext_width(K, k))
    np.testing.assert_array_equal(codes, wp["cw"])
    np.testing.assert_array_equal(sf, wp["sw"])
    assert pad_ok


def _gpu_kext_linear(fmt, k, x, mask, wp, path, out_dtype=torch.float32):
    M, K = x.shape
    N = wp["cw"].shape[0]
    xg = x.to(DEV)
    mg = torch.from_numpy(mask).to(DEV)
    ax = gpu_tensor_scale(xg) if fmt == 0 else None
    y = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    if path == "prequantized":
        xq = torch.empty(rs.rs_kext_act_bytes(fmt, M, K, k), dtype=torch.uint8, device=DEV)
        rs.rs_quantize_kext(fmt, xg, k, ax, mg, xq)
        rs.rs_linear_kext(fmt, M, N, K, k, xq=xq, alpha_x=ax, wq=wp["wq"], alpha_w=wp["aw"], y=y)
    else:
        ws = torch.empty(rs.rs_kext_workspace_bytes(fmt, M, N, K, k), dtype=torch.uint8, device=DEV)
        rs.rs_linear_kext(fmt, M, N, K, k, x=xg, alpha_x=None if path == "own_scale" else ax, mask=mg,
                          wq=wp["wq"], alpha_w=wp["aw"], y=y, workspace=ws)
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    return y


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("k", [1, 2, 4, 8])
@pytest.mark.parametrize("M,N,K", [(64, 384, 512), (300, 256, 256), (520, 640, 1024)])
def test_kext_linear_parity(fmt, k, M, N, K):
    import oracle
    x = workloads.make_x("prefill_k8192", M, K=K, seed=M + k)
    w = workloads.make_w("prefill_k8192", N=N, K=K, seed=N + k)
    mask = _mask(x, k, k)
    wp = _prep_weight(fmt, w, k, mask)
    xb = workloads.bf16_bits(x)
    ax = oracle.tensor_scale(xb) if fmt == 0 else np.float32(0)
    ref = oracle.linear_kext(fmt, xb, k, mask, ax, wp["cw"], wp["sw"], wp["aw_or"])
    y = _gpu_kext_linear(fmt, k, x, mask, wp, "x")
    assert_close_f32(y, ref)
    y2 = _gpu_kext_linear(fmt, k, x, mask, wp, "prequantized")
    assert torch.equal(y, y2)


def test_kext_own_scale_and_bf16():
    import oracle
    M, N, K, k = 200, 256, 1024, 2
    x = workloads.make_x("prefill_k8192", M, K=K, seed=9)
    w = workloads.make_w("prefill_k8192", N=N, K=K, seed=10)
    mask = _mask(x, k, 3)
    wp = _prep_weight(0, w, k, mask)
    y_given = _gpu_kext_linear(0, k, x, mask, wp, "x")
    y_own = _gpu_kext_linear(0, k, x, mask, wp, "own_scale")
    assert torch.equal(y_given, y_own)
    yb = _gpu_kext_linear(0, k, x, mask, wp, "x", out_dtype=torch.bfloat16)
    assert torch.equal(yb, y_given.to(torch.bfloat16))


def test_channel_mean_abs():
    x = workloads.make_x("prefill_k8192", 96, K=512, seed=4)
    score = torch.empty(512, dtype=torch.float32, device=DEV)
    rs.rs_channel_mean_abs(x.to(DEV), score)
    torch.cuda.synchronize()
    ref = np.abs(x.float().numpy()).astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(score.cpu().numpy(), ref, rtol=2e-6)


def test_kext_full_prefill_shape_sampled_rows():
    """M = 4096, K = N = 8192, rho = 0.125 (k = 1): every output checked on
    32 sampled token rows (quantization is row-local, so the oracle runs on
    those rows alone)."""
    import oracle
    M, K, k = 4096, 8192, 1
    x = workloads.make_x("prefill_k8192", M)
    w = workloads.make_w("prefill_k8192")
    N = w.shape[0]
    mask = _mask(x[:256], k, 1)
    wp = _prep_weight(0, w, k, mask)
    xg = x.to(DEV)
    ax = gpu_tensor_scale(xg)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    ws = torch.empty(rs.rs_kext_workspace_bytes(0, M, N, K, k), dtype=torch.uint8, device=DEV)
    rs.rs_linear_kext(0, M, N, K, k, x=xg, alpha_x=ax, mask=torch.from_numpy(mask).to(DEV), wq=wp["wq"],
                      alpha_w=wp["aw"], y=y, workspace=ws)
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    rows = np.random.default_rng(0).choice(M, 32, replace=False)
    xb = workloads.bf16_bits(x[torch.from_numpy(rows)])
    ref = oracle.linear_kext(0, xb, k, mask, ax.cpu().numpy()[0], wp["cw"], wp["sw"], wp["aw_or"])
    assert_close_f32(y[torch.from_numpy(rows).to(DEV)], ref)


# Large NVFP4 operands (rows x K/256 >= 128 per SM, K a multiple of 512)
# take the quantizer with one 16-element base block (two selection groups)
# per lane: the extended operand must be the same, bit for bit, on every row.
@pytest.mark.parametrize("k", [1, 2, 4, 8])
@pytest.mark.parametrize("rows,K", [(700, 8192), (3300, 1536)])
def test_extended_operand_bit_exact_large(k, rows, K):
    import oracle
    x = workloads.make_x("prefill_k8192", rows, K=K, seed=rows + k)
    mask = _mask(x[:256], k, rows + k)
    xb = workloads.bf16_bits(x)
    a_or = oracle.tensor_scale(xb)
    Ke = K + rs.rs_kext_width(K, k)
    buf = torch.full((rs.rs_kext_act_bytes(0, rows, K, k),), 0xAB, dtype=torch.uint8, device=DEV)
    rs.rs_quantize_kext(0, x.to(DEV), k, torch.tensor([a_or], dtype=torch.float32, device=DEV),
                        torch.from_numpy(mask).to(DEV), buf)
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    host = buf.cpu().numpy()
    codes, sf = layout.unpack_operand(host, 0, rows, Ke)
    cx, sx = oracle.quantize_kext(0, xb, k, mask, a_or)
    np.testing.assert_array_equal(codes, cx)
    np.testing.assert_array_equal(sf, sx)
    assert not np.any(layout.padding_sf_bytes(host, 0, rows, Ke))


# Large K-Ext operands outside the one-block-per-lane kernel (MXFP4, or NVFP4
# with K not a multiple of 512): four chunks per warp step, ragged last group.
@pytest.mark.parametrize("fmt,k,rows,K", [(1, 1, 700, 8192), (1, 4, 600, 8448), (0, 2, 600, 8448)])
def test_extended_operand_bit_exact_large_four_chunk_steps(fmt, k, rows, K):
    import oracle
    x = workloads.make_x("prefill_k8192", rows, K=K, seed=rows + k + fmt)
    mask = _mask(x[:256], k, rows + k)
    xb = workloads.bf16_bits(x)
    a_or = oracle.tensor_scale(xb) if fmt == 0 else np.float32(0)
    a_gpu = torch.tensor([a_or], dtype=torch.float32, device=DEV) if fmt == 0 else None
    Ke = K + rs.rs_kext_width(K, k)
    buf = torch.full((rs.rs_kext_act_bytes(fmt, rows, K, k),), 0xAB, dtype=torch.uint8, device=DEV)
    rs.rs_quantize_kext(fmt, x.to(DEV), k, a_gpu, torch.from_numpy(mask).to(DEV), buf)
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    host = buf.cpu().numpy()
    codes, sf = layout.unpack_operand(host, fmt, rows, Ke)
    cx, sx = oracle.quantize_kext(fmt, xb, k, mask, a_or)
    np.testing.assert_array_equal(codes, cx)
    np.testing.assert_array_equal(sf, sx)
    assert not np.any(layout.padding_sf_bytes(host, fmt, rows, Ke))
