"""GPU parity of the quantizers through the C ABI: codes and scale bytes
bit-exact against the oracle (ResServe App. B.2 Eq. 8-10, Alg. 1), padding
scale bytes zero, tensor scale bit-exact."""
import numpy as np
import pytest
import torch

import layout
from gpu_util import DEV, gpu_quantize, gpu_tensor_scale, unpack
from block_scaled_quantized_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()


@pytest.mark.parametrize("recipe", ["gauss_outlier_k2048", "attn_proj_k4096", "mlp_down",
                                    "mx_k5120_n27648", "prefill_k8192"])
def test_tensor_scale_bit_exact(recipe):
    import oracle
    x = workloads.make_x(recipe, 8)
    a = gpu_tensor_scale(x.to(DEV)).cpu().numpy()[0]
    assert a == oracle.tensor_scale(workloads.bf16_bits(x))
    w = workloads.make_w(recipe, N=256)
    a = gpu_tensor_scale(w.to(DEV)).cpu().numpy()[0]
    assert a == oracle.tensor_scale(workloads.bf16_bits(w))


def _check(fmt, x, paired, alpha=None):
    import oracle
    rows, K = x.shape
    xb = workloads.bf16_bits(x.cpu())
    a_or = oracle.tensor_scale(xb) if (fmt == 0 and alpha is None) else np.float32(alpha or 0)
    a_gpu = torch.tensor([a_or], dtype=torch.float32, device=DEV) if fmt == 0 else None
    buf = gpu_quantize(fmt, x.to(DEV) if not x.is_cuda else x, a_gpu, paired)
    host = buf.cpu().numpy()
    if paired:
        ref = oracle.quantize_residue(fmt, xb, a_or)
        codes, sf = layout.unpack_operand(host, fmt, 2 * rows, K)
        np.testing.assert_array_equal(codes[0::2], ref["codes_x"])
        np.testing.assert_array_equal(sf[0::2], ref["sf_x"])
        np.testing.assert_array_equal(codes[1::2], ref["codes_r"])
        np.testing.assert_array_equal(sf[1::2], ref["sf_r"])
        assert not np.any(layout.padding_sf_bytes(host, fmt, 2 * rows, K))
    else:
        cx, sx, _ = oracle.quantize(fmt, xb, a_or)
        codes, sf = layout.unpack_operand(host, fmt, rows, K)
        np.testing.assert_array_equal(codes, cx)
        np.testing.assert_array_equal(sf, sx)
        assert not np.any(layout.padding_sf_bytes(host, fmt, rows, K))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("paired", [False, True])
@pytest.mark.parametrize("rows,K", [(1, 32), (1, 2048), (2, 96), (3, 288), (7, 1024), (8, 4096),
                                    (64, 160), (130, 512), (257, 64)])
def test_quantizer_bit_exact_ragged(fmt, paired, rows, K):
    x = workloads.make_x("attn_proj_k4096", rows, K=K, seed=rows * 1000 + K)
    _check(fmt, x, paired)


@pytest.mark.parametrize("fmt,recipe,M", [(0, "gauss_outlier_k2048", 1), (0, "attn_proj_k4096", 8),
                                          (0, "mlp_gate_up", 8), (0, "mlp_down", 8),
                                          (1, "mx_k5120_n27648", 128), (0, "prefill_k8192", 64)])
def test_quantizer_bit_exact_workloads(fmt, recipe, M):
    x = workloads.make_x(recipe, M)
    _check(fmt, x, True)
    _check(fmt, x, False)


def _check_weight(fmt, w):
    import oracle
    from block_scaled_quantized_gb300 import rs
    N, K = w.shape
    wb = workloads.bf16_bits(w)
    a_or = oracle.tensor_scale(wb) if fmt == 0 else np.float32(0)
    a_gpu = torch.tensor([a_or], dtype=torch.float32, device=DEV) if fmt == 0 else None
    buf = torch.full((rs.rs_weight_bytes(fmt, N, K),), 0xAB, dtype=torch.uint8, device=DEV)
    assert buf.numel() == layout.weight_bytes(fmt, N, K)
    rs.rs_quantize_weight(fmt, w.to(DEV), a_gpu, buf)
    torch.cuda.synchronize()
    codes, sf, pad_ok = layout.unpack_weight(buf.cpu().numpy(), fmt, N, K)
    cw, sw, _ = oracle.quantize(fmt, wb, a_or)
    np.testing.assert_array_equal(codes, cw)
    np.testing.assert_array_equal(sf, sw)
    assert pad_ok


@pytest.mark.parametrize("fmt,recipe", [(0, "attn_proj_k4096"), (0, "mlp_gate_up"), (1, "mx_k5120_n27648"),
                                        (0, "prefill_k8192")])
def test_weight_quantization_bit_exact(fmt, recipe):
    _check_weight(fmt, workloads.make_w(recipe, N=384))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("N,K", [(1, 32), (100, 288), (129, 96), (256, 1024), (300, 4128)])
def test_weight_quantization_ragged(fmt, N, K):
    _check_weight(fmt, workloads.random_bf16((N, K), seed=N + K, scale=0.02))


def test_quantizer_strided_rows_and_edge_values():
    import oracle
    # rows of a wider buffer (ldx > K), plus zeros, -0, tiny and huge values
    wide = workloads.random_bf16((5, 320), seed=3).to(DEV)
    x = wide[:, :256]
    assert x.stride(0) == 320
    xc = x.cpu().clone()
    xc[0, :16] = 0.0
    xc[1, :16] = -0.0
    xc[2, 16] = 1e-30
    xc[2, 17] = 3e30
    xc[3, 32:64] = 1.0
    wide[:, :256] = xc.to(DEV)
    for fmt in (0, 1):
        for paired in (False, True):
            xb = workloads.bf16_bits(xc)
            a = oracle.tensor_scale(xb) if fmt == 0 else np.float32(0)
            ag = torch.tensor([a], device=DEV) if fmt == 0 else None
            buf = gpu_quantize(fmt, x, ag, paired)
            rows_out = 10 if paired else 5
            codes, sf = unpack(buf, fmt, rows_out, 256)
            if paired:
                ref = oracle.quantize_residue(fmt, xb, a)
                np.testing.assert_array_equal(codes[0::2], ref["codes_x"])
                np.testing.assert_array_equal(codes[1::2], ref["codes_r"])
                np.testing.assert_array_equal(sf[0::2], ref["sf_x"])
                np.testing.assert_array_equal(sf[1::2], ref["sf_r"])
            else:
                cx, sx, _ = oracle.quantize(fmt, xb, a)
                np.testing.assert_array_equal(codes, cx)
                np.testing.assert_array_equal(sf, sx)


def test_alpha_zero_gives_zero_operand():
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device=DEV)
    a = gpu_tensor_scale(x)
    assert a.item() == 0.0
    buf = gpu_quantize(0, x, a, paired=True)
    codes, sf = unpack(buf, 0, 8, 64)
    assert not codes.any() and not sf.any()


# The NVFP4 block scale byte E4M3(fl(fl(amax/6)/alpha)) for every positive
# finite bf16 value as a block amax (ResServe App. B.2 Eq. 8-9): blocks whose
# scale lies next to an E4M3 rounding boundary (ties included) and blocks far
# from one, saturation, underflow to zero, subnormal block amaxes, and the
# ends of the supported tensor-scale range (2^-117 and a scale so large that
# the quantizer's estimate of 1/(6 alpha) would be subnormal).
ALPHAS = [1.0, 2.0 ** -10, 0.012345678, 3.7e-5, 1.5e-30, 2.0 ** -110, 2.0 ** -117, 2.0e30, 3.0e37]


@pytest.mark.parametrize("alpha", ALPHAS)
@pytest.mark.parametrize("paired", [False, True])
def test_nvfp4_scale_every_bf16_amax(alpha, paired):
    K = 4096
    amax_bits = torch.arange(1, 0x7F80, dtype=torch.int32)            # 0x0001 .. 0x7F7F
    nblk = (amax_bits.numel() + K // 16 - 1) // (K // 16) * (K // 16)
    amax = torch.zeros(nblk, dtype=torch.int32)
    amax[: amax_bits.numel()] = amax_bits
    amax = amax.to(torch.int16).view(torch.bfloat16).float()
    g = torch.Generator().manual_seed(2024)
    u = torch.rand((nblk, 16), generator=g) * 2.0 - 1.0
    blocks = amax[:, None] * u
    blocks[:, 0] = amax                                                # the block amax itself
    sign = torch.where(torch.rand((nblk, 16), generator=g) < 0.5, -1.0, 1.0)
    sign[:, 0] = torch.where(torch.arange(nblk) % 2 == 0, 1.0, -1.0)
    x = (blocks * sign).to(torch.bfloat16).reshape(-1, K)
    _check(0, x, paired, alpha=np.float32(alpha))


@pytest.mark.parametrize("alpha", [1.0e-39, 2.0 ** -118, float("inf"), -1.0])
def test_unsupported_tensor_scale_flagged(alpha):
    """An NVFP4 tensor scale outside {0} and [2^-117, max float] sets the
    device error word (RS_ERR_INVALID_ARG); a supported one does not."""
    from block_scaled_quantized_gb300 import rs
    x = workloads.make_x("attn_proj_k4096", 4, K=512)
    assert rs.rs_get_device_error() == 0
    gpu_quantize(0, x.to(DEV), torch.tensor([alpha], dtype=torch.float32, device=DEV), False)
    assert rs.rs_get_device_error() == rs.RS_ERR_INVALID_ARG
    gpu_quantize(0, x.to(DEV), torch.tensor([2.0 ** -117], dtype=torch.float32, device=DEV), True)
    assert rs.rs_get_device_error() == 0


# Large NVFP4 operands (rows x K/256 >= 128 per SM, K a multiple of 512) take
# the quantizer that derives each block scale on one lane: the same codes and
# scale bytes, checked on every row, with ragged row tiles, a chunk group
# whose second half is past K, sub-normal and huge values, and the full bf16
# amax sweep.
@pytest.mark.parametrize("paired", [False, True])
@pytest.mark.parametrize("rows,K", [(700, 8192), (3300, 1536)])
def test_quantizer_large_nvfp4_operand(paired, rows, K):
    x = workloads.make_x("prefill_k8192", rows, K=K, seed=rows + K)
    x[1, :16] = 0.0
    x[2, :16] = -0.0
    x[3, 16] = 1e-40                     # bf16 sub-normal
    x[3, 17] = 3e30
    x[4, 32:64] = 1.0
    _check(0, x, paired)


@pytest.mark.parametrize("alpha", [1.0, 0.012345678, 2.0 ** -117, 3.0e37])
def test_nvfp4_scale_every_bf16_amax_large_operand(alpha):
    K = 4096
    amax_bits = torch.arange(1, 0x7F80, dtype=torch.int32)
    nblk = (amax_bits.numel() + K // 16 - 1) // (K // 16) * (K // 16)
    amax = torch.zeros(nblk, dtype=torch.int32)
    amax[: amax_bits.numel()] = amax_bits
    amax = amax.to(torch.int16).view(torch.bfloat16).float()
    g = torch.Generator().manual_seed(7)
    blocks = amax[:, None] * (torch.rand((nblk, 16), generator=g) * 2.0 - 1.0)
    blocks[:, 0] = amax
    sign = torch.where(torch.rand((nblk, 16), generator=g) < 0.5, -1.0, 1.0)
    x = (blocks * sign).to(torch.bfloat16).reshape(-1, K)
    x = torch.cat([x.roll(i, dims=1) for i in range(10)])    # 1280 rows: the large-operand quantizer
    _check(0, x, True, alpha=np.float32(alpha))


# Large operands that the one-block-per-lane kernel does not take (MXFP4, or
# NVFP4 with K not a multiple of 512) use the two-lanes-per-block kernel with
# four chunks per warp step: K = 8448 leaves a last group of one chunk.
@pytest.mark.parametrize("fmt,rows,K", [(1, 700, 8192), (0, 600, 8448), (1, 600, 8448)])
@pytest.mark.parametrize("paired", [False, True])
def test_quantizer_large_operand_four_chunk_steps(fmt, rows, K, paired):
    x = workloads.make_x("prefill_k8192", rows, K=K, seed=rows + K + fmt)
    _check(fmt, x, paired)
