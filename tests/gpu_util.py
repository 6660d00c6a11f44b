"""Helpers shared by the GPU parity tests: run the CUDA path through the
C-ABI binding and the oracle on the same seeded inputs."""
import numpy as np
import torch

import layout
from block_scaled_quantized_gb300 import rs, workloads

DEV = "cuda"


def gpu_tensor_scale(x_gpu):
    a = torch.empty(1, dtype=torch.float32, device=DEV)
    rs.rs_compute_tensor_scale(x_gpu, a)
    return a


def gpu_quantize(fmt, x_gpu, alpha, paired):
    rows, K = x_gpu.shape
    out_rows = 2 * rows if paired else rows
    buf = torch.full((rs.rs_operand_bytes(fmt, out_rows, K),), 0xAB, dtype=torch.uint8, device=DEV)
    if paired:
        rs.rs_quantize_residue(fmt, x_gpu, alpha, buf)
    else:
        rs.rs_quantize_fp4(fmt, x_gpu, alpha, buf)
    torch.cuda.synchronize()
    return buf


def unpack(buf, fmt, rows, K):
    return layout.unpack_operand(buf.cpu().numpy(), fmt, rows, K)


def prepare_weight(fmt, w_bf16):
    """GPU weight operand + alpha_w, and the oracle's own quantization of W."""
    import oracle
    N, K = w_bf16.shape
    w_gpu = w_bf16.to(DEV)
    aw = gpu_tensor_scale(w_gpu) if fmt == 0 else None
    wq = torch.full((rs.rs_weight_bytes(fmt, N, K),), 0xCD, dtype=torch.uint8, device=DEV)
    rs.rs_quantize_weight(fmt, w_gpu, aw, wq)
    torch.cuda.synchronize()
    wb = workloads.bf16_bits(w_bf16)
    aw_or = oracle.tensor_scale(wb) if fmt == 0 else np.float32(0)
    cw, sw, _ = oracle.quantize(fmt, wb, aw_or)
    return dict(w_gpu=w_gpu, aw=aw, wq=wq, aw_or=aw_or, cw=cw, sw=sw)


def gpu_linear(fmt, compensated, x_bf16, wprep, out_dtype=torch.float32, prequantized=False, ax=None):
    M, K = x_bf16.shape
    N = wprep["w_gpu"].shape[0]
    x_gpu = x_bf16.to(DEV)
    if fmt == 0 and ax is None:
        ax = gpu_tensor_scale(x_gpu)
    y = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    ws = rs.empty_workspace(fmt, M, N, K, compensated)
    fn = rs.rs_linear_compensated if compensated else rs.rs_linear_w4a4
    if prequantized:
        xq = gpu_quantize(fmt, x_gpu, ax, paired=compensated)
        kw = {"xq_paired" if compensated else "xq": xq}
        fn(fmt, M, N, K, alpha_x=ax, wq=wprep["wq"], alpha_w=wprep["aw"], y=y, workspace=ws, **kw)
    else:
        fn(fmt, M, N, K, x=x_gpu, alpha_x=ax, wq=wprep["wq"], alpha_w=wprep["aw"], y=y, workspace=ws)
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    # the split-K tile counters are re-armed at the end of every call
    return y, ws


def oracle_linear(fmt, compensated, x_bf16, wprep):
    import oracle
    xb = workloads.bf16_bits(x_bf16)
    ax = oracle.tensor_scale(xb) if fmt == 0 else np.float32(0)
    return oracle.linear(fmt, compensated, xb, ax, wprep["cw"], wprep["sw"], wprep["aw_or"])


def assert_close_f32(y_gpu, y_ref, rel=1e-3):
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(y))
    bound = rel * np.max(np.abs(y_ref))
    err = np.max(np.abs(y - y_ref))
    assert err <= bound, f"max|dY| {err:.3e} > {bound:.3e}"


def assert_close_bf16(y_gpu, y_ref, rel=1e-3):
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(y))
    ref_b = torch.from_numpy(y_ref.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)
    ulp = np.abs(ref_b) * 2.0 ** -7
    bound = ulp + rel * np.max(np.abs(y_ref))
    assert np.all(np.abs(y - ref_b) <= bound), f"max excess {np.max(np.abs(y - ref_b) - bound):.3e}"
