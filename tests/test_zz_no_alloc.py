"""rs_linear_compensated_noalloc: the compensated linear layer for callers
that cannot allocate device memory (for example a plugin that another
framework hands only its input and output buffers).  Its quantized
activations live in a fixed device array inside librs instead of a
workspace; these tests check, through the C ABI, that two calls in a row
give the same output as rs_linear_compensated (the array keeps the previous
call's contents, which must not leak into the next result), and that sizes
beyond the array are refused before any work is enqueued.

This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import layout
from gpu_util import DEV, assert_close_f32, gpu_tensor_scale, prepare_weight
from block_scaled_quantized_gb300 import rs, workloads

SCRATCH_BYTES = 4 << 20


def test_noalloc_refuses_sizes_beyond_the_array():
    """Host-side check, no GPU needed: the operand of 2*M rows must fit."""
    from block_scaled_quantized_gb300 import build
    lib = rs.load_library(build.build())
    fake = 1 << 20
    K = 4096
    M_fit = 904
    assert layout.operand_bytes(0, 2 * M_fit, K) <= SCRATCH_BYTES < layout.operand_bytes(0, 2 * (M_fit + 1), K)
    f = lib.rs_linear_compensated_noalloc
    assert f(0, M_fit + 1, 128, K, fake, fake, fake, fake, fake, 0, None) == 5  # RS_ERR_WORKSPACE
    assert f(0, M_fit + 1, 128, K, fake, None, fake, fake, fake, 0, None) == 5  # also without alpha_x
    # the largest size fits with and without alpha_x: validation goes on to the
    # alignment check (a misaligned output stops the call before any launch)
    assert f(0, M_fit, 128, K, fake, fake, fake, fake, fake + 2, 0, None) == 2  # RS_ERR_ALIGNMENT
    assert f(0, M_fit, 128, K, fake, None, fake, fake, fake + 2, 0, None) == 2
    assert f(0, 4, 128, 48, fake, fake, fake, fake, fake, 0, None) == 3         # K % 32
    assert f(0, 4, 128, K, None, fake, fake, fake, fake, 0, None) == 1          # no input
    assert f(0, 0, 128, K, None, None, None, None, None, 0, None) == 0          # nothing to do


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", [0, 1])
def test_noalloc_matches_compensated_twice(fmt):
    from block_scaled_quantized_gb300 import build
    build.build()
    M, N, K = 24, 640, 1536
    w = workloads.make_w("attn_proj_k4096", N=N, K=K, seed=41)
    wp = prepare_weight(fmt, w)
    for call, seed in enumerate((42, 43)):  # two calls in a row on the shared array
        x = workloads.make_x("attn_proj_k4096", M, K=K, seed=seed).to(DEV)
        ax = gpu_tensor_scale(x) if fmt == 0 else None
        y_ref = torch.empty((M, N), dtype=torch.float32, device=DEV)
        ws = rs.empty_workspace(fmt, M, N, K, True)
        rs.rs_linear_compensated(fmt, M, N, K, x=x, alpha_x=ax, wq=wp["wq"], alpha_w=wp["aw"], y=y_ref,
                                 workspace=ws)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        rs.rs_linear_compensated_noalloc(fmt, M, N, K, x=x, alpha_x=ax, wq=wp["wq"], alpha_w=wp["aw"], y=y)
        torch.cuda.synchronize()
        assert rs.rs_get_device_error() == 0
        assert_close_f32(y, y_ref.cpu().numpy().astype(np.float64))


@pytest.mark.gpu
def test_noalloc_finds_tensor_scale():
    """Without alpha_x the no-allocation call uses the input's own tensor
    scale: the same Y as with rs_compute_tensor_scale's value."""
    M, N, K = 8, 512, 2048
    x = workloads.make_x("attn_proj_k4096", M, K=K, seed=21).to(DEV)
    wp = prepare_weight(0, workloads.make_w("attn_proj_k4096", N=N, K=K, seed=22))
    y1 = torch.empty((M, N), dtype=torch.float32, device=DEV)
    y2 = torch.empty_like(y1)
    rs.rs_linear_compensated_noalloc(0, M, N, K, x=x, alpha_x=gpu_tensor_scale(x), wq=wp["wq"], alpha_w=wp["aw"],
                                     y=y1)
    rs.rs_linear_compensated_noalloc(0, M, N, K, x=x, alpha_x=None, wq=wp["wq"], alpha_w=wp["aw"], y=y2)
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    assert torch.equal(y1, y2)
