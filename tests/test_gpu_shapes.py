"""GPU parity on the 22 projection shapes (N, K) that ResServe times one by one
(Fig. 18 NVFP4 and Fig. 19 MXFP4, M-Ext latency per shape): compensated
NVFP4 with the activation tensor scale found in the call (M = 8 and 64),
compensated MXFP4 (M = 8) and W4A4 NVFP4 (M = 1), each against the oracle on
192 sampled output channels.  The weight is quantized row by row with the
tensor scale of the whole W, so the oracle quantizes the sampled rows alone;
the bar is max|dY| <= 1e-3 max|Y| over those channels."""
import numpy as np
import pytest
import torch

from gpu_util import DEV, assert_close_f32, gpu_tensor_scale
from block_scaled_quantized_gb300 import rs, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()


# (format, compensated, M, tensor scale found in the call)
VARIANTS = [(0, True, 8, True), (0, True, 64, True), (1, True, 8, False), (0, False, 1, False)]


@pytest.mark.parametrize("N,K", workloads.PROJECTION_SHAPES)
def test_projection_shape_parity(N, K):
    import oracle
    seed = N + K
    w = workloads.make_w("proj_shapes", N=N, K=K, seed=seed)
    wb = workloads.bf16_bits(w)
    wg = w.to(DEV)
    cols = np.sort(np.random.default_rng(seed).choice(N, 192, replace=False))
    cols_dev = torch.from_numpy(cols).to(DEV)
    for fmt, comp, M, own_scale in VARIANTS:
        aw = gpu_tensor_scale(wg) if fmt == 0 else None
        wq = torch.empty(rs.rs_weight_bytes(fmt, N, K), dtype=torch.uint8, device=DEV)
        rs.rs_quantize_weight(fmt, wg, aw, wq)
        x = workloads.make_x("proj_shapes", M, K=K, seed=seed + M)
        xg = x.to(DEV)
        ax = None if (fmt == 1 or own_scale) else gpu_tensor_scale(xg)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        ws = rs.empty_workspace(fmt, M, N, K, comp)
        fn = rs.rs_linear_compensated if comp else rs.rs_linear_w4a4
        fn(fmt, M, N, K, x=xg, alpha_x=ax, wq=wq, alpha_w=aw, y=y, workspace=ws)
        torch.cuda.synchronize()
        assert rs.rs_get_device_error() == 0, (fmt, comp, M)
        aw_or = oracle.tensor_scale(wb) if fmt == 0 else np.float32(0)
        cw, sw, _ = oracle.quantize(fmt, np.ascontiguousarray(wb[cols]), aw_or)
        xb = workloads.bf16_bits(x)
        ax_or = oracle.tensor_scale(xb) if fmt == 0 else np.float32(0)
        ref = oracle.linear(fmt, comp, xb, ax_or, cw, sw, aw_or)
        assert_close_f32(y[:, cols_dev], ref)
        del wq, ws
