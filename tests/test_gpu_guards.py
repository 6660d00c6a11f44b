"""Every device output stays inside its buffer (guard regions in place of a
memory checker): the output Y, the workspace and the quantized operands are
allocated with a sentinel tail that must be untouched after the call, for
ragged M, N and K across fused, split-K, two-kernel, MXFP4 and W4A4 plans."""
import pytest
import torch

from gpu_util import DEV, gpu_tensor_scale
from block_scaled_quantized_gb300 import rs, workloads

pytestmark = pytest.mark.gpu

GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_quantized_gb300 import build
    build.build()


@pytest.mark.parametrize("fmt,comp,M,N,K", [(0, True, 3, 300, 512), (0, False, 7, 200, 256), (1, True, 5, 384, 1024),
                                            (0, True, 40, 256, 768), (0, True, 600, 640, 1024), (1, False, 130, 128, 288)])
@pytest.mark.parametrize("out_f32", [True, False])
def test_outputs_stay_inside_their_buffers(fmt, comp, M, N, K, out_f32):
    x = workloads.make_x("attn_proj_k4096", M, K=K, seed=M + N)
    w = workloads.make_w("attn_proj_k4096", N=N, K=K, seed=N + K)
    wg = w.to(DEV)
    aw = gpu_tensor_scale(wg) if fmt == 0 else None
    wbytes = rs.rs_weight_bytes(fmt, N, K)
    wbig = torch.full((wbytes + GUARD,), 0x5A, dtype=torch.uint8, device=DEV)
    rs.rs_quantize_weight(fmt, wg, aw, wbig[:wbytes])
    xg = x.to(DEV)
    ax = gpu_tensor_scale(xg) if fmt == 0 else None
    dt = torch.float32 if out_f32 else torch.bfloat16
    ybig = torch.full((M * N + GUARD,), 12288.0, dtype=dt, device=DEV)
    y = ybig[:M * N].view(M, N)
    wsb = max(rs.rs_workspace_bytes(fmt, M, N, K, comp), 16)
    wsbig = torch.full((wsb + GUARD,), 0xA5, dtype=torch.uint8, device=DEV)
    fn = rs.rs_linear_compensated if comp else rs.rs_linear_w4a4
    fn(fmt, M, N, K, x=xg, alpha_x=ax, wq=wbig[:wbytes], alpha_w=aw, y=y, workspace=wsbig[:wsb])
    # the quantized operand on its own, also with a guard
    rows = 2 * M if comp else M
    qbytes = rs.rs_operand_bytes(fmt, rows, K)
    qbig = torch.full((qbytes + GUARD,), 0x3C, dtype=torch.uint8, device=DEV)
    (rs.rs_quantize_residue if comp else rs.rs_quantize_fp4)(fmt, xg, ax, qbig[:qbytes])
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == rs.RS_OK
    assert torch.all(wbig[wbytes:] == 0x5A)
    assert torch.all(ybig[M * N:] == 12288.0)
    assert torch.all(wsbig[wsb:] == 0xA5)
    assert torch.all(qbig[qbytes:] == 0x3C)
    assert torch.isfinite(y.float()).all() and not torch.any(y.float() == 12288.0)
