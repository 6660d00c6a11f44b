"""Bit-exact pin of the quantizing prologue of the one-launch GEMM (ResServe
Sec. 4.4: Algorithm 1 of App. B.2 fused into the linear layer for small M).

rs_debug_linear_dump runs the same call rs_linear_compensated /
rs_linear_w4a4 make with a bf16 input and copies every CTA's quantized
activation slice (codes in the 128-byte-swizzled tile, scale atoms) as the
MMAs read it.  The expected image is built here from the oracle's logical
codes and scale bytes with the layout include/rs.h documents, and every CTA's
slice must equal it byte for byte: codes, scale bytes, and the zero padding
rows, blocks and bytes.  Each CTA of a K split quantizes its slice on its own,
so all of them are compared.  Shapes: the attention projection at M = 1, 4, 8
(compensated and W4A4), the MLP gate/up (three tiles per CTA) and down
projections, wider activation tiles (2M = 32, W4A4 M = 32), ragged K tails,
split counts that do not divide the outputs, MXFP4, and the call that finds
its own tensor scale (alpha_x = NULL) in both formats."""
import numpy as np
import pytest
import torch

from gpu_util import DEV
from block_scaled_quantized_gb300 import rs, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()


def chunks_of_split(chunks, splits, z):
    per, rem = divmod(chunks, splits)
    c0 = z * per + min(z, rem)
    return list(range(c0, c0 + per + (1 if z < rem else 0)))


def expected_image(fmt, codes_log, sf_log, K, bn, stage, chunk_ids):
    """Shared-memory image of the listed 256-element K chunks of the paired
    (or plain) activation rows: codes of row r, byte b at r * 128 +
    ((b / 16) ^ (r % 8)) * 16 + b % 16, then scale atoms at bn * 128."""
    bs = 16 if fmt == 0 else 32
    bpc = 256 // bs
    rows = codes_log.shape[0]
    img = np.zeros(len(chunk_ids) * stage, np.uint8)
    r = np.arange(rows)[:, None]
    b = np.arange(128)[None, :]
    cpos = r * 128 + ((b // 16) ^ (r % 8)) * 16 + b % 16
    kb = np.arange(bpc)[None, :]
    spos = bn * 128 + (kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    for i, c in enumerate(chunk_ids):
        blk = np.zeros((rows, 128), np.uint8)
        lo, hi = c * 128, min(K // 2, c * 128 + 128)
        blk[:, :hi - lo] = codes_log[:, lo:hi]
        img[i * stage + cpos] = blk
        sblk = np.zeros((rows, bpc), np.uint8)
        b0, b1 = c * bpc, min(K // bs, c * bpc + bpc)
        sblk[:, :b1 - b0] = sf_log[:, b0:b1]
        img[i * stage + spos] = sblk
    return img


def oracle_rows(fmt, compensated, xb, alpha):
    """Logical operand rows the GEMM consumes: paired (base 2j, residue
    2j + 1) for the compensated layer, the base rows for W4A4."""
    import oracle
    if not compensated:
        codes, sf, _ = oracle.quantize(fmt, xb, alpha)
        return codes, sf
    q = oracle.quantize_residue(fmt, xb, alpha)
    M = xb.shape[0]
    codes = np.empty((2 * M,) + q["codes_x"].shape[1:], np.uint8)
    sf = np.empty((2 * M,) + q["sf_x"].shape[1:], np.uint8)
    codes[0::2], codes[1::2] = q["codes_x"], q["codes_r"]
    sf[0::2], sf[1::2] = q["sf_x"], q["sf_r"]
    return codes, sf


def make_weight(fmt, N, K, seed):
    w = workloads.make_w("attn_proj_k4096", N=N, K=K, seed=seed).to(DEV)
    aw = None
    if fmt == 0:
        aw = torch.empty(1, dtype=torch.float32, device=DEV)
        rs.rs_compute_tensor_scale(w, aw)
    wq = torch.empty(rs.rs_weight_bytes(fmt, N, K), dtype=torch.uint8, device=DEV)
    rs.rs_quantize_weight(fmt, w, aw, wq)
    return wq, aw


def run_dump(fmt, compensated, x_bf16, wq, aw, N, alpha_x):
    M, K = x_bf16.shape
    x = x_bf16.to(DEV)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    ws = rs.empty_workspace(fmt, M, N, K, compensated)
    lay = rs.rs_debug_linear_dump(fmt, compensated, M, N, K)
    assert lay["fused"] in (1, 2), "the shape must take the one-launch plan"
    nbytes = lay["grid_x"] * lay["splits"] * lay["slots"] * lay["stage_bytes"]
    dump = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device=DEV)
    lay2 = rs.rs_debug_linear_dump(fmt, compensated, M, N, K, x=x, alpha_x=alpha_x, wq=wq, alpha_w=aw, y=y,
                                   workspace=ws, dump=dump)
    torch.cuda.synchronize()
    assert lay2 == lay
    assert rs.rs_get_device_error() == 0
    return lay, dump.cpu().numpy()


def check_slices(fmt, lay, dump, codes_log, sf_log, K):
    stage, slots = lay["stage_bytes"], lay["slots"]
    for z in range(lay["splits"]):
        ids = chunks_of_split(lay["chunks"], lay["splits"], z)
        want = expected_image(fmt, codes_log, sf_log, K, lay["bn"], stage, ids)
        for x in range(lay["grid_x"]):
            off = (z * lay["grid_x"] + x) * slots * stage
            got = dump[off:off + len(ids) * stage]
            if not np.array_equal(got, want):
                bad = np.flatnonzero(got != want)
                raise AssertionError(f"CTA (x={x}, split={z}): {bad.size} bytes differ, first at "
                                     f"{bad[0]} (chunk {bad[0] // stage}, byte {bad[0] % stage}): "
                                     f"got {got[bad[0]]:#04x} want {want[bad[0]]:#04x}")


CASES = [
    # (fmt, compensated, M, N, K, recipe)
    (0, True, 8, 4096, 4096, "attn_proj_k4096"),
    (0, True, 4, 4096, 4096, "attn_proj_k4096"),
    (0, True, 1, 4096, 4096, "attn_proj_k4096"),
    (0, False, 8, 4096, 4096, "attn_proj_k4096"),
    (0, True, 1, 2048, 2048, "gauss_outlier_k2048"),
    (0, True, 8, 28672, 4096, "mlp_gate_up"),
    (0, True, 8, 4096, 14336, "mlp_down"),
    (0, True, 16, 1024, 2048, "attn_proj_k4096"),
    (0, False, 32, 2048, 1024, "attn_proj_k4096"),
    (0, True, 5, 640, 1056, "gauss_outlier_k2048"),
    (1, True, 8, 27648, 5120, "mx_k5120_n27648"),
    (1, False, 16, 2048, 5120, "mx_k5120_n27648"),
    (1, True, 3, 384, 800, "gauss_outlier_k2048"),
]


@pytest.fixture(params=["shipped", "paired", "unpaired"])
def prologue_mode(request):
    """Which prologue runs: the shipped tactic table's choice, the analytic
    plan (CTA pairs share the quantization of a K slice when the grid allows),
    or the same plan with every CTA quantizing its whole slice."""
    yield request.param
    rs.rs_reset_tactics(True)


def set_mode(mode, fmt, compensated, M, N, K):
    rs.rs_reset_tactics(mode == "shipped")
    if mode == "unpaired":
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        p = rs.rs_plan_linear(fmt, compensated, M, N, K, sms)
        rs.rs_set_tactic(fmt, compensated, M, N, K, sms, p["splits"], 1, p["bn"])
    lay = rs.rs_debug_linear_dump(fmt, compensated, M, N, K)
    if mode == "unpaired":
        assert lay["fused"] == 1
    if mode == "shipped" and lay["fused"] == 0:
        pytest.skip("the shipped tactic quantizes this shape in a separate kernel")


@pytest.mark.parametrize("own_scale", [False, True])
@pytest.mark.parametrize("fmt,compensated,M,N,K,recipe", CASES)
def test_fused_slices_bit_exact(fmt, compensated, M, N, K, recipe, own_scale, prologue_mode):
    import oracle
    if own_scale and fmt == 1:
        pytest.skip("MXFP4 has no tensor scale")
    set_mode(prologue_mode, fmt, compensated, M, N, K)
    x = workloads.make_x(recipe, M, K=K, seed=M * 31 + K)
    xb = workloads.bf16_bits(x)
    ax = oracle.tensor_scale(xb) if fmt == 0 else np.float32(0)
    wq, aw = make_weight(fmt, N, K, seed=N + K)
    ax_dev = None
    if fmt == 0 and not own_scale:
        ax_dev = torch.tensor([ax], dtype=torch.float32, device=DEV)
    lay, dump = run_dump(fmt, compensated, x, wq, aw, N, ax_dev)
    codes, sf = oracle_rows(fmt, compensated, xb, ax)
    check_slices(fmt, lay, dump, codes, sf, K)


# slices of more than 32 chunks (up to the shared memory's limit) and ragged
# K tails, forced by tactics: (fmt, compensated, M, N, K, recipe, splits, fused)
LONG_CASES = [
    (0, True, 4, 384, 16640, "gauss_outlier_k2048", 2, 1),     # 33 chunks per slice
    (0, False, 1, 5120, 25600, "proj_shapes", 3, 1),           # 34
    (1, True, 3, 256, 12320, "gauss_outlier_k2048", 1, 1),     # 49, ragged tail
    (0, False, 5, 768, 12320, "gauss_outlier_k2048", 2, 2),    # CTA pairs, ragged tail
    (1, False, 8, 512, 12320, "gauss_outlier_k2048", 2, 2),
]


@pytest.mark.parametrize("fmt,compensated,M,N,K,recipe,splits,fused", LONG_CASES)
def test_fused_long_slices_bit_exact(fmt, compensated, M, N, K, recipe, splits, fused):
    import oracle
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rs.rs_reset_tactics(False)
    try:
        rs.rs_set_tactic(fmt, compensated, M, N, K, sms, splits, fused, 16, 1)
        lay = rs.rs_debug_linear_dump(fmt, compensated, M, N, K)
        assert lay["fused"] == fused and lay["splits"] == splits
        assert lay["slots"] == (lay["chunks"] + splits - 1) // splits
        x = workloads.make_x(recipe, M, K=K, seed=M * 13 + K)
        xb = workloads.bf16_bits(x)
        ax = oracle.tensor_scale(xb) if fmt == 0 else np.float32(0)
        wq, aw = make_weight(fmt, N, K, seed=N + 2 * K)
        ax_dev = torch.tensor([ax], dtype=torch.float32, device=DEV) if fmt == 0 else None
        lay, dump = run_dump(fmt, compensated, x, wq, aw, N, ax_dev)
        codes, sf = oracle_rows(fmt, compensated, xb, ax)
        check_slices(fmt, lay, dump, codes, sf, K)
    finally:
        rs.rs_reset_tactics(True)


def test_dump_layout_query_and_refusals():
    # layout only (no launch) and the documented refusals
    lay = rs.rs_debug_linear_dump(0, True, 8, 4096, 4096)
    assert lay["fused"] in (1, 2) and lay["splits"] * lay["grid_x"] <= 304
    lay = rs.rs_debug_linear_dump(0, True, 512, 4096, 4096)
    assert lay["fused"] == 0
    wq, aw = make_weight(0, 256, 512, seed=3)
    x = workloads.make_x("attn_proj_k4096", 512, K=512, seed=3).to(DEV)
    y = torch.empty((512, 256), dtype=torch.float32, device=DEV)
    ws = rs.empty_workspace(0, 512, 256, 512, True)
    dump = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    with pytest.raises(rs.RsError) as e:
        rs.rs_debug_linear_dump(0, True, 512, 256, 512, x=x, alpha_x=None, wq=wq, alpha_w=aw, y=y, workspace=ws,
                                dump=dump)
    assert e.value.status == rs.RS_ERR_UNSUPPORTED
    x8 = x[:8].contiguous()
    with pytest.raises(rs.RsError) as e:
        rs.rs_debug_linear_dump(0, True, 8, 256, 512, x=x8, alpha_x=None, wq=wq, alpha_w=aw, y=y, workspace=ws,
                                dump=dump[:16])
    assert e.value.status == rs.RS_ERR_WORKSPACE


def test_residue_scale_boundaries_standalone_and_fused():
    """Blocks whose residue block scale t lies within 4 fp32 ulps of every
    E4M3 rounding boundary a residue reaches, at three tensor-scale families
    (tests/scale_boundary_cases.py): the standalone paired quantizer and the
    GEMM's quantizing prologue give the oracle's codes and scale bytes."""
    import layout
    import oracle
    import scale_boundary_cases as sbc
    cases = sbc.all_cases()
    n, K, N = len(cases), sbc.K_ROW, 128
    rows = np.stack([c[0] for c in cases])
    alphas = np.array([c[1] for c in cases], np.float32)
    x = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).to(DEV)
    a_dev = torch.from_numpy(alphas).to(DEV)
    wq, aw = make_weight(0, N, K, seed=11)
    opb = rs.rs_operand_bytes(0, 2, K)
    q_all = torch.full((n * opb,), 0xAB, dtype=torch.uint8, device=DEV)
    lay = rs.rs_debug_linear_dump(0, True, 1, N, K)
    assert lay["fused"] in (1, 2) and lay["splits"] == 1 and lay["grid_x"] == 1
    stage = lay["stage_bytes"] * lay["slots"]
    d_all = torch.full((n * stage,), 0x5A, dtype=torch.uint8, device=DEV)
    y = torch.empty((n, N), dtype=torch.float32, device=DEV)
    ws = rs.empty_workspace(0, 1, N, K, True)
    for i in range(n):
        xi, ai = x[i:i + 1], a_dev[i:i + 1]
        rs.rs_quantize_residue(0, xi, ai, q_all[i * opb:(i + 1) * opb])
        rs.rs_debug_linear_dump(0, True, 1, N, K, x=xi, alpha_x=ai, wq=wq, alpha_w=aw, y=y[i:i + 1],
                                workspace=ws, dump=d_all[i * stage:(i + 1) * stage])
    torch.cuda.synchronize()
    assert rs.rs_get_device_error() == 0
    q_all, d_all = q_all.cpu().numpy(), d_all.cpu().numpy()
    for i, (row, alpha, m, fam) in enumerate(cases):
        q = oracle.quantize_residue(0, row[None, :], alpha)
        assert abs(sbc.residue_offset(q["resid"][0], alpha, m)) <= 4
        codes, sf = layout.unpack_operand(q_all[i * opb:(i + 1) * opb], 0, 2, K)
        ctx = f"case {i}: midpoint {float(m)}, family {fam}, alpha {float(alpha)!r}"
        assert np.array_equal(sf[0], q["sf_x"][0]) and np.array_equal(sf[1], q["sf_r"][0]), ctx
        assert np.array_equal(codes[0], q["codes_x"][0]) and np.array_equal(codes[1], q["codes_r"][0]), ctx
        lcodes = np.stack([q["codes_x"][0], q["codes_r"][0]])
        lsf = np.stack([q["sf_x"][0], q["sf_r"][0]])
        want = expected_image(0, lcodes, lsf, K, lay["bn"], lay["stage_bytes"], [0])
        assert np.array_equal(d_all[i * stage:i * stage + len(want)], want), ctx


# (fmt, compensated, M, N, K, splits, recipe): CTA pairs with odd chunk counts
# per K slice (one CTA of a pair quantizes one chunk more), a single K split
# (clusters of one pair), and MXFP4
PAIRED = [
    (0, True, 3, 1024, 1280, 2, "gauss_outlier_k2048"),
    (0, True, 8, 512, 768, 1, "attn_proj_k4096"),
    (0, False, 6, 768, 2560, 3, "attn_proj_k4096"),
    (1, True, 5, 768, 2560, 3, "mx_k5120_n27648"),
    (1, False, 7, 512, 1280, 1, "gauss_outlier_k2048"),
]


@pytest.mark.parametrize("own_scale", [False, True])
@pytest.mark.parametrize("fmt,compensated,M,N,K,splits,recipe", PAIRED)
def test_paired_prologue_bit_exact(fmt, compensated, M, N, K, splits, recipe, own_scale):
    """Tactic fused = 2 forces CTA pairs to share the quantization of each K
    slice; every CTA's slice image still equals the oracle's codes and scale
    bytes, and Y matches a plan without pairs exactly (same MMAs, same order)."""
    import oracle
    if own_scale and fmt == 1:
        pytest.skip("MXFP4 has no tensor scale")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    x = workloads.make_x(recipe, M, K=K, seed=M + 7 * K)
    xb = workloads.bf16_bits(x)
    ax = oracle.tensor_scale(xb) if fmt == 0 else np.float32(0)
    wq, aw = make_weight(fmt, N, K, seed=N + 3)
    ax_dev = None if (fmt == 1 or own_scale) else torch.tensor([ax], dtype=torch.float32, device=DEV)
    ys = {}
    try:
        for fused in (2, 1):
            rs.rs_reset_tactics(False)
            rs.rs_set_tactic(fmt, compensated, M, N, K, sms, splits, fused, 16)
            lay, dump = run_dump(fmt, compensated, x, wq, aw, N, ax_dev)
            assert lay["fused"] == fused and lay["splits"] == splits
            codes, sf = oracle_rows(fmt, compensated, xb, ax)
            check_slices(fmt, lay, dump, codes, sf, K)
            y = torch.empty((M, N), dtype=torch.float32, device=DEV)
            fn = rs.rs_linear_compensated if compensated else rs.rs_linear_w4a4
            fn(fmt, M, N, K, x=x.to(DEV), alpha_x=ax_dev, wq=wq, alpha_w=aw, y=y,
               workspace=rs.empty_workspace(fmt, M, N, K, compensated))
            torch.cuda.synchronize()
            assert rs.rs_get_device_error() == 0
            ys[fused] = y.cpu()
    finally:
        rs.rs_reset_tactics(True)
    assert torch.equal(ys[1], ys[2])
