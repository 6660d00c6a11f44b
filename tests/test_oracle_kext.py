"""Pins of the oracle's selective prefill compensation (K-Ext): ResServe
Sec. 5.3 Eq. 6, App. A Eq. 7, App. B.2 Alg. 1.  The oracle is checked
against a block worked by hand, the full-compensation special case (which
must equal the already pinned M-Ext residue path), the base parts (which
must equal the plain quantizers), Eq. 6's split into a base and an
extension GEMM, the selection invariants of Eq. 7, and the error ordering
against plain W4A4."""
import numpy as np
import pytest
import torch

from conftest import read_golden
from block_scaled_quantized_gb300 import workloads


def _bits(vals):
    return workloads.bf16_bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


def test_kext_block_worked_by_hand(oracle_mod):
    g = read_golden("kext_nvfp4_block.txt")
    x = _bits([[float(v) for v in g["x"]]])
    mask = np.array([int(v, 16) for v in g["mask"]], np.uint8)
    codes, sf = oracle_mod.quantize_kext(0, x, 4, mask, alpha=1.0)
    assert codes.shape == (1, (32 + 16) // 2) and sf.shape == (1, 3)
    assert sf[0, 2] == int(g["ext_sf"][0], 16)
    assert list(codes[0, 16:]) == [int(v, 16) for v in g["ext_codes"]]
    # the base part is the plain quantizer's
    cb, sb, _ = oracle_mod.quantize(0, x, 1.0)
    assert np.array_equal(codes[:, :16], cb) and np.array_equal(sf[:, :2], sb)
    assert list(sb[0]) == [0x38, 0x38]


@pytest.mark.parametrize("fmt", [0, 1])
def test_full_ratio_equals_full_compensation(oracle_mod, fmt):
    """k = 8 selects every channel: the extension is the residue operand of
    M-Ext (Sec. 4.2: full compensation reuses the base weight) and Eq. 6
    equals Eq. 1 with all channels."""
    M, N, K = 5, 24, 256
    x = workloads.make_x("gauss_outlier_k2048", M, K=K, seed=7)
    w = workloads.make_w("gauss_outlier_k2048", N=N, K=K, seed=8)
    xb, wb = workloads.bf16_bits(x), workloads.bf16_bits(w)
    ax = oracle_mod.tensor_scale(xb) if fmt == 0 else 0.0
    aw = oracle_mod.tensor_scale(wb) if fmt == 0 else 0.0
    mask = np.full(K // 8, 0xFF, np.uint8)
    codes, sf = oracle_mod.quantize_kext(fmt, xb, 8, mask, ax)
    ref = oracle_mod.quantize_residue(fmt, xb, ax)
    bs = oracle_mod.block_size(fmt)
    assert np.array_equal(codes[:, :K // 2], ref["codes_x"]) and np.array_equal(sf[:, :K // bs], ref["sf_x"])
    assert np.array_equal(codes[:, K // 2:], ref["codes_r"]) and np.array_equal(sf[:, K // bs:], ref["sf_r"])
    cw, sw = oracle_mod.quantize_weight_kext(fmt, wb, 8, mask, aw)
    cw0, sw0, _ = oracle_mod.quantize(fmt, wb, aw)
    for h in (0, 1):  # both halves of [W | W[:, S]] are the plain weight
        assert np.array_equal(cw[:, h * K // 2:(h + 1) * K // 2], cw0)
        assert np.array_equal(sw[:, h * K // bs:(h + 1) * K // bs], sw0)
    y = oracle_mod.linear_kext(fmt, xb, 8, mask, ax, cw, sw, aw)
    y_m = oracle_mod.linear(fmt, True, xb, ax, cw0, sw0, aw)
    np.testing.assert_allclose(y, y_m, rtol=1e-12, atol=1e-12 * np.abs(y_m).max())


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("k", [1, 2, 4])
def test_extended_gemm_splits_into_base_and_extension(oracle_mod, fmt, k):
    """Eq. 6: [X^ | R^_S][W^ | W^_S]^T = X^ W^T + R^_S W^_S^T, and the base
    parts of both extended operands are the plain quantizations."""
    M, N, K = 3, 16, 512
    x = workloads.make_x("gauss_outlier_k2048", M, K=K, seed=10 + k)
    w = workloads.make_w("gauss_outlier_k2048", N=N, K=K, seed=20 + k)
    xb, wb = workloads.bf16_bits(x), workloads.bf16_bits(w)
    ax = oracle_mod.tensor_scale(xb) if fmt == 0 else 0.0
    aw = oracle_mod.tensor_scale(wb) if fmt == 0 else 0.0
    score = np.abs(x.float().numpy()).mean(axis=0)
    mask = oracle_mod.kext_select(score, k)
    ca, sa = oracle_mod.quantize_kext(fmt, xb, k, mask, ax)
    cw, sw = oracle_mod.quantize_weight_kext(fmt, wb, k, mask, aw)
    bs = oracle_mod.block_size(fmt)
    cb, sb, _ = oracle_mod.quantize(fmt, xb, ax)
    cw0, sw0, _ = oracle_mod.quantize(fmt, wb, aw)
    assert np.array_equal(ca[:, :K // 2], cb) and np.array_equal(sa[:, :K // bs], sb)
    assert np.array_equal(cw[:, :K // 2], cw0) and np.array_equal(sw[:, :K // bs], sw0)
    g = float(ax) * float(aw) if fmt == 0 else 1.0
    z_base = oracle_mod.block_gemm(fmt, ca[:, :K // 2], sa[:, :K // bs], cw[:, :K // 2], sw[:, :K // bs])
    z_ext = oracle_mod.block_gemm(fmt, ca[:, K // 2:], sa[:, K // bs:], cw[:, K // 2:], sw[:, K // bs:])
    y = oracle_mod.linear_kext(fmt, xb, k, mask, ax, cw, sw, aw)
    ref = g * (z_base + z_ext)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert ca.shape[1] * 2 == K + oracle_mod.kext_width(K, k)


@pytest.mark.parametrize("k", [0, 1, 2, 4, 8])
def test_selection_invariants(oracle_mod, k):
    """Eq. 7: exactly k channels per group of 8, and no unselected channel
    scores above a selected one of its group."""
    rng = np.random.default_rng(k)
    score = rng.random(256).astype(np.float32)
    mask = oracle_mod.kext_select(score, k)
    for gi, m in enumerate(mask):
        sel = [t for t in range(8) if m >> t & 1]
        assert len(sel) == k
        rest = [t for t in range(8) if not m >> t & 1]
        if sel and rest:
            assert min(score[8 * gi + t] for t in sel) >= max(score[8 * gi + t] for t in rest)


def test_selection_known_groups(oracle_mod):
    score = np.array([0, 1, 2, 3, 4, 5, 6, 7,       # increasing: the top two are 6, 7
                      5, 5, 5, 5, 5, 5, 5, 5,       # all equal: the lower channels
                      9, 0, 0, 0, 0, 0, 0, 8], np.float32)
    assert list(oracle_mod.kext_select(score, 2)) == [0xC0, 0x03, 0x81]
    assert list(oracle_mod.kext_select(score, 8)) == [0xFF] * 3
    assert list(oracle_mod.kext_select(score, 0)) == [0] * 3


def test_selected_compensation_lowers_error(oracle_mod):
    """App. A / Sec. 5.3: compensating the calibration-salient channels lowers
    the linear-layer error against the bf16 product, and full compensation
    (k = 8) lowers it at least as much as the smallest ratio."""
    M, N, K = 16, 64, 1024
    x = workloads.make_x("mlp_gate_up", M, K=K, seed=3)
    w = workloads.make_w("mlp_gate_up", N=N, K=K, seed=4)
    xb, wb = workloads.bf16_bits(x), workloads.bf16_bits(w)
    ref = x.double().numpy() @ w.double().numpy().T
    ax, aw = oracle_mod.tensor_scale(xb), oracle_mod.tensor_scale(wb)
    cw0, sw0, _ = oracle_mod.quantize(0, wb, aw)
    e_plain = oracle_mod.nmse(oracle_mod.linear(0, False, xb, ax, cw0, sw0, aw), ref)
    calib = workloads.make_x("mlp_gate_up", 64, K=K, seed=5)  # calibration rows, same recipe
    score = np.abs(calib.float().numpy()).mean(axis=0)
    errs = {}
    for k in (1, 8):
        mask = oracle_mod.kext_select(score, k)
        cw, sw = oracle_mod.quantize_weight_kext(0, wb, k, mask, aw)
        errs[k] = oracle_mod.nmse(oracle_mod.linear_kext(0, xb, k, mask, ax, cw, sw, aw), ref)
    assert errs[1] < e_plain
    assert errs[8] <= errs[1]
