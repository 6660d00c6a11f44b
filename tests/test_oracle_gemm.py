"""Pins for the oracle's block-scaled GEMM and the compensated linear layer.

* brute force with exact rational arithmetic on tiny shapes, decoding every
  element through the library casts (ml_dtypes E2M1, torch E4M3/E8M0);
* the double-precision product of dequantized operands from numpy's matmul;
* Eq. 4's operand swap: Z(W, A) = Z(A, W)^T;
* Eq. 2's stacked GEMM + Fold equals Eq. 1's sum of two GEMMs;
* App. C.2's pooled NMSE: the compensated layer is closer than W4A4 to the
  FP32 product of the original bf16 operands (Table 3's direction).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from block_scaled_quantized_gb300 import workloads


def _lib_decode(fmt, codes, sf):
    """Dequantize with library decoders (no oracle code involved)."""
    mld = pytest.importorskip("ml_dtypes")
    rows, half = codes.shape
    q = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(rows, 2 * half)
    vals = q.astype(np.uint8).view(mld.float4_e2m1fn).astype(np.float64)
    dt = torch.float8_e4m3fn if fmt == 0 else torch.float8_e8m0fnu
    s = torch.from_numpy(np.ascontiguousarray(sf)).view(dt).to(torch.float64).numpy()
    bs = 16 if fmt == 0 else 32
    return vals * np.repeat(s, bs, axis=1)


def _random_operand(rng, fmt, rows, K):
    codes = rng.integers(0, 256, size=(rows, K // 2)).astype(np.uint8)
    if fmt == 0:
        sf = rng.integers(0, 0x7F, size=(rows, K // 16)).astype(np.uint8)
    else:
        sf = rng.integers(100, 150, size=(rows, K // 32)).astype(np.uint8)
    return codes, sf


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (2, 3, 32), (4, 8, 64), (3, 5, 96)])
def test_block_gemm_brute_force_exact(oracle_mod, fmt, M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K + fmt)
    ca, sa = _random_operand(rng, fmt, M, K)
    cb, sb = _random_operand(rng, fmt, N, K)
    Z = oracle_mod.block_gemm(fmt, ca, sa, cb, sb)
    A = _lib_decode(fmt, ca, sa)
    B = _lib_decode(fmt, cb, sb)
    for m in range(M):
        for n in range(N):
            exact = sum((Fraction(float(A[m, k])) * Fraction(float(B[n, k])) for k in range(K)),
                        Fraction(0))
            assert abs(Fraction(float(Z[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + \
                Fraction(1, 2 ** 200)


@pytest.mark.parametrize("fmt", [0, 1])
def test_block_gemm_matches_numpy_matmul_and_swap(oracle_mod, fmt):
    rng = np.random.default_rng(7 + fmt)
    ca, sa = _random_operand(rng, fmt, 6, 256)
    cb, sb = _random_operand(rng, fmt, 40, 256)
    Z = oracle_mod.block_gemm(fmt, ca, sa, cb, sb)
    ref = _lib_decode(fmt, ca, sa) @ _lib_decode(fmt, cb, sb).T
    np.testing.assert_allclose(Z, ref, rtol=1e-12, atol=1e-300)
    Zt = oracle_mod.block_gemm(fmt, cb, sb, ca, sa)           # Eq. 4 swap
    np.testing.assert_array_equal(Zt, Z.T)


@pytest.mark.parametrize("fmt", [0, 1])
def test_linear_equals_stacked_gemm_and_fold(oracle_mod, fmt):
    o = oracle_mod
    M, N, K = 5, 48, 512
    x = workloads.make_x("gauss_outlier_k2048", M, K=K, seed=11)
    w = workloads.make_w("gauss_outlier_k2048", N=N, K=K, seed=12)
    xb, wb = workloads.bf16_bits(x), workloads.bf16_bits(w)
    ax = o.tensor_scale(xb) if fmt == 0 else np.float32(0)
    aw = o.tensor_scale(wb) if fmt == 0 else np.float32(0)
    cw, sw, _ = o.quantize(fmt, wb, aw)
    q = o.quantize_residue(fmt, xb, ax)
    # Eq. 2: stack [X^; R^] as 2M rows, one GEMM, then Fold rows j and M+j.
    Zs = o.block_gemm(fmt, np.vstack([q["codes_x"], q["codes_r"]]),
                      np.vstack([q["sf_x"], q["sf_r"]]), cw, sw)
    g = float(ax) * float(aw) if fmt == 0 else 1.0
    folded = g * (Zs[:M] + Zs[M:])
    Y = o.linear(fmt, True, xb, ax, cw, sw, aw)
    np.testing.assert_array_equal(Y, folded)
    Yp = o.linear(fmt, False, xb, ax, cw, sw, aw)
    np.testing.assert_array_equal(Yp, g * Zs[:M])
    # Eq. 1 with the dequantized operands as values.
    xh = _lib_decode(fmt, q["codes_x"], q["sf_x"])
    rh = _lib_decode(fmt, q["codes_r"], q["sf_r"])
    wh = _lib_decode(fmt, cw, sw)
    np.testing.assert_allclose(Y, g * (xh @ wh.T + rh @ wh.T), rtol=1e-12, atol=1e-30)


@pytest.mark.parametrize("fmt,recipe", [(0, "gauss_outlier_k2048"), (0, "attn_proj_k4096"),
                                        (0, "mlp_down"), (1, "mx_k5120_n27648")])
def test_compensation_lowers_nmse(oracle_mod, fmt, recipe):
    o = oracle_mod
    M, N, K = 8, 256, 1024
    x = workloads.make_x(recipe, M, K=K, seed=21)
    w = workloads.make_w(recipe, N=N, K=K, seed=22)
    xb, wb = workloads.bf16_bits(x), workloads.bf16_bits(w)
    ax = o.tensor_scale(xb) if fmt == 0 else np.float32(0)
    aw = o.tensor_scale(wb) if fmt == 0 else np.float32(0)
    cw, sw, wq = o.quantize(fmt, wb, aw)
    # App. C.2: FP32 product of the original bf16 operands.
    ref = (x.float() @ w.float().T).double().numpy()
    plain = o.linear(fmt, False, xb, ax, cw, sw, aw)
    comp = o.linear(fmt, True, xb, ax, cw, sw, aw)
    assert o.nmse(comp, ref) < o.nmse(plain, ref)
    # With the weight error removed the activation error shrinks sharply.
    ref_w = x.double().numpy() @ wq.astype(np.float64).T
    assert o.nmse(comp, ref_w) < 0.1 * o.nmse(plain, ref_w)


def test_thread_count_does_not_change_results():
    """The all-core baseline runs the same k-ordered double sums: outputs are
    bit-identical for any number of oracle threads."""
    import oracle
    from block_scaled_quantized_gb300 import workloads
    x = workloads.make_x("attn_proj_k4096", 5, K=512, seed=9)
    w = workloads.make_w("attn_proj_k4096", N=300, K=512, seed=9)
    xb, wb = workloads.bf16_bits(x), workloads.bf16_bits(w)
    aw = oracle.tensor_scale(wb)
    cw, sw, _ = oracle.quantize(0, wb, aw)
    ax = oracle.tensor_scale(xb)
    ys = []
    for t in (1, 3, 8):
        oracle.set_threads(t)
        ys.append(oracle.linear(0, True, xb, ax, cw, sw, aw))
    oracle.set_threads(1)
    assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])
