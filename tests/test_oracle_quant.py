"""Pins for the oracle's NVFP4 / MXFP4 quantizers (base and residue).

What pins them (ResServe App. B.2 Eq. 8-10, Algorithm 1, Sec. 2):
* a block worked out by hand (tests/golden/nvfp4_tie_block.txt);
* inputs that are exactly representable quantize to themselves with a zero
  residue and all-zero residue codes;
* Eq. 8's tensor-scale form max_i(Max_i/6)/448 agrees with amax/2688;
* the block scale is the E4M3 value nearest to (Max/6)/alpha (or its
  saturation), checked against a torch float8 cast;
* the codes are the E2M1 values nearest to x * fl(1/s~), checked against an
  ml_dtypes cast; the reconstruction and the residue satisfy their
  definitions exactly; the MXFP4 scale keeps the block maximum in [4, 8);
* the compensated reconstruction X^ + R^ is closer to X than X^ alone.
"""
import numpy as np
import pytest
import torch

from conftest import read_golden
from block_scaled_quantized_gb300 import workloads


def _bits(a):
    return workloads.bf16_bits(workloads.to_bf16(np.asarray(a, np.float32)))


def _unpack(codes):
    lo = codes & 0xF
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def _e2m1_value(c):
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float64)
    v = mags[c & 7]
    return np.where(c & 8, -v, v)


def test_hand_worked_block(oracle_mod):
    o = oracle_mod
    g = read_golden("nvfp4_tie_block.txt")
    x = np.array([float(v) for v in g["x"]], np.float32)[None, :]
    alpha = float(g["alpha"][0])
    out = o.quantize_residue(o.NVFP4, _bits(x), alpha)
    assert out["sf_x"][0, 0] == int(g["base_sf"][0], 16)
    np.testing.assert_array_equal(_unpack(out["codes_x"])[0], [int(v) for v in g["base_codes"]])
    np.testing.assert_array_equal(out["resid"][0], [float(v) for v in g["resid"]])
    assert out["sf_r"][0, 0] == int(g["resid_sf"][0], 16)
    np.testing.assert_array_equal(_unpack(out["codes_r"])[0], [int(v) for v in g["resid_codes"]])
    _, _, xhat = o.quantize(o.NVFP4, _bits(x), alpha)
    np.testing.assert_array_equal(xhat[0], [float(v) for v in g["base_xhat"]])
    assert np.signbit(xhat[0, 15])

    xm = np.concatenate([x, x], axis=1)
    mx = o.quantize_residue(o.MXFP4, _bits(xm))
    assert mx["sf_x"][0, 0] == int(g["mx_base_sf"][0], 16)
    np.testing.assert_array_equal(_unpack(mx["codes_x"])[0, :16], [int(v) for v in g["base_codes"]])
    assert mx["sf_r"][0, 0] == int(g["mx_resid_sf"][0], 16)
    np.testing.assert_array_equal(_unpack(mx["codes_r"])[0, :16], [int(v) for v in g["mx_resid_codes"]])
    np.testing.assert_array_equal(_unpack(mx["codes_r"])[0, 16:], [int(v) for v in g["mx_resid_codes"]])


@pytest.mark.parametrize("log2_alpha", [-12, -5, 0, 3])
def test_nvfp4_representable_inputs_have_zero_residue(oracle_mod, log2_alpha):
    o = oracle_mod
    rng = np.random.default_rng(100 + log2_alpha)
    rows, K = 6, 256
    nb = K // 16
    alpha = 2.0 ** log2_alpha
    # block scales: any finite non-zero E4M3 byte (normal and subnormal)
    sf = rng.integers(1, 0x7F, size=(rows, nb)).astype(np.uint8)
    q = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
    # one element of every block carries the E2M1 maximum (+-6)
    pos = rng.integers(0, 16, size=(rows, nb))
    for r in range(rows):
        for b in range(nb):
            q[r, b * 16 + pos[r, b]] = 7 | (q[r, b * 16 + pos[r, b]] & 8)
    sfv = np.array([o.e4m3_decode(int(b)) for b in range(256)])[sf]
    x = alpha * np.repeat(sfv, 16, axis=1) * _e2m1_value(q)
    x32 = x.astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x)           # exact in fp32
    bits = _bits(x32)
    assert np.array_equal(workloads.to_bf16(x32).float().numpy(), x32)  # exact in bf16
    out = o.quantize_residue(o.NVFP4, bits, np.float32(alpha))
    np.testing.assert_array_equal(out["sf_x"], sf)
    np.testing.assert_array_equal(_unpack(out["codes_x"]), q)
    assert not np.any(out["resid"])
    assert not np.any(_unpack(out["codes_r"]))
    assert not np.any(out["sf_r"])


def test_mxfp4_representable_inputs_have_zero_residue(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(3)
    rows, K = 5, 256
    nb = K // 32
    e = rng.integers(-100, 100, size=(rows, nb))
    q = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
    pos = rng.integers(0, 32, size=(rows, nb))
    top = rng.choice([6, 7], size=(rows, nb))                  # |q| = 4 or 6
    for r in range(rows):
        for b in range(nb):
            i = b * 32 + pos[r, b]
            q[r, i] = top[r, b] | (q[r, i] & 8)
    x = np.ldexp(_e2m1_value(q), np.repeat(e, 32, axis=1)).astype(np.float32)
    out = o.quantize_residue(o.MXFP4, _bits(x))
    np.testing.assert_array_equal(out["sf_x"], (e + 127).astype(np.uint8))
    np.testing.assert_array_equal(_unpack(out["codes_x"]), q)
    assert not np.any(out["resid"])
    assert not np.any(_unpack(out["codes_r"]))


def test_tensor_scale_matches_eq8(oracle_mod):
    o = oracle_mod
    for seed in range(5):
        x = workloads.make_x("attn_proj_k4096", 4, seed=seed)
        bits = workloads.bf16_bits(x)
        alpha = o.tensor_scale(bits)
        xf = x.float().numpy()
        blocks = np.abs(xf).reshape(-1, 16).max(axis=1)
        eq8 = np.float32(np.float32(blocks.max()) / np.float32(6)) / np.float32(448)
        assert abs(float(alpha) - float(eq8)) <= float(np.spacing(np.float32(eq8)))
        assert alpha == np.float32(np.float32(np.abs(xf).max()) / np.float32(2688))


def _library_nvfp4_rows(xf, alpha):
    """NVFP4 QDQ with the two roundings done by library casts: torch's
    float8_e4m3fn cast for the block scale and ml_dtypes' float4_e2m1fn cast
    for the elements."""
    mld = pytest.importorskip("ml_dtypes")
    rows, K = xf.shape
    blk = xf.reshape(rows, K // 16, 16)
    amax = np.abs(blk).max(axis=2)
    s = (amax / np.float32(6)).astype(np.float32)
    t = (s / np.float32(alpha)).astype(np.float32) if alpha > 0 else np.zeros_like(s)
    t = np.minimum(t, np.float32(448))
    sf = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    sfv = torch.from_numpy(sf).view(torch.float8_e4m3fn).float().numpy()
    st = (np.float32(alpha) * sfv).astype(np.float32)
    with np.errstate(divide="ignore"):
        mul = np.where(st == 0, np.float32(0), (np.float32(1) / st)).astype(np.float32)
    v = (blk * mul[:, :, None]).astype(np.float32)
    v = np.clip(v, -6, 6)
    q = v.astype(mld.float4_e2m1fn).view(np.uint8).reshape(rows, K) & 0xF
    return sf, q


@pytest.mark.parametrize("recipe", ["gauss_outlier_k2048", "attn_proj_k4096", "mlp_gate_up"])
def test_nvfp4_codes_against_library_casts(oracle_mod, recipe):
    o = oracle_mod
    x = workloads.make_x(recipe, 8, K=1024, seed=5)
    bits = workloads.bf16_bits(x)
    alpha = o.tensor_scale(bits)
    out = o.quantize_residue(o.NVFP4, bits, alpha)
    xf = x.float().numpy()
    sf, q = _library_nvfp4_rows(xf, alpha)
    np.testing.assert_array_equal(out["sf_x"], sf)
    np.testing.assert_array_equal(_unpack(out["codes_x"]), q)
    sf_r, q_r = _library_nvfp4_rows(out["resid"], alpha)
    np.testing.assert_array_equal(out["sf_r"], sf_r)
    np.testing.assert_array_equal(_unpack(out["codes_r"]), q_r)


@pytest.mark.parametrize("fmt", [0, 1])
def test_reconstruction_and_residue_definitions(oracle_mod, fmt):
    o = oracle_mod
    bs = o.block_size(fmt)
    x = workloads.make_x("attn_proj_k4096", 4, K=512, seed=9)
    bits = workloads.bf16_bits(x)
    alpha = o.tensor_scale(bits) if fmt == 0 else np.float32(0)
    out = o.quantize_residue(fmt, bits, alpha)
    xf = x.float().numpy()
    if fmt == 0:
        sfv = torch.from_numpy(out["sf_x"]).view(torch.float8_e4m3fn).float().numpy()
        st = (np.float32(alpha) * sfv).astype(np.float32)
    else:
        st = torch.from_numpy(out["sf_x"]).view(torch.float8_e8m0fnu).float().numpy()
    st_el = np.repeat(st, bs, axis=1)
    xhat = (st_el * _e2m1_value(_unpack(out["codes_x"])).astype(np.float32)).astype(np.float32)
    np.testing.assert_array_equal(out["resid"], (xf - xhat).astype(np.float32))
    # E2M1 step is at most 2 (between 4 and 6): an unsaturated element is
    # within one scale unit of its reconstruction.
    v = np.abs(xf) / np.where(st_el == 0, np.inf, st_el)
    ok = v <= 6
    assert np.all(np.abs(xf - xhat)[ok] <= st_el[ok] * (1 + 2 ** -20))


def test_mxfp4_scale_keeps_block_max_in_range(oracle_mod):
    o = oracle_mod
    x = workloads.make_x("mx_k5120_n27648", 8, K=1024, seed=2)
    bits = workloads.bf16_bits(x)
    out = o.quantize_residue(o.MXFP4, bits)
    xf = x.float().numpy().astype(np.float64)
    amax = np.abs(xf).reshape(8, -1, 32).max(axis=2)
    e = out["sf_x"].astype(np.int64) - 127
    ratio = amax / np.ldexp(1.0, e)
    nz = amax > 0
    assert np.all((ratio[nz] >= 4) & (ratio[nz] < 8))
    r = out["resid"].astype(np.float64)
    ramax = np.abs(r).reshape(8, -1, 32).max(axis=2)
    er = out["sf_r"].astype(np.int64) - 127
    nzr = ramax > 2.0 ** -100
    rr = ramax[nzr] / np.ldexp(1.0, er[nzr])
    assert np.all((rr >= 4) & (rr < 8))


@pytest.mark.parametrize("fmt", [0, 1])
def test_residue_reduces_reconstruction_error(oracle_mod, fmt):
    o = oracle_mod
    x = workloads.make_x("attn_proj_k4096", 8, K=1024, seed=4)
    bits = workloads.bf16_bits(x)
    alpha = o.tensor_scale(bits) if fmt == 0 else 0.0
    out = o.quantize_residue(fmt, bits, alpha)
    _, _, xhat = o.quantize(fmt, bits, alpha)
    xf = x.float().numpy().astype(np.float64)
    e_base = np.sum((xf - xhat) ** 2)
    e_comp = np.sum((xf - xhat - out["rhat"]) ** 2)
    assert e_comp < 0.1 * e_base


def test_zero_and_tiny_blocks(oracle_mod):
    o = oracle_mod
    x = np.zeros((2, 32), np.float32)
    x[1, :16] = -0.0
    x[1, 16] = 1e-30                       # far below alpha * 2^-9
    x[1, 17] = 1.0
    bits = _bits(x)
    alpha = o.tensor_scale(bits)
    out = o.quantize_residue(o.NVFP4, bits, alpha)
    assert out["sf_x"][0, 0] == 0 and out["sf_x"][0, 1] == 0
    assert np.all(_unpack(out["codes_x"])[0] == 0)
    assert np.all(_unpack(out["codes_x"])[1, :16] == 8)      # -0 keeps its sign
    # alpha = 0 (all-zero tensor) quantizes to zero scales and +-0 codes
    z = o.quantize_residue(o.NVFP4, _bits(np.zeros((1, 16), np.float32)), 0.0)
    assert not np.any(z["sf_x"]) and not np.any(z["codes_x"])


def test_division_reading_differs_rarely_by_one_step(oracle_mod):
    """Eq. 10 divides, x / s~; Alg. 1 multiplies by the fp32 reciprocal (the
    reading the quantizers take, R3).  Both give the same scale bytes; codes
    differ only where the two fp32 values straddle an E2M1 rounding boundary,
    by one step and with the same sign, and rarely.  The first difference is
    recomputed by hand in numpy fp32."""
    o = oracle_mod
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    total = changed = 0
    example = None
    for rec in ["gauss_outlier_k2048", "attn_proj_k4096", "mlp_down", "prefill_k8192"]:
        x = workloads.make_x(rec, 64, seed=3)
        xb = workloads.bf16_bits(x)
        a = o.tensor_scale(xb)
        cm, sm, _ = o.quantize(0, xb, a)
        cd, sd = o.quantize_nvfp4_div(xb, a)
        assert np.array_equal(sm, sd)
        qm = np.stack([cm & 15, cm >> 4], axis=-1).reshape(cm.shape[0], -1)
        qd = np.stack([cd & 15, cd >> 4], axis=-1).reshape(cd.shape[0], -1)
        diff = np.argwhere(qm != qd)
        for r, k in diff:
            assert (qm[r, k] & 8) == (qd[r, k] & 8) and abs(int(qm[r, k] & 7) - int(qd[r, k] & 7)) == 1
        if len(diff) and example is None:
            r, k = diff[0]
            example = (x[r, k].item(), float(a), int(sm[r, k // 16]), int(qm[r, k]), int(qd[r, k]))
        total += qm.size
        changed += len(diff)
    assert changed / total < 1e-3 and example is not None
    xv, alpha, sfb, code_mul, code_div = example
    st = np.float32(np.float32(alpha) * np.float32(o.e4m3_decode(sfb)))
    v_mul = np.float32(np.float32(xv) * np.float32(np.float32(1.0) / st))
    v_div = np.float32(np.float32(xv) / st)
    assert v_mul != v_div
    for v, code in ((v_mul, code_mul), (v_div, code_div)):
        mag = abs(float(v))
        i = int(np.argmin(np.abs(grid - mag)))
        d = np.abs(grid - mag)
        if np.sum(d == d[i]) > 1:  # a tie: the even code
            i = [j for j in np.flatnonzero(d == d[i]) if j % 2 == 0][0]
        assert (code & 7) == i


def test_alg1_reconstruction_reading_differs_rarely(oracle_mod):
    """Eq. 10 writes x^ = s~ x_FP4 (reading R5: fl(s~ dec(q))); Alg. 1 line 6
    forms the residue as x - x_q / scale with the fp32 multiplier, i.e.
    x^ = fl(dec(q) / fl(1/s~)).  The base operand is the same under both.
    The two reconstructions are recomputed here in numpy fp32: where they
    agree on a whole block, the residue codes and scale byte of that block
    agree too; where they differ, it is by one ulp of x^, and a residue code
    moves by at most one E2M1 step (or only its sign, at zero).  That happens
    for about 1e-5 of the elements on the recipes (bounded by 1e-3 here)."""
    o = oracle_mod
    f32 = np.float32
    total = changed = 0
    for rec in ["gauss_outlier_k2048", "attn_proj_k4096", "mlp_down", "prefill_k8192"]:
        x = workloads.make_x(rec, 64, seed=3)
        xb = workloads.bf16_bits(x)
        a = o.tensor_scale(xb)
        q = o.quantize_residue(0, xb, a)
        r = o.quantize_residue_nvfp4_recon_div(xb, a)
        assert np.array_equal(q["codes_x"], r["codes_x"]) and np.array_equal(q["sf_x"], r["sf_x"])
        rows, K = xb.shape
        nib = lambda c: np.stack([c & 15, c >> 4], axis=-1).reshape(rows, K)
        d = np.array([o.e2m1_decode(c) for c in range(16)], np.float32)[nib(q["codes_x"])]
        st = (f32(a) * np.array([o.e4m3_decode(b) for b in range(256)], np.float32)[q["sf_x"]]).astype(f32)
        st = np.repeat(st, 16, axis=1)
        mul = np.where(st == 0, f32(0), (f32(1) / np.where(st == 0, f32(1), st)).astype(f32)).astype(f32)
        xh_eq10 = (st * d).astype(f32)
        with np.errstate(divide="ignore", invalid="ignore"):
            xh_alg1 = np.where(mul == 0, f32(0), (d / np.where(mul == 0, f32(1), mul)).astype(f32)).astype(f32)
        differ = xh_eq10 != xh_alg1
        ulps = np.abs(xh_eq10.view(np.int32).astype(np.int64) - xh_alg1.view(np.int32).astype(np.int64))
        assert np.all(ulps[differ] == 1)
        same_block = ~differ.reshape(rows, K // 16, 16).any(axis=2)
        assert np.array_equal(q["sf_r"][same_block], r["sf_r"][same_block])
        cq, cr = nib(q["codes_r"]), nib(r["codes_r"])
        same_el = np.repeat(same_block, 16, axis=1)
        assert np.array_equal(cq[same_el], cr[same_el])
        for rr, k in np.argwhere(cq != cr):
            a_, b_ = int(cq[rr, k]), int(cr[rr, k])
            assert abs((a_ & 7) - (b_ & 7)) <= 1
            assert (a_ & 8) == (b_ & 8) or (a_ & 7) == (b_ & 7) == 0
        total += cq.size
        changed += int(np.sum(cq != cr))
    assert 0 < changed and changed / total < 1e-3
