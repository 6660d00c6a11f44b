"""Pins of the ResAttn oracle (ResServe Sec. 4.3, Fig. 3, Sec. 5.2): closed
forms (one cached token; equal scores; two tokens whose FP8 softmax weight is
worked out by hand), the online softmax and split combination against the
plain softmax, the base + residue score fold against the effective query,
the GQA head mapping, empty and ragged sequences, and the error ordering of
the compensated query against the plain FP4 query."""
import math

import numpy as np
import pytest
import torch

from block_scaled_quantized_gb300 import workloads

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _bits(a):
    return workloads.bf16_bits(torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16))


def _grid_rows(rng, shape):
    """Rows of E2M1 grid values whose every 16-element block has amax 6: with
    tensor scale 1.0 their NVFP4 block scale is E4M3(1.0) and they quantize
    to themselves, and every value is also an E4M3 value (R14, R17)."""
    v = rng.choice(E2M1, size=shape) * rng.choice([-1.0, 1.0], size=shape)
    v[..., ::16] = 6.0
    return v


def _kv(oracle_mod, k_vals, v_vals):
    from oracle import resattn as ra
    B, L, H, D = k_vals.shape
    kc, ks = ra.kv_quantize(_bits(k_vals.reshape(-1, D)))
    vc, vs = ra.kv_quantize(_bits(v_vals.reshape(-1, D)))
    return (kc.reshape(B, L, H, D // 2), ks.reshape(B, L, H, D // 16),
            vc.reshape(B, L, H, D // 2), vs.reshape(B, L, H, D // 16))


def _e4m3_by_hand(p):
    """Nearest-even E4M3 of 0 < p <= 1 from its binary expansion (normal
    range: 3 fraction bits; below 2^-6 the step is 2^-9)."""
    e = max(math.floor(math.log2(p)), -6)
    step = 2.0 ** (e - 3)
    q = p / step
    r = math.floor(q + 0.5)
    if q + 0.5 == r and r % 2 == 1:  # a tie goes to the even multiple
        r -= 1
    return r * step


def test_one_cached_token_returns_its_value(oracle_mod):
    from oracle import resattn as ra
    rng = np.random.default_rng(1)
    D, Hq = 32, 4
    k = _grid_rows(rng, (1, 1, 1, D))
    v = _grid_rows(rng, (1, 1, 1, D))
    q = rng.standard_normal((1, Hq, D)).astype(np.float32)
    qb = _bits(q)
    O = ra.resattn_decode(qb, oracle_mod.tensor_scale(qb), *_kv(oracle_mod, k, v), np.array([1]))
    for g in range(Hq):
        np.testing.assert_array_equal(O[0, g], v[0, 0, 0])


@pytest.mark.parametrize("split", [None, 128, 256])
def test_equal_scores_average_the_values(oracle_mod, split):
    """Q = 0: every score is 0, every weight exp(0) = 1 is exact in E4M3, so O
    is the plain mean of the values over the sequence (300 tokens: three
    tiles, the last one ragged)."""
    from oracle import resattn as ra
    rng = np.random.default_rng(2)
    B, L, H, D, G = 1, 300, 2, 32, 3
    k = _grid_rows(rng, (B, L, H, D))
    v = _grid_rows(rng, (B, L, H, D))
    qb = _bits(np.zeros((B, H * G, D)))
    O = ra.resattn_decode(qb, 0.0, *_kv(oracle_mod, k, v), np.array([L]), split_tokens=split)
    for g in range(H * G):
        np.testing.assert_allclose(O[0, g], v[0, :, g // G].mean(axis=0), rtol=0, atol=1e-13)


@pytest.mark.parametrize("fp8_p", [True, False])
def test_two_tokens_worked_by_hand(oracle_mod, fp8_p):
    """D = 16, alpha_q = 2^-8: a query on the E2M1 grid with block amax 6 gets
    block scale E4M3(256) = 256, so Q^ = Q and R^ = 0 exactly.  Scores:
    s0 = <q, k0>/4 = 0 and s1 = <q, k1>/4 = 6 * (-0.5) / 4 = -0.75.  Weights
    1 and exp(-0.75) = 0.47237..., whose E4M3 value is 0.46875 (1.875 x 2^-2);
    O = (v0 + w v1) / (1 + w)."""
    from oracle import resattn as ra
    D = 16
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = 6.0
    k = np.zeros((1, 2, 1, D))
    k[0, :, 0, 5] = 6.0              # block amax 6 on a dimension the query ignores
    k[0, 1, 0, 0] = -0.5
    rng = np.random.default_rng(3)
    v = _grid_rows(rng, (1, 2, 1, D))
    O = ra.resattn_decode(_bits(q), 2.0 ** -8, *_kv(oracle_mod, k, v), np.array([2]), fp8_p=fp8_p)
    w = math.exp(-0.75)
    if fp8_p:
        w = _e4m3_by_hand(w)
        assert w == 0.46875
    np.testing.assert_allclose(O[0, 0], (v[0, 0, 0] + w * v[0, 1, 0]) / (1.0 + w), rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("split,tile", [(None, 128), (128, 128), (256, 128), (512, 64)])
@pytest.mark.parametrize("compensated", [True, False])
def test_online_softmax_and_splits_equal_plain_softmax(oracle_mod, split, tile, compensated):
    """With exact weights (fp8_p off) the tile-by-tile online softmax and the
    split combination (R18, R19) must give the plain softmax over the whole
    sequence; the scores are those of the effective query Q^ + R^ (the base
    and residue scores added before the softmax, R16), or Q^ alone."""
    from oracle import resattn as ra
    B, Hq, Hkv, D = 2, 8, 2, 64
    q, k, v = workloads.make_attention(B, Hq, Hkv, D, 700, seed=4)
    qb, kb, vb = workloads.bf16_bits(q), workloads.bf16_bits(k), workloads.bf16_bits(v)
    kc, ks = ra.kv_quantize(kb.reshape(-1, D))
    vc, vs = ra.kv_quantize(vb.reshape(-1, D))
    shp = (B, 700, Hkv)
    kc, ks, vc, vs = kc.reshape(*shp, D // 2), ks.reshape(*shp, D // 16), vc.reshape(*shp, D // 2), vs.reshape(*shp, D // 16)
    a = oracle_mod.tensor_scale(qb)
    lens = np.array([700, 333])
    O = ra.resattn_decode(qb, a, kc, ks, vc, vs, lens, compensated=compensated, split_tokens=split, tile=tile,
                          fp8_p=False)
    qh, rh = ra.query_operands(qb.reshape(-1, D), a, compensated)
    q_eff = (qh + rh).reshape(B, Hq, D)
    K = ra.kv_dequantize(kc.reshape(-1, D // 2), ks.reshape(-1, D // 16)).reshape(B, 700, Hkv, D)
    V8 = ra.v_to_fp8(vc.reshape(-1, D // 2), vs.reshape(-1, D // 16)).reshape(B, 700, Hkv, D)
    ref = ra.attention_reference(q_eff, K, V8, lens, Hq // Hkv)
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


def test_gqa_heads_read_their_kv_head(oracle_mod):
    """Query head g reads KV head g // G: swapping the two KV heads swaps the
    outputs of the two query groups."""
    from oracle import resattn as ra
    B, Hq, Hkv, D, L = 1, 6, 2, 32, 200
    q, k, v = workloads.make_attention(B, Hq, Hkv, D, L, seed=5)
    qb, kb, vb = workloads.bf16_bits(q), workloads.bf16_bits(k), workloads.bf16_bits(v)
    ops = _kv(oracle_mod, k.float().numpy(), v.float().numpy())
    a = oracle_mod.tensor_scale(qb)
    O = ra.resattn_decode(qb, a, *ops, np.array([L]))
    swapped = [x[:, :, ::-1].copy() for x in ops]
    q_sw = np.concatenate([qb[:, 3:], qb[:, :3]], axis=1)     # groups swapped too
    O_sw = ra.resattn_decode(q_sw, a, *swapped, np.array([L]))
    np.testing.assert_array_equal(O_sw[:, :3], O[:, 3:])
    np.testing.assert_array_equal(O_sw[:, 3:], O[:, :3])


def test_empty_and_ragged_sequences(oracle_mod):
    from oracle import resattn as ra
    B, Hq, Hkv, D, L = 3, 4, 1, 32, 260
    q, k, v = workloads.make_attention(B, Hq, Hkv, D, L, seed=6)
    qb = workloads.bf16_bits(q)
    ops = _kv(oracle_mod, k.float().numpy(), v.float().numpy())
    a = oracle_mod.tensor_scale(qb)
    O = ra.resattn_decode(qb, a, *ops, np.array([0, 129, 260]), split_tokens=128)
    assert not O[0].any()
    # the rows past a sequence's length are never read
    ops2 = [x.copy() for x in ops]
    for x in ops2:
        x[1, 129:] = 0x77
    O2 = ra.resattn_decode(qb, a, *ops2, np.array([0, 129, 260]), split_tokens=128)
    np.testing.assert_array_equal(O2[1], O[1])


def test_fp8_weights_stay_close(oracle_mod):
    """Rounding the weights to E4M3 (R18) perturbs each by at most 2^-4
    relative (or drops weights below 2^-10); the output stays close to the
    exact-weight output."""
    from oracle import resattn as ra
    B, Hq, Hkv, D, L = 2, 8, 1, 128, 1000
    q, k, v = workloads.make_attention(B, Hq, Hkv, D, L, seed=7)
    qb = workloads.bf16_bits(q)
    ops = _kv(oracle_mod, k.float().numpy(), v.float().numpy())
    a = oracle_mod.tensor_scale(qb)
    lens = np.array([L, 517])
    O8 = ra.resattn_decode(qb, a, *ops, lens, split_tokens=256)
    O = ra.resattn_decode(qb, a, *ops, lens, split_tokens=256, fp8_p=False)
    assert oracle_mod.nmse(O8, O) < 1e-3
    assert np.abs(O8 - O).max() <= 0.1 * np.abs(O).max()


def test_compensated_query_lowers_attention_error(oracle_mod):
    """Against attention with the BF16 query and the same NVFP4 K/V (the
    reference the paper uses to isolate attention-computation error), the
    compensated query's pooled NMSE is below the plain FP4 query's."""
    from oracle import resattn as ra
    errs = {True: [], False: []}
    for seed in range(3):
        B, Hq, Hkv, D, L = 2, 8, 1, 128, 512
        q, k, v = workloads.make_attention(B, Hq, Hkv, D, L, seed=10 + seed)
        qb = workloads.bf16_bits(q)
        kc, ks, vc, vs = _kv(oracle_mod, k.float().numpy(), v.float().numpy())
        a = oracle_mod.tensor_scale(qb)
        lens = np.array([L, L])
        K = ra.kv_dequantize(kc.reshape(-1, D // 2), ks.reshape(-1, D // 16)).reshape(B, L, Hkv, D)
        V = ra.kv_dequantize(vc.reshape(-1, D // 2), vs.reshape(-1, D // 16)).reshape(B, L, Hkv, D)
        ref = ra.attention_reference(q.float().numpy(), K, V, lens, Hq // Hkv)
        for comp in (True, False):
            errs[comp].append((ra.resattn_decode(qb, a, kc, ks, vc, vs, lens, compensated=comp), ref))
    pooled = {c: oracle_mod.nmse(np.concatenate([o for o, _ in e]), np.concatenate([r for _, r in e]))
              for c, e in errs.items()}
    assert pooled[True] < pooled[False]
