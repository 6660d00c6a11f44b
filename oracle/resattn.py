"""Plain CPU oracle for residue-compensated decode attention (ResAttn).

TEST INFRASTRUCTURE ONLY, like the rest of this package: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may use it.

Source: "ResServe: Accurate and Efficient FP4 LLM Inference with Residue
Compensation", Sec. 4.3 (ResAttn: the BF16 query of a query-head group is
split into an FP4 base and a quantized residue; their scores against the
cached FP4 keys are added before the softmax), Fig. 3, and Sec. 5.2 (ResAttn
execution: a query-quantization step produces the base and residue rows; the
keys are used directly from the paged NVFP4 cache with scale groups along the
head dimension; base and residue scores are added in FP32 before an online
softmax; V is converted from NVFP4 to FP8 on chip and PV runs with FP8
operands, FP32 accumulation and normalization; the sequence is split into
parts whose partial outputs and softmax statistics are combined).

Readings taken where the paper leaves a step open (also listed in the design
notes):

  R14  K and V are NVFP4 (16-element blocks along the head dimension, E4M3
       block scales) with tensor scale 1.0, quantized row by row (one token
       of one KV head per row) exactly as the activation quantizer does.
  R15  The query is quantized with Alg. 1 (base and residue, own block
       scales, one tensor scale alpha_q for the whole Q tensor of the call);
       query head g of a group of G reads KV head g // G.
  R16  Scores: s = (<Q^, K^> + <R^, K^>) * alpha_q * alpha_k / sqrt(D) with
       the dequantized operands; the oracle sums in double.
  R17  V on chip: each dequantized element fl(s~ * dec(q)) (exact in fp32)
       is rounded to E4M3, nearest-even, saturating to 448.
  R18  Online softmax over tiles of T tokens (T = 128) inside each split: the
       running maximum m is updated with the tile's scores, the weights are
       p = exp(s - m), rounded to E4M3 (fp32 p, nearest-even) for PV, and the
       normalizer l sums the rounded weights, so O = sum(p8 v8) / sum(p8) in
       every split.  Earlier partial sums are rescaled by exp(m_old - m_new).
  R19  Splits are consecutive ranges of S tokens (a multiple of T); their
       partial outputs o_s and normalizers l_s combine as
       O = sum_s exp(m_s - M) o_s / sum_s exp(m_s - M) l_s, M = max_s m_s.
       A sequence of length 0 gives O = 0.
"""
from __future__ import annotations

import math

import numpy as np

from . import NVFP4, dequantize, e4m3_decode, e4m3_encode_array, quantize, quantize_residue

TILE = 128  # tokens per online-softmax step (R18)


_E4M3_TABLE = None


def _e4m3_values(v) -> np.ndarray:
    """E4M3 nearest-even, saturating (R17/R18), of fp32 values, as float64."""
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        _E4M3_TABLE = np.array([e4m3_decode(b) for b in range(256)], np.float64)
    v32 = np.asarray(v, np.float32)
    codes = e4m3_encode_array(v32.ravel())
    return _E4M3_TABLE[codes].reshape(v32.shape)


def kv_quantize(x_u16):
    """NVFP4 codes and block scales of bf16 K or V rows [rows][D] with tensor
    scale 1.0 (R14).  Returns (codes [rows][D/2], sf [rows][D/16])."""
    codes, sf, _ = quantize(NVFP4, x_u16, 1.0)
    return codes, sf


def kv_dequantize(codes, sf) -> np.ndarray:
    """Values of NVFP4 K/V rows (tensor scale 1.0): s~ * dec(q), float64."""
    return dequantize(NVFP4, codes, sf)


def v_to_fp8(codes, sf) -> np.ndarray:
    """V converted from NVFP4 to FP8 on chip (R17), as float64 values."""
    return _e4m3_values(kv_dequantize(codes, sf).astype(np.float32))


def query_operands(q_u16, alpha_q: float, compensated: bool = True):
    """Dequantized base Q^ and residue R^ of bf16 query rows [rows][D]
    (Alg. 1, R15), tensor scale applied.  R^ is zero without compensation."""
    out = quantize_residue(NVFP4, q_u16, alpha_q)
    qh = float(alpha_q) * dequantize(NVFP4, out["codes_x"], out["sf_x"])
    rh = float(alpha_q) * dequantize(NVFP4, out["codes_r"], out["sf_r"])
    return qh, (rh if compensated else np.zeros_like(rh))


def resattn_decode(q_u16, alpha_q: float, k_codes, k_sf, v_codes, v_sf, seq_lens, compensated: bool = True,
                   split_tokens: int | None = None, tile: int = TILE, fp8_p: bool = True) -> np.ndarray:
    """One decode step of ResAttn (Sec. 4.3, Sec. 5.2).

    q_u16:   bf16 bits [B][Hq][D]
    k_codes, v_codes: [B][L][Hkv][D/2] NVFP4 codes (logical token order)
    k_sf, v_sf:       [B][L][Hkv][D/16] E4M3 block scales (tensor scale 1.0)
    seq_lens: [B] tokens per sequence (<= L)
    split_tokens: tokens per split (a multiple of tile); None: one split
    fp8_p: round the softmax weights to E4M3 for PV (R18); False keeps them
           exact (used to check the online softmax against the plain one)
    Returns O [B][Hq][D] float64."""
    q = np.asarray(q_u16, np.uint16)
    B, Hq, D = q.shape
    Hkv = k_codes.shape[2]
    G = Hq // Hkv
    assert Hq == G * Hkv and D % 16 == 0
    S = split_tokens or max(int(np.max(seq_lens)) if len(seq_lens) else 0, 1)
    assert S % tile == 0 or split_tokens is None
    qh, rh = query_operands(q.reshape(B * Hq, D), alpha_q, compensated)
    qh = qh.reshape(B, Hq, D)
    rh = rh.reshape(B, Hq, D)
    c = 1.0 / math.sqrt(D)  # alpha_k = 1.0 (R14)
    O = np.zeros((B, Hq, D), np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        for h in range(Hkv):
            K = kv_dequantize(k_codes[b, :L, h], k_sf[b, :L, h])           # [L][D]
            V = v_to_fp8(v_codes[b, :L, h], v_sf[b, :L, h])                # [L][D]
            heads = range(h * G, (h + 1) * G)
            # base and residue scores added before the softmax (R16)
            s_all = (qh[b, heads] @ K.T + rh[b, heads] @ K.T) * c         # [G][L]
            parts = []
            for t0 in range(0, L, S):
                t1 = min(L, t0 + S)
                m = np.full(G, -np.inf)
                l = np.zeros(G)
                o = np.zeros((G, D))
                for u0 in range(t0, t1, tile):                             # online softmax (R18)
                    u1 = min(t1, u0 + tile)
                    s = s_all[:, u0:u1]
                    m_new = np.maximum(m, s.max(axis=1))
                    a = np.exp(m - m_new)
                    p = np.exp(s - m_new[:, None])
                    p = _e4m3_values(p) if fp8_p else p
                    o = o * a[:, None] + p @ V[u0:u1]
                    l = l * a + p.sum(axis=1)
                    m = m_new
                parts.append((m, l, o))
            M = np.max([pt[0] for pt in parts], axis=0)                    # split combination (R19)
            num = sum(np.exp(pt[0] - M)[:, None] * pt[2] for pt in parts)
            den = sum(np.exp(pt[0] - M) * pt[1] for pt in parts)
            O[b, heads] = num / den[:, None]
    return O


def attention_reference(q_values, k_values, v_values, seq_lens, groups: int) -> np.ndarray:
    """Plain softmax attention in double on given (already dequantized or
    bf16) values: q [B][Hq][D], k, v [B][L][Hkv][D].  ResServe measures
    ResAttn's error against an FP32 attention on the same dequantized KV
    (decode-attention evaluation, Fig. 10d); this is that reference in double."""
    q = np.asarray(q_values, np.float64)
    B, Hq, D = q.shape
    O = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        for g in range(Hq):
            h = g // groups
            s = np.asarray(k_values[b, :L, h], np.float64) @ q[b, g] / math.sqrt(D)
            p = np.exp(s - s.max())
            O[b, g] = p @ np.asarray(v_values[b, :L, h], np.float64) / p.sum()
    return O
