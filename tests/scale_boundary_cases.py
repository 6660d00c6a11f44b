"""Inputs that put an NVFP4 residue block scale next to an E4M3 rounding
boundary (test input generator; the expected codes and scale bytes come from
the oracle).

The residue block scale of Eq. 9 (App. B.2) is t = fl(fl(Max / 6) / alpha),
rounded to E4M3, where Max is the largest |r| of the block and r = fl(x - x^)
is an fp32 value.  For every midpoint m between consecutive E4M3 values that
a residue can reach (t <= 448 / 6: a residue is at most one base step s~ and
s~ <= 448 alpha), and for three families of tensor scales, a row of 256 bf16
values is built whose first block has t within a few fp32 ulps of m:

* m <= 17 ("small"): the block is [x_max, y, 0, ...]; x_max = bf16(6 s~)
  fixes the base scale byte E, and |y| < 0.25 s~ quantizes to code 0, so
  its residue is y itself.  alpha is tuned ulp by ulp until
  fl(fl(y / 6) / alpha) equals m + k ulps exactly, k = -4..4.
* 17 < m <= 74.67 ("large"): y = 4 s~ + r quantizes to code 4 and leaves
  r = fl(y - 4 s~) with r / (6 alpha) near m; y runs over bf16 values and
  alpha over a few ulps, keeping the pairs that land within 4 ulps.

Each case is (row bf16 bits [256], alpha, m, family); `residue_offset`
measures, from the oracle's residues, where t actually falls."""
import numpy as np

F = np.float32
K_ROW = 256
FAMILIES = 3


def e4m3_values() -> np.ndarray:
    """The 127 finite non-negative E4M3 values, indexed by byte."""
    out = []
    for b in range(127):
        e, mant = b >> 3, b & 7
        out.append(mant * 2.0 ** -9 if e == 0 else (8 + mant) * 2.0 ** (e - 10))
    return np.array(out, np.float64)


def midpoints(limit: float) -> list:
    v = e4m3_values()
    mids = (v[:-1] + v[1:]) / 2  # exact in fp32
    return [F(m) for m in mids if m <= limit]


def step(x, k: int):
    x = F(x)
    d = F(np.inf) if k > 0 else F(-np.inf)
    for _ in range(abs(k)):
        x = np.nextafter(x, d, dtype=F)
    return x


def ulp_distance(a, b) -> int:
    """Signed distance in fp32 ulps between positive finite a and b."""
    return int(np.array(a, F).view(np.int32)) - int(np.array(b, F).view(np.int32))


def t_of(amax, alpha):
    return F(F(F(amax) / F(6)) / F(alpha))


def bf16_bits(v: float) -> int:
    """Round-to-nearest-even fp32 -> bf16 bits."""
    u = int(np.array(v, F).view(np.uint32))
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF


def bf16_value(bits: int) -> F:
    return np.array(bits << 16, np.uint32).view(F)[()]


def _row(x_max_bits: int, y_bits: int) -> np.ndarray:
    row = np.zeros(K_ROW, np.uint16)
    row[0], row[1] = x_max_bits, y_bits
    return row


def small_cases():
    vals = e4m3_values()
    ys = [F(0.3984375), F(5.0), F(-96.5)]  # bf16 values; one family each
    out = []
    for m in midpoints(17.0):
        for fam, y in enumerate(ys):
            q6 = F(y / F(6)) if y > 0 else F(-y / F(6))
            ay = F(abs(y))
            for k in range(-4, 5):
                T = step(m, k)
                a0 = F(q6 / T)
                alpha = None
                for d in (0, 1, -1, 2, -2, 3, -3, 4, -4):
                    a = step(a0, d)
                    if F(q6 / a) == T:
                        alpha = a
                        break
                if alpha is None:
                    continue
                big = [v for v in vals if v > 0 and F(alpha * F(v)) >= F(4.2) * ay]
                if not big:
                    continue
                st = F(alpha * F(big[0]))
                xm = bf16_bits(F(F(6) * st))
                out.append((_row(xm, bf16_bits(y)), alpha, m, fam))
    return out


def large_cases():
    vals = e4m3_values()
    scales = [F(2.0 ** -7), F(1.0), F(37.0)]  # tensor-scale magnitude of each family
    out = []
    for m in midpoints(74.6):
        if m <= 17.0:
            continue
        E = next((v for v in vals if v >= 6.0 * float(m) / 0.95), None)
        if E is None:
            continue
        E = F(E)
        for fam, lam in enumerate(scales):
            y_nom = F(lam * (F(4) * E + F(6) * m))
            b0 = bf16_bits(y_nom)
            seen = set()
            for j in range(-24, 25):
                y = bf16_value(b0 + j)
                a_star = F(y / (F(4) * E + F(6) * m))
                for d in range(-6, 7):
                    a = step(a_star, d)
                    st = F(a * E)
                    v = F(y * F(F(1) / st))
                    if not (F(3.5) < v < F(5.0)):
                        continue
                    r = F(y - F(st * F(4)))
                    off = ulp_distance(t_of(r, a), m)
                    if abs(off) <= 4 and off not in seen:
                        seen.add(off)
                        out.append((_row(bf16_bits(F(F(6) * st)), b0 + j), a, m, fam))
    return out


def all_cases():
    return small_cases() + large_cases()


def residue_offset(resid_row, alpha, m) -> int:
    """ulp distance of the first block's residue scale t from m, from the
    oracle's fp32 residues of that row."""
    amax = F(np.max(np.abs(np.asarray(resid_row, F)[:16])))
    return ulp_distance(t_of(amax, alpha), m)
