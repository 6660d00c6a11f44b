"""The residue-scale boundary inputs (tests/scale_boundary_cases.py) do what
the GPU pin relies on, checked with the oracle's own residues (CPU):

* every E4M3 midpoint a residue block scale can reach (up to 448 / 6) has
  cases on both sides, within 4 fp32 ulps, at each of three tensor-scale
  families;
* the oracle rounds those scales as Eq. 9's round-to-nearest-even says: a t
  below the midpoint gives the lower E4M3 neighbour, above it the upper one,
  and exactly on it the neighbour with the even mantissa."""
import numpy as np

import scale_boundary_cases as sbc


def _cases_with_offsets():
    import oracle
    oracle.build()
    out = []
    for row, alpha, m, fam in sbc.all_cases():
        q = oracle.quantize_residue(0, row[None, :], alpha)
        out.append((row, alpha, m, fam, sbc.residue_offset(q["resid"][0], alpha, m), int(q["sf_r"][0, 0])))
    return out


def test_cases_cover_every_reachable_midpoint():
    cover = {}
    for row, alpha, m, fam, off, _ in _cases_with_offsets():
        assert abs(off) <= 4, (float(m), fam, off)
        cover.setdefault((float(m), fam), set()).add(off)
    mids = sbc.midpoints(448.0 / 6.0)
    assert float(mids[-1]) == 68.0  # midpoint of 64 and 72; the next one (76) is out of reach
    for m in mids:
        for fam in range(sbc.FAMILIES):
            offs = cover[(float(m), fam)]
            assert min(offs) < 0 < max(offs), (float(m), fam, sorted(offs))


def test_oracle_rounds_residue_scales_to_the_right_neighbour():
    vals = sbc.e4m3_values()
    for row, alpha, m, fam, off, byte in _cases_with_offsets():
        lo = int(np.searchsorted(vals, float(m)) - 1)  # byte of the lower neighbour
        if off < 0:
            assert byte == lo, (float(m), off, byte)
        elif off > 0:
            assert byte == lo + 1, (float(m), off, byte)
        else:
            assert byte == (lo if lo % 2 == 0 else lo + 1), (float(m), byte)
