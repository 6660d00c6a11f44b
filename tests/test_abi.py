"""librs loads and exports every entry point include/rs.h declares, its size
functions follow the documented layout, and host-side argument checks reject
bad calls before anything reaches a GPU (no compute call needs a device here:
every call below fails validation first)."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT
import layout


@pytest.fixture(scope="module")
def librs():
    from block_scaled_quantized_gb300 import build, rs
    build.build()
    return rs.load_library()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "rs.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(rs_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for want in ["rs_quantize_fp4", "rs_quantize_residue", "rs_linear_w4a4", "rs_linear_compensated"]:
        assert want in names


def test_library_exports_every_declared_symbol(librs):
    from block_scaled_quantized_gb300 import rs
    names = _declared_functions()
    for name in names:
        assert hasattr(librs, name), name
    assert sorted(rs.EXPORTS) == names


def test_status_strings(librs):
    for code, name in [(0, b"RS_OK"), (3, b"RS_ERR_SHAPE"), (7, b"RS_ERR_DEVICE_TIMEOUT")]:
        assert librs.rs_status_string(code) == name
    assert librs.rs_version() >= 1


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("rows,K", [(1, 32), (3, 96), (16, 4096), (130, 288), (4096, 8192), (28672, 4096)])
def test_operand_sizes_follow_documented_layout(librs, fmt, rows, K):
    assert librs.rs_operand_bytes(fmt, rows, K) == layout.operand_bytes(fmt, rows, K)
    assert librs.rs_operand_sf_offset(fmt, rows, K) == layout.sf_offset(rows, K)
    assert librs.rs_act_bytes(fmt, rows, K) == librs.rs_operand_bytes(fmt, rows, K)
    assert librs.rs_weight_bytes(fmt, rows, K) == layout.weight_bytes(fmt, rows, K)


def test_size_functions_reject_bad_shapes(librs):
    assert librs.rs_operand_bytes(0, 4, 48) == 0       # K % 32 != 0
    assert librs.rs_operand_bytes(2, 4, 64) == 0       # bad format
    assert librs.rs_operand_bytes(0, -1, 64) == 0
    assert librs.rs_workspace_bytes(0, 0, 128, 64, 1) == 0
    assert librs.rs_workspace_bytes(0, 8, 4096, 4096, 1) >= librs.rs_act_bytes(0, 16, 4096)


FAKE = 1 << 20          # 16-byte aligned fake device address (never dereferenced)
FAKE_ODD = FAKE + 8


def _lin(librs, fn="rs_linear_compensated", fmt=0, M=8, N=256, K=256, x=FAKE, xq=None, ax=FAKE, w=FAKE,
         aw=FAKE, y=FAKE, out=0, ws=FAKE, wsb=None):
    if wsb is None:
        wsb = librs.rs_workspace_bytes(fmt, M, N, K, 1)
    return getattr(librs, fn)(fmt, M, N, K, x, xq, ax, w, aw, y, out, ws, wsb, None)


def test_linear_argument_checks(librs):
    assert _lin(librs, fmt=5) == 1                            # bad format
    assert _lin(librs, K=48) == 3                             # K % 32
    assert _lin(librs, K=0) == 3
    assert _lin(librs, M=-1) == 1
    assert _lin(librs, M=0) == 0                              # nothing to do
    assert _lin(librs, N=0) == 0
    assert _lin(librs, x=None, xq=None) == 1                  # need exactly one input
    assert _lin(librs, x=FAKE, xq=FAKE) == 1
    assert _lin(librs, w=None) == 1
    assert _lin(librs, y=None) == 1
    assert _lin(librs, aw=None) == 1                          # NVFP4 needs the weight scale
    assert _lin(librs, ax=None) not in (1, 2, 3, 5)           # bf16 input: alpha_x may be NULL
    assert _lin(librs, x=None, xq=FAKE, ax=None) == 1         # a quantized input needs its scale
    assert _lin(librs, out=3) == 1
    assert _lin(librs, x=FAKE_ODD) == 2                       # alignment
    assert _lin(librs, y=FAKE_ODD) == 2
    assert _lin(librs, w=FAKE_ODD) == 2
    assert _lin(librs, wsb=16) == 5                           # workspace too small
    assert _lin(librs, ws=None) == 5
    assert _lin(librs, fn="rs_linear_w4a4", wsb=0) == 5
    assert _lin(librs, x=None, xq=FAKE, ws=None, wsb=0, w=FAKE_ODD) == 2  # xq path needs no workspace


def test_quantizer_argument_checks(librs):
    q = librs.rs_quantize_residue
    assert q(3, 4, 64, FAKE, 64, FAKE, FAKE, None) == 1
    assert q(0, 4, 40, FAKE, 64, FAKE, FAKE, None) == 3
    assert q(0, 4, 64, FAKE, 32, FAKE, FAKE, None) == 1       # ldx < K
    assert q(0, 4, 64, FAKE, 68, FAKE, FAKE, None) == 2       # row pitch not 16-byte aligned
    assert q(0, 4, 64, FAKE_ODD, 64, FAKE, FAKE, None) == 2
    assert q(0, 4, 64, FAKE, 64, None, FAKE, None) == 1       # NVFP4 needs alpha
    assert q(0, 0, 64, None, 64, None, None, None) == 0       # empty input
    f = librs.rs_quantize_fp4
    assert f(0, 4, 64, None, 64, FAKE, FAKE, None) == 1
    wq = librs.rs_quantize_weight
    assert wq(0, 4, 48, FAKE, 64, FAKE, FAKE, None) == 3
    assert wq(0, 4, 64, FAKE, 64, None, FAKE, None) == 1
    assert wq(1, 4, 64, FAKE, 64, None, FAKE_ODD, None) == 2
    assert wq(0, 0, 64, None, 64, None, None, None) == 0
    assert f(1, 4, 64, FAKE, 64, None, FAKE_ODD, None) == 2
    assert librs.rs_compute_tensor_scale(FAKE, -1, FAKE, None) == 1
    assert librs.rs_compute_tensor_scale(FAKE, 16, None, None) == 1


def test_kext_host_selection_matches_oracle(librs, oracle_mod):
    """rs_kext_select (Eq. 7, host code of librs) against the oracle's."""
    import ctypes
    rng = np.random.default_rng(5)
    for k in (1, 2, 4, 8):
        score = rng.random(512).astype(np.float32)
        score[::7] = score[3]  # ties
        mask = np.zeros(64, np.uint8)
        assert librs.rs_kext_select(512, k, score.ctypes.data_as(ctypes.c_void_p),
                                    mask.ctypes.data_as(ctypes.c_void_p)) == 0
        assert np.array_equal(mask, oracle_mod.kext_select(score, k))


def test_kext_argument_checks(librs):
    assert librs.rs_kext_width(512, 2) == 128
    assert librs.rs_kext_width(500, 2) == 0 and librs.rs_kext_width(512, 3) == 0
    assert librs.rs_kext_act_bytes(0, 4, 512, 2) == librs.rs_operand_bytes(0, 4, 640)
    assert librs.rs_kext_weight_bytes(1, 256, 512, 8) == librs.rs_weight_bytes(1, 256, 1024)
    f = librs.rs_linear_kext
    ws = librs.rs_kext_workspace_bytes(0, 8, 256, 512, 2)
    assert f(0, 8, 256, 512, 3, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, ws, None) == 1   # k
    assert f(0, 8, 256, 288, 2, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, ws, None) == 3   # K % 256
    assert f(0, 8, 256, 512, 2, FAKE, None, FAKE, None, FAKE, FAKE, FAKE, 0, FAKE, ws, None) == 1   # mask
    assert f(0, 8, 256, 512, 2, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 16, None) == 5   # workspace
    q = librs.rs_quantize_kext
    assert q(0, 4, 512, 5, FAKE, 512, FAKE, FAKE, FAKE, None) == 3
    assert q(0, 4, 512, 2, FAKE, 512, FAKE, None, FAKE, None) == 1


def test_wait_probe_rejects_out_of_range_limits():
    from block_scaled_quantized_gb300 import rs
    for bad in (0, 2_000_000_000):
        with pytest.raises(rs.RsError) as e:
            rs.rs_debug_wait_probe(bad, stream=0)  # argument checks come before any CUDA call
        assert e.value.status == rs.RS_ERR_INVALID_ARG


def test_resattn_sizes_and_argument_checks(librs):
    from block_scaled_quantized_gb300 import rs
    f = librs.rs_resattn_decode
    P = ctypes.c_void_p
    f.argtypes = [ctypes.c_int] * 6 + [P] * 7 + [ctypes.c_int, P, ctypes.c_size_t, P]
    dummy = P(1 << 20)  # aligned, never dereferenced: every call fails validation first
    ok = (2, 8, 2, 128, 4, 128)
    # workspace: partials (o, m, l) of up to ceil(max_len/128) splits
    B, Hq, Hkv, D, L = 2, 8, 2, 128, 1000
    assert librs.rs_resattn_workspace_bytes(B, Hq, Hkv, D, L) == B * Hkv * 8 * (Hq // Hkv) * (D + 2) * 4
    assert librs.rs_resattn_workspace_bytes(B, Hq, Hkv, 64, L) == 0      # head size
    assert librs.rs_resattn_workspace_bytes(B, 18, 2, D, L) == 0         # 9 query heads per KV head
    assert librs.rs_resattn_split_tokens(1, 8, 128, 4096, 152) % 128 == 0
    assert librs.rs_resattn_split_tokens(1, 1, 128, 4096, 152) == 128   # one tile per split covers the SMs
    assert librs.rs_resattn_split_tokens(1, 8, 96, 4096, 152) == 0      # head size
    # splits fill one wave of resident CTAs (two per SM at D = 128, one at 256)
    # rather than spill a few CTAs into a second one
    assert librs.rs_resattn_split_tokens(8, 8, 128, 8192, 152) == 2048  # 4 splits: 256 CTAs <= 304
    assert librs.rs_resattn_split_tokens(4, 8, 256, 16384, 152) == 1920  # 9 splits: 2 waves x 15 tiles < 1 x 32
    assert librs.rs_resattn_split_tokens(32, 8, 128, 2048, 152) == 2048  # 256 sequence-heads: no split

    def call(shape, ptrs=None, dtype=0, ws=1 << 30):
        pp = ptrs or [dummy] * 7
        return f(*shape, *pp, dtype, dummy, ws, None)

    assert call((2, 8, 2, 96, 4, 128)) == rs.RS_ERR_SHAPE             # D
    assert call((2, 8, 3, 128, 4, 128)) == rs.RS_ERR_SHAPE            # Hq % Hkv
    assert call((2, 8, 2, 128, 4, 129)) == rs.RS_ERR_SHAPE            # max_len > 32 * max_pages
    assert call((0, 8, 2, 128, 4, 128)) == rs.RS_ERR_SHAPE            # B
    assert call(ok, dtype=7) == rs.RS_ERR_INVALID_ARG
    assert call(ok, ptrs=[None] + [dummy] * 6) == rs.RS_ERR_INVALID_ARG
    assert call(ok, ptrs=[P((1 << 20) + 8)] + [dummy] * 6) == rs.RS_ERR_ALIGNMENT
    assert call(ok, ws=16) == rs.RS_ERR_WORKSPACE
