"""Plain CPU oracle for residue-compensated block-scaled FP4 linear layers.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library never loads it, and it shares no code with the CUDA library.

The arithmetic lives in ``rs_oracle.c`` (plain C, fp32 quantizer steps as
Algorithm 1 of the ResServe paper names them, double-precision GEMM); this
module compiles it with ``-ffp-contract=off`` and wraps it with numpy arrays
on the logical layouts:

* codes: ``uint8 [rows][K/2]``, element ``2j`` in the low nibble of byte ``j``;
* block scales: ``uint8 [rows][K/bs]`` (E4M3 bytes for NVFP4, E8M0 for MXFP4);
* tensor scale (NVFP4 only): one fp32 value.

Formats: ``NVFP4 = 0`` (block 16, E4M3 scale, fp32 tensor scale) and
``MXFP4 = 1`` (block 32, E8M0 scale), ResServe Sec. 2 and Fig. 1.

``oracle.resattn`` holds the decode-attention oracle (ResAttn, Sec. 4.3 and
5.2) in numpy on top of these quantizers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

NVFP4 = 0
MXFP4 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rs_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc, no fast-math, no FMA
    contraction) if it is missing or older than its source."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i, i64, f = ctypes.c_int, ctypes.c_int64, ctypes.c_float
        u8 = ctypes.c_uint8
        lib.or_e2m1_decode.argtypes = [u8]
        lib.or_e2m1_decode.restype = ctypes.c_double
        lib.or_e2m1_encode.argtypes = [f]
        lib.or_e2m1_encode.restype = u8
        lib.or_e4m3_decode.argtypes = [u8]
        lib.or_e4m3_decode.restype = ctypes.c_double
        lib.or_e4m3_encode_satfinite.argtypes = [f]
        lib.or_e4m3_encode_satfinite.restype = u8
        lib.or_e8m0_decode.argtypes = [u8]
        lib.or_e8m0_decode.restype = ctypes.c_double
        lib.or_tensor_scale.argtypes = [P, i64]
        lib.or_tensor_scale.restype = f
        lib.or_block_size.argtypes = [i]
        lib.or_block_size.restype = i
        lib.or_quantize.argtypes = [i, i, i, P, f, P, P, P]
        lib.or_quantize.restype = i
        lib.or_quantize_residue.argtypes = [i, i, i, P, f, P, P, P, P, P, P]
        lib.or_quantize_residue.restype = i
        lib.or_dequantize.argtypes = [i, i, i, P, P, P]
        lib.or_dequantize.restype = None
        lib.or_block_gemm.argtypes = [i, i, i, i, P, P, P, P, P]
        lib.or_block_gemm.restype = i
        lib.or_linear.argtypes = [i, i, i, i, i, P, f, P, P, f, P]
        lib.or_linear.restype = i
        lib.or_e2m1_encode_array.argtypes = [P, i64, P]
        lib.or_e2m1_encode_array.restype = None
        lib.or_e4m3_encode_array.argtypes = [P, i64, P]
        lib.or_e4m3_encode_array.restype = None
        lib.or_kext_width.argtypes = [i, i]
        lib.or_kext_width.restype = i
        lib.or_kext_select.argtypes = [i, i, P, P]
        lib.or_kext_select.restype = i
        lib.or_quantize_kext.argtypes = [i, i, i, i, P, f, P, P, P]
        lib.or_quantize_kext.restype = i
        lib.or_quantize_weight_kext.argtypes = [i, i, i, i, P, f, P, P, P]
        lib.or_quantize_weight_kext.restype = i
        lib.or_linear_kext.argtypes = [i, i, i, i, i, P, f, P, P, P, f, P]
        lib.or_quantize_nvfp4_div.argtypes = [i, i, P, f, P, P]
        lib.or_quantize_nvfp4_div.restype = i
        lib.or_set_threads.argtypes = [i]
        lib.or_set_threads.restype = None
        lib.or_quantize_residue_nvfp4_recon_div.argtypes = [i, i, P, f, P, P, P, P]
        lib.or_quantize_residue_nvfp4_recon_div.restype = i
        lib.or_linear_kext.restype = i
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_u16(x) -> np.ndarray:
    """bf16 input as its raw uint16 bit pattern (numpy has no bf16)."""
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return x


def block_size(fmt: int) -> int:
    return 16 if fmt == NVFP4 else 32


# ---------------------------------------------------------------- codecs ---

def e2m1_decode(code: int) -> float:
    return _load().or_e2m1_decode(code & 0xFF)


def e2m1_encode(v: float) -> int:
    return int(_load().or_e2m1_encode(v))


def e2m1_encode_array(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().or_e2m1_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode(b: int) -> float:
    return _load().or_e4m3_decode(b & 0xFF)


def e4m3_encode(t: float) -> int:
    return int(_load().or_e4m3_encode_satfinite(t))


def e4m3_encode_array(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().or_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e8m0_decode(b: int) -> float:
    return _load().or_e8m0_decode(b & 0xFF)


# ------------------------------------------------------------- quantizer ---

def set_threads(n: int) -> None:
    """Threads of the oracle's dequantization and GEMM loops (default 1);
    results do not depend on it (each output is the same ordered sum)."""
    _load().or_set_threads(int(n))


def tensor_scale(x_u16) -> np.float32:
    """alpha = fl(amax / 2688) over the whole tensor (App. B.2 Eq. 8)."""
    x = _as_u16(x_u16)
    return np.float32(_load().or_tensor_scale(_ptr(x), x.size))


def quantize(fmt: int, x_u16, alpha: float = 0.0):
    """QDQ of bf16 rows [rows][K].  Returns (codes, sf, xhat_f32)."""
    x = _as_u16(x_u16)
    rows, K = x.shape
    bs = block_size(fmt)
    codes = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // bs), np.uint8)
    xhat = np.zeros((rows, K), np.float32)
    rc = _load().or_quantize(fmt, rows, K, _ptr(x), float(alpha),
                             _ptr(codes), _ptr(sf), _ptr(xhat))
    if rc:
        raise ValueError("oracle quantize: bad shape")
    return codes, sf, xhat


def quantize_nvfp4_div(x_u16, alpha: float):
    """NVFP4 codes and scale bytes with Eq. 10's division v = fl(x / s~)
    instead of Alg. 1's multiplier (the alternative reading; parity uses the
    multiplier)."""
    x = _as_u16(x_u16)
    rows, K = x.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 16), np.uint8)
    if _load().or_quantize_nvfp4_div(rows, K, _ptr(x), float(alpha), _ptr(codes), _ptr(sf)):
        raise ValueError("oracle quantize_nvfp4_div: bad shape")
    return codes, sf


def quantize_residue_nvfp4_recon_div(x_u16, alpha: float):
    """NVFP4 base and residue operands with Alg. 1's reconstruction
    x^ = fl(dec(q) / fl(1/s~)) in place of Eq. 10's fl(s~ dec(q)) (the
    alternative reading; parity uses Eq. 10).  Returns dict with codes_x,
    sf_x, codes_r, sf_r."""
    x = _as_u16(x_u16)
    rows, K = x.shape
    out = dict(codes_x=np.zeros((rows, K // 2), np.uint8), sf_x=np.zeros((rows, K // 16), np.uint8),
               codes_r=np.zeros((rows, K // 2), np.uint8), sf_r=np.zeros((rows, K // 16), np.uint8))
    if _load().or_quantize_residue_nvfp4_recon_div(rows, K, _ptr(x), float(alpha), _ptr(out["codes_x"]),
                                                   _ptr(out["sf_x"]), _ptr(out["codes_r"]), _ptr(out["sf_r"])):
        raise ValueError("oracle quantize_residue_nvfp4_recon_div: bad shape")
    return out


def quantize_residue(fmt: int, x_u16, alpha: float = 0.0):
    """Base and residue operands of bf16 rows [rows][K] (Alg. 1).
    Returns dict with codes_x, sf_x, codes_r, sf_r, resid (fp32 R), rhat."""
    x = _as_u16(x_u16)
    rows, K = x.shape
    bs = block_size(fmt)
    out = dict(codes_x=np.zeros((rows, K // 2), np.uint8),
               sf_x=np.zeros((rows, K // bs), np.uint8),
               codes_r=np.zeros((rows, K // 2), np.uint8),
               sf_r=np.zeros((rows, K // bs), np.uint8),
               resid=np.zeros((rows, K), np.float32),
               rhat=np.zeros((rows, K), np.float32))
    rc = _load().or_quantize_residue(
        fmt, rows, K, _ptr(x), float(alpha), _ptr(out["codes_x"]), _ptr(out["sf_x"]),
        _ptr(out["codes_r"]), _ptr(out["sf_r"]), _ptr(out["resid"]), _ptr(out["rhat"]))
    if rc:
        raise ValueError("oracle quantize_residue: bad shape")
    return out


def dequantize(fmt: int, codes, sf) -> np.ndarray:
    """Values represented by codes and block scales (tensor scale excluded)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8)
    rows, half = codes.shape
    out = np.zeros((rows, 2 * half), np.float64)
    _load().or_dequantize(fmt, rows, 2 * half, _ptr(codes), _ptr(sf), _ptr(out))
    return out


def block_gemm(fmt: int, codes_a, sf_a, codes_b, sf_b) -> np.ndarray:
    """Z[m][n] = sum_k deq(A)[m][k] * deq(B)[n][k] in double."""
    codes_a = np.ascontiguousarray(codes_a, np.uint8)
    sf_a = np.ascontiguousarray(sf_a, np.uint8)
    codes_b = np.ascontiguousarray(codes_b, np.uint8)
    sf_b = np.ascontiguousarray(sf_b, np.uint8)
    M, half = codes_a.shape
    N = codes_b.shape[0]
    Z = np.zeros((M, N), np.float64)
    rc = _load().or_block_gemm(fmt, M, N, 2 * half, _ptr(codes_a), _ptr(sf_a),
                               _ptr(codes_b), _ptr(sf_b), _ptr(Z))
    if rc:
        raise ValueError("oracle block_gemm: bad shape")
    return Z


def linear(fmt: int, compensated: bool, x_u16, alpha_x: float,
           codes_w, sf_w, alpha_w: float) -> np.ndarray:
    """Y [M][N] (double) of one W4A4 or fully compensated linear layer."""
    x = _as_u16(x_u16)
    codes_w = np.ascontiguousarray(codes_w, np.uint8)
    sf_w = np.ascontiguousarray(sf_w, np.uint8)
    M, K = x.shape
    N = codes_w.shape[0]
    Y = np.zeros((M, N), np.float64)
    rc = _load().or_linear(fmt, int(bool(compensated)), M, N, K, _ptr(x), float(alpha_x),
                           _ptr(codes_w), _ptr(sf_w), float(alpha_w), _ptr(Y))
    if rc:
        raise ValueError("oracle linear: bad shape")
    return Y


# ---- selective prefill compensation, K-Ext (Sec. 5.3 Eq. 6, App. A Eq. 7) ----

def kext_width(K: int, k: int) -> int:
    """Extension length K * rho with rho = k / 8 (k channels per group of 8)."""
    return K // 8 * k


def kext_select(score, k: int) -> np.ndarray:
    """Eq. 7: per group of 8 channels the k channels with the largest
    calibration score (mean |x|); equal scores keep the lower channel.
    Returns one uint8 mask per group (bit t = channel 8g + t)."""
    score = np.ascontiguousarray(score, np.float32)
    K = score.size
    mask = np.zeros(K // 8, np.uint8)
    if _load().or_kext_select(K, int(k), _ptr(score), _ptr(mask)):
        raise ValueError("oracle kext_select: bad shape")
    return mask


def quantize_kext(fmt: int, x_u16, k: int, mask, alpha: float = 0.0):
    """Extended activation operand [X^ | R^_S] of bf16 rows [rows][K]:
    codes [rows][K_eff/2], scales [rows][K_eff/bs]."""
    x = _as_u16(x_u16)
    mask = np.ascontiguousarray(mask, np.uint8)
    rows, K = x.shape
    Ke = K + kext_width(K, k)
    bs = block_size(fmt)
    codes = np.zeros((rows, Ke // 2), np.uint8)
    sf = np.zeros((rows, Ke // bs), np.uint8)
    if _load().or_quantize_kext(fmt, rows, K, int(k), _ptr(x), float(alpha), _ptr(mask), _ptr(codes), _ptr(sf)):
        raise ValueError("oracle quantize_kext: bad shape or mask")
    return codes, sf


def quantize_weight_kext(fmt: int, w_u16, k: int, mask, alpha_w: float = 0.0):
    """Extended weight [W | W[:, S]] of bf16 [N][K] quantized as one tensor:
    codes [N][K_eff/2], scales [N][K_eff/bs]."""
    w = _as_u16(w_u16)
    mask = np.ascontiguousarray(mask, np.uint8)
    N, K = w.shape
    Ke = K + kext_width(K, k)
    bs = block_size(fmt)
    codes = np.zeros((N, Ke // 2), np.uint8)
    sf = np.zeros((N, Ke // bs), np.uint8)
    if _load().or_quantize_weight_kext(fmt, N, K, int(k), _ptr(w), float(alpha_w), _ptr(mask), _ptr(codes),
                                       _ptr(sf)):
        raise ValueError("oracle quantize_weight_kext: bad shape or mask")
    return codes, sf


def linear_kext(fmt: int, x_u16, k: int, mask, alpha_x: float, codes_w, sf_w, alpha_w: float) -> np.ndarray:
    """Y [M][N] (double) of the K-Ext linear layer, one GEMM over K_eff."""
    x = _as_u16(x_u16)
    mask = np.ascontiguousarray(mask, np.uint8)
    codes_w = np.ascontiguousarray(codes_w, np.uint8)
    sf_w = np.ascontiguousarray(sf_w, np.uint8)
    M, K = x.shape
    N = codes_w.shape[0]
    Y = np.zeros((M, N), np.float64)
    if _load().or_linear_kext(fmt, M, N, K, int(k), _ptr(x), float(alpha_x), _ptr(mask), _ptr(codes_w),
                              _ptr(sf_w), float(alpha_w), _ptr(Y)):
        raise ValueError("oracle linear_kext: bad shape or mask")
    return Y


def nmse(y, ref) -> float:
    """Pooled NMSE: summed squared error over summed squared reference
    (ResServe App. C.2)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.sum((y - ref) ** 2) / np.sum(ref ** 2))
