"""ctypes binding of librs (include/rs.h): argument marshalling only.

Every function here has the name of the C entry point it calls.  Tensors are
torch tensors on the current CUDA device; their data pointers and the current
torch stream are passed straight through, and a non-OK status raises
``RsError``.  All arithmetic runs in librs's CUDA kernels; there is no CPU
fallback, and importing the binding fails loudly when librs.so is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

NVFP4 = 0
MXFP4 = 1
OUT_BF16 = 0
OUT_F32 = 1

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "librs.so")

STATUS = {0: "RS_OK", 1: "RS_ERR_INVALID_ARG", 2: "RS_ERR_ALIGNMENT", 3: "RS_ERR_SHAPE",
          4: "RS_ERR_UNSUPPORTED", 5: "RS_ERR_WORKSPACE", 6: "RS_ERR_CUDA", 7: "RS_ERR_DEVICE_TIMEOUT"}
globals().update({name: code for code, name in STATUS.items()})  # RS_OK, RS_ERR_INVALID_ARG, ...

# Every symbol include/rs.h declares.
EXPORTS = ["rs_status_string", "rs_version", "rs_operand_bytes", "rs_operand_sf_offset", "rs_act_bytes",
           "rs_weight_bytes", "rs_workspace_bytes", "rs_compute_tensor_scale", "rs_quantize_fp4",
           "rs_quantize_weight", "rs_quantize_residue", "rs_linear_w4a4", "rs_linear_compensated",
           "rs_linear_compensated_noalloc", "rs_get_device_error", "rs_kext_width", "rs_kext_select",
           "rs_channel_mean_abs", "rs_kext_act_bytes", "rs_kext_weight_bytes", "rs_kext_workspace_bytes",
           "rs_quantize_weight_kext", "rs_quantize_kext", "rs_linear_kext", "rs_plan_linear", "rs_debug_wait_probe",
           "rs_get_device_error_async", "rs_debug_linear_dump", "rs_fold_pairs", "rs_resattn_workspace_bytes",
           "rs_resattn_split_tokens", "rs_resattn_decode", "rs_debug_pair_gemm", "rs_set_tactic",
           "rs_reset_tactics", "rs_tactic_count"]


class RsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


def load_library(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"librs.so not found at {path}: build it with "
                           "block_scaled_quantized_gb300.build.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "rs_status_string": ([I], ctypes.c_char_p),
        "rs_version": ([], I),
        "rs_operand_bytes": ([I, I, I], SZ),
        "rs_operand_sf_offset": ([I, I, I], SZ),
        "rs_act_bytes": ([I, I, I], SZ),
        "rs_weight_bytes": ([I, I, I], SZ),
        "rs_workspace_bytes": ([I, I, I, I, I], SZ),
        "rs_compute_tensor_scale": ([P, I64, P, P], I),
        "rs_quantize_fp4": ([I, I, I, P, I64, P, P, P], I),
        "rs_quantize_weight": ([I, I, I, P, I64, P, P, P], I),
        "rs_quantize_residue": ([I, I, I, P, I64, P, P, P], I),
        "rs_linear_w4a4": ([I, I, I, I, P, P, P, P, P, P, I, P, SZ, P], I),
        "rs_linear_compensated": ([I, I, I, I, P, P, P, P, P, P, I, P, SZ, P], I),
        "rs_linear_compensated_noalloc": ([I, I, I, I, P, P, P, P, P, I, P], I),
        "rs_get_device_error": ([P], I),
        "rs_kext_width": ([I, I], I),
        "rs_kext_select": ([I, I, P, P], I),
        "rs_channel_mean_abs": ([P, I, I, I64, P, P], I),
        "rs_kext_act_bytes": ([I, I, I, I], SZ),
        "rs_kext_weight_bytes": ([I, I, I, I], SZ),
        "rs_kext_workspace_bytes": ([I, I, I, I, I], SZ),
        "rs_quantize_weight_kext": ([I, I, I, I, P, I64, P, P, P, P], I),
        "rs_quantize_kext": ([I, I, I, I, P, I64, P, P, P, P], I),
        "rs_linear_kext": ([I, I, I, I, I, P, P, P, P, P, P, P, I, P, SZ, P], I),
        "rs_plan_linear": ([I, I, I, I, I, I, I, P, I], I),
        "rs_debug_wait_probe": ([ctypes.c_uint64, P], I),
        "rs_get_device_error_async": ([P, P], I),
        "rs_fold_pairs": ([I, I, P, P, I, P], I),
        "rs_resattn_workspace_bytes": ([I, I, I, I, I], SZ),
        "rs_resattn_split_tokens": ([I, I, I, I, I], I),
        "rs_debug_pair_gemm": ([I], None),
        "rs_set_tactic": ([I, I, I, I, I, I, I, I, I, I], I),
        "rs_reset_tactics": ([I], I),
        "rs_tactic_count": ([], I),
        "rs_resattn_decode": ([I, I, I, I, I, I, P, P, P, P, P, P, P, I, P, SZ, P], I),
        "rs_debug_linear_dump": ([I, I, I, I, I, P, P, P, P, P, I, P, SZ, P, SZ, P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("librs takes CUDA tensors")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, status: int):
    if status != 0:
        raise RsError(fn, status)


# -------------------------------------------------------------- sizes ----

def rs_operand_bytes(fmt: int, rows: int, K: int) -> int:
    return lib().rs_operand_bytes(fmt, rows, K)


def rs_operand_sf_offset(fmt: int, rows: int, K: int) -> int:
    return lib().rs_operand_sf_offset(fmt, rows, K)


def rs_act_bytes(fmt: int, rows: int, K: int) -> int:
    return lib().rs_act_bytes(fmt, rows, K)


def rs_weight_bytes(fmt: int, N: int, K: int) -> int:
    return lib().rs_weight_bytes(fmt, N, K)


def rs_workspace_bytes(fmt: int, M: int, N: int, K: int, compensated: bool) -> int:
    return lib().rs_workspace_bytes(fmt, M, N, K, int(bool(compensated)))


def rs_debug_wait_probe(limit_ns: int, stream=None):
    """One bounded wait that runs out after limit_ns on the device (see rs.h)."""
    _check("rs_debug_wait_probe", lib().rs_debug_wait_probe(int(limit_ns), _stream(stream)))


PLAN_FIELDS = ("bn", "n_tiles", "b_tiles", "chunks", "splits", "grid_x", "stages", "fused", "slots", "nacc",
               "tmem_cols", "smem_bytes", "tuned", "mcast")


def rs_plan_linear(fmt: int, compensated: bool, M: int, N: int, K: int, num_sms: int, x_in_call: bool = True) -> dict:
    """The launch plan of a linear call of this shape (host only)."""
    out = (ctypes.c_int * len(PLAN_FIELDS))()
    n = lib().rs_plan_linear(fmt, int(bool(compensated)), M, N, K, num_sms, int(bool(x_in_call)), out, len(out))
    if n < 0:
        raise RsError("rs_plan_linear", -n)
    return dict(zip(PLAN_FIELDS, out[:n]))


def rs_version() -> int:
    return lib().rs_version()


# -------------------------------------------------------- entry points ----

def rs_compute_tensor_scale(x: torch.Tensor, alpha_out: torch.Tensor, stream=None):
    _check("rs_compute_tensor_scale",
           lib().rs_compute_tensor_scale(_ptr(x), x.numel(), _ptr(alpha_out), _stream(stream)))


def rs_quantize_fp4(fmt: int, x: torch.Tensor, alpha: torch.Tensor | None, q_out: torch.Tensor,
                    stream=None):
    rows, K = x.shape
    _check("rs_quantize_fp4", lib().rs_quantize_fp4(fmt, rows, K, _ptr(x), x.stride(0), _ptr(alpha),
                                                    _ptr(q_out), _stream(stream)))


def rs_quantize_weight(fmt: int, w: torch.Tensor, alpha: torch.Tensor | None, wq_out: torch.Tensor,
                       stream=None):
    N, K = w.shape
    _check("rs_quantize_weight", lib().rs_quantize_weight(fmt, N, K, _ptr(w), w.stride(0), _ptr(alpha),
                                                          _ptr(wq_out), _stream(stream)))


def rs_quantize_residue(fmt: int, x: torch.Tensor, alpha: torch.Tensor | None, q_paired_out: torch.Tensor,
                        stream=None):
    M, K = x.shape
    _check("rs_quantize_residue", lib().rs_quantize_residue(fmt, M, K, _ptr(x), x.stride(0), _ptr(alpha),
                                                            _ptr(q_paired_out), _stream(stream)))


def _linear(name: str, fmt: int, M: int, N: int, K: int, x, xq, alpha_x, wq, alpha_w, y, workspace,
            stream):
    out = OUT_F32 if y.dtype == torch.float32 else OUT_BF16
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    fn = getattr(lib(), name)
    _check(name, fn(fmt, M, N, K, _ptr(x), _ptr(xq), _ptr(alpha_x), _ptr(wq), _ptr(alpha_w), _ptr(y), out,
                    _ptr(workspace), ws_bytes, _stream(stream)))


def rs_linear_w4a4(fmt: int, M: int, N: int, K: int, x=None, xq=None, alpha_x=None, wq=None, alpha_w=None,
                   y=None, workspace=None, stream=None):
    _linear("rs_linear_w4a4", fmt, M, N, K, x, xq, alpha_x, wq, alpha_w, y, workspace, stream)


def rs_linear_compensated(fmt: int, M: int, N: int, K: int, x=None, xq_paired=None, alpha_x=None, wq=None,
                          alpha_w=None, y=None, workspace=None, stream=None):
    _linear("rs_linear_compensated", fmt, M, N, K, x, xq_paired, alpha_x, wq, alpha_w, y, workspace, stream)


def rs_linear_compensated_noalloc(fmt: int, M: int, N: int, K: int, x=None, alpha_x=None, wq=None,
                                  alpha_w=None, y=None, stream=None):
    """Compensated linear without a workspace, for callers that cannot
    allocate device memory: the quantized activations go to librs's fixed
    device array (see include/rs.h)."""
    out = OUT_F32 if y.dtype == torch.float32 else OUT_BF16
    _check("rs_linear_compensated_noalloc",
           lib().rs_linear_compensated_noalloc(fmt, M, N, K, _ptr(x), _ptr(alpha_x), _ptr(wq), _ptr(alpha_w),
                                               _ptr(y), out, _stream(stream)))


def rs_resattn_workspace_bytes(B: int, Hq: int, Hkv: int, D: int, max_len: int) -> int:
    return lib().rs_resattn_workspace_bytes(B, Hq, Hkv, D, max_len)


def rs_resattn_split_tokens(B: int, Hkv: int, D: int, max_len: int, num_sms: int) -> int:
    return lib().rs_resattn_split_tokens(B, Hkv, D, max_len, num_sms)


def rs_resattn_decode(q: torch.Tensor, alpha_q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_table: torch.Tensor, seq_lens: torch.Tensor, max_len: int, out: torch.Tensor,
                      workspace: torch.Tensor, Hkv: int, stream=None):
    """One ResAttn decode step (see rs.h): q [B][Hq][D] bf16, paged NVFP4
    caches, block_table [B][max_pages] int32, seq_lens [B] int32."""
    B, Hq, D = q.shape
    dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check("rs_resattn_decode",
           lib().rs_resattn_decode(B, Hq, Hkv, D, block_table.shape[1], max_len, _ptr(q), _ptr(alpha_q),
                                   _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(out),
                                   dtype, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)))


def rs_debug_pair_gemm(enable: bool):
    """Route eligible large calls to the paired-CTA GEMM (see rs.h)."""
    lib().rs_debug_pair_gemm(int(bool(enable)))


def rs_set_tactic(fmt: int, compensated: bool, M: int, N: int, K: int, num_sms: int, splits: int, fused: int,
                  bn: int, deep: int = 0):
    """Install a measured launch tactic for one shape (see rs.h)."""
    _check("rs_set_tactic", lib().rs_set_tactic(fmt, int(bool(compensated)), M, N, K, num_sms, splits,
                                                int(fused), bn, int(deep)))


def rs_reset_tactics(builtin: bool = True):
    _check("rs_reset_tactics", lib().rs_reset_tactics(int(bool(builtin))))


def rs_tactic_count() -> int:
    return lib().rs_tactic_count()


def rs_fold_pairs(M: int, N: int, z: torch.Tensor, y: torch.Tensor, stream=None):
    """y[j] = z[2j] + z[2j+1] (separate Fold kernel, for the ablation)."""
    out = OUT_F32 if y.dtype == torch.float32 else OUT_BF16
    _check("rs_fold_pairs", lib().rs_fold_pairs(M, N, _ptr(z), _ptr(y), out, _stream(stream)))


def rs_get_device_error(stream=None) -> int:
    return lib().rs_get_device_error(_stream(stream))


def rs_get_device_error_async(out: torch.Tensor, stream=None):
    """Enqueue the read-and-clear of the device error word into out (one
    int32/uint32 element, device or pinned host memory); no synchronization."""
    ptr = out.data_ptr()
    _check("rs_get_device_error_async", lib().rs_get_device_error_async(ptr, _stream(stream)))


DUMP_FIELDS = ("fused", "bn", "grid_x", "splits", "slots", "stage_bytes", "chunks")


def rs_debug_linear_dump(fmt: int, compensated: bool, M: int, N: int, K: int, x=None, alpha_x=None, wq=None,
                         alpha_w=None, y=None, workspace=None, dump=None, stream=None) -> dict:
    """The linear call with its quantizing prologue's slices copied to dump
    (see rs.h); with dump None, only the layout is returned."""
    layout = (ctypes.c_int * len(DUMP_FIELDS))()
    out = OUT_F32 if (y is not None and y.dtype == torch.float32) else OUT_BF16
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    dump_bytes = dump.numel() * dump.element_size() if dump is not None else 0
    _check("rs_debug_linear_dump",
           lib().rs_debug_linear_dump(fmt, int(bool(compensated)), M, N, K, _ptr(x), _ptr(alpha_x), _ptr(wq),
                                      _ptr(alpha_w), _ptr(y), out, _ptr(workspace), ws_bytes, _ptr(dump),
                                      dump_bytes, layout, _stream(stream)))
    return dict(zip(DUMP_FIELDS, layout[:]))


# -------------------------------------------------- buffer conveniences ----

def empty_operand(fmt: int, rows: int, K: int, device=None) -> torch.Tensor:
    """Uninitialised byte buffer for an rs operand of rows x K."""
    return torch.empty(rs_operand_bytes(fmt, rows, K), dtype=torch.uint8, device=device or "cuda")


def empty_weight(fmt: int, N: int, K: int, device=None) -> torch.Tensor:
    """Uninitialised byte buffer for an rs weight of W [N][K]."""
    return torch.empty(rs_weight_bytes(fmt, N, K), dtype=torch.uint8, device=device or "cuda")


def empty_workspace(fmt: int, M: int, N: int, K: int, compensated: bool, device=None) -> torch.Tensor:
    """Workspace for a linear call with bf16 input (no initialisation needed)."""
    n = max(rs_workspace_bytes(fmt, M, N, K, compensated), 16)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


# ------------------------------------- selective compensation (K-Ext) ----

def rs_kext_width(K: int, k: int) -> int:
    return lib().rs_kext_width(K, k)


def rs_kext_select(score, k: int):
    """Eq. 7 on the host: numpy float32 scores [K] -> uint8 masks [K/8]."""
    import numpy as np
    score = np.ascontiguousarray(score, np.float32)
    mask = np.zeros(score.size // 8, np.uint8)
    _check("rs_kext_select", lib().rs_kext_select(score.size, k, score.ctypes.data_as(ctypes.c_void_p),
                                                  mask.ctypes.data_as(ctypes.c_void_p)))
    return mask


def rs_channel_mean_abs(x: torch.Tensor, score_out: torch.Tensor, stream=None):
    rows, K = x.shape
    _check("rs_channel_mean_abs", lib().rs_channel_mean_abs(_ptr(x), rows, K, x.stride(0), _ptr(score_out),
                                                            _stream(stream)))


def rs_kext_act_bytes(fmt: int, rows: int, K: int, k: int) -> int:
    return lib().rs_kext_act_bytes(fmt, rows, K, k)


def rs_kext_weight_bytes(fmt: int, N: int, K: int, k: int) -> int:
    return lib().rs_kext_weight_bytes(fmt, N, K, k)


def rs_kext_workspace_bytes(fmt: int, M: int, N: int, K: int, k: int) -> int:
    return lib().rs_kext_workspace_bytes(fmt, M, N, K, k)


def rs_quantize_weight_kext(fmt: int, w: torch.Tensor, k: int, alpha: torch.Tensor | None, mask: torch.Tensor,
                            wq_out: torch.Tensor, stream=None):
    N, K = w.shape
    _check("rs_quantize_weight_kext", lib().rs_quantize_weight_kext(fmt, N, K, k, _ptr(w), w.stride(0), _ptr(alpha),
                                                                    _ptr(mask), _ptr(wq_out), _stream(stream)))


def rs_quantize_kext(fmt: int, x: torch.Tensor, k: int, alpha: torch.Tensor | None, mask: torch.Tensor,
                     q_out: torch.Tensor, stream=None):
    rows, K = x.shape
    _check("rs_quantize_kext", lib().rs_quantize_kext(fmt, rows, K, k, _ptr(x), x.stride(0), _ptr(alpha),
                                                      _ptr(mask), _ptr(q_out), _stream(stream)))


def rs_linear_kext(fmt: int, M: int, N: int, K: int, k: int, x=None, xq=None, alpha_x=None, mask=None,
                   wq=None, alpha_w=None, y=None, workspace=None, stream=None):
    out = OUT_F32 if y.dtype == torch.float32 else OUT_BF16
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("rs_linear_kext", lib().rs_linear_kext(fmt, M, N, K, k, _ptr(x), _ptr(xq), _ptr(alpha_x), _ptr(mask),
                                                  _ptr(wq), _ptr(alpha_w), _ptr(y), out, _ptr(workspace), ws_bytes,
                                                  _stream(stream)))
