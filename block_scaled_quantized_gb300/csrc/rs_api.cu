// Host entry points of librs (include/rs.h): argument validation, the device
// error word, and the launch sequence of each call.
#include <mutex>

#include "rs.h"
#include "rs_device.cuh"
#include "rs_internal.h"

namespace rs {

// Written by kernels whose bounded waits ran out (or on a non-finite tensor
// amax); read and cleared by rs_get_device_error().
__device__ uint32_t g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    uint32_t* err = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Properties of the current device, queried once per device.
const DeviceInfo* current_device(cudaError_t* why) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *why = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
            *why = e;
            return nullptr;
        }
        d.supported = (major == 10 && minor == 3);  // kernels are built for sm_103a only
        if (d.supported) {
            void* p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_device_error)) != cudaSuccess) {
                *why = e;
                return nullptr;
            }
            d.err = static_cast<uint32_t*>(p);
        }
        d.ready = true;
    }
    *why = cudaSuccess;
    return &d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool fmt_ok(int fmt) { return fmt == RS_NVFP4 || fmt == RS_MXFP4; }
bool k_ok(int K) { return K > 0 && K % 32 == 0; }

rs_status from_cuda(cudaError_t e) { return e == cudaSuccess ? RS_OK : RS_ERR_CUDA; }

// Common checks of the quantizer entry points.
rs_status check_quant(int fmt, int rows, int K, const void* x, int64_t ldx, const float* alpha, const void* q) {
    if (!fmt_ok(fmt) || rows < 0) return RS_ERR_INVALID_ARG;
    if (!k_ok(K)) return RS_ERR_SHAPE;
    if (rows == 0) return RS_OK;
    if (!x || !q) return RS_ERR_INVALID_ARG;
    if (ldx < K) return RS_ERR_INVALID_ARG;
    if (fmt == RS_NVFP4 && !alpha) return RS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || (ldx % 8) != 0) return RS_ERR_ALIGNMENT;
    if (fmt == RS_NVFP4 && !aligned4(alpha)) return RS_ERR_ALIGNMENT;
    if ((int64_t)rows * 2 > (int64_t)0x7FFFFFFF) return RS_ERR_SHAPE;
    return RS_OK;
}

bool kext_ok(int K, int k) { return (k == 1 || k == 2 || k == 4 || k == 8) && K > 0 && K % 256 == 0; }
int kext_cols(int K, int k) { return K + K / 8 * k; }

// kext_k > 0: selective compensation (K-Ext): the operand and the weight are
// the extended ones with K_eff columns and no Fold (compensated == false).
rs_status linear_impl(int fmt, bool compensated, int M, int N, int K, const void* x, const void* xq,
                      const float* alpha_x, const void* wq, const float* alpha_w, void* y, int out_dtype,
                      void* ws, size_t ws_bytes, cudaStream_t stream, int kext_k = 0,
                      const uint8_t* kext_mask = nullptr, void* qdump = nullptr) {
    if (!fmt_ok(fmt) || M < 0 || N < 0) return RS_ERR_INVALID_ARG;
    if (out_dtype != RS_OUT_BF16 && out_dtype != RS_OUT_F32) return RS_ERR_INVALID_ARG;
    if (!k_ok(K)) return RS_ERR_SHAPE;
    if (kext_k > 0 && !kext_ok(K, kext_k)) return RS_ERR_SHAPE;
    const int Kg = kext_k > 0 ? kext_cols(K, kext_k) : K;  // GEMM reduction length
    if ((int64_t)M * 2 > (int64_t)0x7FFFFFFF) return RS_ERR_SHAPE;
    if (M == 0 || N == 0) return RS_OK;
    if ((x == nullptr) == (xq == nullptr)) return RS_ERR_INVALID_ARG;
    if (!wq || !y) return RS_ERR_INVALID_ARG;
    // NVFP4: alpha_w is required; alpha_x may be NULL with a bf16 input (the
    // call then computes the activation tensor scale itself)
    const bool dyn_alpha = fmt == RS_NVFP4 && alpha_x == nullptr;
    if (fmt == RS_NVFP4 && !alpha_w) return RS_ERR_INVALID_ARG;
    if (dyn_alpha && x == nullptr) return RS_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (xq && !aligned16(xq)) || !aligned16(wq) || !aligned16(y) ||
        (ws && !aligned16(ws)))
        return RS_ERR_ALIGNMENT;
    if (fmt == RS_NVFP4 && ((alpha_x && !aligned4(alpha_x)) || !aligned4(alpha_w))) return RS_ERR_ALIGNMENT;
    const bool quantize_input = x != nullptr;
    if (kext_k > 0 && quantize_input && !kext_mask) return RS_ERR_INVALID_ARG;
    if (quantize_input && (!ws || ws_bytes < workspace_bytes(fmt, compensated, M, Kg))) return RS_ERR_WORKSPACE;

    cudaError_t why;
    const DeviceInfo* dev = current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;

    const GemmPlan plan =
        make_gemm_plan(fmt, compensated, M, N, Kg, dev->num_sms, /*allow_fused=*/quantize_input && kext_k == 0);
    GemmCall c{};
    c.wq = wq;
    c.alpha_x = alpha_x;
    c.alpha_w = alpha_w;
    c.y = y;
    c.out_f32 = out_dtype == RS_OUT_F32 ? 1 : 0;
    c.err = dev->err;
    if (quantize_input && plan.fused) {
        c.x = x;  // the GEMM quantizes its own K slices (and finds the tensor scale): one launch
        c.dyn_alpha = dyn_alpha ? 1 : 0;
        c.qdump = qdump;
    } else if (quantize_input) {
        void* act = ws;
        const float* ax = alpha_x;
        if (dyn_alpha) {
            // the tensor scale goes to the workspace slot after the operand
            float* a = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + alpha_slot_offset(fmt, compensated, M, Kg));
            if (launch_tensor_scale(x, (int64_t)M * K, a, dev->err, stream, dev->num_sms) != cudaSuccess)
                return RS_ERR_CUDA;
            ax = a;
            c.alpha_x = a;
        }
        cudaError_t e = kext_k > 0 ? launch_quantize_kext(fmt, kext_k, M, K, x, K, ax, kext_mask, act, stream,
                                                          dev->num_sms, /*pdl=*/true)
                                   : launch_quantize(fmt, compensated, M, K, x, K, ax, act, stream, dev->num_sms,
                                                     /*pdl=*/true);
        if (e != cudaSuccess) return RS_ERR_CUDA;
        c.xq = act;
    } else {
        c.xq = xq;
    }
    return from_cuda(launch_gemm(plan, c, stream));
}

}  // namespace

rs_status current_device_status(int* num_sms, uint32_t** err) {
    cudaError_t why;
    const DeviceInfo* d = current_device(&why);
    if (!d) return RS_ERR_CUDA;
    if (!d->supported) return RS_ERR_UNSUPPORTED;
    *num_sms = d->num_sms;
    *err = d->err;
    return RS_OK;
}

uint32_t* device_error_word() {
    cudaError_t why;
    const DeviceInfo* d = current_device(&why);
    return d ? d->err : nullptr;
}

}  // namespace rs

using namespace rs;

extern "C" {

const char* rs_status_string(rs_status s) {
    switch (s) {
        case RS_OK: return "RS_OK";
        case RS_ERR_INVALID_ARG: return "RS_ERR_INVALID_ARG";
        case RS_ERR_ALIGNMENT: return "RS_ERR_ALIGNMENT";
        case RS_ERR_SHAPE: return "RS_ERR_SHAPE";
        case RS_ERR_UNSUPPORTED: return "RS_ERR_UNSUPPORTED";
        case RS_ERR_WORKSPACE: return "RS_ERR_WORKSPACE";
        case RS_ERR_CUDA: return "RS_ERR_CUDA";
        case RS_ERR_DEVICE_TIMEOUT: return "RS_ERR_DEVICE_TIMEOUT";
    }
    return "RS_ERR_UNKNOWN";
}

int rs_version(void) { return 1; }

size_t rs_operand_bytes(rs_format fmt, int rows, int K) {
    if (!fmt_ok(fmt) || rows < 0 || !k_ok(K)) return 0;
    return operand_bytes(fmt, rows, K);
}

size_t rs_operand_sf_offset(rs_format fmt, int rows, int K) {
    if (!fmt_ok(fmt) || rows < 0 || !k_ok(K)) return 0;
    return operand_sf_offset(fmt, rows, K);
}

size_t rs_act_bytes(rs_format fmt, int rows, int K) { return rs_operand_bytes(fmt, rows, K); }

size_t rs_weight_bytes(rs_format fmt, int N, int K) {
    if (!fmt_ok(fmt) || N < 0 || !k_ok(K)) return 0;
    return weight_bytes(fmt, N, K);
}

size_t rs_workspace_bytes(rs_format fmt, int M, int N, int K, int compensated) {
    if (!fmt_ok(fmt) || M < 0 || N < 0 || !k_ok(K)) return 0;
    if (M == 0 || N == 0) return 0;
    return workspace_bytes(fmt, compensated != 0, M, K);
}

int rs_plan_linear(rs_format fmt, int compensated, int M, int N, int K, int num_sms, int x_in_call, int* out,
                   int n_out) {
    if (!fmt_ok(fmt) || M < 1 || N < 1 || num_sms < 1 || n_out < 0 || (n_out > 0 && !out))
        return -(int)RS_ERR_INVALID_ARG;
    if (!k_ok(K) || (int64_t)M * 2 > (int64_t)0x7FFFFFFF) return -(int)RS_ERR_SHAPE;
    const GemmPlan p = make_gemm_plan(fmt, compensated != 0, M, N, K, num_sms, x_in_call != 0);
    const int fused = p.fused ? (p.qpair ? 2 : 1) : 0;
    const int v[] = {p.bn,  p.n_tiles, p.b_tiles, p.chunks,    p.splits,          p.grid_x, p.stages,
                     fused, p.slots,   p.nacc,    p.tmem_cols, (int)p.smem_bytes, p.tuned,
                     multicast_eligible(p) ? 1 : 0};
    const int n = n_out < (int)(sizeof(v) / sizeof(v[0])) ? n_out : (int)(sizeof(v) / sizeof(v[0]));
    for (int i = 0; i < n; ++i) out[i] = v[i];
    return n;
}

rs_status rs_set_tactic(rs_format fmt, int compensated, int M, int N, int K, int num_sms, int splits, int fused,
                        int bn, int deep) {
    if (!fmt_ok(fmt) || M < 1 || N < 1 || num_sms < 1) return RS_ERR_INVALID_ARG;
    if (!k_ok(K)) return RS_ERR_SHAPE;
    return set_tactic(fmt, compensated != 0, M, N, K, num_sms, Tactic{splits, fused, bn, deep}) ? RS_OK
                                                                                               : RS_ERR_INVALID_ARG;
}

rs_status rs_reset_tactics(int builtin) {
    reset_tactics(builtin != 0);
    return RS_OK;
}

int rs_tactic_count(void) { return tactic_count(); }

rs_status rs_compute_tensor_scale(const void* x_bf16, int64_t n, float* alpha_out, rs_stream_t stream) {
    if (n < 0 || !alpha_out || (n > 0 && !x_bf16)) return RS_ERR_INVALID_ARG;
    if ((x_bf16 && (reinterpret_cast<uintptr_t>(x_bf16) & 1u)) || !aligned4(alpha_out)) return RS_ERR_ALIGNMENT;
    cudaError_t why;
    const DeviceInfo* dev = current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    return from_cuda(launch_tensor_scale(x_bf16, n, alpha_out, dev->err, (cudaStream_t)stream, dev->num_sms));
}

rs_status rs_quantize_fp4(rs_format fmt, int rows, int K, const void* x_bf16, int64_t ldx, const float* alpha,
                          void* q_out, rs_stream_t stream) {
    rs_status s = check_quant(fmt, rows, K, x_bf16, ldx, alpha, q_out);
    if (s != RS_OK || rows == 0) return s;
    cudaError_t why;
    const DeviceInfo* dev = current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    return from_cuda(launch_quantize(fmt, false, rows, K, x_bf16, ldx, alpha, q_out, (cudaStream_t)stream,
                                     dev->num_sms, /*pdl=*/false));
}

rs_status rs_quantize_weight(rs_format fmt, int N, int K, const void* w_bf16, int64_t ldw, const float* alpha,
                             void* wq_out, rs_stream_t stream) {
    rs_status s = check_quant(fmt, N, K, w_bf16, ldw, alpha, wq_out);
    if (s != RS_OK || N == 0) return s;
    cudaError_t why;
    const DeviceInfo* dev = current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    return from_cuda(launch_quantize_weight(fmt, N, K, w_bf16, ldw, alpha, wq_out, (cudaStream_t)stream,
                                            dev->num_sms));
}

rs_status rs_quantize_residue(rs_format fmt, int M, int K, const void* x_bf16, int64_t ldx, const float* alpha,
                              void* q_paired_out, rs_stream_t stream) {
    rs_status s = check_quant(fmt, M, K, x_bf16, ldx, alpha, q_paired_out);
    if (s != RS_OK || M == 0) return s;
    cudaError_t why;
    const DeviceInfo* dev = current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    return from_cuda(launch_quantize(fmt, true, M, K, x_bf16, ldx, alpha, q_paired_out, (cudaStream_t)stream,
                                     dev->num_sms, /*pdl=*/false));
}

rs_status rs_linear_w4a4(rs_format fmt, int M, int N, int K, const void* x_bf16, const void* xq,
                         const float* alpha_x, const void* wq, const float* alpha_w, void* y,
                         rs_out_dtype out_dtype, void* workspace, size_t ws_bytes, rs_stream_t stream) {
    return linear_impl(fmt, false, M, N, K, x_bf16, xq, alpha_x, wq, alpha_w, y, out_dtype, workspace, ws_bytes,
                       (cudaStream_t)stream);
}

rs_status rs_linear_compensated(rs_format fmt, int M, int N, int K, const void* x_bf16, const void* xq_paired,
                                const float* alpha_x, const void* wq, const float* alpha_w, void* y,
                                rs_out_dtype out_dtype, void* workspace, size_t ws_bytes, rs_stream_t stream) {
    return linear_impl(fmt, true, M, N, K, x_bf16, xq_paired, alpha_x, wq, alpha_w, y, out_dtype, workspace,
                       ws_bytes, (cudaStream_t)stream);
}

int rs_kext_width(int K, int k) { return kext_ok(K, k) ? K / 8 * k : 0; }

rs_status rs_kext_select(int K, int k, const float* score, uint8_t* mask) {
    // Eq. 7: per group of 8 channels the k largest scores; equal scores keep
    // the lower channel.
    if (!score || !mask || K <= 0 || K % 8 != 0 || k < 0 || k > 8) return RS_ERR_INVALID_ARG;
    for (int g = 0; g < K / 8; ++g) {
        unsigned chosen = 0;
        for (int j = 0; j < k; ++j) {
            int top = -1;
            for (int t = 0; t < 8; ++t)
                if (!(chosen >> t & 1u) && (top < 0 || score[8 * g + t] > score[8 * g + top])) top = t;
            chosen |= 1u << top;
        }
        mask[g] = (uint8_t)chosen;
    }
    return RS_OK;
}

rs_status rs_channel_mean_abs(const void* x_bf16, int rows, int K, int64_t ldx, float* score, rs_stream_t stream) {
    if (rows < 0 || K <= 0 || !x_bf16 || !score || ldx < K) return RS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x_bf16) & 1u) || !aligned4(score)) return RS_ERR_ALIGNMENT;
    cudaError_t why;
    const DeviceInfo* dev = current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    return from_cuda(launch_channel_mean_abs(x_bf16, rows, K, ldx, score, (cudaStream_t)stream));
}

size_t rs_kext_act_bytes(rs_format fmt, int rows, int K, int k) {
    if (!fmt_ok(fmt) || rows < 0 || !kext_ok(K, k)) return 0;
    return operand_bytes(fmt, rows, kext_cols(K, k));
}

size_t rs_kext_weight_bytes(rs_format fmt, int N, int K, int k) {
    if (!fmt_ok(fmt) || N < 0 || !kext_ok(K, k)) return 0;
    return weight_bytes(fmt, N, kext_cols(K, k));
}

size_t rs_kext_workspace_bytes(rs_format fmt, int M, int N, int K, int k) {
    if (!fmt_ok(fmt) || M <= 0 || N <= 0 || !kext_ok(K, k)) return 0;
    return workspace_bytes(fmt, false, M, kext_cols(K, k));
}

rs_status rs_quantize_weight_kext(rs_format fmt, int N, int K, int k, const void* w_bf16, int64_t ldw,
                                  const float* alpha_w, const uint8_t* mask, void* wq_out, rs_stream_t stream) {
    rs_status s = check_quant(fmt, N, K, w_bf16, ldw, alpha_w, wq_out);
    if (s != RS_OK || N == 0) return s;
    if (!kext_ok(K, k)) return RS_ERR_SHAPE;
    if (!mask) return RS_ERR_INVALID_ARG;
    cudaError_t why;
    const DeviceInfo* dev = current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    return from_cuda(launch_quantize_weight(fmt, N, K, w_bf16, ldw, alpha_w, wq_out, (cudaStream_t)stream,
                                            dev->num_sms, k, mask));
}

rs_status rs_quantize_kext(rs_format fmt, int rows, int K, int k, const void* x_bf16, int64_t ldx, const float* alpha,
                           const uint8_t* mask, void* q_out, rs_stream_t stream) {
    rs_status s = check_quant(fmt, rows, K, x_bf16, ldx, alpha, q_out);
    if (s != RS_OK || rows == 0) return s;
    if (!kext_ok(K, k)) return RS_ERR_SHAPE;
    if (!mask) return RS_ERR_INVALID_ARG;
    cudaError_t why;
    const DeviceInfo* dev = current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    return from_cuda(launch_quantize_kext(fmt, k, rows, K, x_bf16, ldx, alpha, mask, q_out, (cudaStream_t)stream,
                                          dev->num_sms, /*pdl=*/false));
}

rs_status rs_linear_kext(rs_format fmt, int M, int N, int K, int k, const void* x_bf16, const void* xq,
                         const float* alpha_x, const uint8_t* mask, const void* wq_ext, const float* alpha_w,
                         void* y, rs_out_dtype out_dtype, void* workspace, size_t ws_bytes, rs_stream_t stream) {
    if (k != 1 && k != 2 && k != 4 && k != 8) return RS_ERR_INVALID_ARG;
    return linear_impl(fmt, false, M, N, K, x_bf16, xq, alpha_x, wq_ext, alpha_w, y, out_dtype, workspace,
                       ws_bytes, (cudaStream_t)stream, k, mask);
}

namespace rs {
// Failure detection without a fault: one CTA waits on an mbarrier that
// nothing arrives on, with the bounded wait every kernel uses; the wait runs
// out after limit_ns, sets the device error word (RS_ERR_DEVICE_TIMEOUT) and
// returns, and the kernel exits normally.
__global__ void wait_probe_kernel(uint64_t limit_ns, uint32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0u;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait_bounded(smem_u32(&bar), 0u, &abort_flag, err, limit_ns);
}
}  // namespace rs

rs_status rs_debug_wait_probe(uint64_t limit_ns, rs_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return RS_ERR_INVALID_ARG;
    cudaError_t why;
    const rs::DeviceInfo* dev = rs::current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    rs::wait_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_ns, dev->err);
    return cudaGetLastError() == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

namespace rs {
// One thread: hand the error word to the caller's buffer and clear it.
__global__ void read_error_kernel(uint32_t* err, uint32_t* out) { *out = atomicExch(err, 0u); }
}  // namespace rs

namespace {
bool attn_shape_ok(int B, int Hq, int Hkv, int D, int max_pages, int max_len) {
    return B >= 1 && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 && Hq / Hkv <= 8 && (D == 128 || D == 256) &&
           max_pages >= 1 && max_len >= 0 && (int64_t)max_len <= (int64_t)max_pages * 32 &&
           (int64_t)B * Hq * 2 <= 0x7FFFFFFF;
}
}  // namespace

size_t rs_resattn_workspace_bytes(int B, int Hq, int Hkv, int D, int max_len) {
    if (!attn_shape_ok(B, Hq, Hkv, D, (max_len + 31) / 32 + 1, max_len)) return 0;
    const int max_splits = max_len > 0 ? (max_len + 127) / 128 : 1;
    return (size_t)B * Hkv * max_splits * (Hq / Hkv) * (D + 2) * sizeof(float);
}

int rs_resattn_split_tokens(int B, int Hkv, int D, int max_len, int num_sms) {
    if (B < 1 || Hkv < 1 || (D != 128 && D != 256) || max_len < 0 || num_sms < 1) return 0;
    return rs::resattn_split_tokens(B, Hkv, D, max_len, num_sms);
}

rs_status rs_resattn_decode(int B, int Hq, int Hkv, int D, int max_pages, int max_len, const void* q_bf16,
                            const float* alpha_q, const void* k_cache, const void* v_cache, const int* block_table,
                            const int* seq_lens, void* out, rs_out_dtype out_dtype, void* workspace, size_t ws_bytes,
                            rs_stream_t stream) {
    if (!attn_shape_ok(B, Hq, Hkv, D, max_pages, max_len)) return RS_ERR_SHAPE;
    if (out_dtype != RS_OUT_BF16 && out_dtype != RS_OUT_F32) return RS_ERR_INVALID_ARG;
    if (!q_bf16 || !alpha_q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !workspace)
        return RS_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace) ||
        !aligned4(alpha_q) || !aligned4(block_table) || !aligned4(seq_lens))
        return RS_ERR_ALIGNMENT;
    if (ws_bytes < rs_resattn_workspace_bytes(B, Hq, Hkv, D, max_len)) return RS_ERR_WORKSPACE;
    cudaError_t why;
    const rs::DeviceInfo* dev = rs::current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    // (the query-quantization step of Sec. 5.2 runs inside the split kernel)
    rs::AttnArgs a{};
    a.q = static_cast<const uint16_t*>(q_bf16);
    a.alpha_q = alpha_q;
    a.k_cache = static_cast<const uint8_t*>(k_cache);
    a.v_cache = static_cast<const uint8_t*>(v_cache);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.part = static_cast<float*>(workspace);
    a.err = dev->err;
    a.trace = rs::trace_buffer();
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.max_pages = max_pages;
    a.max_len = max_len;
    a.split_tokens = rs::resattn_split_tokens(B, Hkv, D, max_len, dev->num_sms);
    a.splits = max_len > 0 ? (max_len + a.split_tokens - 1) / a.split_tokens : 1;
    return from_cuda(rs::launch_resattn(D, a, out, out_dtype == RS_OUT_F32 ? 1 : 0, (cudaStream_t)stream));
}

void rs_debug_pair_gemm(int enable) { rs::set_pair_gemm(enable); }

rs_status rs_fold_pairs(int M, int N, const float* z, void* y, rs_out_dtype out_dtype, rs_stream_t stream) {
    if (M < 0 || N < 0 || (out_dtype != RS_OUT_BF16 && out_dtype != RS_OUT_F32)) return RS_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return RS_OK;
    if (!z || !y) return RS_ERR_INVALID_ARG;
    if (!aligned16(z) || !aligned16(y)) return RS_ERR_ALIGNMENT;
    cudaError_t why;
    const rs::DeviceInfo* dev = rs::current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    return from_cuda(launch_fold_pairs(z, y, M, N, out_dtype == RS_OUT_F32 ? 1 : 0, (cudaStream_t)stream,
                                       dev->num_sms));
}

rs_status rs_get_device_error_async(uint32_t* out, rs_stream_t stream) {
    if (!out) return RS_ERR_INVALID_ARG;
    if (!aligned4(out)) return RS_ERR_ALIGNMENT;
    cudaError_t why;
    const rs::DeviceInfo* dev = rs::current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    rs::read_error_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(dev->err, out);
    return cudaGetLastError() == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

rs_status rs_debug_linear_dump(rs_format fmt, int compensated, int M, int N, int K, const void* x_bf16,
                               const float* alpha_x, const void* wq, const float* alpha_w, void* y,
                               rs_out_dtype out_dtype, void* workspace, size_t ws_bytes, void* dump,
                               size_t dump_bytes, int* layout, rs_stream_t stream) {
    if (!layout || !fmt_ok(fmt) || M < 1 || N < 1) return RS_ERR_INVALID_ARG;
    if (!k_ok(K) || (int64_t)M * 2 > (int64_t)0x7FFFFFFF) return RS_ERR_SHAPE;
    cudaError_t why;
    const rs::DeviceInfo* dev = rs::current_device(&why);
    if (!dev) return RS_ERR_CUDA;
    if (!dev->supported) return RS_ERR_UNSUPPORTED;
    const GemmPlan p = make_gemm_plan(fmt, compensated != 0, M, N, K, dev->num_sms, /*allow_fused=*/true);
    const size_t stage = plan_b_stage_bytes(p);
    const int v[7] = {p.fused ? (p.qpair ? 2 : 1) : 0, p.bn, p.grid_x, p.splits, p.slots, (int)stage, p.chunks};
    for (int i = 0; i < 7; ++i) layout[i] = v[i];
    if (!dump) return RS_OK;  // layout query only
    if (!p.fused) return RS_ERR_UNSUPPORTED;
    if (!aligned16(dump)) return RS_ERR_ALIGNMENT;
    if (dump_bytes < (size_t)p.grid_x * (size_t)p.splits * (size_t)p.slots * stage) return RS_ERR_WORKSPACE;
    if (!x_bf16) return RS_ERR_INVALID_ARG;
    return linear_impl(fmt, compensated != 0, M, N, K, x_bf16, nullptr, alpha_x, wq, alpha_w, y, out_dtype,
                       workspace, ws_bytes, (cudaStream_t)stream, 0, nullptr, dump);
}

rs_status rs_get_device_error(rs_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return RS_ERR_CUDA;
    uint32_t* p = device_error_word();
    if (!p) return RS_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return RS_ERR_CUDA;
    if (v != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return RS_ERR_CUDA;
    }
    return (rs_status)v;
}

}  // extern "C"
