// rs_linear_compensated_noalloc: the compensated linear layer for callers that
// cannot allocate device memory.
//
// Who needs it: code that runs where no allocator is available or allowed,
// e.g. a plugin called from inside another framework's execution graph that
// is handed only its input and output buffers, or a process that must keep
// its device-memory footprint fixed after start-up.  rs_linear_compensated
// asks such a caller for a workspace it cannot provide.
//
// How: the quantized activations (the paired base + residue operand) live in
// a fixed device array of this library, below, instead of a caller
// workspace.  The call runs the two-kernel form of the compensated layer:
// the paired quantizer into that array, then the GEMM reading it (the
// workspace call may instead quantize inside the GEMM, so the outputs agree
// within the output tolerance, not bit for bit).  No cudaMalloc, cudaFree
// or allocating library routine is called.
#include <mutex>

#include "rs.h"
#include "rs_internal.h"

namespace {

// Every GPU that loads librs holds this array until the process exits: the
// largest accepted operand, its 1024-byte alignment and the 256-byte tensor
// scale slot after it.
constexpr size_t kScratchBytes = (size_t)RS_NOALLOC_SCRATCH_BYTES + 1024 + 256;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device.  In host code the
// array's name only stands for it, so the address is looked up once per
// device, with that device current, and cached.
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            (void)cudaGetLastError();  // leave no error behind for the caller's next CUDA call
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" rs_status rs_linear_compensated_noalloc(rs_format fmt, int M, int N, int K, const void* x_bf16,
                                                   const float* alpha_x, const void* wq, const float* alpha_w,
                                                   void* y, rs_out_dtype out_dtype, rs_stream_t stream) {
    if ((fmt != RS_NVFP4 && fmt != RS_MXFP4) || M < 0 || N < 0) return RS_ERR_INVALID_ARG;
    if (K <= 0 || K % 32 != 0) return RS_ERR_SHAPE;
    if (M == 0 || N == 0) return RS_OK;
    if (!x_bf16 || !wq || !y || (fmt == RS_NVFP4 && !alpha_w)) return RS_ERR_INVALID_ARG;
    if (out_dtype != RS_OUT_BF16 && out_dtype != RS_OUT_F32) return RS_ERR_INVALID_ARG;
    // the paired operand of 2*M rows must fit the documented maximum (the
    // array also holds the tensor-scale slot after the largest operand)
    if ((int64_t)M * 2 > (int64_t)0x7FFFFFFF || rs::operand_bytes(fmt, 2 * M, K) > (size_t)RS_NOALLOC_SCRATCH_BYTES)
        return RS_ERR_WORKSPACE;
    const size_t a_off = rs::alpha_slot_offset(fmt, true, M, K);
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (!a16(x_bf16) || !a16(wq) || !a16(y) || (alpha_x && !a4(alpha_x)) || (alpha_w && !a4(alpha_w)))
        return RS_ERR_ALIGNMENT;
    int num_sms = 0;
    uint32_t* err = nullptr;
    const rs_status dev = rs::current_device_status(&num_sms, &err);
    if (dev != RS_OK) return dev;
    void* scratch = scratch_on_current_device();
    if (!scratch) return RS_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    if (fmt == RS_NVFP4 && !alpha_x) {
        float* a = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + a_off);
        if (rs::launch_tensor_scale(x_bf16, (int64_t)M * K, a, err, st, num_sms) != cudaSuccess) return RS_ERR_CUDA;
        alpha_x = a;
    }
    // The quantizer writes every byte of the operand that the GEMM reads
    // (codes, scales and the zero scale padding), so nothing left over from
    // an earlier call needs clearing.  Programmatic launch, as in the
    // two-kernel plan of rs_linear_compensated.
    if (rs::launch_quantize(fmt, true, M, K, x_bf16, K, alpha_x, scratch, st, num_sms, /*pdl=*/true) != cudaSuccess)
        return RS_ERR_CUDA;
    return rs_linear_compensated(fmt, M, N, K, nullptr, scratch, alpha_x, wq, alpha_w, y, out_dtype, nullptr, 0,
                                 stream);
}
