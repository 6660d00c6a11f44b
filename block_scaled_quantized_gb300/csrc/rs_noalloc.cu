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
// workspace.  The call runs the two existing steps, rs_quantize_residue into
// that array and rs_linear_compensated reading it, so its results are those
// of the existing entry points.  No cudaMalloc, cudaFree or allocating
// library routine is called.
#include <mutex>

#include "rs.h"
#include "rs_internal.h"

namespace {

// Every GPU that loads librs holds this array until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[RS_NOALLOC_SCRATCH_BYTES];

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
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
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
    if (!x_bf16 || !wq || !y) return RS_ERR_INVALID_ARG;
    // the paired operand of 2*M rows (and, without alpha_x, the tensor scale
    // after it) must fit the fixed array
    if (rs::operand_bytes(fmt, 2 * M, K) > (size_t)RS_NOALLOC_SCRATCH_BYTES) return RS_ERR_WORKSPACE;
    const size_t a_off = rs::alpha_slot_offset(fmt, true, M, K);
    if (fmt == RS_NVFP4 && !alpha_x && a_off + 256 > (size_t)RS_NOALLOC_SCRATCH_BYTES) return RS_ERR_WORKSPACE;
    void* scratch = scratch_on_current_device();
    if (!scratch) return RS_ERR_CUDA;
    if (fmt == RS_NVFP4 && !alpha_x) {
        float* a = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + a_off);
        const rs_status st = rs_compute_tensor_scale(x_bf16, (int64_t)M * K, a, stream);
        if (st != RS_OK) return st;
        alpha_x = a;
    }
    // The quantizer writes every byte of the operand that the GEMM reads
    // (codes, scales and the zero scale padding), so nothing left over from
    // an earlier call needs clearing.
    rs_status s = rs_quantize_residue(fmt, M, K, x_bf16, K, alpha_x, scratch, stream);
    if (s != RS_OK) return s;
    return rs_linear_compensated(fmt, M, N, K, nullptr, scratch, alpha_x, wq, alpha_w, y, out_dtype, nullptr, 0,
                                 stream);
}
