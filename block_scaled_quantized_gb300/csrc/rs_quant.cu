// Activation / weight quantizers (ResServe Sec. 4.4, App. B.2 Eq. 8-10 and
// Algorithm 1 "Residue NVFP4 quantization: eight inputs per thread").
//
// One warp covers 256 consecutive elements of one row; each lane loads eight
// bf16 inputs with one 16-byte load (the paper's "pack8" mapping).  The block
// amax is a shuffle-max over the 2 (NVFP4, 16-element block) or 4 (MXFP4,
// 32-element block) lanes that share a block.  Codes are written as one
// 32-bit word per lane; the four scale bytes of a scale-atom row are gathered
// into one lane with shuffles and written as one 32-bit word, directly in
// the atom layout the tcgen05 GEMM reads (no reorder kernel).
//
// In paired mode (full compensation) each lane also forms the residue
// r = x - x^ in registers, quantizes it with its own block scales and the
// same tensor scale, and writes it as the odd row of the row pair.
#include <cuda_bf16.h>

#include "rs_device.cuh"
#include "rs_internal.h"

namespace rs {

// ----------------------------------------------------------- tensor scale --

__global__ void tensor_amax_kernel(const uint16_t* __restrict__ x, int64_t n,
                                   uint32_t* __restrict__ amax_bits) {
    uint32_t m = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t a = x[i] & 0x7FFFu;  // |x| as bf16 bits; order-preserving
        m = a > m ? a : m;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint32_t t = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        m = t > m ? t : m;
    }
    if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(amax_bits, m << 16);  // as fp32 bits
}

// alpha = fl(amax / 2688) (App. B.2 Eq. 8: max_i s_i / 448 with s_i = Max_i/6).
__global__ void tensor_scale_finalize_kernel(float* __restrict__ alpha, uint32_t* __restrict__ err) {
    const uint32_t bits = *reinterpret_cast<uint32_t*>(alpha);
    if (bits >= 0x7F800000u) {  // Inf or NaN amax
        atomicExch(err, kErrInvalidArg);
        *alpha = __uint_as_float(0x7FC00000u);
        return;
    }
    *alpha = __fdiv_rn(__uint_as_float(bits), 2688.0f);
}

// ------------------------------------------------------------- quantizer --

struct QuantArgs {
    const uint16_t* x;   // bf16 bits [rows][ldx]
    int64_t ldx;
    int rows;            // input rows
    int K;
    const float* alpha;  // NVFP4 tensor scale (device); unused for MXFP4
    uint8_t* codes;      // [rows_out][K/2]
    uint8_t* sf;         // scale atoms
    int rows_out;        // rows (base) or 2*rows (paired)
    int rows_pad;        // rows_out rounded up to 128
    int n_atoms_k;       // ceil(K / atom_k)
    int chunks;          // ceil(K / 256)
    int early_trigger;   // release the dependent grid once the prior grid is done
};

// Quantize the 8 values of one lane given the block's scale.  Returns the
// packed codes (element 2j in the low nibble of byte j) and writes the
// reconstruction x^ = fl(s~ * dec(q)) into xh.
__device__ __forceinline__ uint32_t quantize8(const float (&xf)[8], float mul, float st,
                                              float (&xh)[8]) {
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t q = e2m1_encode(__fmul_rn(xf[e], mul));
        word |= q << (4 * e);
        xh[e] = __fmul_rn(st, e2m1_decode(q));
    }
    return word;
}

// NVFP4 block scale from the block amax (Eq. 8-9, Alg. 1 line 3):
// sf = E4M3(fl(fl(amax/6)/alpha)), s~ = fl(alpha * dec(sf)), mul = fl(1/s~).
__device__ __forceinline__ uint32_t nv_block_scale(float amax, float alpha, float& st, float& mul) {
    const float s = __fdiv_rn(amax, kE2M1Max);
    const float t = alpha > 0.0f ? __fdiv_rn(s, alpha) : 0.0f;
    const uint32_t sf = e4m3_encode_satfinite(t);
    st = __fmul_rn(alpha, e4m3_decode(sf));
    mul = st == 0.0f ? 0.0f : __fdiv_rn(1.0f, st);
    return sf;
}

// MXFP4 block scale: byte = max(E - 2, 0) where E is the biased fp32
// exponent of amax, i.e. e = floor(log2 amax) - 2 clamped at -127 (amax == 0
// and fp32-subnormal amax give byte 0).  st = 2^e, mul = 2^-e, both exact.
__device__ __forceinline__ uint32_t mx_block_scale(float amax, float& st, float& mul) {
    const int E = (int)(__float_as_uint(amax) >> 23);
    const uint32_t byte = E >= 2 ? (uint32_t)(E - 2) : 0u;
    st = byte >= 1u ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);  // 2^(byte-127)
    mul = __uint_as_float((254u - byte) << 23);                                      // 2^(127-byte)
    return byte;
}

// Shuffle-max over the lanes that share one scale block.
template <int FMT>
__device__ __forceinline__ float block_amax(float a) {
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    if (FMT == 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    return a;
}

// Gather the four scale bytes of one atom row into the first lane of the
// group and store them as one 32-bit word.  NVFP4: lanes 8g..8g+7 hold
// blocks 4g'..4g'+3 (two lanes per block); MXFP4: lanes 16g..16g+15.
template <int FMT>
__device__ __forceinline__ void store_sf_word(uint8_t* sf, int row, int chunk, int lane,
                                              uint32_t sfbyte, const QuantArgs& a) {
    constexpr int kLanesPerBlock = FMT == 0 ? 2 : 4;
    constexpr int kLanesPerAtom = 4 * kLanesPerBlock;
    const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, sfbyte, (lane & ~(kLanesPerAtom - 1)) + 0 * kLanesPerBlock);
    const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, sfbyte, (lane & ~(kLanesPerAtom - 1)) + 1 * kLanesPerBlock);
    const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, sfbyte, (lane & ~(kLanesPerAtom - 1)) + 2 * kLanesPerBlock);
    const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, sfbyte, (lane & ~(kLanesPerAtom - 1)) + 3 * kLanesPerBlock);
    if ((lane & (kLanesPerAtom - 1)) == 0) {
        const int g = chunk * (256 / atom_k(FMT)) + lane / kLanesPerAtom;  // atom index along K
        if (g < a.n_atoms_k) {
            const size_t off = sf_offset(row, g * kAtomBlocks, a.n_atoms_k);
            *reinterpret_cast<uint32_t*>(sf + off) = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
        }
    }
}

template <int FMT, bool PAIRED>
__global__ void __launch_bounds__(256) quantize_kernel(QuantArgs a) {
    // Inputs may come from the previous kernel in the stream.
    pdl_wait_prior_grid();
    if (a.early_trigger) pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps_total = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t tasks = (int64_t)a.rows * a.chunks;
    const float alpha = FMT == 0 ? *a.alpha : 0.0f;

    for (int64_t task = warp; task < tasks; task += n_warps_total) {
        const int row = (int)(task / a.chunks);
        const int chunk = (int)(task % a.chunks);
        const int k0 = chunk * 256 + lane * 8;
        const bool valid = k0 < a.K;

        float xf[8];
        if (valid) {
            const uint4 v = *reinterpret_cast<const uint4*>(a.x + row * a.ldx + k0);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xf[2 * i] = __uint_as_float(w[i] << 16);
                xf[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) xf[e] = 0.0f;
        }

        // ---- base (Alg. 1 lines 1-5)
        float am = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(xf[e]));
        am = block_amax<FMT>(am);
        float st, mul;
        const uint32_t sfb = FMT == 0 ? nv_block_scale(am, alpha, st, mul) : mx_block_scale(am, st, mul);
        float xh[8];
        const uint32_t word = quantize8(xf, mul, st, xh);
        const int out_row = PAIRED ? 2 * row : row;
        if (valid)
            *reinterpret_cast<uint32_t*>(a.codes + (size_t)out_row * (a.K / 2) + k0 / 2) = word;
        store_sf_word<FMT>(a.sf, out_row, chunk, lane, valid ? sfb : 0u, a);

        if (PAIRED) {
            // ---- residue in registers (Alg. 1 line 6), same tensor scale
            float r[8];
            float ra = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                r[e] = __fsub_rn(xf[e], xh[e]);
                ra = fmaxf(ra, fabsf(r[e]));
            }
            ra = block_amax<FMT>(ra);
            float rst, rmul;
            const uint32_t sfr = FMT == 0 ? nv_block_scale(ra, alpha, rst, rmul) : mx_block_scale(ra, rst, rmul);
            float rh[8];
            const uint32_t rword = quantize8(r, rmul, rst, rh);
            if (valid)
                *reinterpret_cast<uint32_t*>(a.codes + (size_t)(out_row + 1) * (a.K / 2) + k0 / 2) = rword;
            store_sf_word<FMT>(a.sf, out_row + 1, chunk, lane, valid ? sfr : 0u, a);
        }
    }

    // ---- zero scale words of the padding rows [rows_out, rows_pad)
    const int64_t pad_words = (int64_t)(a.rows_pad - a.rows_out) * a.n_atoms_k;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = tid; i < pad_words; i += nthreads) {
        const int r = a.rows_out + (int)(i / a.n_atoms_k);
        const int g = (int)(i % a.n_atoms_k);
        *reinterpret_cast<uint32_t*>(a.sf + sf_offset(r, g * kAtomBlocks, a.n_atoms_k)) = 0u;
    }
}

// ---------------------------------------------------------------- launch --

static int quant_grid(int64_t warps_needed, int pad_words, int num_sms) {
    int64_t blocks = (warps_needed + 7) / 8;
    const int64_t pad_blocks = (pad_words + 255) / 256;
    if (pad_blocks > blocks) blocks = pad_blocks;
    const int64_t cap = (int64_t)num_sms * 32;
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

cudaError_t launch_tensor_scale(const void* x, int64_t n, float* alpha, uint32_t* err,
                                cudaStream_t stream, int num_sms) {
    cudaError_t e = cudaMemsetAsync(alpha, 0, sizeof(float), stream);
    if (e != cudaSuccess) return e;
    if (n > 0) {
        int64_t blocks = (n + 1023) / 1024;
        if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
        tensor_amax_kernel<<<(int)blocks, 256, 0, stream>>>(static_cast<const uint16_t*>(x), n,
                                                             reinterpret_cast<uint32_t*>(alpha));
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    tensor_scale_finalize_kernel<<<1, 1, 0, stream>>>(alpha, err);
    return cudaGetLastError();
}

template <int FMT, bool PAIRED>
static cudaError_t launch_quant_typed(const QuantArgs& a, int grid, cudaStream_t stream, bool pdl) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, quantize_kernel<FMT, PAIRED>, a);
}

cudaError_t launch_quantize(int fmt, bool paired, int rows, int K, const void* x, int64_t ldx,
                            const float* alpha, void* q_out, cudaStream_t stream, int num_sms, bool pdl) {
    QuantArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.ldx = ldx;
    a.rows = rows;
    a.K = K;
    a.alpha = alpha;
    a.rows_out = paired ? 2 * rows : rows;
    a.rows_pad = (a.rows_out + kAtomRows - 1) / kAtomRows * kAtomRows;
    a.n_atoms_k = (K + atom_k(fmt) - 1) / atom_k(fmt);
    a.chunks = (K + 255) / 256;
    a.codes = static_cast<uint8_t*>(q_out);
    a.sf = static_cast<uint8_t*>(q_out) + operand_sf_offset(fmt, a.rows_out, K);
    a.early_trigger = pdl ? 1 : 0;
    const int64_t warps = (int64_t)rows * a.chunks;
    const int pad_words = (a.rows_pad - a.rows_out) * a.n_atoms_k;
    const int grid = quant_grid(warps, pad_words, num_sms);
    if (fmt == 0) return paired ? launch_quant_typed<0, true>(a, grid, stream, pdl)
                                : launch_quant_typed<0, false>(a, grid, stream, pdl);
    return paired ? launch_quant_typed<1, true>(a, grid, stream, pdl) : launch_quant_typed<1, false>(a, grid, stream, pdl);
}

}  // namespace rs
