// Activation / weight quantizers (ResServe Sec. 4.4, App. B.2 Eq. 8-10 and
// Algorithm 1 "Residue NVFP4 quantization: eight inputs per thread").
//
// One warp covers 256 consecutive elements of one row; each lane loads eight
// bf16 inputs with one 16-byte load.  Codes are written as one 32-bit word
// per lane; the four scale bytes of a scale-atom row are gathered into one
// lane with shuffles and written as one 32-bit word, directly in the layout
// the tcgen05 GEMM reads, so no reorder pass follows.
//
// Three output layouts:
//  * ROWS    activation operand, row-major codes + scale atoms;
//  * PAIRED  the same with base row 2j and residue row 2j+1 (full
//            compensation: the residue is formed in registers from x and the
//            decoded base and quantized with its own block scales and the same
//            tensor scale);
//  * WEIGHT  the tiled weight operand: one contiguous block per 128 output
//            channels x 256 K holding the codes in the 128-byte-swizzled
//            shared-memory image the MMA reads, followed by the block's scale
//            atoms, so the GEMM streams each block with a single bulk copy.
#include <cuda_bf16.h>

#include <algorithm>

#include "rs_device.cuh"
#include "rs_internal.h"
#include "rs_quant_core.cuh"

namespace rs {

// ----------------------------------------------------------- tensor scale --

__global__ void tensor_amax_kernel(const uint16_t* __restrict__ x, int64_t n,
                                   uint32_t* __restrict__ amax_bits) {
    // |x| as bf16 bits (sign cleared) orders like |x|; two halves per word
    // are compared at once with an unsigned 16-bit SIMD max.
    uint32_t m2 = 0;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // elements before the first 16-byte boundary take element loads
    int64_t head = (int64_t)((16 - (reinterpret_cast<uintptr_t>(x) & 15)) & 15) / 2;
    if (head > n) head = n;
    const uint4* v = reinterpret_cast<const uint4*>(x + head);
    const int64_t nv = (n - head) / 8;
    int64_t i = tid;
    for (; i + 3 * stride < nv; i += 4 * stride) {  // four independent 16-byte loads in flight
        uint4 a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) a[u] = v[i + u * stride];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            m2 = __vmaxu2(__vmaxu2(m2, a[u].x & 0x7FFF7FFFu),
                          __vmaxu2(__vmaxu2(a[u].y & 0x7FFF7FFFu, a[u].z & 0x7FFF7FFFu), a[u].w & 0x7FFF7FFFu));
    }
    for (; i < nv; i += stride) {
        const uint4 a = v[i];
        m2 = __vmaxu2(__vmaxu2(m2, a.x & 0x7FFF7FFFu),
                      __vmaxu2(__vmaxu2(a.y & 0x7FFF7FFFu, a.z & 0x7FFF7FFFu), a.w & 0x7FFF7FFFu));
    }
    for (int64_t j = head + nv * 8 + tid; j < n; j += stride) m2 = __vmaxu2(m2, x[j] & 0x7FFFu);
    for (int64_t j = tid; j < head; j += stride) m2 = __vmaxu2(m2, x[j] & 0x7FFFu);
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
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
    const float a = __fdiv_rn(__uint_as_float(bits), 2688.0f);
    if (!nv_alpha_supported(a)) atomicExch(err, kErrInvalidArg);  // tensor amax below about 4e-32
    *alpha = a;
}

// ------------------------------------------------------------- quantizer --

enum QuantMode { kRows = 0, kPaired = 1, kWeight = 2 };

struct QuantArgs {
    const uint16_t* x;   // bf16 bits [rows][ldx]
    int64_t ldx;
    int rows;            // input rows
    int K;
    const float* alpha;  // NVFP4 tensor scale (device); unused for MXFP4
    uint8_t* out;        // operand base
    uint8_t* sf;         // ROWS / PAIRED: scale-atom region
    int rows_out;        // ROWS / PAIRED: rows or 2*rows
    int rows_pad;        // ROWS / PAIRED: rows_out rounded up to 128
    int task_rows;       // rows iterated over (WEIGHT: padded to 128)
    int n_atoms_k;       // ceil(K / atom_k)
    int chunks;          // ceil(K / 256)
    int early_trigger;   // release the dependent grid once the prior grid is done
    uint32_t* err;       // device error word
    // WEIGHT with a K-Ext extension (Eq. 6; [W | W[:, S]] in bf16): columns k_base..K-1
    // are W[:, S] -- column k_base + g*kext_k + j is the j-th selected channel
    // of group g (kext_mask[g], device)
    int k_base;
    int kext_k;
    const uint8_t* kext_mask;
};

// U > 1 (large activation operands): a warp takes U consecutive 256-element
// chunks of one row per step and issues their U loads before quantizing any
// of them, so that each lane keeps U x 16 bytes in flight.
template <int FMT, int MODE, int U>
__global__ void __launch_bounds__(256, U > 1 ? 3 : 1) quantize_kernel(QuantArgs a) {
    static_assert(U == 1 || MODE != kWeight, "the weight quantizer takes one chunk per step");
    // Inputs may come from the previous kernel in the stream.
    pdl_wait_prior_grid();
    if (a.early_trigger) pdl_launch_dependents();
    constexpr int LPA = lanes_per_atom<FMT>();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps_total = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int n_cg = (a.chunks + U - 1) / U;  // chunk groups per row
    const int64_t tasks = (int64_t)a.task_rows * n_cg;
    const NvScaleConst ksc = nv_scale_const(FMT == 0 ? *a.alpha : 0.0f);
    if (FMT == 0 && blockIdx.x == 0 && threadIdx.x == 0 && !nv_alpha_supported(ksc.alpha))
        atomicExch(a.err, kErrInvalidArg);

    // task = row * n_cg + cg, advanced by n_warps_total without a division
    const int dstep_row = (int)(n_warps_total / n_cg), dstep_cg = (int)(n_warps_total % n_cg);
    int row = (int)(warp / n_cg), cg = (int)(warp % n_cg);
    for (int64_t task = warp; task < tasks; task += n_warps_total) {
        if (task != warp) {
            row += dstep_row;
            cg += dstep_cg;
            if (cg >= n_cg) {
                cg -= n_cg;
                ++row;
            }
        }
        uint4 raw[U];  // the U input words, widened when processed
        float xw[8];   // the weight path's gathered extension columns
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int chunk = cg * U + u;
            const int k0 = chunk * 256 + lane * 8;
            if (MODE == kWeight && a.kext_k > 0 && k0 >= a.k_base) {
                // appended columns of the extended weight: gathered
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int e = k0 - a.k_base + i;
                    float v = 0.0f;
                    if (row < a.rows && e < a.K - a.k_base) {
                        const int grp = e / a.kext_k;
                        const uint32_t t = __fns(a.kext_mask[grp], 0, e - grp * a.kext_k + 1);
                        if (t < 8u) v = __uint_as_float((uint32_t)a.x[(int64_t)row * a.ldx + 8 * grp + (int)t] << 16);
                        else atomicExch(a.err, kErrInvalidArg);  // fewer than k channels in the group
                    }
                    xw[i] = v;
                }
                raw[u] = make_uint4(0u, 0u, 0u, 0u);
            } else {
                raw[u] = load16_or_zero(a.x + (int64_t)row * a.ldx + k0, k0 < a.K && row < a.rows);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int chunk = cg * U + u;
            if (U > 1 && chunk >= a.chunks) break;  // ragged last group (warp-uniform)
            const int k0 = chunk * 256 + lane * 8;
            const bool valid = k0 < a.K && row < a.rows;
            float xf[8];
            if (MODE == kWeight && a.kext_k > 0 && k0 >= a.k_base) {
#pragma unroll
                for (int i = 0; i < 8; ++i) xf[i] = xw[i];
            } else {
                unpack8_bf16(raw[u], xf);
            }

            uint32_t sfb;
            float xh[8];
            const uint32_t codes = quant_lane<FMT, MODE == kPaired>(xf, ksc, sfb, xh);
            const uint32_t sfw = gather_sf_word<FMT>(sfb, lane);
            const int g = chunk * (256 / atom_k(FMT)) + lane / LPA;  // atom index along K
            const bool leader = (lane % LPA) == 0;

            if (MODE == kWeight) {
                const int t = row / 128, r = row % 128;
                uint8_t* blk = a.out + ((size_t)t * a.chunks + chunk) * weight_block_bytes(FMT);
                *reinterpret_cast<uint32_t*>(blk + sw128_offset((uint32_t)r, (uint32_t)lane * 4u)) = codes;
                if (leader)
                    *reinterpret_cast<uint32_t*>(blk + kWeightCodeBytes + (lane / LPA) * kAtomBytes + (r % 32) * 16 +
                                                 ((r / 32) % 4) * 4) = sfw;
            } else {
                const int out_row = MODE == kPaired ? 2 * row : row;
                if (valid)
                    *reinterpret_cast<uint32_t*>(a.out + (size_t)out_row * (a.K / 2) + k0 / 2) = codes;
                if (leader && g < a.n_atoms_k)
                    *reinterpret_cast<uint32_t*>(a.sf + sf_offset(out_row, g * kAtomBlocks, a.n_atoms_k)) = sfw;
                if (MODE == kPaired) {
                    float r[8];
                    residue8(xf, xh, r);
                    uint32_t sfr;
                    float rh[8];
                    const uint32_t rcodes = quant_lane<FMT, false>(r, ksc, sfr, rh);
                    const uint32_t sfrw = gather_sf_word<FMT>(sfr, lane);
                    if (valid)
                        *reinterpret_cast<uint32_t*>(a.out + (size_t)(out_row + 1) * (a.K / 2) + k0 / 2) = rcodes;
                    if (leader && g < a.n_atoms_k)
                        *reinterpret_cast<uint32_t*>(a.sf + sf_offset(out_row + 1, g * kAtomBlocks, a.n_atoms_k)) =
                            sfrw;
                }
            }
        }
    }

    if (MODE != kWeight) {
        // zero scale words of the padding rows [rows_out, rows_pad)
        const int64_t pad_words = (int64_t)(a.rows_pad - a.rows_out) * a.n_atoms_k;
        const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
        for (int64_t i = tid; i < pad_words; i += nthreads) {
            const int r = a.rows_out + (int)(i / a.n_atoms_k);
            const int g = (int)(i % a.n_atoms_k);
            *reinterpret_cast<uint32_t*>(a.sf + sf_offset(r, g * kAtomBlocks, a.n_atoms_k)) = 0u;
        }
    }
}

// NVFP4, one whole 16-element block held as two raw bf16 words: base codes
// (two words, element e in bits 4(e%8).. of word e/8) and scale byte, and,
// when `resid`, the residue's codes and scale byte (Eq. 8-10, Alg. 1).
// s~ and fl(1/s~) come from a table of the 127 finite E4M3 bytes built with
// nv_scale_table_entry; the block amax is taken on the packed bf16 bits.
// Same codes and bytes as quant_block; the reconstruction and the residue use
// the never-fused scalar intrinsics.
__device__ __forceinline__ void nv_quant16(const uint4 (&raw)[2], const NvScaleConst& k, const float* tab_st,
                                           const float* tab_mul, bool resid, uint32_t (&cb)[2], uint32_t& sfb,
                                           uint32_t (&cr)[2], uint32_t& sfr) {
    const uint32_t w[8] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w};
    sfb = nv_block_byte(amax16_bf16(w), k);
    const float st = tab_st[sfb], mul = tab_mul[sfb];
    float xf[16], v[16];
    unpack8_bf16(raw[0], *reinterpret_cast<float(*)[8]>(&xf[0]));
    unpack8_bf16(raw[1], *reinterpret_cast<float(*)[8]>(&xf[8]));
#pragma unroll
    for (int e = 0; e < 16; e += 2) fmul2_rn(xf[e], xf[e + 1], mul, mul, v[e], v[e + 1]);
    cb[0] = e2m1_encode8(*reinterpret_cast<const float(*)[8]>(&v[0]));
    cb[1] = e2m1_encode8(*reinterpret_cast<const float(*)[8]>(&v[8]));
    if (!resid) return;
    float d[16];
    e2m1_decode8(cb[0], *reinterpret_cast<float(*)[8]>(&d[0]));
    e2m1_decode8(cb[1], *reinterpret_cast<float(*)[8]>(&d[8]));
#pragma unroll
    for (int e = 0; e < 16; ++e) xf[e] = __fsub_rn(xf[e], __fmul_rn(st, d[e]));  // r = fl(x - fl(s~ dec(q)))
    float am0 = 0.0f, am1 = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
        am0 = fmaxf(am0, fabsf(xf[e]));
        am1 = fmaxf(am1, fabsf(xf[e + 1]));
    }
    sfr = nv_block_byte(fmaxf(am0, am1), k);
    const float mulr = tab_mul[sfr];
#pragma unroll
    for (int e = 0; e < 16; e += 2) fmul2_rn(xf[e], xf[e + 1], mulr, mulr, v[e], v[e + 1]);
    cr[0] = e2m1_encode8(*reinterpret_cast<const float(*)[8]>(&v[0]));
    cr[1] = e2m1_encode8(*reinterpret_cast<const float(*)[8]>(&v[8]));
}

// ------------------------------------------- NVFP4, one block per lane --
//
// Large NVFP4 activation operands (ROWS / PAIRED, K a multiple of 512): lane
// l of a warp quantizes the whole 16-element block 16l..16l+15 of a
// 512-element chunk, so each block scale is derived once (not on both lanes
// of a block pair), its amax is taken on the packed bf16 bits, and s~ and
// fl(1/s~) come from a per-CTA table of the 127 finite E4M3 bytes.  Same
// arithmetic per element as quant_lane (Eq. 8-10, Alg. 1), identical codes
// and scale bytes.  U chunks per warp step, loads first.
template <int MODE, int U>
__global__ void __launch_bounds__(256, 3) quantize_nv_wide_kernel(QuantArgs a) {
    __shared__ float tab_st[128], tab_mul[128];
    pdl_wait_prior_grid();
    if (a.early_trigger) pdl_launch_dependents();
    const NvScaleConst ksc = nv_scale_const(*a.alpha);
    if (threadIdx.x < 128) nv_scale_table_entry(threadIdx.x, ksc.alpha, tab_st[threadIdx.x], tab_mul[threadIdx.x]);
    if (blockIdx.x == 0 && threadIdx.x == 0 && !nv_alpha_supported(ksc.alpha)) atomicExch(a.err, kErrInvalidArg);
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps_total = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int chunks = a.K / 512;
    const int n_cg = (chunks + U - 1) / U;
    const int64_t tasks = (int64_t)a.rows * n_cg;
    const int dstep_row = (int)(n_warps_total / n_cg), dstep_cg = (int)(n_warps_total % n_cg);
    int row = (int)(warp / n_cg), cg = (int)(warp % n_cg);
    for (int64_t task = warp; task < tasks; task += n_warps_total) {
        if (task != warp) {
            row += dstep_row;
            cg += dstep_cg;
            if (cg >= n_cg) {
                cg -= n_cg;
                ++row;
            }
        }
        const uint16_t* xrow = a.x + (int64_t)row * a.ldx + lane * 16;
        uint4 raw[U][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool ok = cg * U + u < chunks;
            raw[u][0] = load16_or_zero(xrow + (cg * U + u) * 512, ok);
            raw[u][1] = load16_or_zero(xrow + (cg * U + u) * 512 + 8, ok);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int chunk = cg * U + u;
            if (U > 1 && chunk >= chunks) break;  // ragged last group (warp-uniform)
            uint32_t c[2], rc[2], sf, sfr = 0;
            nv_quant16(raw[u], ksc, tab_st, tab_mul, MODE == kPaired, c, sf, rc, sfr);
            // the atom row word of blocks 4j..4j+3 lands on lane 4j
            uint32_t t = sf | (__shfl_down_sync(0xFFFFFFFFu, sf, 1) << 8);
            const uint32_t sfw = t | (__shfl_down_sync(0xFFFFFFFFu, t, 2) << 16);
            const int out_row = MODE == kPaired ? 2 * row : row;
            const size_t code_off = (size_t)chunk * 256 + (size_t)lane * 8;
            *reinterpret_cast<uint2*>(a.out + (size_t)out_row * (a.K / 2) + code_off) = make_uint2(c[0], c[1]);
            if ((lane & 3) == 0)
                *reinterpret_cast<uint32_t*>(a.sf + sf_offset(out_row, chunk * 32 + lane, a.n_atoms_k)) = sfw;
            if (MODE == kPaired) {
                t = sfr | (__shfl_down_sync(0xFFFFFFFFu, sfr, 1) << 8);
                const uint32_t sfrw = t | (__shfl_down_sync(0xFFFFFFFFu, t, 2) << 16);
                *reinterpret_cast<uint2*>(a.out + (size_t)(out_row + 1) * (a.K / 2) + code_off) =
                    make_uint2(rc[0], rc[1]);
                if ((lane & 3) == 0)
                    *reinterpret_cast<uint32_t*>(a.sf + sf_offset(out_row + 1, chunk * 32 + lane, a.n_atoms_k)) =
                        sfrw;
            }
        }
    }

    // zero scale words of the padding rows [rows_out, rows_pad)
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

// Blocks of 256 threads (no dynamic shared memory) of `kernel` that one SM
// holds at once.
template <typename Kern>
static int resident_blocks_per_sm(Kern kernel) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, 0) != cudaSuccess || n < 1) n = 1;
    return n;
}

// Chunks per warp step: 4 once every SM has at least 128 warp tasks of one
// chunk to share, else 1 (small operands need every warp they can get).
static int quant_unroll(int64_t chunk_tasks, int num_sms) { return chunk_tasks >= (int64_t)num_sms * 128 ? 4 : 1; }

static int quant_grid(int64_t warps_needed, int64_t pad_words, int num_sms) {
    int64_t blocks = (warps_needed + 7) / 8;
    const int64_t pad_blocks = (pad_words + 255) / 256;
    if (pad_blocks > blocks) blocks = pad_blocks;
    const int64_t cap = (int64_t)num_sms * 32;
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

cudaError_t launch_tensor_scale(const void* x, int64_t n, float* alpha, uint32_t* err, cudaStream_t stream,
                                int num_sms) {
    cudaError_t e = cudaMemsetAsync(alpha, 0, sizeof(float), stream);
    if (e != cudaSuccess) return e;
    if (n > 0) {
        // one wave of resident blocks, each thread looping (no partial last wave)
        static const int occ = resident_blocks_per_sm(tensor_amax_kernel);
        int64_t blocks = (n / 8 + 255) / 256;
        if (blocks > (int64_t)num_sms * occ) blocks = (int64_t)num_sms * occ;
        if (blocks < 1) blocks = 1;
        tensor_amax_kernel<<<(int)blocks, 256, 0, stream>>>(static_cast<const uint16_t*>(x), n,
                                                             reinterpret_cast<uint32_t*>(alpha));
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    tensor_scale_finalize_kernel<<<1, 1, 0, stream>>>(alpha, err);
    return cudaGetLastError();
}

template <int FMT, int MODE, int U>
static cudaError_t launch_quant_typed(const QuantArgs& a, int grid, cudaStream_t stream, bool pdl, int num_sms) {
    if (U > 1) {  // large operands: one wave of resident blocks whose warps loop over the tasks
        static const int occ = resident_blocks_per_sm(quantize_kernel<FMT, MODE, U>);
        if (grid > num_sms * occ) grid = num_sms * occ;
    }
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
    return cudaLaunchKernelEx(&cfg, quantize_kernel<FMT, MODE, U>, a);
}

template <int MODE, int U = 1>
static cudaError_t launch_mode(int fmt, const QuantArgs& a, int grid, cudaStream_t stream, bool pdl, int num_sms) {
    return fmt == 0 ? launch_quant_typed<0, MODE, U>(a, grid, stream, pdl, num_sms)
                    : launch_quant_typed<1, MODE, U>(a, grid, stream, pdl, num_sms);
}

cudaError_t launch_quantize(int fmt, bool paired, int rows, int K, const void* x, int64_t ldx, const float* alpha,
                            void* q_out, cudaStream_t stream, int num_sms, bool pdl) {
    QuantArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.ldx = ldx;
    a.rows = rows;
    a.K = K;
    a.alpha = alpha;
    a.err = device_error_word();
    a.rows_out = paired ? 2 * rows : rows;
    a.rows_pad = (a.rows_out + kAtomRows - 1) / kAtomRows * kAtomRows;
    a.task_rows = rows;
    a.n_atoms_k = (K + atom_k(fmt) - 1) / atom_k(fmt);
    a.chunks = (K + 255) / 256;
    a.out = static_cast<uint8_t*>(q_out);
    a.sf = static_cast<uint8_t*>(q_out) + operand_sf_offset(fmt, a.rows_out, K);
    a.early_trigger = pdl ? 1 : 0;
    if (fmt == 0 && K % 512 == 0 && (int64_t)rows * a.chunks >= (int64_t)num_sms * 128) {
        // large NVFP4 operand: one scale block per lane, one wave of resident CTAs
        static const int occ_rows = resident_blocks_per_sm(quantize_nv_wide_kernel<kRows, 2>);
        static const int occ_paired = resident_blocks_per_sm(quantize_nv_wide_kernel<kPaired, 2>);
        const int64_t warps = (int64_t)rows * ((K / 512 + 1) / 2);
        int grid = (int)std::min<int64_t>((warps + 7) / 8, (int64_t)num_sms * (paired ? occ_paired : occ_rows));
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)std::max(grid, 1), 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        return paired ? cudaLaunchKernelEx(&cfg, quantize_nv_wide_kernel<kPaired, 2>, a)
                      : cudaLaunchKernelEx(&cfg, quantize_nv_wide_kernel<kRows, 2>, a);
    }
    const int U = quant_unroll((int64_t)rows * a.chunks, num_sms);
    const int64_t warps = (int64_t)rows * ((a.chunks + U - 1) / U);
    const int64_t pad_words = (int64_t)(a.rows_pad - a.rows_out) * a.n_atoms_k;
    const int grid = quant_grid(warps, pad_words, num_sms);
    if (U == 4)
        return paired ? launch_mode<kPaired, 4>(fmt, a, grid, stream, pdl, num_sms)
                      : launch_mode<kRows, 4>(fmt, a, grid, stream, pdl, num_sms);
    return paired ? launch_mode<kPaired>(fmt, a, grid, stream, pdl, num_sms)
                  : launch_mode<kRows>(fmt, a, grid, stream, pdl, num_sms);
}

cudaError_t launch_quantize_weight(int fmt, int N, int K, const void* w, int64_t ldw, const float* alpha,
                                   void* wq_out, cudaStream_t stream, int num_sms, int kext_k,
                                   const uint8_t* kext_mask) {
    QuantArgs a{};
    if (kext_k > 0) {  // extended weight [W | W[:, S]] with K_eff columns
        a.k_base = K;
        a.kext_k = kext_k;
        a.kext_mask = kext_mask;
        K = K + K / 8 * kext_k;
    }
    a.x = static_cast<const uint16_t*>(w);
    a.ldx = ldw;
    a.rows = N;
    a.K = K;
    a.alpha = alpha;
    a.err = device_error_word();
    a.task_rows = (N + 127) / 128 * 128;  // padding rows quantize as zeros
    a.n_atoms_k = (K + atom_k(fmt) - 1) / atom_k(fmt);
    a.chunks = (K + 255) / 256;
    a.out = static_cast<uint8_t*>(wq_out);
    const int64_t warps = (int64_t)a.task_rows * a.chunks;
    const int grid = quant_grid(warps, 0, num_sms);
    return launch_mode<kWeight>(fmt, a, grid, stream, false, num_sms);
}

}  // namespace rs
