// Selective prefill compensation, K-Ext (ResServe Sec. 5.3 Eq. 6, App. A
// Eq. 7, App. B.2 Alg. 1 for the partial residues): the quantizer that
// writes the extended activation operand [X^ | R^_S] of K_eff = K + K k / 8
// columns in the rs operand layout, so that the block-scaled GEMM over K_eff
// adds the base and the selected-residue products in one accumulator.
//
// One warp takes one token row x 256 channels; lane l holds channels
// 8l .. 8l+7 of the chunk, which are exactly one 8-channel selection group
// (Eq. 7), so its byte of the mask says which of its residues are kept.
// Base: as the plain quantizer (two lanes per 16-element block).  Residues
// r = fl(x - x^) of the k selected channels, in increasing channel order,
// are extension elements g k .. g k + k - 1 (g = group index); a block of
// 16 (NVFP4) / 32 (MXFP4) extension elements spans 16/k (32/k) consecutive
// lanes, whose block amax is a shuffle reduction; the block scale uses the
// base operand's tensor scale.
#include <cuda_bf16.h>

#include "rs_device.cuh"
#include "rs_internal.h"
#include "rs_quant_core.cuh"

namespace rs {

struct KextArgs {
    const uint16_t* x;      // bf16 [rows][ldx]
    int64_t ldx;
    int rows, K;            // K: base channels (a multiple of 256)
    const float* alpha;     // NVFP4 tensor scale (device)
    const uint8_t* mask;    // [K/8] selection bytes (device), k bits set each
    uint8_t* out;           // operand base (codes [rows][K_eff/2])
    uint8_t* sf;            // its scale atoms
    int rows_pad;           // rows rounded up to 128
    int n_atoms_k;          // scale atoms per row tile along K_eff
    int early_trigger;      // release the dependent grid once the prior grid is done
    uint32_t* err;
};

// U > 1: a warp takes U consecutive chunks of one row per step and issues
// their loads before quantizing any of them (large operands).
template <int FMT, int KS, int U>
__global__ void __launch_bounds__(256, U > 1 ? 3 : 1) kext_quantize_kernel(KextArgs a) {
    pdl_wait_prior_grid();
    if (a.early_trigger) pdl_launch_dependents();
    constexpr int BS = block_elems(FMT);
    constexpr int L = BS / KS;               // lanes per extension block
    constexpr int LPA = lanes_per_atom<FMT>();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps_total = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int chunks = a.K / 256;
    const int n_cg = (chunks + U - 1) / U;
    const int64_t tasks = (int64_t)a.rows * n_cg;
    const int Ke = a.K + a.K / 8 * KS;
    const NvScaleConst ksc = nv_scale_const(FMT == 0 ? *a.alpha : 0.0f);
    if (FMT == 0 && blockIdx.x == 0 && threadIdx.x == 0 && !nv_alpha_supported(ksc.alpha))
        atomicExch(a.err, kErrInvalidArg);

    for (int64_t task = warp; task < tasks; task += n_warps_total) {
        const int row = (int)(task / n_cg);
        const int cg = (int)(task - (int64_t)row * n_cg);
        uint4 raw[U];  // the U input words, widened when processed
#pragma unroll
        for (int u = 0; u < U; ++u)
            raw[u] = load16_or_zero(a.x + (int64_t)row * a.ldx + (cg * U + u) * 256 + lane * 8, cg * U + u < chunks);
        uint8_t* orow = a.out + (size_t)row * (size_t)(Ke / 2);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int chunk = cg * U + u;
            if (U > 1 && chunk >= chunks) break;  // ragged last group (warp-uniform)
            const int k0 = chunk * 256 + lane * 8;
            float xf[8];
            unpack8_bf16(raw[u], xf);

            // base operand (Eq. 8-10)
            uint32_t sfb;
            float xh[8];
            const uint32_t codes = quant_lane<FMT, true>(xf, ksc, sfb, xh);
            const uint32_t sfw = gather_sf_word<FMT>(sfb, lane);
            *reinterpret_cast<uint32_t*>(orow + k0 / 2) = codes;
            if (lane % LPA == 0)
                *reinterpret_cast<uint32_t*>(a.sf + sf_offset(row, (chunk * (256 / atom_k(FMT)) + lane / LPA) * kAtomBlocks,
                                                              a.n_atoms_k)) = sfw;

            // the group's selected residues, in channel order (Alg. 1 lines 6-7)
            float r[8];
            residue8(xf, xh, r);
            const int grp = chunk * 32 + lane;
            const uint32_t m = a.mask[grp];
            if (__popc(m) != KS) atomicExch(a.err, kErrInvalidArg);  // a mask must keep k channels per group
            float sel[KS];
    #pragma unroll
            for (int j = 0; j < KS; ++j) {
                const uint32_t idx = __fns(m, 0, j + 1);  // position of the (j+1)-th set bit
                float v = 0.0f;
    #pragma unroll
                for (int t = 0; t < 8; ++t) v = idx == (uint32_t)t ? r[t] : v;
                sel[j] = v;
            }
            // block amax over the L lanes of this extension block (lines 8-9)
            float am = 0.0f;
    #pragma unroll
            for (int j = 0; j < KS; ++j) am = fmaxf(am, fabsf(sel[j]));
    #pragma unroll
            for (int o = 1; o < L; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
            float st, mul;
            const uint32_t sfr = FMT == 0 ? nv_block_scale_fast(am, ksc, st, mul) : mx_block_scale(am, st, mul);
            float v8[8];
    #pragma unroll
            for (int e = 0; e < 8; ++e) v8[e] = e < KS ? __fmul_rn(sel[e], mul) : 0.0f;
            const uint32_t rc = e2m1_encode8(v8);  // element j in nibble j
            const int c = a.K + grp * KS;          // K_eff column of this lane's first extension element
            if constexpr (KS == 8) {
                *reinterpret_cast<uint32_t*>(orow + c / 2) = rc;
            } else if constexpr (KS == 4) {
                *reinterpret_cast<uint16_t*>(orow + c / 2) = (uint16_t)(rc & 0xFFFFu);
            } else if constexpr (KS == 2) {
                orow[c / 2] = (uint8_t)(rc & 0xFFu);
            } else {
                const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, rc & 0xFu, 1);
                if ((lane & 1) == 0) orow[c / 2] = (uint8_t)((rc & 0xFu) | (hi << 4));
            }
            if (lane % L == 0) a.sf[sf_offset(row, c / BS, a.n_atoms_k)] = (uint8_t)sfr;
            // padding blocks of the row's last, partly filled scale atom
            const int nb = Ke / BS;
            if (chunk == chunks - 1 && lane < a.n_atoms_k * kAtomBlocks - nb)
                a.sf[sf_offset(row, nb + lane, a.n_atoms_k)] = 0;
        }
    }

    // zero scale words of the padding rows [rows, rows_pad)
    const int64_t pad_words = (int64_t)(a.rows_pad - a.rows) * a.n_atoms_k;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = tid; i < pad_words; i += nthreads) {
        const int rr = a.rows + (int)(i / a.n_atoms_k);
        const int gg = (int)(i % a.n_atoms_k);
        *reinterpret_cast<uint32_t*>(a.sf + sf_offset(rr, gg * kAtomBlocks, a.n_atoms_k)) = 0u;
    }
}

// Large NVFP4 operands (K a multiple of 512): lane l takes the 16-element
// base block 16l..16l+15 of a 512-element chunk, i.e. two selection groups.
// The block scale is derived once per block (packed-bf16 amax, s~ and
// fl(1/s~) from a per-CTA table of the 127 finite E4M3 bytes); the lane's
// 2k selected residues are consecutive extension elements, so an extension
// block of 16 spans L = 8/k lanes.  Same arithmetic per element as
// kext_quantize_kernel; U chunks per warp step, loads first; one wave of
// resident CTAs.
template <int KS, int U>
__global__ void __launch_bounds__(256, 3) kext_quantize_nv_wide_kernel(KextArgs a) {
    __shared__ float tab_st[128], tab_mul[128];
    pdl_wait_prior_grid();
    if (a.early_trigger) pdl_launch_dependents();
    constexpr int L = 8 / KS;  // lanes per extension block
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
    const int Ke = a.K + a.K / 8 * KS;
    const int nb = Ke / 16;  // scale blocks per row along K_eff
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
        uint8_t* orow = a.out + (size_t)row * (size_t)(Ke / 2);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int chunk = cg * U + u;
            if (U > 1 && chunk >= chunks) break;  // ragged last group (warp-uniform)
            // base block (Eq. 8-10)
            const uint32_t w[8] = {raw[u][0].x, raw[u][0].y, raw[u][0].z, raw[u][0].w,
                                   raw[u][1].x, raw[u][1].y, raw[u][1].z, raw[u][1].w};
            const uint32_t sf = nv_block_byte(amax16_bf16(w), ksc);
            const float st = tab_st[sf], mul = tab_mul[sf];
            float xf[16];
            unpack8_bf16(raw[u][0], *reinterpret_cast<float(*)[8]>(&xf[0]));
            unpack8_bf16(raw[u][1], *reinterpret_cast<float(*)[8]>(&xf[8]));
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; e += 2) fmul2_rn(xf[e], xf[e + 1], mul, mul, v[e], v[e + 1]);
            const uint32_t c0 = e2m1_encode8(*reinterpret_cast<const float(*)[8]>(&v[0]));
            const uint32_t c1 = e2m1_encode8(*reinterpret_cast<const float(*)[8]>(&v[8]));
            const uint32_t t = sf | (__shfl_down_sync(0xFFFFFFFFu, sf, 1) << 8);
            const uint32_t sfw = t | (__shfl_down_sync(0xFFFFFFFFu, t, 2) << 16);
            *reinterpret_cast<uint2*>(orow + (size_t)chunk * 256 + (size_t)lane * 8) = make_uint2(c0, c1);
            if ((lane & 3) == 0)
                *reinterpret_cast<uint32_t*>(a.sf + sf_offset(row, chunk * 32 + lane, a.n_atoms_k)) = sfw;

            // residues r = fl(x - fl(s~ dec(q))) (never fused), the selected
            // ones of the lane's two groups in channel order (Alg. 1 lines 6-7)
            float d[16];
            e2m1_decode8(c0, *reinterpret_cast<float(*)[8]>(&d[0]));
            e2m1_decode8(c1, *reinterpret_cast<float(*)[8]>(&d[8]));
            const int grp0 = chunk * 64 + 2 * lane;
            float sel[2 * KS];
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                float r[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) r[e] = __fsub_rn(xf[8 * g + e], __fmul_rn(st, d[8 * g + e]));
                const uint32_t m = a.mask[grp0 + g];
                if (__popc(m) != KS) atomicExch(a.err, kErrInvalidArg);  // a mask must keep k channels per group
#pragma unroll
                for (int j = 0; j < KS; ++j) {
                    const uint32_t idx = __fns(m, 0, j + 1);  // position of the (j+1)-th set bit
                    float sv = 0.0f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) sv = idx == (uint32_t)e ? r[e] : sv;
                    sel[g * KS + j] = sv;
                }
            }
            // extension block amax over its L lanes (lines 8-9)
            float am = 0.0f;
#pragma unroll
            for (int j = 0; j < 2 * KS; ++j) am = fmaxf(am, fabsf(sel[j]));
#pragma unroll
            for (int o = 1; o < L; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
            const uint32_t sfr = nv_block_byte(am, ksc);
            const float mulr = tab_mul[sfr];
            float vr[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) vr[e] = e < 2 * KS ? __fmul_rn(sel[e < 2 * KS ? e : 0], mulr) : 0.0f;
            const uint32_t r0 = e2m1_encode8(*reinterpret_cast<const float(*)[8]>(&vr[0]));
            const int c = a.K + grp0 * KS;  // K_eff column of the lane's first extension element
            if constexpr (KS == 8) {
                const uint32_t r1 = e2m1_encode8(*reinterpret_cast<const float(*)[8]>(&vr[8]));
                *reinterpret_cast<uint2*>(orow + c / 2) = make_uint2(r0, r1);
            } else if constexpr (KS == 4) {
                *reinterpret_cast<uint32_t*>(orow + c / 2) = r0;
            } else if constexpr (KS == 2) {
                *reinterpret_cast<uint16_t*>(orow + c / 2) = (uint16_t)(r0 & 0xFFFFu);
            } else {
                orow[c / 2] = (uint8_t)(r0 & 0xFFu);
            }
            if (lane % L == 0) a.sf[sf_offset(row, c / 16, a.n_atoms_k)] = (uint8_t)sfr;
            // padding blocks of the row's last, partly filled scale atom
            if (chunk == chunks - 1 && lane < a.n_atoms_k * kAtomBlocks - nb)
                a.sf[sf_offset(row, nb + lane, a.n_atoms_k)] = 0;
        }
    }

    // zero scale words of the padding rows [rows, rows_pad)
    const int64_t pad_words = (int64_t)(a.rows_pad - a.rows) * a.n_atoms_k;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = tid; i < pad_words; i += nthreads) {
        const int rr = a.rows + (int)(i / a.n_atoms_k);
        const int gg = (int)(i % a.n_atoms_k);
        *reinterpret_cast<uint32_t*>(a.sf + sf_offset(rr, gg * kAtomBlocks, a.n_atoms_k)) = 0u;
    }
}

// Calibration score of Eq. 7: mean |x| of every channel over `rows` rows,
// one thread per channel summing in row order (deterministic).
__global__ void channel_mean_abs_kernel(const uint16_t* __restrict__ x, int rows, int K, int64_t ldx,
                                        float* __restrict__ score) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= K) return;
    float s = 0.0f;
    for (int r = 0; r < rows; ++r) s += fabsf(__uint_as_float((uint32_t)x[(int64_t)r * ldx + c] << 16));
    score[c] = rows > 0 ? s / (float)rows : 0.0f;
}

template <int FMT, int KS, int U>
static cudaError_t launch_kext_typed(const KextArgs& a, int grid, cudaStream_t stream, bool pdl, int num_sms) {
    if (U > 1) {  // large operands: one wave of resident blocks whose warps loop over the tasks
        static const int occ = [] {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kext_quantize_kernel<FMT, KS, U>, 256, 0) !=
                    cudaSuccess || n < 1)
                n = 1;
            return n;
        }();
        if (grid > num_sms * occ) grid = num_sms * occ;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kext_quantize_kernel<FMT, KS, U>, a);
}

cudaError_t launch_quantize_kext(int fmt, int k, int rows, int K, const void* x, int64_t ldx, const float* alpha,
                                 const uint8_t* mask, void* q_out, cudaStream_t stream, int num_sms, bool pdl) {
    const int Ke = K + K / 8 * k;
    KextArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.ldx = ldx;
    a.rows = rows;
    a.K = K;
    a.alpha = alpha;
    a.mask = mask;
    a.out = static_cast<uint8_t*>(q_out);
    a.sf = static_cast<uint8_t*>(q_out) + operand_sf_offset(fmt, rows, Ke);
    a.rows_pad = (rows + kAtomRows - 1) / kAtomRows * kAtomRows;
    a.n_atoms_k = n_atoms_k_host(fmt, Ke);
    a.early_trigger = pdl ? 1 : 0;
    a.err = device_error_word();
    if (fmt == 0 && K % 512 == 0 && (int64_t)rows * (K / 256) >= (int64_t)num_sms * 128) {
        // large NVFP4 operand: one base block per lane
        const int64_t wwarps = (int64_t)rows * ((K / 512 + 1) / 2);
        cudaLaunchConfig_t cfg{};
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
#define RS_KEXT_WIDE(S)                                                                                      \
    if (k == S) {                                                                                            \
        static const int occ = [] {                                                                          \
            int n = 0;                                                                                       \
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kext_quantize_nv_wide_kernel<S, 2>, 256, 0) != \
                    cudaSuccess || n < 1)                                                                    \
                n = 1;                                                                                       \
            return n;                                                                                        \
        }();                                                                                                 \
        int64_t g = (wwarps + 7) / 8;                                                                        \
        if (g > (int64_t)num_sms * occ) g = (int64_t)num_sms * occ;                                          \
        cfg.gridDim = dim3((unsigned)(g < 1 ? 1 : g), 1, 1);                                                 \
        return cudaLaunchKernelEx(&cfg, kext_quantize_nv_wide_kernel<S, 2>, a);                              \
    }
        RS_KEXT_WIDE(1) RS_KEXT_WIDE(2) RS_KEXT_WIDE(4) RS_KEXT_WIDE(8)
#undef RS_KEXT_WIDE
        return cudaErrorInvalidValue;
    }
    // chunks per warp step: 4 once every SM has 128 single-chunk warp tasks
    const int U = (int64_t)rows * (K / 256) >= (int64_t)num_sms * 128 ? 4 : 1;
    const int64_t warps = (int64_t)rows * ((K / 256 + U - 1) / U);
    int64_t blocks = (warps + 7) / 8;
    const int64_t pad_blocks = ((int64_t)(a.rows_pad - rows) * a.n_atoms_k + 255) / 256;
    if (pad_blocks > blocks) blocks = pad_blocks;
    if (blocks > (int64_t)num_sms * 32) blocks = (int64_t)num_sms * 32;
    const int grid = (int)(blocks < 1 ? 1 : blocks);
#define RS_KEXT(F, S) \
    if (fmt == F && k == S)   \
        return U == 4 ? launch_kext_typed<F, S, 4>(a, grid, stream, pdl, num_sms) \
                      : launch_kext_typed<F, S, 1>(a, grid, stream, pdl, num_sms);
    RS_KEXT(0, 1) RS_KEXT(0, 2) RS_KEXT(0, 4) RS_KEXT(0, 8)
    RS_KEXT(1, 1) RS_KEXT(1, 2) RS_KEXT(1, 4) RS_KEXT(1, 8)
#undef RS_KEXT
    return cudaErrorInvalidValue;
}

cudaError_t launch_channel_mean_abs(const void* x, int rows, int K, int64_t ldx, float* score, cudaStream_t stream) {
    channel_mean_abs_kernel<<<(K + 255) / 256, 256, 0, stream>>>(static_cast<const uint16_t*>(x), rows, K, ldx, score);
    return cudaGetLastError();
}

}  // namespace rs
