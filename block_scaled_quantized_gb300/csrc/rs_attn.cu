// Residue-compensated decode attention (ResAttn; ResServe Sec. 4.3, Fig. 3,
// Sec. 5.2) over a paged NVFP4 KV cache.
//
// Cache layout: page p of KV head h holds 32 tokens: codes [32][D/2] then
// E4M3 scales [32][D/16], tensor scale 1.0; page bytes = 32 (D/2 + D/16).
// A block table [B][max_pages] (int32) maps a sequence's logical pages.
//
// One CTA per (split, KV head, sequence); tiles of 128 tokens (4 pages):
//   * QK on the tensor cores: kind::mxf4nvf4, A = the key tile (M = 128
//     tokens, K-major 128-byte-swizzled rows; D = 128 uses two 64-element
//     k-steps), B = the group's 2G <= 16 query rows (base 2g, residue 2g+1,
//     from the paired quantizer), accumulator 128 x 16 fp32;
//   * fold, online softmax: thread t of warps 0-3 reads token t's 2G scores,
//     s_g = fl(fl(z_2g + z_2g+1) c), the tile maximum per head through warp
//     shuffles and shared memory, p = exp(s - m), rounded to E4M3;
//   * V: NVFP4 -> E4M3 (R17) into shared memory as fp16 (exact), then
//     O[g][d] = O[g][d] a_g + sum_t p8[g][t] v8[t][d] in fp32 (the products
//     are exact); the normalizer sums the rounded weights (R18);
//   * the split's o, m, l go to a workspace; a second kernel combines the
//     splits (R19) and writes bf16 or fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "rs_device.cuh"
#include "rs_internal.h"
#include "rs_quant_core.cuh"

namespace rs {

constexpr int kAttnThreads = 256;
constexpr int kAttnTile = 128;
constexpr int kPage = 32;


__host__ __device__ constexpr int page_bytes(int D) { return kPage * (D / 2 + D / 16); }

// Tokens of sequence b the kernels attend to: its length, clamped to
// [0, max_len] (a longer one is reported in the device error word, so that
// no block-table entry beyond max_len is ever read).
__device__ __forceinline__ int attn_len(const AttnArgs& g, int b) {
    const int L = g.seq_lens[b];
    if (L > g.max_len && threadIdx.x == 0 && blockIdx.x == 0) atomicExch(g.err, kErrInvalidArg);
    return L < 0 ? 0 : (L > g.max_len ? g.max_len : L);
}

// E4M3 value of an fp32 value (nearest-even, saturating, sign kept) as float.
__device__ __forceinline__ float e4m3_round(float p) { return e4m3_decode_hw(e4m3x2_encode_hw(0.0f, p) & 0xFFu); }

// Dynamic shared memory of one CTA.
__host__ __device__ constexpr size_t attn_smem_bytes(int D) {
    return 1024 + kAttnTile * 128 + 16 * 128 + 2 * (D / 64) * 512 + (size_t)kAttnTile * D * 2 + 8 * kAttnTile * 4 +
           4 * 8 * 4 + 3 * 8 * 4 + 64;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) resattn_split_kernel(const AttnArgs g) {
    constexpr int CB = D / 2, SB = D / 16;          // code / scale bytes per token row
    constexpr int NKS = D / 64;                     // 64-element k-steps
    constexpr int NA = D / 64;                      // scale atoms (4 blocks each) per row
    constexpr int HPT = 8 * D / kAttnThreads;       // heads per PV thread (4 at D = 128, 8 at D = 256)
    constexpr uint32_t TCOLS = D == 128 ? 32 : 64;  // accumulator 16 + scale atoms 2 x 4 NA
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ktile = sm;                                         // 128 SW128 rows, D/2 bytes used
    uint8_t* qtile = ktile + kAttnTile * 128;                    // 16 SW128 rows
    uint8_t* ksf = qtile + 16 * 128;                             // NA key scale atoms
    uint8_t* qsf = ksf + NA * 512;                               // NA query scale atoms
    __half* vt = reinterpret_cast<__half*>(qsf + NA * 512);      // V8 values [token][d]
    float (*pw)[kAttnTile] = reinterpret_cast<float (*)[kAttnTile]>(vt + kAttnTile * D);  // p8 [head][token]
    float (*red)[8] = reinterpret_cast<float (*)[8]>(&pw[8][0]);
    float* m_run = &red[4][0];
    float* l_run = m_run + 8;
    float* a_fac = l_run + 8;
    uint64_t* mma_done = reinterpret_cast<uint64_t*>(a_fac + 8);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = g.Hq / g.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = attn_len(g, b);
    const int t0 = split * g.split_tokens, t1 = min(L, t0 + g.split_tokens);
    float* part = g.part + (((size_t)b * g.Hkv + h) * g.splits + split) * (size_t)G * (D + 2);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(mma_done), 1);
        *abort_flag = 0u;
        fence_mbarrier_init();
    }
    if (threadIdx.x < 8) {
        m_run[threadIdx.x] = -INFINITY;
        l_run[threadIdx.x] = 0.0f;
    }
    // the group's 2G query rows (zero rows up to 16) and their scale bytes
    for (int i = threadIdx.x; i < 16 * 8; i += kAttnThreads) {  // 16 rows x 8 chunks of 16 bytes
        const int r = i / 8, c = i % 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        const int row = 2 * (b * g.Hq + h * G) + r;
        if (r < 2 * G && c * 16 < CB) v = *reinterpret_cast<const uint4*>(g.q_op + (size_t)row * CB + c * 16);
        *reinterpret_cast<uint4*>(qtile + sw128_offset((uint32_t)r, (uint32_t)c * 16u)) = v;
    }
    for (int i = threadIdx.x; i < NA * 512; i += kAttnThreads) qsf[i] = 0;
    __syncthreads();
    {
        const uint8_t* qsf_src = g.q_sf;
        for (int i = threadIdx.x; i < 2 * G * SB; i += kAttnThreads) {
            const int r = i / SB, blk = i % SB;
            const int row = 2 * (b * g.Hq + h * G) + r;
            qsf[(blk / 4) * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + blk % 4] =
                qsf_src[sf_offset(row, blk, g.q_atoms_k)];
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;                 // accumulator: columns 0-15
    const uint32_t tsfa = tmem + 16, tsfb = tmem + 16 + 4 * NA;
    const float c = __fmul_rn(*g.alpha_q, __frsqrt_rn((float)D));  // alpha_q / sqrt(D), alpha_k = 1
    float o[HPT];                                      // thread: d = tid % D, heads og0 .. og0 + HPT - 1
#pragma unroll
    for (int q = 0; q < HPT; ++q) o[q] = 0.0f;
    const int od = threadIdx.x % D, og0 = (threadIdx.x / D) * HPT;
    uint32_t ph = 0;

    for (int u0 = t0; *abort_flag == 0u && u0 < t1; u0 += kAttnTile) {
        const int nt = min(kAttnTile, t1 - u0);
        // K tile: codes into the swizzled rows, scales into the atoms
        for (int i = threadIdx.x; i < kAttnTile * (CB / 16); i += kAttnThreads) {
            const int r = i / (CB / 16), cc = i % (CB / 16);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < nt) {
                const int t = u0 + r;
                const int page = g.block_table[(size_t)b * g.max_pages + t / kPage];
                const uint8_t* pg = g.k_cache + ((size_t)page * g.Hkv + h) * page_bytes(D);
                v = *reinterpret_cast<const uint4*>(pg + (size_t)(t % kPage) * CB + cc * 16);
            }
            *reinterpret_cast<uint4*>(ktile + sw128_offset((uint32_t)r, (uint32_t)cc * 16u)) = v;
        }
        for (int i = threadIdx.x; i < kAttnTile * NA; i += kAttnThreads) {
            const int r = i / NA, a = i % NA;
            uint32_t w = 0u;
            if (r < nt) {
                const int t = u0 + r;
                const int page = g.block_table[(size_t)b * g.max_pages + t / kPage];
                const uint8_t* pg = g.k_cache + ((size_t)page * g.Hkv + h) * page_bytes(D) + kPage * CB;
                w = *reinterpret_cast<const uint32_t*>(pg + (size_t)(t % kPage) * SB + a * 4);
            }
            *reinterpret_cast<uint32_t*>(ksf + a * 512 + (r % 32) * 16 + (r / 32) * 4) = w;
        }
        // V tile -> E4M3 values (as fp16, exact) in [token][d]
        for (int i = threadIdx.x; i < kAttnTile * SB; i += kAttnThreads) {
            const int r = i / SB, blk = i % SB;
            __half hv[16];
            if (r < nt) {
                const int t = u0 + r;
                const int page = g.block_table[(size_t)b * g.max_pages + t / kPage];
                const uint8_t* pg = g.v_cache + ((size_t)page * g.Hkv + h) * page_bytes(D);
                const uint2 cw = *reinterpret_cast<const uint2*>(pg + (size_t)(t % kPage) * CB + blk * 8);
                const float s = e4m3_decode_hw(pg[kPage * CB + (t % kPage) * SB + blk]);
                float d8[8];
                e2m1_decode8(cw.x, d8);
#pragma unroll
                for (int e = 0; e < 8; ++e) hv[e] = __float2half_rn(e4m3_round(__fmul_rn(s, d8[e])));
                e2m1_decode8(cw.y, d8);
#pragma unroll
                for (int e = 0; e < 8; ++e) hv[8 + e] = __float2half_rn(e4m3_round(__fmul_rn(s, d8[e])));
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) hv[e] = __float2half_rn(0.0f);
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) vt[r * D + blk * 16 + e] = hv[e];
        }
        fence_proxy_async_smem();
        __syncthreads();

        // QK: base and residue scores of the group against the tile
        if (warp == 1) {
            tc_fence_after();
            if (elect_one_sync()) {
                const uint64_t ad = kmajor_sw128_desc(smem_u32(ktile)), bd = kmajor_sw128_desc(smem_u32(qtile));
                for (int a = 0; a < NA; ++a) {
                    tc_cp_sf_atom(tsfa + a * 4, sf_atom_desc(smem_u32(ksf + a * 512)));
                    tc_cp_sf_atom(tsfb + a * 4, sf_atom_desc(smem_u32(qsf + a * 512)));
                }
                for (int ks = 0; ks < NKS; ++ks)
                    mma_nvfp4(tmem, ad + (uint32_t)ks * 2u, bd + (uint32_t)ks * 2u, mxf4_idesc(16, false, 0),
                              tsfa + ks * 4, tsfb + ks * 4, ks > 0 ? 1u : 0u);
                tc_commit(smem_u32(mma_done));
            }
            __syncwarp();
        }
        // fold, tile maximum, weights (warps 0-3: token = thread)
        float sc[8];
        if (warp < 4) {
            const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(mma_done), ph, abort_flag, g.err));
            tc_fence_after();
            float z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0.0f;
            if (ok) tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16), z);
            const int r = threadIdx.x;
#pragma unroll
            for (int gg = 0; gg < 8; ++gg) {
                sc[gg] = (gg < G && r < nt) ? __fmul_rn(__fadd_rn(z[2 * gg], z[2 * gg + 1]), c) : -INFINITY;
                float mx = sc[gg];
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o2));
                if (lane == 0) red[warp][gg] = mx;
            }
        }
        ph ^= 1u;
        __syncthreads();
        if (threadIdx.x < 8) {
            const int gg = threadIdx.x;
            const float tm = fmaxf(fmaxf(red[0][gg], red[1][gg]), fmaxf(red[2][gg], red[3][gg]));
            const float mn = fmaxf(m_run[gg], tm);
            a_fac[gg] = m_run[gg] == -INFINITY ? 0.0f : __expf(m_run[gg] - mn);
            m_run[gg] = mn;
        }
        __syncthreads();
        if (warp < 4) {
            const int r = threadIdx.x;
#pragma unroll
            for (int gg = 0; gg < 8; ++gg) {
                const float p8 = (gg < G && r < nt) ? e4m3_round(__expf(sc[gg] - m_run[gg])) : 0.0f;
                pw[gg][r] = p8;
                float sm = p8;
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) sm += __shfl_xor_sync(0xFFFFFFFFu, sm, o2);
                if (lane == 0) red[warp][gg] = sm;
            }
        }
        __syncthreads();
        if (threadIdx.x < 8) {
            const int gg = threadIdx.x;
            l_run[gg] = l_run[gg] * a_fac[gg] + ((red[0][gg] + red[1][gg]) + (red[2][gg] + red[3][gg]));
        }
        // PV: thread (d, 4 heads), exact fp32 products of E4M3 values
        __syncthreads();  // l_run and a_fac are final for this tile
#pragma unroll
        for (int q = 0; q < HPT; ++q) o[q] *= a_fac[og0 + q];
        for (int t = 0; t < nt; ++t) {
            const float v = __half2float(vt[t * D + od]);
#pragma unroll
            for (int q = 0; q < HPT; ++q) o[q] = fmaf(pw[og0 + q][t], v, o[q]);
        }
        __syncthreads();
    }

    // this split's o, m, l
#pragma unroll
    for (int q = 0; q < HPT; ++q)
        if (og0 + q < G) part[(size_t)(og0 + q) * (D + 2) + od] = o[q];
    if (threadIdx.x < G) {
        part[(size_t)threadIdx.x * (D + 2) + D] = m_run[threadIdx.x];
        part[(size_t)threadIdx.x * (D + 2) + D + 1] = l_run[threadIdx.x];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TCOLS);
}

// O = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s (R19); empty sequences give 0.
__global__ void resattn_combine_kernel(const AttnArgs g, void* out, int out_f32) {
    const int B = g.B, Hq = g.Hq, Hkv = g.Hkv, D = g.D, splits = g.splits, split_tokens = g.split_tokens;
    const float* part = g.part;
    (void)B;
    const int G = Hq / Hkv;
    const int b = blockIdx.y, hq = blockIdx.x, d = threadIdx.x;
    if (d >= D) return;
    const int h = hq / G, gg = hq % G;
    const int L = attn_len(g, b);
    const int ns = min(splits, (L + split_tokens - 1) / split_tokens);
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s)
        M = fmaxf(M, part[((((size_t)b * Hkv + h) * splits + s) * G + gg) * (D + 2) + D]);
    float num = 0.0f, den = 0.0f;
    for (int s = 0; s < ns; ++s) {
        const float* p = part + ((((size_t)b * Hkv + h) * splits + s) * G + gg) * (D + 2);
        const float w = __expf(p[D] - M);
        num = fmaf(w, p[d], num);
        den = fmaf(w, p[D + 1], den);
    }
    const float val = ns > 0 ? num / den : 0.0f;
    const size_t idx = ((size_t)b * Hq + hq) * D + d;
    if (out_f32) reinterpret_cast<float*>(out)[idx] = val;
    else reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(val);
}

// ---------------------------------------------------------------- launch --

// Splits: enough (split, KV head, sequence) CTAs for every SM, in multiples
// of the tile, at least one tile per split (the preset rule of Sec. 5.2 from
// batch, KV heads, sequence length and SM count).
int resattn_split_tokens(int B, int Hkv, int max_len, int num_sms) {
    const int tiles = (max_len + kAttnTile - 1) / kAttnTile;
    int splits = (num_sms + B * Hkv - 1) / (B * Hkv);
    if (splits > tiles) splits = tiles;
    if (splits < 1) splits = 1;
    const int tiles_per_split = (tiles + splits - 1) / splits;
    return (tiles_per_split < 1 ? 1 : tiles_per_split) * kAttnTile;
}

cudaError_t launch_resattn(int D, const AttnArgs& a, void* out, int out_f32, cudaStream_t stream) {
    const size_t smem = attn_smem_bytes(D);
    dim3 grid((unsigned)a.splits, (unsigned)a.Hkv, (unsigned)a.B);
    cudaError_t e;
    if (D == 128) {
        e = cudaFuncSetAttribute(resattn_split_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) resattn_split_kernel<128><<<grid, kAttnThreads, smem, stream>>>(a);
    } else if (D == 256) {
        e = cudaFuncSetAttribute(resattn_split_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) resattn_split_kernel<256><<<grid, kAttnThreads, smem, stream>>>(a);
    } else {
        return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    resattn_combine_kernel<<<dim3((unsigned)a.Hq, (unsigned)a.B), D, 0, stream>>>(a, out, out_f32);
    return cudaGetLastError();
}

}  // namespace rs
