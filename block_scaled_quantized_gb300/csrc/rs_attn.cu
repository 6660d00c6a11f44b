// Residue-compensated decode attention (ResAttn; ResServe Sec. 4.3, Fig. 3,
// Sec. 5.2) over a paged NVFP4 KV cache.
//
// Cache layout: page p of KV head h holds 32 tokens: codes [32][D/2] then
// E4M3 scales [32][D/16], tensor scale 1.0; page bytes = 32 (D/2 + D/16).
// A block table [B][max_pages] (int32) maps a sequence's logical pages.
//
// One CTA per (split, KV head, sequence); tiles of 128 tokens (four pages):
//   * warp 0 streams the tile's K and V pages with bulk copies into a ring
//     of stages, ahead of the compute (pages taken from the block table);
//   * the group's G query rows are quantized in the kernel (Alg. 1: base and
//     residue rows with the call's tensor scale), straight into the QK operand;
//   * warps 1-7 rearrange a landed stage in shared memory: K codes into the
//     128-byte-swizzled rows of the MMA operand, K scales into atoms, and V
//     from NVFP4 to E4M3 (each dequantized element rounded to nearest-even,
//     saturating) in its own token-major order (128 head dimensions per
//     128-byte-swizzled row);
//   * QK on the tensor cores: kind::mxf4nvf4, A = the key tile (M = 128
//     tokens), B = the group's 2G <= 16 query rows (base 2g, residue 2g+1),
//     accumulator 128 x 16 fp32;
//   * fold and online softmax (warps 4-7, one token per thread):
//     s_g = fl(fl(z_2g + z_2g+1) c), the tile maximum per head, p = exp(s - m)
//     rounded to E4M3 and written as the PV operand P [head][token];
//   * PV on the tensor cores: kind::f8f6f4 (E4M3 x E4M3, fp32 accumulation),
//     A = V^T read as an MN-major operand (M = 128 head dimensions per MMA,
//     contiguous in each token row), B = P (N = 16), K = 128 tokens in four
//     steps of 32 rows; warps 4-7 add the tile's accumulator into their
//     running outputs after rescaling them by exp(m_old - m_new), and the
//     normalizer sums the rounded weights;
//   * the split's o, m, l go to a workspace; a second kernel combines the
//     splits (O = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s) and writes
//     bf16 or fp32.
// Several CTAs share an SM (head size 128), so one CTA's rearranging and
// softmax overlap another's MMAs and copies.  Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "rs_device.cuh"
#include "rs_internal.h"
#include "rs_quant_core.cuh"

namespace rs {

constexpr int kAttnThreads = 256;     // warp 0 copies, warp 1 MMAs, warps 1-7 rearrange, warps 4-7 softmax/PV
constexpr int kAttnCompute = 224;     // warps 1-7
constexpr int kAttnTile = 128;
constexpr int kPage = 32;

__host__ __device__ constexpr int page_bytes(int D) { return kPage * (D / 2 + D / 16); }

// Shared-memory layout of one CTA (offsets from a 1024-byte aligned base).
template <int D>
struct AttnLayout {
    static constexpr int CB = D / 2, SB = D / 16;      // code / scale bytes per token
    static constexpr int NA = D / 64;                  // scale atoms (4 blocks) per token row; = QK k-steps
    static constexpr int PB = page_bytes(D);
    static constexpr int STAGES = D == 128 ? 3 : 2;
    static constexpr uint32_t STG = 8u * (uint32_t)PB;         // four K pages, then four V pages
    static constexpr uint32_t OFF_K = (uint32_t)STAGES * STG;  // key tile: 128 SW128 rows
    static constexpr uint32_t OFF_V = OFF_K + 16384u;          // V (E4M3): per 128 dims, 128 SW128 token rows
    static constexpr uint32_t OFF_Q = OFF_V + (uint32_t)D * 128u;  // query rows: 16 SW128 rows
    static constexpr uint32_t OFF_P = OFF_Q + 2048u;           // P: 16 SW128 rows of 128 tokens
    static constexpr uint32_t OFF_KSF = OFF_P + 2048u;         // key scale atoms
    static constexpr uint32_t OFF_QSF = OFF_KSF + (uint32_t)NA * 512u;
    static constexpr uint32_t OFF_LUT = OFF_QSF + (uint32_t)NA * 512u;  // V: E4M3 of s~ x |E2M1| per scale byte
    static constexpr uint32_t OFF_CTRL = OFF_LUT + 1024u;
    static constexpr size_t SMEM = 1024 + OFF_CTRL + 512;
    // tensor memory: QK accumulator (16 columns), PV accumulators (16 per
    // 128 head dimensions), then the key and query scale atoms
    static constexpr uint32_t T_PV = 16u, T_SFK = T_PV + 16u * (D / 128), T_SFQ = T_SFK + 4u * NA;
    static constexpr uint32_t TCOLS = D == 128 ? 64u : 128u;
    static_assert(STG % 1024 == 0 && OFF_K % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static_assert(T_SFQ + 4u * NA <= TCOLS, "tensor-memory columns");
};

// Instruction descriptor of kind::f8f6f4: A and B E4M3 (format 0), fp32
// accumulator (bit 4), A MN-major (bit 15: M contiguous), B K-major,
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t f8_idesc_amn(int n, int m) {
    return (1u << 4) | (1u << 15) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D[128 x N] (+)= A[128 x 32] * B[N x 32]^T, E4M3 operands, fp32 accumulation.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Tokens of sequence b the kernels attend to: its length, clamped to
// [0, max_len] (a longer one is reported in the device error word, so that
// no block-table entry beyond max_len is ever read).
__device__ __forceinline__ int attn_len(const AttnArgs& g, int b) {
    const int L = g.seq_lens[b];
    if (L > g.max_len && threadIdx.x == 0 && blockIdx.x == 0) atomicExch(g.err, kErrInvalidArg);
    return L < 0 ? 0 : (L > g.max_len ? g.max_len : L);
}

// V from NVFP4 to E4M3 (each dequantized element rounded to nearest-even, saturating).  The E4M3 value of s~ x dec(q) depends only
// on the block's scale byte and the code's magnitude, so each CTA first
// builds lut[byte][m] = E4M3(s~(byte) x |dec(m)|), m = 0..7: the product of an
// E4M3 and an E2M1 value has at most five significant bits and lies within
// [2^-10, 2688], so it is exact in fp16 and its E4M3 rounding (nearest even,
// saturating) is that of the exact product.  A block's sixteen bytes are then
// byte permutations of its table row selected by the code nibbles, with the
// code's sign bit as the E4M3 sign.
__device__ __forceinline__ void build_v_lut(uint8_t* lut, int tid, int nthreads) {
    for (int i = tid; i < 128 * 4; i += nthreads) {
        const uint32_t byte = (uint32_t)(i >> 2), pair = (uint32_t)(i & 3);
        uint32_t s2, p2;
        uint16_t e2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"((uint16_t)(byte | (byte << 8))));
        // |dec(m)| for m = 2 pair, 2 pair + 1 as f16x2 (low half first): {0, .5}, {1, 1.5}, {2, 3}, {4, 6}
        const uint32_t d2 = pair == 0 ? 0x38000000u : pair == 1 ? 0x3E003C00u : pair == 2 ? 0x42004000u : 0x46004400u;
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p2) : "r"(d2), "r"(s2));
        asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(e2) : "r"(p2));
        *reinterpret_cast<uint16_t*>(lut + byte * 8 + pair * 2) = e2;
    }
}

// The sixteen E4M3 bytes of one V block (codes: element e in nibble e;
// row: its scale byte's table row), byte e of the block in byte e % 4 of w[e / 4].
__device__ __forceinline__ void v_block_e4m3(uint2 codes, uint2 row, uint32_t (&w)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t c = ((k < 2 ? codes.x : codes.y) >> (16 * (k & 1))) & 0xFFFFu;
        const uint32_t mag = __byte_perm(row.x, row.y, c & 0x7777u);          // magnitude bytes
        const uint32_t sgn = __byte_perm(0x8000u, 0u, (c >> 3) & 0x1111u);    // 0x00 or 0x80 per byte
        w[k] = mag | sgn;
    }
}

// Warp maximum of a float (NaN-free inputs; -inf allowed) with one redux.sync
// on an order-preserving integer image of its bits.
__device__ __forceinline__ float warp_max_f32(float x) {
    const int i = __float_as_int(x);
    int key = i >= 0 ? i : (i ^ 0x7FFFFFFF);
    key = __reduce_max_sync(0xFFFFFFFFu, key);
    return __int_as_float(key >= 0 ? key : (key ^ 0x7FFFFFFF));
}

// GM: the query heads per KV head the softmax and output loops cover (4 or
// 8, at least G; groups of at most four take the shorter loops).
template <int D, int GM>
__global__ void __launch_bounds__(kAttnThreads, D == 128 ? 2 : 1) resattn_split_kernel(const AttnArgs g) {
    using Ly = AttnLayout<D>;
    constexpr int CB = Ly::CB, SB = Ly::SB, NA = Ly::NA, PB = Ly::PB, S = Ly::STAGES;
    constexpr int MB = D / 128;  // PV MMAs of 128 head dimensions
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stg = sm;
    uint8_t* ktile = sm + Ly::OFF_K;
    uint8_t* vt = sm + Ly::OFF_V;
    uint8_t* qtile = sm + Ly::OFF_Q;
    uint8_t* ptile = sm + Ly::OFF_P;
    uint8_t* ksf = sm + Ly::OFF_KSF;
    uint8_t* qsf = sm + Ly::OFF_QSF;
    uint8_t* vlut = sm + Ly::OFF_LUT;
    if (threadIdx.x == 0) RS_TRACE_MARK(g.trace, 30);  // CTA start
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + Ly::OFF_CTRL);  // [S]: a stage's pages landed
    uint64_t* empty = full + 3;                                       // [S]: a stage was read
    uint64_t* qk_done = empty + 3;                                    // the tile's QK MMAs are done
    uint64_t* pv_done = qk_done + 1;                                  // the tile's PV MMAs are done
    float* red = reinterpret_cast<float*>(pv_done + 1);               // [4][8] tile maxima per warp
    int* red2 = reinterpret_cast<int*>(red + 32);                      // [4][8] weight sums per warp (2^-9 units)
    float* m_run = red + 64;                                          // [8] running maxima
    float* l_run = m_run + 8;                                         // [8] running normalizers
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(l_run + 8);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    volatile uint32_t* issued = tmem_slot + 2;    // tiles whose copies were issued
    volatile uint32_t* consumed = tmem_slot + 3;  // tiles whose stage was released

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = g.Hq / g.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* part = g.part + (((size_t)b * g.Hkv + h) * g.splits + split) * (size_t)G * (D + 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(qk_done), 1);
        mbar_init(smem_u32(pv_done), 1);
        *abort_flag = 0u;
        *issued = 0u;
        *consumed = 0u;
        fence_mbarrier_init();
    }
    if (threadIdx.x < 8) {
        m_run[threadIdx.x] = -INFINITY;
        l_run[threadIdx.x] = 0.0f;
    }
    build_v_lut(vlut, threadIdx.x, kAttnThreads);
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Ly::TCOLS);
        tmem_relinquish();
    }
    // Set-up above overlaps the previous kernel (programmatic launch); the
    // query operand, sequence lengths, block table and cache come after it.
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    const int L = attn_len(g, b);
    const int t0 = split * g.split_tokens, t1 = min(L, t0 + g.split_tokens);
    const int ntiles = t1 > t0 ? (t1 - t0 + kAttnTile - 1) / kAttnTile : 0;
    // The query-quantization step (Sec. 5.2) inside this kernel: the
    // group's G query rows, one 16-element block per thread (Alg. 1: base,
    // then residue with its own block scale and the same tensor scale), into
    // rows 2g (base) and 2g + 1 (residue) of the QK operand and its scale
    // atoms; every other byte zero (rows up to 16, head dimensions up to the
    // 256-element chunk), P all zero (rows >= G stay zero).
    for (int i = threadIdx.x; i < 16 * 8; i += kAttnThreads) {
        *reinterpret_cast<uint4*>(qtile + (size_t)i * 16) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(ptile + (size_t)i * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int i = threadIdx.x; i < NA * 128; i += kAttnThreads) reinterpret_cast<uint32_t*>(qsf)[i] = 0u;
    __syncthreads();
    {
        const NvScaleConst qsc = nv_scale_const(*g.alpha_q);
        if (threadIdx.x == 0 && split == 0 && h == 0 && b == 0 && !nv_alpha_supported(qsc.alpha))
            atomicExch(g.err, kErrInvalidArg);
        for (int i = threadIdx.x; i < G * SB; i += kAttnThreads) {
            const int gq = i / SB, blk = i % SB;
            const uint16_t* src = g.q + ((size_t)b * g.Hq + h * G + gq) * D + blk * 16;
            const uint4 raw[2] = {*reinterpret_cast<const uint4*>(src), *reinterpret_cast<const uint4*>(src + 8)};
            uint32_t sf, sfr, codes[2], rcodes[2];
            quant_block_raw<0, 16, true>(raw, qsc, sf, codes, sfr, rcodes);
            const uint32_t rb = 2u * (uint32_t)gq;
            *reinterpret_cast<uint2*>(qtile + sw128_offset(rb, (uint32_t)blk * 8u)) = make_uint2(codes[0], codes[1]);
            *reinterpret_cast<uint2*>(qtile + sw128_offset(rb + 1u, (uint32_t)blk * 8u)) =
                make_uint2(rcodes[0], rcodes[1]);
            qsf[(blk / 4) * 512 + rb * 16 + blk % 4] = (uint8_t)sf;
            qsf[(blk / 4) * 512 + (rb + 1u) * 16 + blk % 4] = (uint8_t)sfr;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_qk = tmem, t_pv = tmem + Ly::T_PV, t_sfk = tmem + Ly::T_SFK, t_sfq = tmem + Ly::T_SFQ;

    if (warp == 0) {
        // ------------------------------------------------ page copies
        const uint64_t pol = l2_policy_evict_first();  // the cache is read once
        int s = 0;
        uint32_t ph = 0;
        for (int it = 0; it < ntiles; ++it) {
            if (it >= S &&
                !__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort_flag, g.err)))
                break;
            if (elect_one_sync()) {
                const int u0 = t0 + it * kAttnTile, nt = min(kAttnTile, t1 - u0), np = (nt + kPage - 1) / kPage;
                uint8_t* st = stg + (size_t)s * Ly::STG;
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, 2u * (uint32_t)np * (uint32_t)PB);
                for (int p = 0; p < np; ++p) {
                    const int page = g.block_table[(size_t)b * g.max_pages + u0 / kPage + p];
                    const size_t off = ((size_t)page * g.Hkv + h) * (size_t)PB;
                    bulk_load(smem_u32(st + p * PB), g.k_cache + off, (uint32_t)PB, fb, pol);
                    bulk_load(smem_u32(st + (4 + p) * PB), g.v_cache + off, (uint32_t)PB, fb, pol);
                }
                *issued = (uint32_t)(it + 1);
            }
            __syncwarp();
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
    } else {
        // ------------------------------------------------ warps 1-7
        const int ct = threadIdx.x - 32;               // 0..223: rearranging thread
        const bool smw = warp >= 4;                    // softmax / PV warps
        const int r = (warp & 3) * 32 + lane;          // token (softmax), head dimension (PV)
        const uint32_t quarter = (uint32_t)((warp & 3) * 32) << 16;
        const float c = __fmul_rn(*g.alpha_q, __frsqrt_rn((float)D));  // alpha_q / sqrt(D), alpha_k = 1
        const uint64_t kdesc = kmajor_sw128_desc(smem_u32(ktile)), qdesc = kmajor_sw128_desc(smem_u32(qtile));
        const uint64_t vdesc = kmajor_sw128_desc(smem_u32(vt)), pdesc = kmajor_sw128_desc(smem_u32(ptile));
        float o[MB][GM];
#pragma unroll
        for (int mb = 0; mb < MB; ++mb)
#pragma unroll
            for (int q = 0; q < GM; ++q) o[mb][q] = 0.0f;
        float a_t[GM];  // this tile's rescale factors exp(m_old - m_new)
        if (warp == 1) {
            // (only with tiles to process: every copy must be complete, through the
            // last PV commit that warps 4-7 wait for, before the tensor memory is freed)
            if (ntiles > 0 && elect_one_sync())
                for (int a = 0; a < NA; ++a) tc_cp_sf_atom(t_sfq + a * 4, sf_atom_desc(smem_u32(qsf + a * 512)));
            __syncwarp();
        }
        int s = 0;
        uint32_t ph = 0;
        for (int it = 0; it < ntiles; ++it) {
            const int u0 = t0 + it * kAttnTile, nt = min(kAttnTile, t1 - u0);
            // the previous tile's MMAs have read the key tile, V^T and P
            if (it > 0) (void)mbar_wait_bounded(smem_u32(pv_done), (uint32_t)(it - 1) & 1u, abort_flag, g.err);
            const bool landed = mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, g.err);
            if (ct == 0 && it < 6) RS_TRACE_MARK(g.trace, 5 * it);  // stage landed
            const uint8_t* st = stg + (size_t)s * Ly::STG;
            if (landed) {
                // every load of this thread's share first, then the stores
                constexpr int NKC = (kAttnTile * (CB / 16) + kAttnCompute - 1) / kAttnCompute;  // key code chunks
                constexpr int NKS = (kAttnTile * NA + kAttnCompute - 1) / kAttnCompute;        // key scale words
                constexpr int NV = (kAttnTile * SB + kAttnCompute - 1) / kAttnCompute;         // V blocks
                uint4 kc[NKC];
                uint32_t ks[NKS];
                uint2 vc[NV];
                uint32_t vs[NV];
#pragma unroll
                for (int j = 0; j < NKC; ++j) {
                    const int i = ct + j * kAttnCompute, rr = i / (CB / 16), cc = i % (CB / 16);
                    kc[j] = make_uint4(0u, 0u, 0u, 0u);
                    if (i < kAttnTile * (CB / 16) && rr < nt)
                        kc[j] = *reinterpret_cast<const uint4*>(st + (rr / kPage) * PB + (rr % kPage) * CB + cc * 16);
                }
#pragma unroll
                for (int j = 0; j < NKS; ++j) {
                    const int i = ct + j * kAttnCompute, rr = i / NA, a = i % NA;
                    ks[j] = 0u;
                    if (i < kAttnTile * NA && rr < nt)
                        ks[j] = *reinterpret_cast<const uint32_t*>(st + (rr / kPage) * PB + kPage * CB +
                                                                   (rr % kPage) * SB + a * 4);
                }
#pragma unroll
                for (int j = 0; j < NV; ++j) {
                    const int i = ct + j * kAttnCompute, t = i / SB, bb = i % SB;
                    vc[j] = make_uint2(0u, 0u);
                    vs[j] = 0u;
                    if (i < kAttnTile * SB && t < nt) {
                        const uint8_t* pg = st + (4 + t / kPage) * PB;
                        vc[j] = *reinterpret_cast<const uint2*>(pg + (t % kPage) * CB + bb * 8);
                        vs[j] = pg[kPage * CB + (t % kPage) * SB + bb];
                    }
                }
                uint2 vrow[NV];  // each V block's table row (its scale byte's E4M3 magnitudes)
#pragma unroll
                for (int j = 0; j < NV; ++j) vrow[j] = *reinterpret_cast<const uint2*>(vlut + vs[j] * 8);
                // key codes -> 128-byte-swizzled rows (tokens past the end: zero)
#pragma unroll
                for (int j = 0; j < NKC; ++j) {
                    const int i = ct + j * kAttnCompute, rr = i / (CB / 16), cc = i % (CB / 16);
                    if (i < kAttnTile * (CB / 16))
                        *reinterpret_cast<uint4*>(ktile + sw128_offset((uint32_t)rr, (uint32_t)cc * 16u)) = kc[j];
                }
                // key scales -> atoms (the four blocks of an atom are one word per token)
#pragma unroll
                for (int j = 0; j < NKS; ++j) {
                    const int i = ct + j * kAttnCompute, rr = i / NA, a = i % NA;
                    if (i < kAttnTile * NA)
                        *reinterpret_cast<uint32_t*>(ksf + a * 512 + (rr % 32) * 16 + (rr / 32) * 4) = ks[j];
                }
                // V -> E4M3: token row t holds its head dimensions, 128 per tile
#pragma unroll
                for (int j = 0; j < NV; ++j) {
                    const int i = ct + j * kAttnCompute, t = i / SB, bb = i % SB;
                    uint32_t w[4];
                    v_block_e4m3(vc[j], vrow[j], w);
                    if (i < kAttnTile * SB)
                        *reinterpret_cast<uint4*>(vt + (bb / 8) * 16384 +
                                                  sw128_offset((uint32_t)t, (uint32_t)(bb % 8) * 16u)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(1, kAttnCompute);
            if (ct == 0 && it < 6) RS_TRACE_MARK(g.trace, 5 * it + 1);  // rearranged
            if (warp == 1) {
                // stage free again; QK of the group's base and residue rows
                tc_fence_after();
                if (elect_one_sync()) {
                    mbar_arrive(smem_u32(&empty[s]));
                    *consumed = (uint32_t)(it + 1);
                    if (*abort_flag == 0u) {
                        for (int a = 0; a < NA; ++a)
                            tc_cp_sf_atom(t_sfk + a * 4, sf_atom_desc(smem_u32(ksf + a * 512)));
                        for (int ks = 0; ks < NA; ++ks)
                            mma_nvfp4(t_qk, kdesc + (uint32_t)ks * 2u, qdesc + (uint32_t)ks * 2u, mxf4_idesc(16, false, 0),
                                      t_sfk + ks * 4, t_sfq + ks * 4, ks > 0 ? 1u : 0u);
                        tc_commit(smem_u32(qk_done));
                    }
                }
                __syncwarp();
            }
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
            if (smw) {
                // fold, tile maximum, E4M3 weights, normalizer (token r per thread)
                const bool ok =
                    __all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(qk_done), (uint32_t)it & 1u, abort_flag, g.err));
                tc_fence_after();
                float z[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) z[e] = 0.0f;
                if (ok) tmem_ld16(t_qk + quarter, z);
                if (r == 0 && it < 6) RS_TRACE_MARK(g.trace, 5 * it + 2);  // QK done
                float sc[GM];
#pragma unroll
                for (int q = 0; q < GM; ++q) {
                    sc[q] = (q < G && r < nt) ? __fmul_rn(__fadd_rn(z[2 * q], z[2 * q + 1]), c) : -INFINITY;
                    const float mx = warp_max_f32(sc[q]);
                    if (lane == 0) red[(warp - 4) * 8 + q] = mx;
                }
                named_bar_sync(2, 128);
                float m_new[GM];
#pragma unroll
                for (int q = 0; q < GM; ++q) {
                    const float tm = fmaxf(fmaxf(red[q], red[8 + q]), fmaxf(red[16 + q], red[24 + q]));
                    const float mo = m_run[q];
                    m_new[q] = fmaxf(mo, tm);
                    a_t[q] = mo == -INFINITY ? 0.0f : __expf(mo - m_new[q]);
                    // exp(-inf - m) = 0 for padded tokens; heads beyond G have m = -inf: weight 0
                    const float e = m_new[q] == -INFINITY ? 0.0f : __expf(sc[q] - m_new[q]);
                    const uint32_t pb = e4m3x2_encode_hw(0.0f, e) & 0xFFu;
                    if (q < G) ptile[sw128_offset((uint32_t)q, (uint32_t)r)] = (uint8_t)pb;
                    // E4M3 weights in [0, 1] are multiples of 2^-9: their sum is exact in integers
                    const int units = __float2int_rn(__fmul_rn(e4m3_decode_hw(pb), 512.0f));
                    const int sum = __reduce_add_sync(0xFFFFFFFFu, units);
                    if (lane == 0) red2[(warp - 4) * 8 + q] = sum;
                }
                named_bar_sync(2, 128);
                if (r == 0)
#pragma unroll
                    for (int q = 0; q < GM; ++q) {
                        const int tile_sum = (red2[q] + red2[8 + q]) + (red2[16 + q] + red2[24 + q]);
                        l_run[q] = l_run[q] * a_t[q] + __fmul_rn((float)tile_sum, 0x1p-9f);
                        m_run[q] = m_new[q];
                    }
                fence_proxy_async_smem();  // P for the tensor pipe
            }
            if (warp == 1 || smw) named_bar_sync(3, 160);  // warps 1 and 4-7: P is in shared memory
            if (r == 0 && smw && it < 6) RS_TRACE_MARK(g.trace, 5 * it + 3);  // softmax done
            if (warp == 1) {
                // PV: V^T (128 head dimensions per MMA) x P^T over the tile's tokens
                tc_fence_after();
                if (elect_one_sync() && *abort_flag == 0u) {
#pragma unroll
                    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
                        for (int kt = 0; kt < kAttnTile / 32; ++kt)
                            mma_e4m3(t_pv + (uint32_t)(mb * 16),
                                     vdesc + (uint32_t)(mb * (16384 >> 4)) + (uint32_t)kt * (4096u >> 4),
                                     pdesc + (uint32_t)kt * 2u, f8_idesc_amn(16, 128), kt > 0 ? 1u : 0u);
                    tc_commit(smem_u32(pv_done));
                }
                __syncwarp();
            }
            if (smw) {
                // running outputs: o = o exp(m_old - m_new) + the tile's P V (head dimension r)
                const bool ok =
                    __all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(pv_done), (uint32_t)it & 1u, abort_flag, g.err));
                tc_fence_after();
#pragma unroll
                for (int mb = 0; mb < MB; ++mb) {
                    float pv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) pv[e] = 0.0f;
                    if (ok) tmem_ld16(t_pv + (uint32_t)(mb * 16) + quarter, pv);
                    if (r == 0 && mb == 0 && it < 6) RS_TRACE_MARK(g.trace, 5 * it + 4);  // PV done
#pragma unroll
                    for (int q = 0; q < GM; ++q) o[mb][q] = fmaf(o[mb][q], a_t[q], pv[q]);
                }
            }
        }
        // this split's o, m, l
        if (smw) {
#pragma unroll
            for (int mb = 0; mb < MB; ++mb)
#pragma unroll
                for (int q = 0; q < GM; ++q)
                    if (q < G) part[(size_t)q * (D + 2) + mb * 128 + r] = o[mb][q];
            if (r < G) {
                part[(size_t)r * (D + 2) + D] = m_run[r];
                part[(size_t)r * (D + 2) + D + 1] = l_run[r];
            }
            if (r == 0) RS_TRACE_MARK(g.trace, 31);  // split written
        }
    }

    // teardown: after an abort, let the page copies still in flight land
    // before the shared memory goes away
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            for (uint32_t u = *consumed; u < *issued; ++u) {
                volatile uint32_t no_abort = 0;
                (void)mbar_wait_bounded(smem_u32(&full[u % (uint32_t)S]), (u / (uint32_t)S) & 1u, &no_abort, nullptr,
                                        100000000ull);
            }
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Ly::TCOLS);
    }
}

// O = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s; empty sequences give 0.
// Split combination, one CTA of P x D threads per (query head,
// sequence), P = 4 groups when there are many splits and 1 otherwise: the
// CTA's maximum M of the splits' m_s, then group p sums w_s o_s[d] and
// w_s l_s over the splits s = p, p + P, ... (w_s = e^(m_s - M), four splits'
// loads in flight per thread), and the groups' sums are added in group order:
// a fixed order, so the result does not depend on timing.
constexpr int kCombineGroups = 4;

__global__ void __launch_bounds__(kCombineGroups * 256) resattn_combine_kernel(const AttnArgs g, void* out,
                                                                               int out_f32) {
    __shared__ float red_m[32];
    __shared__ float num_p[kCombineGroups][256];
    __shared__ float den_p[kCombineGroups];
    pdl_wait_prior_grid();  // the splits' partial results
    pdl_launch_dependents();
    const int Hq = g.Hq, Hkv = g.Hkv, D = g.D, splits = g.splits, split_tokens = g.split_tokens;
    const int G = Hq / Hkv;
    const int b = blockIdx.y, hq = blockIdx.x;
    const int d = threadIdx.x % D, grp = threadIdx.x / D, P = (int)blockDim.x / D;
    const int h = hq / G, gg = hq % G;
    const int L = attn_len(g, b);
    const int ns = min(splits, (L + split_tokens - 1) / split_tokens);
    const size_t stride = (size_t)G * (D + 2);  // floats from one split's row of this head to the next
    const float* base = g.part + ((((size_t)b * Hkv + h) * splits) * G + gg) * (D + 2);
    // M = max_s m_s over the whole CTA
    float m = -INFINITY;
    for (int s = threadIdx.x; s < ns; s += blockDim.x) m = fmaxf(m, base[(size_t)s * stride + D]);
    m = warp_max_f32(m);
    if ((threadIdx.x & 31) == 0) red_m[threadIdx.x >> 5] = m;
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) M = fmaxf(M, red_m[w]);
    // this group's splits
    float num = 0.0f, den = 0.0f;
    int s = grp;
    for (; s + 3 * P < ns; s += 4 * P) {
        float mv[4], ov[4], lv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float* p = base + (size_t)(s + u * P) * stride;
            mv[u] = p[D];
            ov[u] = p[d];
            lv[u] = p[D + 1];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float w = __expf(mv[u] - M);
            num = fmaf(w, ov[u], num);
            den = fmaf(w, lv[u], den);
        }
    }
    for (; s < ns; s += P) {
        const float* p = base + (size_t)s * stride;
        const float w = __expf(p[D] - M);
        num = fmaf(w, p[d], num);
        den = fmaf(w, p[D + 1], den);
    }
    num_p[grp][d] = num;
    if (d == 0) den_p[grp] = den;
    __syncthreads();
    if (grp != 0) return;
    float nsum = 0.0f, dsum = 0.0f;
    for (int p = 0; p < P; ++p) {
        nsum += num_p[p][d];
        dsum += den_p[p];
    }
    const float val = ns > 0 ? nsum / dsum : 0.0f;
    const size_t idx = ((size_t)b * Hq + hq) * D + d;
    if (out_f32) reinterpret_cast<float*>(out)[idx] = val;
    else reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(val);
}

// ---------------------------------------------------------------- launch --

// Split count: the (split, KV head, sequence) CTAs run in waves of `slots`
// (resident CTAs per SM x SMs: two at head size 128, one at 256); a CTA's
// time is about its tiles plus one tile's worth of set-up and teardown.  The
// split minimising waves x (tiles per split + 1) wins, the fewer splits on a
// tie (fewer partial results to combine).
int resattn_split_tokens(int B, int Hkv, int D, int max_len, int num_sms) {
    const int tiles = (max_len + kAttnTile - 1) / kAttnTile;
    if (tiles <= 1) return kAttnTile;
    const int64_t slots = (int64_t)(D <= 128 ? 2 : 1) * num_sms;
    const int64_t groups = (int64_t)B * Hkv;
    int best = 1;
    int64_t best_cost = -1;
    for (int s = 1; s <= tiles; ++s) {
        const int per = (tiles + s - 1) / s;
        if (s > 1 && (tiles + per - 1) / per < s) continue;  // the same split size as a smaller s
        const int64_t waves = (groups * s + slots - 1) / slots;
        const int64_t cost = waves * (per + 1);
        if (best_cost < 0 || cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return ((tiles + best - 1) / best) * kAttnTile;
}

template <int D, int GM>
static cudaError_t launch_split(const AttnArgs& a, cudaStream_t stream) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(resattn_split_kernel<D, GM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)AttnLayout<D>::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)a.splits, (unsigned)a.Hkv, (unsigned)a.B);
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
    cfg.dynamicSmemBytes = AttnLayout<D>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, resattn_split_kernel<D, GM>, a);
}

cudaError_t launch_resattn(int D, const AttnArgs& a, void* out, int out_f32, cudaStream_t stream) {
    const bool g4 = a.Hq / a.Hkv <= 4;
    cudaError_t e = D == 128   ? (g4 ? launch_split<128, 4>(a, stream) : launch_split<128, 8>(a, stream))
                    : D == 256 ? (g4 ? launch_split<256, 4>(a, stream) : launch_split<256, 8>(a, stream))
                               : cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)a.Hq, (unsigned)a.B, 1);
    cfg.blockDim = dim3((unsigned)((a.splits >= 2 * kCombineGroups ? kCombineGroups : 1) * D), 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, resattn_combine_kernel, a, out, out_f32);
}

}  // namespace rs
