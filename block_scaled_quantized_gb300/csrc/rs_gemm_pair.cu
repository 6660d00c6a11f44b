// Paired-CTA block-scaled GEMM for large activation operands.
//
// Two CTAs of a (2,1,1) cluster share one tcgen05.mma.cta_group::2 of
// M = 256 output channels x N = 256 activation rows: each CTA stages its own
// 128 weight channels (A) and its own 128 activation rows (B) per 256-K chunk,
// so a CTA's stage holds 16 KB of activation codes instead of 32 KB, and the
// ring is one stage deeper.  The even CTA of the pair (leader) issues the
// scale copies and the MMAs; each CTA's tensor memory holds the accumulator
// rows of its 128 channels; both epilogues read their own accumulator.
//
// Barriers (same offsets in both CTAs):
//   full[s]       own copies of stage s landed (both CTAs)
//   pfull[s]      leader: the peer's copies of stage s landed (the peer's
//                 relay warp waits on its own full[s] and arrives remotely)
//   empty[s]      both: the pair's MMAs of stage s are done (multicast commit)
//   accum_full    both: the tile's MMAs are done (multicast commit)
//   accum_empty   leader: both epilogues have read the accumulator (16 warp
//                 arrivals; the stores of a tile overlap the next tile's MMAs)
// Every wait is bounded; a wait that runs out sets the error word and the
// abort flag, and the CTA goes to the pair's final cluster barrier.
#include <cuda.h>
#include <cuda_bf16.h>

#include "rs_device.cuh"
#include "rs_internal.h"

#include <algorithm>

namespace rs {

constexpr int kPairThreads = 384;  // warp 0 producer, warp 1 MMA (leader) / relay (peer), warps 4-11 epilogue
constexpr int kPairMaxStages = 6;

struct PairArgs {
    const uint8_t* wq;    // tiled weight operand ([n_tile][chunk] blocks of WB bytes)
    const uint8_t* sfb;   // activation scale atoms (rs operand layout)
    const float* alpha_x;
    const float* alpha_w;
    void* y;
    uint32_t* err;
    uint64_t* trace;      // trace builds only: 32 timer stamps per CTA
    int N, K, M, Rb;      // Rb: activation rows (2M when folded)
    int n_atoms_k, b_row_tiles, n_tiles, b_tiles, chunks;
    int fold, out_f32, stages;
};

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Scale atom shared -> tensor memory of both CTAs of the pair, each from its
// own shared memory at the same address.
__device__ __forceinline__ void tc_cp_sf_atom_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void mma_pair(int fmt, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    if (fmt == 0)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
            " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X"
            " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
}
// Arrive on `bar` in both CTAs of the pair once this thread's MMAs are done.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
// kind::mxf4nvf4 instruction descriptor with M = 256 (the pair's rows).
__host__ __device__ constexpr uint32_t mxf4_idesc_pair(int n, bool ue8m0, uint32_t sf_id) {
    return (sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((ue8m0 ? 1u : 0u) << 23) |
           ((uint32_t)(256 >> 4) << 24) | (sf_id << 29);
}

template <int FMT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_b, const PairArgs g) {
    constexpr int BN = 256;
    constexpr int APC = FMT == 0 ? 4 : 2;                         // scale atoms per 256-K chunk and 128 rows
    constexpr uint32_t WB = 16384u + (uint32_t)APC * 512u;         // weight block: codes + scale atoms
    constexpr uint32_t BH = 128u * 128u;                           // this CTA's activation rows
    constexpr uint32_t SFB_BYTES = 2u * APC * 512u;                // scale atoms of the pair's 256 rows
    constexpr uint32_t STAGE = WB + BH + SFB_BYTES;
    constexpr int SFA_COLS = APC * 4, SFB_COLS = 2 * APC * 4, SF_COLS = SFA_COLS + SFB_COLS;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = g.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * STAGE);
    uint64_t* pfull = full + kPairMaxStages;
    uint64_t* empty = pfull + kPairMaxStages;
    uint64_t* accum_full = empty + kPairMaxStages;
    uint64_t* accum_empty = accum_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_empty + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: leader
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int n_pair_tiles = g.n_tiles / 2;  // launch_gemm_pair requires an even n_tiles
    const int total = n_pair_tiles * g.b_tiles;
    const int ntl = pair < total ? (total - pair + npairs - 1) / npairs : 0;
    const int nu = ntl * g.chunks;
    auto nt_of = [&](int j) { return 2 * ((pair + j * npairs) % n_pair_tiles) + (int)rank; };
    auto bt_of = [&](int j) { return (pair + j * npairs) / n_pair_tiles; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&pfull[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(accum_full), 1);
        mbar_init(smem_u32(accum_empty), 16);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {  // both CTAs take part in the pair's allocation
        tmem_alloc_pair(smem_u32(tmem_slot), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // barriers and tensor memory of both CTAs exist before any remote use
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tm_sf = tmem + (uint32_t)BN;

    if (warp == 0) {
        // ------------------------------------------------ producer (both CTAs)
        pdl_wait_prior_grid();
        int s = 0;
        uint32_t ph = 0;
        for (int u = 0; u < nu; ++u) {
            const int j = u / g.chunks, i = u - j * g.chunks;
            // released by the leader's multicast commit: cluster-scope acquire
            if (u >= S && !__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort_flag, g.err,
                                                                     1000000000ull, true)))
                break;
            if (elect_one_sync()) {
                uint8_t* st = smem + (size_t)s * STAGE;
                const uint32_t fb = smem_u32(&full[s]);
                const int bt = bt_of(j);
                const int nrt = min(2, g.b_row_tiles - 2 * bt);  // scale-atom row tiles of this pair tile
                const int na = min(APC, g.n_atoms_k - i * APC);
                mbar_arrive_expect_tx(fb, WB + BH + (uint32_t)(nrt * na) * 512u);
                bulk_load(smem_u32(st), g.wq + ((size_t)nt_of(j) * g.chunks + i) * WB, WB, fb, 0);
                tma_load_2d(smem_u32(st + WB), &tmap_b, fb, i * 128, bt * BN + (int)rank * 128, 0);
                for (int t = 0; t < nrt; ++t)
                    bulk_load(smem_u32(st + WB + BH + (uint32_t)t * APC * 512u),
                              g.sfb + ((size_t)(2 * bt + t) * g.n_atoms_k + (size_t)i * APC) * 512, (uint32_t)na * 512u,
                              fb, 0);
            }
            __syncwarp();
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
    } else if (warp == 1 && rank == 1) {
        // ------------------------------------------------ relay (peer)
        int s = 0;
        uint32_t ph = 0;
        for (int u = 0; u < nu; ++u) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, g.err))) break;
            if (lane == 0 && u >= g.chunks && u < 2 * g.chunks && u - g.chunks < 32)
                RS_TRACE_MARK(g.trace, u - g.chunks);  // second tile: the peer's stage landed
            if (lane == 0) mbar_arrive_remote(map_dsmem(smem_u32(&pfull[s]), 0));
            __syncwarp();
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader)
        const uint64_t adesc0 = kmajor_sw128_desc(smem_u32(smem));
        const uint64_t bdesc0 = kmajor_sw128_desc(smem_u32(smem + WB));
        const uint64_t sfadesc0 = sf_atom_desc(smem_u32(smem) + 16384u);
        const uint64_t sfbdesc0 = sf_atom_desc(smem_u32(smem + WB + BH));
        constexpr uint32_t kIdesc = mxf4_idesc_pair(BN, FMT == 1, 0);
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int j = 0; ok && j < ntl; ++j) {
            if (j > 0) {  // both epilogues have read the previous tile
                ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(accum_empty), (uint32_t)(j - 1) & 1u,
                                                               abort_flag, g.err, 1000000000ull, true));
                if (!ok) break;
                tc_fence_after();
            }
            for (int i = 0; i < g.chunks; ++i) {
                bool landed = mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, g.err) &&
                              mbar_wait_bounded(smem_u32(&pfull[s]), ph, abort_flag, g.err, 1000000000ull, true);
                ok = __all_sync(0xFFFFFFFFu, landed);
                if (!ok) break;
                if (lane == 0 && j == 1 && i < 32) RS_TRACE_MARK(g.trace, i);  // second tile: both stages in
                tc_fence_after();
                const uint32_t off = (uint32_t)s * (STAGE >> 4);
                const uint32_t tsfa = tm_sf + (uint32_t)(s * SF_COLS), tsfb = tsfa + SFA_COLS;
                const int nks = (i < g.chunks - 1 || (g.K & 255) == 0) ? 4 : (g.K - i * 256 + 63) / 64;
                const int na = FMT == 0 ? nks : (nks + 1) / 2;
                if (elect_one_sync()) {
                    for (int a = 0; a < na; ++a) {
                        tc_cp_sf_atom_pair(tsfa + a * 4, sfadesc0 + off + (uint32_t)a * 32u);
                        for (int t = 0; t < 2; ++t)
                            tc_cp_sf_atom_pair(tsfb + (a * 2 + t) * 4, sfbdesc0 + off + (uint32_t)(t * APC + a) * 32u);
                    }
                    for (int ks = 0; ks < nks; ++ks) {
                        const uint32_t accum = (i > 0 || ks > 0) ? 1u : 0u;
                        if (FMT == 0)
                            mma_pair(0, tmem, adesc0 + off + (uint32_t)ks * 2u, bdesc0 + off + (uint32_t)ks * 2u, kIdesc,
                                     tsfa + ks * 4, tsfb + ks * 8, accum);
                        else
                            mma_pair(1, tmem, adesc0 + off + (uint32_t)ks * 2u, bdesc0 + off + (uint32_t)ks * 2u,
                                     kIdesc | ((uint32_t)(ks & 1) * 2u << 4) | ((uint32_t)(ks & 1) * 2u << 29),
                                     tsfa + (ks >> 1) * 4, tsfb + (ks >> 1) * 8, accum);
                    }
                    tc_commit_pair(smem_u32(&empty[s]));
                }
                __syncwarp();
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (ok) {
                if (elect_one_sync()) tc_commit_pair(smem_u32(accum_full));
                __syncwarp();
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue (both CTAs)
        // Two warps per tensor-memory lane quarter, each taking half of the 256
        // accumulator columns; bf16 results are staged in registers so that
        // the accumulator is released before the stores, which then overlap
        // the next tile's MMAs.
        pdl_wait_prior_grid();
        const int q = warp & 3;                       // tensor-memory lane quarter
        const int half = (warp - 4) >> 2;             // accumulator columns [128 half, 128 half + 128)
        const uint32_t quarter = (uint32_t)(q * 32) << 16;
        const int row = q * 32 + lane;                // channel within this CTA's 128
        const float gsc = FMT == 0 ? __fmul_rn(*g.alpha_x, *g.alpha_w) : 1.0f;
        const int outs = g.fold ? BN / 2 : BN;
        const uint32_t leader_empty = map_dsmem(smem_u32(accum_empty), 0);
        constexpr int NC = BN / 2;                    // columns of this warp
        for (int j = 0; j < ntl; ++j) {
            bool ok = mbar_wait_bounded(smem_u32(accum_full), (uint32_t)j & 1u, abort_flag, g.err, 1000000000ull, true);
            ok = __all_sync(0xFFFFFFFFu, ok && *abort_flag == 0);
            if (!ok) break;
            tc_fence_after();
            const int n = nt_of(j) * 128 + row;
            const int m0 = bt_of(j) * outs;
            const int jmax = n < g.N ? min(outs, g.M - m0) : 0;
            const int obeg = g.fold ? half * NC / 2 : half * NC;   // first output of this warp
            const int nout = g.fold ? NC / 2 : NC;
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0) mbar_arrive(smem_u32(accum_empty));
                    else mbar_arrive_remote(leader_empty);
                }
            };
            if (!g.out_f32) {
                uint32_t pk[NC / 2];  // bf16 pairs: output o of this warp in half o & 1 of pk[o / 2]
#pragma unroll
                for (int t = 0; t < NC / 2; ++t) pk[t] = 0u;
                auto keep = [&](int o, float z) {
                    const uint32_t hb = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(gsc, z)));
                    pk[o >> 1] |= (o & 1) ? (hb << 16) : hb;
                };
#pragma unroll
                for (int c = 0; c < NC; c += 32) {
                    float v[32];
                    tmem_ld32(tmem + quarter + (uint32_t)(half * NC + c), v);
                    if (g.fold) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) keep(c / 2 + e, __fadd_rn(v[2 * e], v[2 * e + 1]));  // Fold (Eq. 2)
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) keep(c + e, v[e]);
                    }
                }
                release();
                __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(g.y) + (size_t)m0 * g.N + n;
#pragma unroll
                for (int o = 0; o < NC; ++o)
                    if (o < nout && obeg + o < jmax)
                        yb[(size_t)(obeg + o) * g.N] =
                            __ushort_as_bfloat16((unsigned short)((o & 1) ? (pk[o >> 1] >> 16) : pk[o >> 1]));
            } else {
                for (int c = 0; c < NC; c += 32) {
                    float v[32];
                    tmem_ld32(tmem + quarter + (uint32_t)(half * NC + c), v);
                    auto put = [&](int jj, float z) {
                        if (jj < jmax) reinterpret_cast<float*>(g.y)[(size_t)(m0 + jj) * g.N + n] = __fmul_rn(gsc, z);
                    };
                    if (g.fold) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) put(obeg + c / 2 + e, __fadd_rn(v[2 * e], v[2 * e + 1]));  // Fold
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) put(obeg + c + e, v[e]);
                    }
                }
                release();
            }
        }
    }

    // Teardown: every MMA of the pair is complete (the epilogues saw the last
    // accumulator, or an abort stopped the pair) before the tensor memory of
    // both CTAs is released and before either CTA's shared memory goes away.
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

// ---------------------------------------------------------------- launch --

size_t pair_smem_bytes(int fmt, int stages) {
    const int apc = fmt == 0 ? 4 : 2;
    const size_t stage = 16384 + (size_t)apc * 512 + 128 * 128 + 2 * (size_t)apc * 512;
    return 1024 + (size_t)stages * stage + 512;
}

// A 2D map over the activation codes [rows][K/2] with 128-row boxes.
typedef CUresult (*PairEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t launch_gemm_pair(int fmt, int M, int Rb, int N, int K, int fold, const void* xq, const void* wq,
                             const float* alpha_x, const float* alpha_w, void* y, int out_f32, uint32_t* err,
                             uint64_t* trace, int num_sms, cudaStream_t stream) {
    if ((N + 127) / 128 % 2 != 0) return cudaErrorInvalidValue;  // pairs of 128-channel tiles
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return cudaErrorNotSupported;
    CUtensorMap tmap;
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)Rb};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    if (reinterpret_cast<PairEncodeFn>(p)(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(xq), dims,
                                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    PairArgs a{};
    a.wq = static_cast<const uint8_t*>(wq);
    a.sfb = static_cast<const uint8_t*>(xq) + operand_sf_offset(fmt, Rb, K);
    a.alpha_x = alpha_x;
    a.alpha_w = alpha_w;
    a.y = y;
    a.err = err;
    a.trace = trace;
    a.N = N;
    a.K = K;
    a.M = M;
    a.Rb = Rb;
    a.n_atoms_k = n_atoms_k_host(fmt, K);
    a.b_row_tiles = (Rb + 127) / 128;
    a.n_tiles = (N + 127) / 128;
    a.b_tiles = (Rb + 255) / 256;
    a.chunks = (K + 255) / 256;
    a.fold = fold;
    a.out_f32 = out_f32;
    // shared memory, and tensor memory: the 256 accumulator columns plus each
    // stage's scale columns (4 per atom: APC for the weights, 2 x APC for the
    // pair's 256 activation rows)
    const int sf_cols = (fmt == 0 ? 4 : 2) * 4 * 3;
    int stages = kPairMaxStages;
    while (stages > 2 && (pair_smem_bytes(fmt, stages) > 232448 || 256 + sf_cols * stages > 512)) --stages;
    a.stages = stages;
    const int pairs = std::min(a.n_tiles / 2 * a.b_tiles, num_sms / 2);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = pair_smem_bytes(fmt, stages);
    cfg.stream = stream;
    cudaError_t e;
    if (fmt == 0) {
        e = cudaFuncSetAttribute(gemm_pair_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, gemm_pair_kernel<0>, tmap, a);
    } else {
        e = cudaFuncSetAttribute(gemm_pair_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, gemm_pair_kernel<1>, tmap, a);
    }
    return e;
}

}  // namespace rs
