// Block-scaled FP4 GEMM on the tcgen05 tensor cores (sm_103a), used by both
// the W4A4 and the residue-compensated linear layer.
//
// Swapped orientation (ResServe Sec. 5.1, Eq. 4): the MMA's 128-row A
// operand is a tile of 128 output channels of W^ [N][K]; the narrow B operand
// is the activation operand (M token rows, or 2M rows when base and residue
// are paired as adjacent rows, Sec. 5.1 "row-pair" layout), so Z^T tiles are
// 128 channels x bn activation rows.  Block scales travel as 512-byte atoms:
// TMA brings them into shared memory next to the code tiles and
// tcgen05.cp (32x128b.warpx4) moves them into tensor memory, where the
// kind::mxf4nvf4 block-scaled MMA reads them.
//
// Fold (Sec. 4.3 Eq. 2; Sec. 5.1): with paired rows, the base and residue
// products of token j land in accumulator columns 2j and 2j+1; a 32x32b
// tensor-memory load hands both to the same thread, which adds them in fp32
// before scaling and storing, so the expanded Z never leaves the SM.
//
// Split-K: when the output tiles alone cannot occupy every SM, each tile's K
// range is split; every split stores its folded fp32 partial to the
// workspace, and the last split to finish (a per-tile counter, no waiting)
// sums the partials in split order and writes Y, then re-arms the counter.
//
// Warp roles (192 threads): warps 0-3 epilogue (tensor-memory lane quarters
// 0-3), warp 4 TMA producer, warp 5 TMEM allocator and MMA issuer.  Every
// wait is bounded (about one second); a wait that runs out sets the device
// error word and an abort flag, and the CTA drains its copies and exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "rs_device.cuh"
#include "rs_internal.h"

namespace rs {

constexpr int kThreads = 192;
constexpr int kMaxStages = 8;
constexpr uint32_t kTileA = 128 * 128;  // 128 channels x 128 bytes (256 K)
constexpr size_t kSmemLimit = 232448;   // 227 KB opt-in per block

__host__ __device__ constexpr int atoms_per_chunk(int fmt) { return 256 / (fmt == 0 ? 64 : 128); }
__host__ __device__ constexpr int b_atom_tiles(int bn) { return (bn + 127) / 128; }
__host__ __device__ constexpr uint32_t stage_bytes(int fmt, int bn) {
    return (kTileA + (uint32_t)bn * 128u + (uint32_t)atoms_per_chunk(fmt) * 512u * (1u + (uint32_t)b_atom_tiles(bn)) + 1023u) /
           1024u * 1024u;
}
__host__ __device__ constexpr int sf_cols_per_stage(int fmt, int bn) {
    return atoms_per_chunk(fmt) * 4 * (1 + b_atom_tiles(bn));
}
constexpr uint32_t kCtrlBytes = 256;

struct GemmArgs {
    const uint8_t* sfa;     // weight scale atoms
    const uint8_t* sfb;     // activation scale atoms
    void* y;
    const float* alpha_x;
    const float* alpha_w;
    float* partials;
    uint32_t* counters;
    uint32_t* err;
    int N, K, Rb, M;
    int n_atoms_k;
    int b_row_tiles;        // scale-atom row tiles of the activation operand
    int chunks;
    int splits;
    int fold;
    int out_f32;
    int stages;
    int tmem_cols;
};

template <int FMT, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                const GemmArgs g) {
    constexpr int APC = atoms_per_chunk(FMT);
    constexpr int BT = b_atom_tiles(BN);
    constexpr uint32_t B_BYTES = BN * 128;
    constexpr uint32_t SFA_BYTES = APC * 512;
    constexpr uint32_t STAGE = stage_bytes(FMT, BN);
    constexpr int SFA_COLS = APC * 4;
    constexpr int SF_COLS = sf_cols_per_stage(FMT, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = g.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * STAGE);
    uint64_t* empty = full + kMaxStages;
    uint64_t* accum_full = empty + kMaxStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_full + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    volatile uint32_t* last_flag = tmem_slot + 2;
    volatile uint32_t* consumed = tmem_slot + 3;
    volatile uint32_t* issued = tmem_slot + 4;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_tile = blockIdx.x, b_tile = blockIdx.y, split = blockIdx.z;
    const int per = g.chunks / g.splits, rem = g.chunks % g.splits;
    const int c0 = split * per + (split < rem ? split : rem);
    const int nck = per + (split < rem ? 1 : 0);

    if (warp == 4 && lane == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(accum_full), 1);
        *abort_flag = 0;
        *last_flag = 0;
        *consumed = 0;
        *issued = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), (uint32_t)g.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tm_acc = tmem;
    const uint32_t tm_sf = tmem + BN;

    // Let the next kernel in the stream start its prologue; it waits for
    // this grid's completion before touching our outputs.
    pdl_launch_dependents();

    if (warp == 4) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();  // weights: streamed once
            const uint64_t pol_x = l2_policy_evict_last();   // activations: re-read by every tile
            const int nb_tiles = min(BT, g.b_row_tiles - b_tile * BT);
            auto atoms_in = [&](int chunk) { return min(APC, g.n_atoms_k - chunk * APC); };
            auto load_w = [&](int i) {
                const int chunk = c0 + i, s = i % S, na = atoms_in(chunk);
                uint8_t* st = smem + (size_t)s * STAGE;
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, kTileA + B_BYTES + (uint32_t)na * 512u * (1u + (uint32_t)nb_tiles));
                tma_load_2d(smem_u32(st), &tmap_a, fb, chunk * 128, n_tile * 128, pol_w);
                bulk_load(smem_u32(st + kTileA + B_BYTES),
                          g.sfa + ((size_t)n_tile * g.n_atoms_k + (size_t)chunk * APC) * 512, (uint32_t)na * 512u, fb,
                          pol_w);
            };
            auto load_x = [&](int i) {
                const int chunk = c0 + i, s = i % S, na = atoms_in(chunk);
                uint8_t* st = smem + (size_t)s * STAGE;
                const uint32_t fb = smem_u32(&full[s]);
                tma_load_2d(smem_u32(st + kTileA), &tmap_b, fb, chunk * 128, b_tile * BN, pol_x);
                for (int t = 0; t < nb_tiles; ++t)
                    bulk_load(smem_u32(st + kTileA + B_BYTES + SFA_BYTES + (uint32_t)t * APC * 512u),
                              g.sfb + ((size_t)(b_tile * BT + t) * g.n_atoms_k + (size_t)chunk * APC) * 512,
                              (uint32_t)na * 512u, fb, pol_x);
            };
            // Weights do not depend on the previous kernel: start them first.
            const int pre = min(S, nck);
            for (int i = 0; i < pre; ++i) load_w(i);
            pdl_wait_prior_grid();
            for (int i = 0; i < pre; ++i) load_x(i);
            int i = pre;
            for (; i < nck; ++i) {
                const int s = i % S;
                const uint32_t ph = (uint32_t)(i / S) & 1u;
                if (!mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort_flag, g.err)) break;
                load_w(i);
                load_x(i);
            }
            *issued = (uint32_t)i;
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int i = 0;
            for (; i < nck; ++i) {
                const int s = i % S;
                const uint32_t ph = (uint32_t)(i / S) & 1u;
                if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, g.err)) break;
                tc_fence_after();
                const int chunk = c0 + i;
                const int na = min(APC, g.n_atoms_k - chunk * APC);
                const int nb_tiles = min(BT, g.b_row_tiles - b_tile * BT);
                const uint32_t sa = smem_u32(smem + (size_t)s * STAGE);
                const uint32_t sb = sa + kTileA;
                const uint32_t ssfa = sb + B_BYTES;
                const uint32_t ssfb = ssfa + SFA_BYTES;
                const uint32_t tsfa = tm_sf + (uint32_t)(s * SF_COLS);
                const uint32_t tsfb = tsfa + SFA_COLS;
                for (int a = 0; a < na; ++a) tc_cp_sf_atom(tsfa + a * 4, sf_atom_desc(ssfa + a * 512));
                for (int t = 0; t < nb_tiles; ++t)
                    for (int a = 0; a < na; ++a)
                        tc_cp_sf_atom(tsfb + (a * BT + t) * 4, sf_atom_desc(ssfb + (t * APC + a) * 512));
                const int kleft = g.K - chunk * 256;
                const int nks = min(4, (kleft + 63) / 64);
                for (int ks = 0; ks < nks; ++ks) {
                    const uint64_t adesc = kmajor_sw128_desc(sa + ks * 32);
                    const uint64_t bdesc = kmajor_sw128_desc(sb + ks * 32);
                    const uint32_t acc = (i > 0 || ks > 0) ? 1u : 0u;
                    if (FMT == 0) {
                        mma_nvfp4(tm_acc, adesc, bdesc, mxf4_idesc(BN, false, 0), tsfa + ks * 4, tsfb + ks * BT * 4,
                                  acc);
                    } else {
                        const int a = ks >> 1;
                        const uint32_t sf_id = (uint32_t)(ks & 1) * 2u;
                        mma_mxfp4(tm_acc, adesc, bdesc, mxf4_idesc(BN, true, sf_id), tsfa + a * 4,
                                  tsfb + a * BT * 4, acc);
                    }
                }
                tc_commit(smem_u32(&empty[s]));
            }
            *consumed = (uint32_t)i;
            tc_commit(smem_u32(accum_full));  // fires once every issued MMA is done
        }
    } else {
        // ------------------------------------------------ epilogue (warps 0-3)
        pdl_wait_prior_grid();
        bool ok = mbar_wait_bounded(smem_u32(accum_full), 0, abort_flag, g.err);
        named_bar_sync(1, 128);
        ok = ok && (*abort_flag == 0);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        tc_fence_after();
        const int row = warp * 32 + lane;  // accumulator lane = channel within the tile
        const int n = n_tile * 128 + row;
        const int outs = g.fold ? BN / 2 : BN;
        const int m0 = b_tile * outs;
        const int tile_id = b_tile * (int)gridDim.x + n_tile;
        const float gsc = FMT == 0 ? __fmul_rn(*g.alpha_x, *g.alpha_w) : 1.0f;
        float* part = g.partials + ((size_t)tile_id * g.splits + split) * (size_t)outs * 128;

        auto store_out = [&](int j, float val) {
            const int m = m0 + j;
            if (m < g.M && n < g.N) {
                const size_t idx = (size_t)m * g.N + n;
                if (g.out_f32) reinterpret_cast<float*>(g.y)[idx] = val;
                else reinterpret_cast<__nv_bfloat16*>(g.y)[idx] = __float2bfloat16_rn(val);
            }
        };

        if (ok) {
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
                float v[16];
                tmem_ld16(tm_acc + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
                if (g.fold) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float z = __fadd_rn(v[2 * u], v[2 * u + 1]);  // Fold: base + residue
                        const int j = c / 2 + u;
                        if (g.splits == 1) store_out(j, __fmul_rn(gsc, z));
                        else part[(size_t)j * 128 + row] = z;
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int j = c + u;
                        if (g.splits == 1) store_out(j, __fmul_rn(gsc, v[u]));
                        else part[(size_t)j * 128 + row] = v[u];
                    }
                }
            }
        }
        if (g.splits > 1) {
            __threadfence();
            named_bar_sync(1, 128);
            if (threadIdx.x == 0) {
                uint32_t prev = 0;
                if (ok) prev = atomicAdd(&g.counters[tile_id], 1u);
                *last_flag = (ok && prev == (uint32_t)g.splits - 1u) ? 1u : 0u;
            }
            named_bar_sync(1, 128);
            if (*last_flag) {
                __threadfence();
                const float* base = g.partials + (size_t)tile_id * g.splits * (size_t)outs * 128;
                for (int j = 0; j < outs && m0 + j < g.M; ++j) {
                    float acc = 0.0f;
                    for (int s = 0; s < g.splits; ++s)
                        acc = __fadd_rn(acc, __ldcg(base + ((size_t)s * outs + j) * 128 + row));
                    store_out(j, __fmul_rn(gsc, acc));
                }
                if (threadIdx.x == 0) g.counters[tile_id] = 0u;  // re-arm for the next call
            }
        }
    }

    // ---------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && warp == 4 && lane == 0) {
        // Let every copy still in flight land before the CTA exits.
        for (uint32_t i = *consumed; i < *issued; ++i) {
            const uint32_t s = i % (uint32_t)S;
            volatile uint32_t no_abort = 0;
            (void)mbar_wait_bounded(smem_u32(&full[s]), (i / (uint32_t)S) & 1u, &no_abort, nullptr, 100000000ull);
        }
    }
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)g.tmem_cols);
    }
}

// ------------------------------------------------------------------- host --

GemmPlan make_gemm_plan(int fmt, bool fold, int M, int N, int K, int num_sms) {
    GemmPlan p{};
    p.fmt = fmt;
    p.fold = fold ? 1 : 0;
    p.M = M;
    p.N = N;
    p.K = K;
    p.Rb = fold ? 2 * M : M;
    p.bn = p.Rb <= 16 ? 16 : p.Rb <= 32 ? 32 : p.Rb <= 64 ? 64 : p.Rb <= 128 ? 128 : 256;
    p.n_tiles = (N + 127) / 128;
    p.b_tiles = (p.Rb + p.bn - 1) / p.bn;
    p.chunks = (K + 255) / 256;
    const int tiles = p.n_tiles * p.b_tiles;
    int splits;
    if (num_sms <= 0) splits = std::min(p.chunks, kMaxSplits);  // sizing bound
    else splits = tiles >= num_sms ? 1 : std::max(1, std::min({p.chunks, kMaxSplits, num_sms / tiles}));
    p.splits = splits;
    const int max_chunks = (p.chunks + splits - 1) / splits;
    const uint32_t st = stage_bytes(fmt, p.bn);
    int stages = (int)((kSmemLimit - 1024 - kCtrlBytes) / st);
    stages = std::min({stages, kMaxStages, max_chunks});
    p.stages = std::max(stages, 1);
    const int cols = p.bn + p.stages * sf_cols_per_stage(fmt, p.bn);
    int alloc = 32;
    while (alloc < cols) alloc *= 2;
    p.tmem_cols = alloc;
    p.smem_bytes = 1024 + (size_t)p.stages * st + kCtrlBytes;
    const int outs = fold ? p.bn / 2 : p.bn;
    p.partial_bytes = splits > 1 ? (size_t)tiles * splits * outs * 128 * sizeof(float) : 0;
    p.counter_bytes = (size_t)tiles * sizeof(uint32_t);
    return p;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        tried = true;
    }
    return fn;
}

// Code tiles: [rows][K/2] bytes, box = 128 bytes (256 K) x box_rows, 128B swizzle.
static bool encode_codes_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The dynamic shared-memory opt-in is set once per kernel and device (to the
// maximum, so later calls never need it again, e.g. during graph capture).
template <int FMT, int BN>
static cudaError_t ensure_smem_attr() {
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(gemm_kernel<FMT, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

template <int FMT, int BN>
static cudaError_t launch_typed(const GemmPlan& p, const GemmCall& c, const CUtensorMap& ta,
                                const CUtensorMap& tb, const GemmArgs& args, cudaStream_t stream) {
    auto kern = gemm_kernel<FMT, BN>;
    cudaError_t e = ensure_smem_attr<FMT, BN>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)p.n_tiles, (unsigned)p.b_tiles, (unsigned)p.splits);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = c.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, args);
}

cudaError_t launch_gemm(const GemmPlan& p, const GemmCall& c, cudaStream_t stream) {
    alignas(64) CUtensorMap ta;
    alignas(64) CUtensorMap tb;
    if (!encode_codes_map(&ta, c.wq, p.N, p.K, 128)) return cudaErrorInvalidValue;
    if (!encode_codes_map(&tb, c.xq, p.Rb, p.K, p.bn)) return cudaErrorInvalidValue;
    GemmArgs a{};
    a.sfa = static_cast<const uint8_t*>(c.wq) + operand_sf_offset(p.fmt, p.N, p.K);
    a.sfb = static_cast<const uint8_t*>(c.xq) + operand_sf_offset(p.fmt, p.Rb, p.K);
    a.y = c.y;
    a.alpha_x = c.alpha_x;
    a.alpha_w = c.alpha_w;
    a.partials = c.partials;
    a.counters = c.counters;
    a.err = c.err;
    a.N = p.N;
    a.K = p.K;
    a.Rb = p.Rb;
    a.M = p.M;
    a.n_atoms_k = n_atoms_k_host(p.fmt, p.K);
    a.b_row_tiles = (p.Rb + 127) / 128;
    a.chunks = p.chunks;
    a.splits = p.splits;
    a.fold = p.fold;
    a.out_f32 = c.out_f32;
    a.stages = p.stages;
    a.tmem_cols = p.tmem_cols;
#define RS_CASE(F, B)                                                   \
    if (p.fmt == F && p.bn == B) return launch_typed<F, B>(p, c, ta, tb, a, stream);
    RS_CASE(0, 16) RS_CASE(0, 32) RS_CASE(0, 64) RS_CASE(0, 128) RS_CASE(0, 256)
    RS_CASE(1, 16) RS_CASE(1, 32) RS_CASE(1, 64) RS_CASE(1, 128) RS_CASE(1, 256)
#undef RS_CASE
    return cudaErrorInvalidValue;
}

}  // namespace rs
