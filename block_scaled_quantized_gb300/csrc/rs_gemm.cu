// Block-scaled FP4 GEMM on the tcgen05 tensor cores (sm_103a), used by both
// the W4A4 and the residue-compensated linear layer.
//
// Swapped orientation (ResServe Sec. 5.1, Eq. 4): the MMA's 128-row A
// operand is a tile of 128 output channels of W^; the narrow B operand holds
// the activation rows (M tokens, or 2M rows when base and residue are paired
// as adjacent rows, the row-pair layout of Sec. 5.1 / Fig. 5a), so each
// accumulator tile is Z^T: 128 channels x bn activation rows.
//
// Data movement:
//  * weights are stored offline as contiguous (128 channels x 256 K) blocks
//    that already hold the 128-byte-swizzled shared-memory image of the codes
//    plus their scale atoms, so each pipeline stage is one bulk copy of
//    18 KB (NVFP4) / 17 KB (MXFP4) of consecutive bytes;
//  * activation codes come either from a TMA tensor load of the row-major
//    activation operand, or, for small M, from a quantizing prologue that
//    converts the CTA's slice of the bf16 input straight into shared memory
//    (Alg. 1 fused into the GEMM: one launch per linear layer);
//  * scale atoms go shared memory -> tensor memory, where the
//    kind::mxf4nvf4 block-scaled MMA reads them: with tcgen05.cp
//    (32x128b.warpx4, issued by the MMA warp ahead of the MMAs that read
//    them; in fused plans the weight atoms of the prefetched stages are
//    copied before the dependency wait), or, for 256-row activation tiles,
//    with tcgen05.st from four scale warps, which keeps the copies out of the
//    tensor pipe.
//
// Fold (Sec. 4.3 Eq. 2): with paired rows, the base and residue products of
// token j are accumulator columns 2j and 2j+1; a 32x32b tensor-memory load
// gives both to one thread, which adds them in fp32 before scaling and
// storing, so the expanded Z never leaves the SM.
//
// Persistent tiles: the grid has at most one CTA per SM and K split; CTA x
// takes output tiles x, x + gridDim.x, ... with its K slice fixed, so the
// weight ring streams across tile boundaries without a gap, a fused plan
// quantizes its activation slice once, and with two tensor-memory
// accumulators the epilogue of one tile overlaps the MMAs of the next.
//
// Split-K: when the output tiles alone cannot keep every SM streaming
// weights, the K range of each tile is split across the CTAs of a thread-
// block cluster (up to 8); each owner CTA sums a slice of the outputs over
// the splits in a fixed partner order and writes Y.  Narrow tiles (at most
// 16 outputs per channel) send their folded fp32 partials straight from
// registers with 16-byte st.async stores into the owner's receive buffer;
// wider tiles stage the partial in shared memory and bulk-copy each owner's
// slice (DSMEM); both complete on the owner's mbarrier.  With several tiles
// per CTA the receive buffers alternate with the accumulators, and an owner
// that has summed a buffer re-arms it and signals every partner (remote
// mbarrier arrive) before they send into it again.
//
// Programmatic dependent launch: the kernel releases its dependents at once
// and starts streaming weights before waiting for the previous grid; only
// the activation / output accesses come after that wait.
//
// Warp roles (384 threads): warp 4 bulk/TMA producer; warp 5 TMEM allocator,
// scale copies and MMA issuer; warps 8-11 (lane quarters 0-3) run the
// epilogue, with warps 0-3 for wide tiles without split-K; in fused plans
// warps 0-3 and 6-11 first run the quantizing prologue.  Kernels for
// 256-row activation tiles have 448 threads: warps 12, 13, 6 and 7 move the
// scale atoms, and warp 5 only issues MMAs.  Every wait is
// bounded (about one second); a wait that runs out sets the device error
// word and an abort flag, and the CTA drains its copies and exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "rs_device.cuh"
#include "rs_internal.h"
#include "rs_quant_core.cuh"

namespace rs {

constexpr int kThreads = 384;       // 12 warps
// Plans with a 256-row activation tile fed by TMA (the large-M GEMMs) bring
// each stage's scale atoms into tensor memory with tcgen05.st from four
// warps of their own (warps 12, 13, 6, 7: lane quarters 0-3), so that the
// tensor pipe runs only MMAs: as tcgen05.cp from the MMA warp the twelve
// copies per chunk took about a third of the pipe's time.  With 128-row tiles
// (six or eight copies per chunk) the extra hand-off per stage cost more than
// it saved, so those keep tcgen05.cp.  These kernels have 448 threads.
__host__ __device__ constexpr bool sf_by_warps(int bn, bool fused) { return !fused && bn >= 256; }
__host__ __device__ constexpr int gemm_threads(int bn, bool fused) { return sf_by_warps(bn, fused) ? 448 : kThreads; }
constexpr int kQuantWarps = 10;     // warps 0-3 and 6-11 quantize in fused plans
constexpr int kQuantThreads = kQuantWarps * 32;
constexpr int kMaxStages = 8;
constexpr size_t kSmemLimit = 232448;   // 227 KB opt-in per block
constexpr uint32_t kCtrlBytes = 2048;  // barriers and flags, then the fused NVFP4 scale table (1 KB)
constexpr int kMaxChunkBars = 64;   // fused plans: one "quantized" mbarrier per resident chunk
// barriers (full, empty: kMaxStages each; accumulator, reduction and receive
// pairs; the chunk barriers; the amax barrier), then the amax slots, the
// tensor-memory slot and the flags: all before the scale table's 1 KB
static_assert((3 * kMaxStages + 8 + kMaxChunkBars + 1) * 8 + (kMaxSplits + 1 + 5) * 4 <= 1024,
              "control words overlap the scale table");

__host__ __device__ constexpr int b_atom_tiles(int bn) { return (bn + 127) / 128; }
// Split-K exchange of a tile with `outs` outputs per channel.  Narrow tiles
// (at most 16 outputs: every one-launch decode plan) send their outputs from
// registers with 16-byte st.async stores, dealt to the first CTAs of the
// cluster in slices of a multiple of four; wider tiles stage a partial in
// shared memory and send each CTA its slice of ceil(outs / splits) outputs
// with one bulk copy (many small remote stores would be slower there).
__host__ __device__ constexpr bool split_async(int outs) { return outs <= 16; }
__host__ __device__ constexpr int split_slice(int outs, int splits) {
    return split_async(outs) ? ((outs + splits - 1) / splits + 3) / 4 * 4 : (outs + splits - 1) / splits;
}
// Shared-memory bytes of one activation stage: codes (bn rows x 128 bytes)
// plus its scale atoms, rounded to the 1024-byte swizzle period.
__host__ __device__ constexpr uint32_t b_stage_bytes(int fmt, int bn) {
    return ((uint32_t)bn * 128u + (uint32_t)weight_atoms_per_block(fmt) * (uint32_t)b_atom_tiles(bn) * 512u + 1023u) /
           1024u * 1024u;
}
__host__ __device__ constexpr int sfa_cols(int fmt) { return weight_atoms_per_block(fmt) * 4; }
__host__ __device__ constexpr int sf_cols_per_stage(int fmt, int bn) {
    return weight_atoms_per_block(fmt) * 4 * (1 + b_atom_tiles(bn));
}

struct GemmArgs {
    const uint8_t* wq;      // tiled weight operand
    const uint16_t* x;      // fused: bf16 activations [M][K]
    const uint8_t* sfb;     // TMA plans: activation scale atoms
    void* y;
    const float* alpha_x;
    const float* alpha_w;
    uint32_t* err;
    uint64_t* trace;        // trace builds only: 32 timer stamps per CTA
    uint8_t* qdump;         // fused plans, test hook: each CTA's quantized slice (null: off)
    int N, K, M, Rb;
    int n_atoms_k;          // activation operand atoms per row tile along K
    int b_row_tiles;        // scale-atom row tiles of the activation operand
    int n_tiles;            // 128-channel output tiles
    int b_tiles;            // bn-row activation tiles
    int chunks;
    int splits;
    int fold;
    int out_f32;
    int stages;
    int slots;              // fused: resident activation chunks
    int nacc;               // accumulator buffers in tensor memory (1 or 2)
    int part_bytes;         // split-K: this CTA's partial
    int recv_bytes;         // split-K: one receive buffer (0 without split)
    int tmem_cols;
    int dyn_alpha;          // fused NVFP4: the tensor scale of X is computed here (alpha_x unused)
    int qpair;              // fused: CTA pairs (x, x ^ 1) share the quantization of their K slice
    int mcast;              // scale-warp plans without split: CTA pairs (x, x ^ 1) of a cluster take
                            // neighbouring channel tiles of one activation tile, each loading half of
                            // it for both by multicast
};

template <int FMT, int BN, bool FUSED>
__global__ void __launch_bounds__(gemm_threads(BN, FUSED), BN >= 128 ? 1 : 2)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmArgs g) {
    constexpr int APC = weight_atoms_per_block(FMT);
    constexpr int BT = b_atom_tiles(BN);
    constexpr uint32_t WB = weight_block_bytes(FMT);
    constexpr uint32_t B_BYTES = BN * 128;
    constexpr uint32_t BSTAGE = b_stage_bytes(FMT, BN);
    constexpr int SFA_COLS = sfa_cols(FMT);
    constexpr int SF_COLS = sf_cols_per_stage(FMT, BN);
    constexpr bool SFW = sf_by_warps(BN, FUSED);
    static_assert(!FUSED || BT == 1, "fused plans keep the activation tile within one scale atom");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = g.stages;
    uint8_t* wring = smem;                                   // S x WB
    uint8_t* bregion = smem + (size_t)S * WB;                // S (or slots) x BSTAGE
    const int nbslots = FUSED ? g.slots : S;
    uint8_t* part_region = bregion + (size_t)nbslots * BSTAGE;    // split-K: our partial
    uint8_t* recv_region = part_region + g.part_bytes;            // split-K: nacc receive buffers
    const uint32_t recv_base = smem_u32(recv_region);
    uint64_t* full = reinterpret_cast<uint64_t*>(recv_region + (size_t)g.nacc * g.recv_bytes);
    uint64_t* empty = full + kMaxStages;
    uint64_t* accum_full = empty + kMaxStages;     // per accumulator: tile's MMAs done
    uint64_t* accum_empty = accum_full + 2;        // per accumulator: drained by the epilogue
    uint64_t* red_full = accum_empty + 2;          // split-K: all partials of a tile received
    uint64_t* recv_free = red_full + 2;            // split-K: every owner's receive buffer free again
    uint64_t* cbar = recv_free + 2;                // fused: chunk i of the slice quantized
    uint64_t* abar = cbar + kMaxChunkBars;         // dynamic tensor scale: every split's slice amax in
    uint64_t* sfr = abar + 1;                      // scale warps: stage s's atoms are in tensor memory
    uint32_t* amax_slot = reinterpret_cast<uint32_t*>(sfr + kMaxStages);  // [kMaxSplits] slice amax (bf16 |x| bits)
    uint32_t* amax_cta = amax_slot + kMaxSplits;   // this CTA's slice amax
    uint32_t* tmem_slot = amax_cta + 1;
    volatile uint32_t* abort_flag = tmem_slot + 1;
    volatile uint32_t* consumed = tmem_slot + 2;
    volatile uint32_t* issued = tmem_slot + 3;
    float* alpha_spec = reinterpret_cast<float*>(tmem_slot + 4);                       // fused: alpha_x before the wait
    float2* sc_tab = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(full) + 1024);  // fused NVFP4: s~, 1/s~ per byte

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) RS_TRACE_MARK(g.trace, 0);
    // Persistent over output tiles: tile t = blockIdx.x + j * gridDim.x, with
    // the channel tile varying fastest so that neighbouring CTAs share the
    // activation tile.  The K slice (split) of a CTA is the same for all of
    // its tiles, so fused plans quantize it once.
    const int split = blockIdx.z;
    // Cluster ranks: (x % 2) + 2 z with CTA pairs sharing a K slice, else z.
    const bool qpair = FUSED && g.qpair != 0;
    // activation tile shared by multicast: cluster rank = x % 2
    const bool mcast = SFW && g.mcast != 0;
    const uint32_t mrank = blockIdx.x & 1u;
    const uint32_t px = qpair ? (blockIdx.x & 1u) : 0u;
    auto krank = [&](uint32_t p) -> uint32_t { return qpair ? px + 2u * p : p; };  // split p, our pair slot
    const int nranks = qpair ? 2 * g.splits : g.splits;
    const uint32_t my_crank = krank((uint32_t)split);
    const int total_tiles = g.n_tiles * g.b_tiles;
    const int ntl = (total_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int per = g.chunks / g.splits, rem = g.chunks % g.splits;
    const int c0 = split * per + (split < rem ? split : rem);
    const int nck = per + (split < rem ? 1 : 0);
    const int nu = ntl * nck;  // (tile, chunk) units, tile-major
    const int pre = nu < S ? nu : S;
    const int nacc = g.nacc;
    const int outs = g.fold ? BN / 2 : BN;
    // split-K: outputs each owner sums, owners, and how the partials travel.
    // Narrow tiles exchange only the outputs of real tokens (rounded up to
    // four) when the operand is one activation tile: the padding columns of
    // a wide MMA are never sent.
    const bool xasync = g.splits > 1 && split_async(outs);
    const int xouts = (xasync && g.b_tiles == 1) ? min(outs, (g.M + 3) / 4 * 4) : outs;
    const int per_cta = split_slice(xouts, g.splits);
    const int owners = xasync ? (xouts + per_cta - 1) / per_cta : g.splits;
    const bool owner = g.splits > 1 && split < owners;
    const uint32_t slice_bytes = (uint32_t)per_cta * 128u * 4u;
    // Wide tiles without split-K: eight epilogue warps (warps 8-11 and 0-3,
    // two per tensor-memory lane quarter) take half of the columns each.
    const bool epi8 = !FUSED && BN >= 64 && g.splits == 1;
    const uint32_t red_bytes = (uint32_t)g.splits * slice_bytes;
    auto n_tile_of = [&](int j) { return ((int)blockIdx.x + j * (int)gridDim.x) % g.n_tiles; };
    auto b_tile_of = [&](int j) { return ((int)blockIdx.x + j * (int)gridDim.x) / g.n_tiles; };
    auto wsrc_of = [&](int u) {
        const int j = u / nck, i = u - j * nck;
        return g.wq + ((size_t)n_tile_of(j) * g.chunks + c0 + i) * WB;
    };
    auto b_tx_of = [&](int u) -> uint32_t {
        if (FUSED) return 0u;
        const int j = u / nck, i = u - j * nck;
        const int nb_tiles = min(BT, g.b_row_tiles - b_tile_of(j) * BT);
        const int na = min(APC, g.n_atoms_k - (c0 + i) * APC);
        return B_BYTES + (uint32_t)na * 512u * (uint32_t)nb_tiles;
    };

    // Producer: barriers, then start streaming weights right away (they do
    // not depend on the previous kernel in the stream).
    // a single activation tile reads each weight block once: stream it;
    // several activation tiles re-read every weight block: keep it
    uint64_t pol_w = 0;
    if (warp == 4) pol_w = g.b_tiles == 1 ? l2_policy_evict_first() : l2_policy_evict_last();
    if (warp == 4 && lane == 0) {
        RS_TRACE_MARK(g.trace, 31);
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), mcast ? 2 : 1);  // (multicast: both CTAs' MMAs)
            if (SFW) mbar_init(smem_u32(&sfr[s]), 4);  // one arrival per scale warp
        }
        // every scale block of chunk i (all token rows) arrives once
        if (FUSED)
            for (int i = 0; i < nck; ++i) mbar_init(smem_u32(&cbar[i]), (uint32_t)(g.M * (256 / block_elems(FMT))));
        // one 4-byte slice amax from every CTA of the cluster (st.async bytes)
        mbar_init(smem_u32(abar), 1);
        if (nranks > 1) mbar_arrive_expect_tx(smem_u32(abar), 4u * (uint32_t)nranks);
        *amax_cta = 0u;
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accum_full[b]), 1);
            mbar_init(smem_u32(&accum_empty[b]), (uint32_t)(epi8 ? 8 : 4));  // one arrival per epilogue warp
            mbar_init(smem_u32(&red_full[b]), 1);
            mbar_init(smem_u32(&recv_free[b]), (uint32_t)owners);  // one arrival per owner
        }
        // the first use of each receive buffer is armed before any partner
        // can send (they send only after the cluster barrier below)
        if (owner)
            for (int b = 0; b < nacc && b < ntl; ++b) mbar_arrive_expect_tx(smem_u32(&red_full[b]), red_bytes);
        *abort_flag = 0;
        *consumed = 0;
        *issued = 0;
        fence_mbarrier_init();
    }
    if (warp == 4) {
        __syncwarp();
        if (elect_one_sync()) {
            for (int u = 0; u < pre; ++u) {
                const uint32_t fb = smem_u32(&full[u]);
                mbar_arrive_expect_tx(fb, WB + b_tx_of(u));
                bulk_load(smem_u32(wring + (size_t)u * WB), wsrc_of(u), WB, fb, pol_w);
            }
            RS_TRACE_MARK(g.trace, 2);
        }
        __syncwarp();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), (uint32_t)g.tmem_cols);
        tmem_relinquish();
    }
    if (FUSED) {
        // The quantizer leaves no byte of the slice unwritten except the padding
        // rows and the scale bytes of a ragged K tail: zeros for those, written
        // before any quantizer (ours or, with CTA pairs, the partner's after the
        // cluster barrier below) stores codes, and visible to the tensor pipe.
        const uint32_t bbytes = (uint32_t)nck * BSTAGE;
        for (uint32_t off = threadIdx.x * 16u; off < bbytes; off += (uint32_t)gemm_threads(BN, FUSED) * 16u)
            *reinterpret_cast<uint4*>(bregion + off) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool tmem_freed = false;  // warp 5: deallocated after the last accumulator was read
    if (threadIdx.x == 0) {
        RS_TRACE_MARK(g.trace, 1);
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        RS_TRACE_VALUE(g.trace, 12, smid);
    }
    const uint32_t tm_sf = tmem + (uint32_t)(nacc * BN);
    // split-K partners copy into our receive buffers and signal red_full:
    // every barrier of the cluster must be initialised before that
    // (multicast: the partner writes into our stages and arrives on our barriers)
    if (g.splits > 1 || qpair || mcast) cluster_sync_all();

    // Dependents may start their prologue now; they wait for our completion
    // before they touch anything we read or write.
    pdl_launch_dependents();

    if (warp == 4) {
        // ------------------------------------------------ producer
        // whole warp runs the loop, one elected lane issues the copies
        // activations are re-read by every channel tile of their row block
        const uint64_t pol_x = g.b_tiles == 1 ? l2_policy_evict_last() : l2_policy_evict_normal();
        auto load_b = [&](int u) {
            if (FUSED) return;
            const int j = u / nck, i = u - j * nck;
            const int chunk = c0 + i, s = u % S, bt = b_tile_of(j);
            const int nb_tiles = min(BT, g.b_row_tiles - bt * BT);
            uint8_t* st = bregion + (size_t)s * BSTAGE;
            const uint32_t fb = smem_u32(&full[s]);
            const int na = min(APC, g.n_atoms_k - chunk * APC);
            if (mcast) {
                // our half of the 256 rows and its atom tile (if the operand
                // has one there), to both CTAs (each CTA's full barrier
                // expects the whole stage)
                static_assert(!SFW || BT == 2, "scale-warp plans have 256-row tiles");
                tma_load_2d_mc(smem_u32(st) + mrank * (B_BYTES / 2), &tmap_b, fb, chunk * 128,
                               bt * BN + (int)mrank * (BN / 2), (uint16_t)3, pol_x);
                if ((int)mrank < nb_tiles)
                    bulk_load_mc(smem_u32(st + B_BYTES + mrank * (uint32_t)APC * 512u),
                                 g.sfb + ((size_t)(bt * BT + (int)mrank) * g.n_atoms_k + (size_t)chunk * APC) * 512,
                                 (uint32_t)na * 512u, fb, (uint16_t)3, pol_x);
                return;
            }
            tma_load_2d(smem_u32(st), &tmap_b, fb, chunk * 128, bt * BN, pol_x);
            for (int t = 0; t < nb_tiles; ++t)
                bulk_load(smem_u32(st + B_BYTES + (uint32_t)t * APC * 512u),
                          g.sfb + ((size_t)(bt * BT + t) * g.n_atoms_k + (size_t)chunk * APC) * 512,
                          (uint32_t)na * 512u, fb, pol_x);
        };
        pdl_wait_prior_grid();
        if (!FUSED && lane == 0) RS_TRACE_MARK(g.trace, 16);
        if (elect_one_sync())
            for (int u = 0; u < pre; ++u) load_b(u);
        __syncwarp();
        int u = pre;
        // stage, phase, and the unit's (tile, chunk) advance incrementally
        int s = pre % S, jj = pre / nck, ii = pre - jj * nck;
        uint32_t ph = (uint32_t)(pre / S) & 1u;
        const uint8_t* wtile = g.wq + ((size_t)n_tile_of(jj) * g.chunks + c0) * WB;
        for (; u < nu; ++u) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort_flag, g.err))) break;
            if (lane == 0 && (u == 8 || u == 16 || u == 24)) RS_TRACE_MARK(g.trace, u == 8 ? 31 : u == 16 ? 29 : 15);
            if (elect_one_sync()) {
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, WB + (FUSED ? 0u : b_tx_of(u)));
                bulk_load(smem_u32(wring + (size_t)s * WB), wtile + (size_t)ii * WB, WB, fb, pol_w);
                load_b(u);
            }
            __syncwarp();
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
            if (++ii == nck) {
                ii = 0;
                ++jj;
                wtile = g.wq + ((size_t)n_tile_of(jj) * g.chunks + c0) * WB;
            }
        }
        if (lane == 0) {
            *issued = (uint32_t)u;
            RS_TRACE_MARK(g.trace, 3);
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs the loop; one elected lane copies the unit's
        // scale atoms shared -> tensor memory (tcgen05.cp, ordered before the
        // MMAs that read them in the tensor pipe) and issues the MMAs.  A
        // stage's scale columns are rewritten only after its full barrier,
        // which the producer re-arms after that stage's previous MMAs are done.
        // Descriptors are formed once and advanced by adding (offset >> 4) to
        // their start-address field (shared addresses stay below 2^18, so the
        // 14-bit field never carries); stage and phase advance incrementally.
        const uint64_t adesc0 = kmajor_sw128_desc(smem_u32(wring));
        const uint64_t bdesc0 = kmajor_sw128_desc(smem_u32(bregion));
        const uint64_t sfadesc0 = sf_atom_desc(smem_u32(wring) + kWeightCodeBytes);
        const uint64_t sfbdesc0 = sf_atom_desc(smem_u32(bregion) + B_BYTES);
        constexpr uint32_t kIdesc = mxf4_idesc(BN, FMT == 1, 0);
        // Fused plans: the weight scale atoms of the stages prefetched ahead of
        // the previous kernel's completion go to tensor memory as soon as they
        // land, so that after the quantizer only the activation scales and the
        // MMAs remain.  (A weight block always holds all of its atoms.)
        const int npre = FUSED ? (nu < S ? nu : S) : 0;
        bool ok = true;
        for (int u0 = 0; ok && u0 < npre; ++u0) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&full[u0]), 0u, abort_flag, g.err));
            if (!ok) break;
            tc_fence_after();
            if (elect_one_sync()) {
#pragma unroll
                for (int a = 0; a < APC; ++a)
                    tc_cp_sf_atom(tm_sf + (uint32_t)(u0 * SF_COLS + a * 4), sfadesc0 + (uint32_t)u0 * (WB >> 4) +
                                                                                 (uint32_t)a * 32u);
            }
            __syncwarp();
        }
        int u = 0, s = 0;
        uint32_t ph = 0;
        for (int j = 0; ok && j < ntl; ++j) {
            const int b = j & (nacc - 1);
            if (j >= nacc) {
                // the epilogue has read this accumulator's previous tile
                ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&accum_empty[b]),
                                                               (uint32_t)(j / nacc - 1) & 1u, abort_flag, g.err));
                if (!ok) break;
                tc_fence_after();
            }
            const uint32_t tm_acc = tmem + (uint32_t)(b * BN);
            const int nb_tiles = min(BT, g.b_row_tiles - b_tile_of(j) * BT);
            for (int i = 0; i < nck; ++i, ++u) {
                bool landed = mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, g.err);
                // (scale warps: the stage's atoms are in tensor memory)
                if (SFW) landed = landed && mbar_wait_bounded(smem_u32(&sfr[s]), ph, abort_flag, g.err);
                if (lane == 0 && (u == 8 || u == 16 || u == 24 || u == 31))
                    RS_TRACE_MARK(g.trace, u == 8 ? 13 : u == 16 ? 14 : u == 24 ? 28 : 30);
                // fused plans: chunk i of the activation slice is quantized
                // (the quantizer finishes chunks in order, so the first MMAs
                // overlap the quantization of the later chunks)
                if (FUSED && j == 0) {
                    // (with CTA pairs, the partner's quantizer arrives on this
                    // barrier from its CTA: a cluster-scope acquire)
                    landed = landed && mbar_wait_bounded(smem_u32(&cbar[i]), 0, abort_flag, g.err, 1000000000ull, qpair);
                    if (qpair) fence_proxy_async_all();
                }
                if (u == 0 && lane == 0) RS_TRACE_MARK(g.trace, 11);
                ok = __all_sync(0xFFFFFFFFu, landed);
                if (!ok) break;
                if (lane == 0) *consumed = (uint32_t)(u + 1);
                if (u == 0 && lane == 0) RS_TRACE_MARK(g.trace, 4);
                if (u == nu - 1 && lane == 0) RS_TRACE_MARK(g.trace, 5);
                tc_fence_after();
                const uint32_t aoff = (uint32_t)s * (WB >> 4);
                const uint32_t boff = (uint32_t)(FUSED ? i : s) * (BSTAGE >> 4);
                const uint64_t ad = adesc0 + aoff, bd = bdesc0 + boff;
                const uint64_t sad = sfadesc0 + aoff, sbd = sfbdesc0 + boff;
                const uint32_t tsfa = tm_sf + (uint32_t)(s * SF_COLS);
                const uint32_t tsfb = tsfa + SFA_COLS;
                const bool whole = c0 + i < g.chunks - 1 || (g.K & 255) == 0;  // all four k-steps
                const bool a_sf = u >= npre;  // weight scales not yet in tensor memory
                if (elect_one_sync()) {
                    if (whole) {
                        if constexpr (!SFW) {
#pragma unroll
                            for (int a = 0; a < APC; ++a) {
                                if (a_sf) tc_cp_sf_atom(tsfa + a * 4, sad + (uint32_t)a * 32u);
                                for (int t = 0; t < nb_tiles; ++t)
                                    tc_cp_sf_atom(tsfb + (a * BT + t) * 4, sbd + (uint32_t)(t * APC + a) * 32u);
                            }
                        }
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint32_t accum = (i > 0 || ks > 0) ? 1u : 0u;
                            if (FMT == 0)
                                mma_nvfp4(tm_acc, ad + (uint32_t)ks * 2u, bd + (uint32_t)ks * 2u, kIdesc,
                                          tsfa + ks * 4, tsfb + ks * BT * 4, accum);
                            else
                                mma_mxfp4(tm_acc, ad + (uint32_t)ks * 2u, bd + (uint32_t)ks * 2u,
                                          kIdesc | ((uint32_t)(ks & 1) * 2u << 4) | ((uint32_t)(ks & 1) * 2u << 29),
                                          tsfa + (ks >> 1) * 4, tsfb + (ks >> 1) * BT * 4, accum);
                        }
                    } else {
                        // ragged K tail: the k-steps (and scale atoms) it covers
                        const int nks = (g.K - (c0 + i) * 256 + 63) / 64;
                        const int na = FMT == 0 ? nks : (nks + 1) / 2;
                        for (int a = 0; !SFW && a < na; ++a) {
                            if (a_sf) tc_cp_sf_atom(tsfa + a * 4, sad + (uint32_t)a * 32u);
                            for (int t = 0; t < nb_tiles; ++t)
                                tc_cp_sf_atom(tsfb + (a * BT + t) * 4, sbd + (uint32_t)(t * APC + a) * 32u);
                        }
                        for (int ks = 0; ks < nks; ++ks) {
                            const uint32_t accum = (i > 0 || ks > 0) ? 1u : 0u;
                            if (FMT == 0)
                                mma_nvfp4(tm_acc, ad + (uint32_t)ks * 2u, bd + (uint32_t)ks * 2u, kIdesc,
                                          tsfa + ks * 4, tsfb + ks * BT * 4, accum);
                            else
                                mma_mxfp4(tm_acc, ad + (uint32_t)ks * 2u, bd + (uint32_t)ks * 2u,
                                          kIdesc | ((uint32_t)(ks & 1) * 2u << 4) | ((uint32_t)(ks & 1) * 2u << 29),
                                          tsfa + (ks >> 1) * 4, tsfb + (ks >> 1) * BT * 4, accum);
                        }
                    }
                    // multicast: the stage is free once both CTAs' MMAs are done
                    // (the last S units' stages are never refilled: local only)
                    if (mcast && u + S < nu) tc_commit_mc(smem_u32(&empty[s]), (uint16_t)3);
                    else tc_commit(smem_u32(&empty[s]));
                }
                __syncwarp();
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (ok) {
                if (elect_one_sync()) tc_commit(smem_u32(&accum_full[b]));  // fires once the tile's MMAs are done
                __syncwarp();
            }
            if (j < 3 && lane == 0) RS_TRACE_MARK(g.trace, 19 + j);
        }
        // Test hook (null on every production call): copy this CTA's quantized
        // activation slice, codes and scale atoms exactly as the MMAs read
        // them, to the dump buffer; every chunk's barrier was waited above.
        if (FUSED && g.qdump != nullptr && ok) {
            uint8_t* dst = g.qdump + ((size_t)split * gridDim.x + blockIdx.x) * (size_t)g.slots * BSTAGE;
            const uint32_t bytes = (uint32_t)nck * BSTAGE;
            for (uint32_t off = (uint32_t)lane * 16u; off < bytes; off += 512u)
                *reinterpret_cast<uint4*>(dst + off) = *reinterpret_cast<const uint4*>(bregion + off);
        }
        // Free the tensor memory as soon as the epilogue has read the last
        // accumulator (it reads the tiles in order), while it still exchanges
        // and stores the outputs.
        if (ok) {
            const int jl = ntl - 1;
            const bool drained = mbar_wait_bounded(smem_u32(&accum_empty[jl & (nacc - 1)]),
                                                   (uint32_t)(jl / nacc) & 1u, abort_flag, g.err);
            if (__all_sync(0xFFFFFFFFu, drained)) {
                tc_fence_after();
                tmem_dealloc(tmem, (uint32_t)g.tmem_cols);
                tmem_freed = true;
                if (lane == 0) RS_TRACE_MARK(g.trace, 10);
            }
        }
    } else if (SFW && (warp == 6 || warp == 7 || warp >= 12)) {
        // ------------------------------------------------ scale warps
        // Once a stage has landed, each warp copies every scale atom of it
        // (32 rows x 16 bytes) into its lane quarter of the stage's scale
        // columns: lane l, columns c..c+3 hold row l of the atom, the image
        // the 32x128b.warpx4 copy gives and the block-scaled MMA reads.  The
        // columns of stage s are rewritten only after its full barrier, which
        // the producer re-arms after that stage's previous MMAs are done.
        const uint32_t tq = tm_sf + ((uint32_t)((warp & 3) * 32) << 16);
        const uint8_t* sa0 = wring + kWeightCodeBytes + lane * 16;
        const uint8_t* sb0 = bregion + B_BYTES + lane * 16;
        int s = 0;
        uint32_t ph = 0;
        for (int u = 0; u < nu; ++u) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag, g.err))) break;
            tc_fence_after();
            const uint32_t col = tq + (uint32_t)(s * SF_COLS);
            uint32_t ra[4 * APC];  // weight atom a -> columns 4a..4a+3
#pragma unroll
            for (int a = 0; a < APC; ++a) {
                const uint4 v = *reinterpret_cast<const uint4*>(sa0 + (size_t)s * WB + (size_t)a * 512);
                ra[4 * a] = v.x, ra[4 * a + 1] = v.y, ra[4 * a + 2] = v.z, ra[4 * a + 3] = v.w;
            }
            uint32_t rb[4 * APC * BT];  // activation atom (a, t) -> columns SFA_COLS + 4 (a BT + t)
#pragma unroll
            for (int a = 0; a < APC; ++a)
#pragma unroll
                for (int t = 0; t < BT; ++t) {
                    const uint4 v = *reinterpret_cast<const uint4*>(sb0 + (size_t)s * BSTAGE + (size_t)(t * APC + a) * 512);
                    const int c = 4 * (a * BT + t);
                    rb[c] = v.x, rb[c + 1] = v.y, rb[c + 2] = v.z, rb[c + 3] = v.w;
                }
            tmem_st_cols(col, ra);
            tmem_st_cols(col + (uint32_t)SFA_COLS, rb);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sfr[s]));
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
    } else {
        // ------------------------------------------------ warps 0-3, 6-11
        const bool epi = warp >= 8 || (epi8 && warp < 4);  // epilogue: lane quarter = warp % 4
        const int qw = warp < 4 ? warp : warp - 2;  // quantizer warp 0..kQuantWarps-1
        const int qtid = qw * 32 + lane;
        float ax_val = 0.0f;  // NVFP4 activation tensor scale of this call
        if (FUSED) {
            // Quantizing prologue (Alg. 1), one scale block per thread: this
            // CTA's K slice of every token -> base (row 2j) and residue
            // (row 2j+1) codes in the swizzled B tiles, scales in the B atoms.
            constexpr int E = block_elems(FMT);  // 16 (NVFP4) or 32 (MXFP4)
            // NVFP4 scale table (s~ and fl(1/s~) of every scale byte): built here
            // from the tensor scale as it reads before the dependency wait (one
            // thread reads it, so that every thread uses the same value), and
            // rebuilt after the wait only if the scale turns out to differ
            const bool spec_tab = FMT == 0 && !g.dyn_alpha;
            if (spec_tab && qtid == 0) *alpha_spec = *g.alpha_x;
            if (spec_tab) named_bar_sync(2, kQuantThreads);  // every thread builds from the value read
            auto build_table = [&](float a) {
                for (int i = qtid; i < 128; i += kQuantThreads) {
                    float st, mul;
                    nv_scale_table_entry((uint32_t)i, a, st, mul);
                    sc_tab[i] = make_float2(st, mul);
                }
            };
            if (spec_tab) {
                build_table(*alpha_spec);
                named_bar_sync(2, kQuantThreads);
            }
            pdl_wait_prior_grid();
            if (qtid == 0) RS_TRACE_MARK(g.trace, 16);
            const int kbeg = c0 * 256, kend = min(g.K, (c0 + nck) * 256);
            // flat chunk-major mapping: thread qtid takes scale blocks qtid,
            // qtid + T, ... (T = quantizer threads) of the order (chunk, token
            // row, block), so chunks complete in order.  With CTA pairs, this
            // CTA's chunks are every other one of the slice, from chunk px.
            constexpr int bpc = 256 / E;    // blocks per token row in one chunk
            constexpr int kWords = E / 8;   // 16-byte words of X per block
            constexpr int kBatch = 32 / E;  // blocks per thread per batch
            const int cb = g.M * bpc;       // blocks per chunk
            // f / cb as a multiply-high: with m = ceil(2^32 / cb) the quotient
            // is exact while f cb < 2^32 (here f < 32 chunks x cb, cb <= 512)
            const uint32_t cb_magic = 0xFFFFFFFFu / (uint32_t)cb + 1u;
            auto div_cb = [&](int f) { return (int)__umulhi((uint32_t)f, cb_magic); };
            const int my_chunks = qpair ? (nck - (int)px + 1) / 2 : nck;
            const int total = my_chunks * cb;
            auto chunk_of = [&](int cl) { return qpair ? 2 * cl + (int)px : cl; };  // local -> slice chunk
            auto block_pos = [&](int f, int& j, int& kk) {
                const int cl = div_cb(f), rem = f - cl * cb;
                j = rem / bpc;
                kk = chunk_of(cl) * 256 + (rem - j * bpc) * E;
            };
            // the partner's copy of this CTA's shared memory (CTA pairs)
            const uint32_t peer = qpair ? krank((uint32_t)split) ^ 1u : 0u;
            // raw bf16 words of this thread's blocks in one batch; the first
            // batch is requested before the tensor scale is read, so that both
            // come back in one round trip
            uint4 raw[kBatch][kWords];
            auto load_batch = [&](int fw) {
#pragma unroll
                for (int r = 0; r < kBatch; ++r) {
                    const int f = fw + lane + r * kQuantThreads;
                    int j, kk;
                    block_pos(f, j, kk);
                    const bool live = f < total && kbeg + kk < kend;
#pragma unroll
                    for (int q = 0; q < kWords; ++q)
                        raw[r][q] = load16_or_zero(g.x + (size_t)j * g.K + kbeg + kk + 8 * q, live);
                }
            };
            const int fw0 = qw * 32;
            if (fw0 < total) load_batch(fw0);
            if (FMT == 0 && g.dyn_alpha) {
                // This call's tensor scale (App. B.2 Eq. 8): a = fl(amax(X) / 2688),
                // the same value rs_compute_tensor_scale gives.  Each CTA takes the
                // max |x| of its K slice; the K splits of the cluster cover K and
                // trade their maxima (one 4-byte st.async into every CTA's slot
                // of this rank, completing bytes on that CTA's barrier).
                // |x| bit patterns, two per word (integer order: NaN > Inf > finite):
                // the words of this thread's first batch are in registers
                // already (zeros for blocks past the slice); later batches'
                // blocks are read here
                uint32_t m2 = 0u;
                if (fw0 < total)
#pragma unroll
                    for (int r = 0; r < kBatch; ++r)
#pragma unroll
                        for (int q = 0; q < kWords; ++q) {
                            m2 = __vmaxu2(m2, raw[r][q].x & 0x7FFF7FFFu);
                            m2 = __vmaxu2(m2, raw[r][q].y & 0x7FFF7FFFu);
                            m2 = __vmaxu2(m2, raw[r][q].z & 0x7FFF7FFFu);
                            m2 = __vmaxu2(m2, raw[r][q].w & 0x7FFF7FFFu);
                        }
                for (int f = kBatch * kQuantThreads + qtid; f < total; f += kQuantThreads) {
                    int j, kk;
                    block_pos(f, j, kk);
                    if (kbeg + kk >= kend) continue;
#pragma unroll
                    for (int q = 0; q < kWords; ++q) {
                        const uint4 v = *reinterpret_cast<const uint4*>(g.x + (size_t)j * g.K + kbeg + kk + 8 * q);
                        m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
                        m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
                        m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
                        m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
                    }
                }
                uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
                m = __reduce_max_sync(0xFFFFFFFFu, m);
                if (lane == 0) atomicMax(amax_cta, m);
                named_bar_sync(2, kQuantThreads);
                const uint32_t cm = *reinterpret_cast<volatile uint32_t*>(amax_cta);
                uint32_t gm = cm;
                if (nranks > 1) {
                    if (qtid < nranks)  // one lane per destination CTA
                        st_async_b32(map_dsmem(smem_u32(&amax_slot[my_crank]), (uint32_t)qtid), cm,
                                     map_dsmem(smem_u32(abar), (uint32_t)qtid));
                    if (mbar_wait_bounded(smem_u32(abar), 0, abort_flag, g.err, 1000000000ull, true))
                        for (int r = 0; r < nranks; ++r)
                            gm = max(gm, reinterpret_cast<volatile uint32_t*>(amax_slot)[r]);
                }
                const uint32_t bits = gm << 16;
                if (qtid == 0) RS_TRACE_MARK(g.trace, 8);  // the cluster's amax is known
                if (bits >= 0x7F800000u) {  // Inf or NaN in X, as rs_compute_tensor_scale reports it
                    if (qtid == 0 && blockIdx.x == 0 && split == 0) atomicExch(g.err, kErrInvalidArg);
                    ax_val = __uint_as_float(0x7FC00000u);
                } else {
                    ax_val = __fdiv_rn(__uint_as_float(bits), 2688.0f);
                }
            } else if (FMT == 0) {
                ax_val = *g.alpha_x;
            }
            const NvScaleConst ksc = nv_scale_const(ax_val);
            if (FMT == 0 && (g.dyn_alpha || __float_as_uint(ax_val) != __float_as_uint(*alpha_spec))) {
                // (the same value on every thread: read after the wait, or found by the
                // cluster; a table built before the wait may still be read until all
                // threads are here, and without one nothing reads it yet)
                if (!g.dyn_alpha) named_bar_sync(2, kQuantThreads);
                build_table(ax_val);
                named_bar_sync(2, kQuantThreads);
            }
#ifdef RS_TRACE
            if (qtid == 0 && fw0 < total) {
                asm volatile("" ::"r"(raw[0][0].x));  // the first block's X words have arrived
                RS_TRACE_MARK(g.trace, 20);
            }
#endif
            if (FMT == 0 && qtid == 0 && blockIdx.x == 0 && blockIdx.z == 0 && !nv_alpha_supported(ksc.alpha))
                atomicExch(g.err, kErrInvalidArg);
            // codes of one block (element offset kk of the slice) and its scale byte
            auto put = [&](uint32_t rowb, int kk, const uint32_t (&codes)[E / 8], uint32_t sfbyte, bool live) {
                if (!live) return;
                const int ci = kk / 256;
                const uint32_t kb = (uint32_t)(kk % 256) / (uint32_t)E;  // block within the chunk
                uint8_t* slot = bregion + (size_t)ci * BSTAGE;
                const uint32_t b = kb * (uint32_t)(E / 2);                // byte within the 128-byte row
                uint8_t* cp = slot + sw128_offset(rowb, b);
                // scale byte: atom kb / 4, byte (row % 32) * 16 + (row / 32 % 4) * 4 + kb % 4
                uint8_t* sp = slot + B_BYTES + (kb / 4) * 512 + (rowb % 32) * 16 + (rowb / 32) * 4 + kb % 4;
                if constexpr (E == 16) {
                    *reinterpret_cast<uint2*>(cp) = make_uint2(codes[0], codes[1]);
                    if (qpair) st_dsmem_v2(map_dsmem(smem_u32(cp), peer), codes[0], codes[1]);
                } else {
                    const uint4 v = make_uint4(codes[0], codes[E / 8 - 3], codes[E / 8 - 2], codes[E / 8 - 1]);
                    *reinterpret_cast<uint4*>(cp) = v;
                    if (qpair) st_dsmem_v4(map_dsmem(smem_u32(cp), peer), v);
                }
                *sp = (uint8_t)sfbyte;
                if (qpair) st_dsmem_u8(map_dsmem(smem_u32(sp), peer), sfbyte);
            };
            // the loop bound is per warp (fw): the warp-wide arrival below
            for (int fw = fw0; fw < total; fw += kBatch * kQuantThreads) {
                if (fw != fw0) load_batch(fw);
#pragma unroll
                for (int r = 0; r < kBatch; ++r) {
                    if (fw + r * kQuantThreads >= total) break;  // whole warp past the end
                    const int f = fw + lane + r * kQuantThreads;
                    int j, kk;
                    block_pos(f, j, kk);
                    const bool live = f < total && kbeg + kk < kend;
                    uint32_t sfq, codes[E / 8], sfr = 0u, rcodes[E / 8];
                    const uint32_t rb = g.fold ? 2u * (uint32_t)j : (uint32_t)j;
                    const float2* tab = FMT == 0 ? sc_tab : nullptr;
                    if (g.fold) {
                        quant_block_raw<FMT, E, true>(raw[r], ksc, sfq, codes, sfr, rcodes, tab);
                        put(rb, kk, codes, sfq, live);
                        put(rb + 1u, kk, rcodes, sfr, live);
                    } else {
                        quant_block_raw<FMT, E, false>(raw[r], ksc, sfq, codes, sfr, rcodes, tab);
                        put(rb, kk, codes, sfq, live);
                    }
#ifdef RS_TRACE
                    if (qtid == 0 && r == 0 && fw == fw0) RS_TRACE_MARK(g.trace, 21);
#endif
                    // these blocks are in shared memory (with CTA pairs in both
                    // CTAs'): make them visible to the tensor pipe, then one
                    // arrival per warp and chunk counts them, on both CTAs
                    if (qpair) fence_proxy_async_all();
                    else fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int lo = fw + r * kQuantThreads, hi = min(lo + 32, total);
                        for (int c = div_cb(lo); c * cb < hi; ++c) {
                            const int n = min(hi, (c + 1) * cb) - max(lo, c * cb);
                            const uint32_t bar = smem_u32(&cbar[chunk_of(c)]);
                            mbar_arrive_cnt(bar, (uint32_t)n);
                            if (qpair) mbar_arrive_remote_cnt(map_dsmem(bar, peer), (uint32_t)n);
                        }
                    }
                }
            }
            if (qtid == 0) RS_TRACE_MARK(g.trace, 17);
            if (qtid == kQuantThreads - 1) RS_TRACE_MARK(g.trace, 18);
        } else if (epi) {
            pdl_wait_prior_grid();  // before writing the output
            if (FMT == 0) ax_val = *g.alpha_x;
        }

        if (epi) {
            // ---------------------------------------------- epilogue
            const int ew = warp & 3;                       // lane quarter
            const uint32_t quarter = (uint32_t)(ew * 32) << 16;
            const int row = ew * 32 + lane;                // accumulator lane = channel within the tile
            const int ctid = row;                          // 0..127
            const float gsc = FMT == 0 ? __fmul_rn(ax_val, *g.alpha_w) : 1.0f;
            float* part = reinterpret_cast<float*>(part_region);  // split-K: [j][channel]
            const uint32_t my_rank = (uint32_t)split;
            // split-K: lane o of warp 8 sends to owner o; its destinations in
            // the cluster (receive buffer b at our rank's slot, owner's red_full[b])
            uint32_t dst_buf0 = 0, dst_buf1 = 0, dst_bar0 = 0, dst_bar1 = 0;
            if (g.splits > 1 && warp == 8 && lane < g.splits) {
                const uint32_t rb = recv_base + my_rank * slice_bytes;
                dst_buf0 = map_dsmem(rb, krank((uint32_t)lane));
                dst_bar0 = map_dsmem(smem_u32(&red_full[0]), krank((uint32_t)lane));
                dst_buf1 = map_dsmem(rb + (uint32_t)g.recv_bytes, krank((uint32_t)lane));
                dst_bar1 = map_dsmem(smem_u32(&red_full[1]), krank((uint32_t)lane));
            }
            for (int j = 0; j < ntl; ++j) {
                const int b = j % nacc;
                const uint32_t use_ph = (uint32_t)(j / nacc) & 1u;
                const int n = n_tile_of(j) * 128 + row;
                const int m0 = b_tile_of(j) * outs;
                auto store_y = [&](int m, float z) {
                    if (n < g.N && m < g.M) {
                        const float val = __fmul_rn(gsc, z);
                        const size_t idx = (size_t)m * g.N + n;
                        if (g.out_f32) reinterpret_cast<float*>(g.y)[idx] = val;
                        else reinterpret_cast<__nv_bfloat16*>(g.y)[idx] = __float2bfloat16_rn(val);
                    }
                };
                auto emit = [&](int jj, float z) {
                    if (g.splits > 1) part[jj * 128 + row] = z;
                    else store_y(m0 + jj, z);
                };
                // narrow tiles: outputs o0 .. o0 + 3 go to owner o0 / per_cta, into
                // its receive buffer b at (our rank, channel row), one st.async
                bool send_ok = true;
                const uint32_t rbuf = recv_base + (uint32_t)b * (uint32_t)g.recv_bytes +
                                      (my_rank * 128u + (uint32_t)row) * (uint32_t)per_cta * 4u;
                const uint32_t rbar = smem_u32(&red_full[b]);
                auto emit4 = [&](int o0, float z0, float z1, float z2, float z3) {
                    if (!send_ok || o0 >= owners * per_cta) return;
                    const int o = o0 / per_cta;
                    st_async_v4(map_dsmem(rbuf + (uint32_t)(o0 - o * per_cta) * 4u, krank((uint32_t)o)),
                                make_uint4(__float_as_uint(z0), __float_as_uint(z1), __float_as_uint(z2),
                                           __float_as_uint(z3)),
                                map_dsmem(rbar, krank((uint32_t)o)));
                };
                bool ok = mbar_wait_bounded(smem_u32(&accum_full[b]), use_ph, abort_flag, g.err);
                if (j == 0 && ctid == 0) RS_TRACE_MARK(g.trace, 6);
                if (j < 3 && ctid == 0) RS_TRACE_MARK(g.trace, 22 + j);
                ok = __all_sync(0xFFFFFFFFu, ok && *abort_flag == 0);  // warp-uniform for tcgen05.ld
                tc_fence_after();
                if (xasync && j >= nacc) {
                    // every owner has summed what was sent into buffer b for tile
                    // j - nacc (after a failed wait nothing is sent: the error is recorded)
                    send_ok = mbar_wait_bounded(smem_u32(&recv_free[b]), (uint32_t)(j / nacc - 1) & 1u, abort_flag,
                                                g.err, 1000000000ull, true);
                } else if (g.splits > 1 && j > 0) {
                    // the previous tile's outgoing copies have read our partial
                    if (warp == 8) bulk_wait_group_read0();  // (the issuing lane's copies; no-op on the rest)
                    named_bar_sync(1, 128);
                }
                bool drained = false;
                if constexpr (!FUSED && BN >= 128) {
                    if (ok && g.splits == 1 && !g.out_f32) {
                        // Wide tile, bf16 output: this warp's BN/2 columns go to
                        // registers as scaled bf16 first, the accumulator is
                        // released, and the stores overlap the next tile's MMAs.
                        constexpr int NC = BN / 2;
                        const int cbeg = warp < 4 ? NC : 0;
                        const int jmax = n < g.N ? min(outs, g.M - m0) : 0;
                        const size_t ybase = (size_t)m0 * g.N + (size_t)n;
                        uint32_t pk[NC / 2];  // bf16 pairs, output o in half o & 1 of pk[o / 2]
#pragma unroll
                        for (int q = 0; q < NC / 2; ++q) pk[q] = 0u;
                        auto keep = [&](int o, float z) {
                            const uint32_t hb =
                                (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(gsc, z)));
                            pk[o >> 1] |= (o & 1) ? (hb << 16) : hb;
                        };
#pragma unroll
                        for (int c = 0; c < NC; c += 32) {
                            float v[32];
                            tmem_ld32(tmem + (uint32_t)(b * BN) + quarter + (uint32_t)(cbeg + c), v);
                            if (g.fold) {
#pragma unroll
                                for (int q = 0; q < 16; ++q) keep(c / 2 + q, __fadd_rn(v[2 * q], v[2 * q + 1]));  // Fold
                            } else {
#pragma unroll
                                for (int q = 0; q < 32; ++q) keep(c + q, v[q]);
                            }
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&accum_empty[b]));
                        drained = true;
                        const int obeg = g.fold ? cbeg / 2 : cbeg;
                        const int nout = g.fold ? NC / 2 : NC;
                        __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(g.y) + ybase;
#pragma unroll
                        for (int o = 0; o < NC; ++o)
                            if (o < nout && obeg + o < jmax)
                                yb[(size_t)(obeg + o) * g.N] =
                                    __ushort_as_bfloat16((unsigned short)((o & 1) ? (pk[o >> 1] >> 16) : pk[o >> 1]));
                    }
                }
                if (drained) {
                    // accumulator already released
                } else if (ok && g.splits == 1) {
                    // this warp's columns; output j of the tile at y + (m0 + j) * N + n
                    const int ncol = epi8 ? BN / 2 : BN;
                    const int cbeg = (epi8 && warp < 4) ? ncol : 0;
                    const int jmax = n < g.N ? min(outs, g.M - m0) : 0;
                    const size_t ybase = (size_t)m0 * g.N + (size_t)n;
                    auto put_y = [&](int jj, float z) {
                        if (jj < jmax) {
                            const float val = __fmul_rn(gsc, z);
                            const size_t idx = ybase + (size_t)jj * g.N;
                            if (g.out_f32) reinterpret_cast<float*>(g.y)[idx] = val;
                            else reinterpret_cast<__nv_bfloat16*>(g.y)[idx] = __float2bfloat16_rn(val);
                        }
                    };
                    if (ncol % 32 == 0) {
#pragma unroll 1
                        for (int c = cbeg; c < cbeg + ncol; c += 32) {
                            float v[32];
                            tmem_ld32(tmem + (uint32_t)(b * BN) + quarter + (uint32_t)c, v);
                            if (g.fold) {
#pragma unroll
                                for (int q = 0; q < 16; ++q) put_y(c / 2 + q, __fadd_rn(v[2 * q], v[2 * q + 1]));  // Fold
                            } else {
#pragma unroll
                                for (int q = 0; q < 32; ++q) put_y(c + q, v[q]);
                            }
                        }
                    } else {
                        float v[16];
                        tmem_ld16(tmem + (uint32_t)(b * BN) + quarter + (uint32_t)cbeg, v);
                        if (g.fold) {
#pragma unroll
                            for (int q = 0; q < 8; ++q) put_y(cbeg / 2 + q, __fadd_rn(v[2 * q], v[2 * q + 1]));  // Fold
                        } else {
#pragma unroll
                            for (int q = 0; q < 16; ++q) put_y(cbeg + q, v[q]);
                        }
                    }
                } else if (ok && xasync) {
#pragma unroll 1
                    for (int c = 0; c < BN; c += 16) {
                        float v[16];
                        tmem_ld16(tmem + (uint32_t)(b * BN) + quarter + (uint32_t)c, v);
                        if (g.fold) {
                            float f[8];
#pragma unroll
                            for (int q = 0; q < 8; ++q) f[q] = __fadd_rn(v[2 * q], v[2 * q + 1]);  // Fold
                            emit4(c / 2, f[0], f[1], f[2], f[3]);
                            emit4(c / 2 + 4, f[4], f[5], f[6], f[7]);
                        } else {
#pragma unroll
                            for (int q = 0; q < 16; q += 4) emit4(c + q, v[q], v[q + 1], v[q + 2], v[q + 3]);
                        }
                    }
                } else if (ok) {
#pragma unroll 1
                    for (int c = 0; c < BN; c += 16) {
                        float v[16];
                        tmem_ld16(tmem + (uint32_t)(b * BN) + quarter + (uint32_t)c, v);
                        if (g.fold) {
#pragma unroll
                            for (int q = 0; q < 8; ++q) emit(c / 2 + q, __fadd_rn(v[2 * q], v[2 * q + 1]));  // Fold
                        } else {
#pragma unroll
                            for (int q = 0; q < 16; ++q) emit(c + q, v[q]);
                        }
                    }
                } else if (xasync) {
                    for (int o0 = 0; o0 < outs; o0 += 4) emit4(o0, 0.0f, 0.0f, 0.0f, 0.0f);
                } else if (g.splits > 1) {
                    for (int jj = 0; jj < outs; ++jj) emit(jj, 0.0f);
                }
                // every owner expects a full slice: pad the last one (emit4 drops
                // the outputs past the owners' slices, so each is sent once)
                if (xasync)
                    for (int o0 = outs; o0 < owners * per_cta; o0 += 4) emit4(o0, 0.0f, 0.0f, 0.0f, 0.0f);
                // accumulator b drained: the MMA warp may start its next tile
                if (!drained) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&accum_empty[b]));
                }
                if (j == 0 && ctid == 0) RS_TRACE_MARK(g.trace, 7);
                if (g.splits > 1 && !xasync) {
                    // send each owner its slice of outputs: one bulk copy per
                    // owner into its receive buffer b at our rank's slot
                    fence_proxy_async_smem();
                    named_bar_sync(1, 128);
                    if (j == 0 && ctid == 0) RS_TRACE_MARK(g.trace, 13);
                    if (warp == 8) {
                        // every owner has consumed what was sent into buffer b
                        // for tile j - nacc (the whole warp waits; one elected
                        // lane issues the copies)
                        bool free_ok = j < nacc || mbar_wait_bounded(smem_u32(&recv_free[b]),
                                                                     (uint32_t)(j / nacc - 1) & 1u, abort_flag, g.err,
                                                                     1000000000ull, true);
                        free_ok = __all_sync(0xFFFFFFFFu, free_ok && *abort_flag == 0);
                        if (free_ok && lane < g.splits) {
                            // lane o sends owner o its slice
                            bulk_copy_to_cluster(b == 0 ? dst_buf0 : dst_buf1,
                                                 smem_u32(part) + (uint32_t)lane * slice_bytes, slice_bytes,
                                                 b == 0 ? dst_bar0 : dst_bar1);
                            bulk_commit_group();
                            if (j == 0 && lane == 0) RS_TRACE_MARK(g.trace, 14);
                        }
                        __syncwarp();
                    }
                }
                if (owner) {
                    // own slice: sum the partners' partials in rank order
                    const bool got = mbar_wait_bounded(smem_u32(&red_full[b]), use_ph, abort_flag, g.err,
                                                       1000000000ull, true);
                    if (j == 0 && ctid == 0) RS_TRACE_MARK(g.trace, 28);
                    const float* recv = reinterpret_cast<const float*>(recv_region + (size_t)b * g.recv_bytes);
                    const bool live = got && *abort_flag == 0;
                    if (xasync) {
                        // receive layout [rank][channel][per_cta], four outputs at a time
                        for (int j4 = 0; live && j4 < per_cta; j4 += 4) {
                            const int jo = split * per_cta + j4;
                            if (jo >= xouts) break;
                            float4 pv[kMaxSplits];
#pragma unroll
                            for (int r = 0; r < kMaxSplits; ++r)
                                pv[r] = r < g.splits ? *reinterpret_cast<const float4*>(
                                                           recv + ((size_t)r * 128 + row) * per_cta + j4)
                                                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                            for (int r = 0; r < kMaxSplits; ++r)
                                if (r < g.splits) {
                                    acc.x = __fadd_rn(acc.x, pv[r].x);
                                    acc.y = __fadd_rn(acc.y, pv[r].y);
                                    acc.z = __fadd_rn(acc.z, pv[r].z);
                                    acc.w = __fadd_rn(acc.w, pv[r].w);
                                }
                            store_y(m0 + jo, acc.x);
                            store_y(m0 + jo + 1, acc.y);
                            store_y(m0 + jo + 2, acc.z);
                            store_y(m0 + jo + 3, acc.w);
                        }
                    } else {
                        // receive layout [rank][output][channel]
                        for (int jj = 0; live && jj < per_cta; ++jj) {
                            const int jo = split * per_cta + jj;
                            if (jo >= outs) break;
                            // all partials first, then the sum in rank order
                            float pv[kMaxSplits];
#pragma unroll
                            for (int r = 0; r < kMaxSplits; ++r)
                                pv[r] = r < g.splits ? recv[(r * per_cta + jj) * 128 + row] : 0.0f;
                            float acc = 0.0f;
#pragma unroll
                            for (int r = 0; r < kMaxSplits; ++r)
                                if (r < g.splits) acc = __fadd_rn(acc, pv[r]);
                            store_y(m0 + jo, acc);
                        }
                    }
                    if (j < 3 && ctid == 0) RS_TRACE_MARK(g.trace, 25 + j);
                    if (j + nacc < ntl) {
                        // buffer b is read: re-arm it for tile j + nacc, then
                        // tell every partner it may send into it again
                        named_bar_sync(1, 128);
                        if (ctid == 0 && *abort_flag == 0) {
                            mbar_arrive_expect_tx(smem_u32(&red_full[b]), red_bytes);
                            for (int p = 0; p < g.splits; ++p)
                                mbar_arrive_remote(map_dsmem(smem_u32(&recv_free[b]), krank((uint32_t)p)));
                        }
                    }
                }
            }
            if (g.splits > 1 && !xasync && warp == 8) bulk_wait_group_read0();  // outgoing copies have read their source
        }
    }

    __syncwarp();
    if (threadIdx.x == 0) RS_TRACE_MARK(g.trace, 9);

    // ---------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {  // CTA-uniform here: every role has finished
        if (warp == 4 && lane == 0) {
            // Let every copy still in flight land before the CTA exits.
            for (uint32_t u = *consumed; u < *issued; ++u) {
                const uint32_t s = u % (uint32_t)S;
                volatile uint32_t no_abort = 0;
                (void)mbar_wait_bounded(smem_u32(&full[s]), (u / (uint32_t)S) & 1u, &no_abort, nullptr,
                                        100000000ull);
            }
        }
        __syncthreads();
    }
    if (warp == 5 && !tmem_freed) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)g.tmem_cols);
        if (lane == 0) RS_TRACE_MARK(g.trace, 10);
    }
    // multicast: neither CTA leaves while the other may still write into it
    if (mcast) cluster_sync_all();
}

// Separate Fold (Sec. 4.3 Eq. 2) for the on-chip Fold ablation (Sec. 5.1,
// Fig. 6b): y[j][n] = z[2j][n] + z[2j+1][n] from an expanded fp32 output of
// the paired rows; four outputs per thread when N % 4 == 0.
__global__ void __launch_bounds__(256) fold_pairs_kernel(const float* __restrict__ z, void* __restrict__ y, int M,
                                                         int N, int out_f32) {
    const bool vec = (N & 3) == 0;
    const int64_t per_row = vec ? N / 4 : N;
    const int64_t total = (int64_t)M * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = i / per_row, c = i - j * per_row;
        if (vec) {
            const float4 a = reinterpret_cast<const float4*>(z + (2 * j) * N)[c];
            const float4 b = reinterpret_cast<const float4*>(z + (2 * j + 1) * N)[c];
            const float4 v = make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
            if (out_f32) {
                reinterpret_cast<float4*>(static_cast<float*>(y) + j * N)[c] = v;
            } else {
                __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
                uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
                reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(y) + j * N)[c] = pk;
            }
        } else {
            const float v = __fadd_rn(z[(2 * j) * N + c], z[(2 * j + 1) * N + c]);
            if (out_f32) static_cast<float*>(y)[j * N + c] = v;
            else static_cast<__nv_bfloat16*>(y)[j * N + c] = __float2bfloat16_rn(v);
        }
    }
}

// ------------------------------------------------------------------- host --

cudaError_t launch_fold_pairs(const float* z, void* y, int M, int N, int out_f32, cudaStream_t stream, int num_sms) {
    const int64_t work = (int64_t)M * (((N & 3) == 0) ? N / 4 : N);
    const int64_t blocks = std::min<int64_t>((work + 255) / 256, (int64_t)num_sms * 8);
    fold_pairs_kernel<<<(unsigned)std::max<int64_t>(blocks, 1), 256, 0, stream>>>(z, y, M, N, out_f32);
    return cudaGetLastError();
}

// Split-K buffers: each receive buffer holds `splits` slices of
// split_slice(outs, splits) outputs x 128 channels (fp32); tiles sent by bulk
// copy also stage their partial (the same size) in shared memory.
static size_t split_buf_bytes(int splits, int outs) {
    if (splits <= 1) return 0;
    return align_up((size_t)splits * split_slice(outs, splits) * 128 * sizeof(float), 1024);
}

static size_t plan_smem(int fmt, int bn, int stages, bool fused, int slots, size_t splitbuf, int nacc,
                        size_t partbuf) {
    const size_t b = fused ? (size_t)slots * b_stage_bytes(fmt, bn) : (size_t)stages * b_stage_bytes(fmt, bn);
    return 1024 + (size_t)stages * weight_block_bytes(fmt) + b + partbuf + splitbuf * (size_t)nacc + kCtrlBytes;
}

// Complete plan for a given split count s; stages == 0 when it does not fit.
// bn_min: the MMA width, at least the one the activation rows need (a measured
// tactic may ask for a wider one; the extra operand rows are zero).  pair_ok:
// a fused plan lets CTA pairs share the quantization of their K slice (only
// on a measured tactic's request: on GB300 the remote stores and the wider
// clusters cost more than the halved quantizer saves for every shape tuned).
// deep: a split plan whose CTAs take one tile each keeps its deepest weight
// ring instead of the shallower one that lets two CTAs share an SM.
static GemmPlan plan_for_splits(int fmt, bool fold, int M, int N, int K, int sms, int s, bool allow_fused,
                                int bn_min = 16, bool pair_ok = false, bool deep = false) {
    GemmPlan p{};
    p.fmt = fmt;
    p.fold = fold ? 1 : 0;
    p.M = M;
    p.N = N;
    p.K = K;
    p.Rb = fold ? 2 * M : M;
    p.bn = p.Rb <= 16 ? 16 : p.Rb <= 32 ? 32 : p.Rb <= 64 ? 64 : p.Rb <= 128 ? 128 : 256;
    p.bn = std::max(p.bn, std::min(bn_min, 256));
    p.n_tiles = (N + 127) / 128;
    p.b_tiles = (p.Rb + p.bn - 1) / p.bn;
    p.chunks = (K + 255) / 256;
    const int tiles = p.n_tiles * p.b_tiles;
    // persistent grid: gridDim.x CTAs per K split, CTA x taking tiles x,
    // x + gridDim.x, ...; one CTA per SM
    p.splits = s;
    p.grid_x = std::min(tiles, std::max(1, sms / s));
    const int max_chunks = (p.chunks + s - 1) / s;
    const int ntl = (tiles + p.grid_x - 1) / p.grid_x;
    const int nu = ntl * max_chunks;
    const int outs = fold ? p.bn / 2 : p.bn;
    const size_t splitbuf = split_buf_bytes(s, outs);
    const size_t partbuf = split_async(outs) ? 0 : splitbuf;
    const int sfc = sf_cols_per_stage(fmt, p.bn);
    bool fused = allow_fused && p.b_tiles == 1 && p.bn <= 32 && max_chunks <= kMaxChunkBars;
    // two accumulators let the epilogue of one tile overlap the next tile's
    // MMAs when a CTA has several tiles
    int nacc = ntl > 1 ? 2 : 1;
    auto fits = [&](int st, bool fu, int na) {
        return plan_smem(fmt, p.bn, st, fu, fu ? max_chunks : 0, splitbuf, na, partbuf) <= kSmemLimit &&
               na * p.bn + st * sfc <= 512;
    };
    auto best_stages = [&](bool fu, int na) {
        int st = std::min(kMaxStages, nu);
        while (st > 1 && !fits(st, fu, na)) --st;
        return fits(st, fu, na) ? st : 0;
    };
    int stages = best_stages(fused, nacc);
    if (nacc == 2 && stages < std::min(4, nu)) {
        const int st1 = best_stages(fused, 1);
        if (st1 > stages) {
            nacc = 1;
            stages = st1;
        }
    }
    // a resident slice that leaves the weight ring fewer than three stages
    // starves the MMAs: quantize in a separate launch then
    if (fused && stages < std::min(3, nu)) {
        fused = false;
        stages = best_stages(false, nacc);
    }
    // A split plan's CTAs form clusters, and a whole cluster must fit into one
    // GPC: with one CTA per SM fewer clusters are resident at once than with
    // two, and the rest wait for a second wave.  A split plan whose CTAs take
    // one tile each keeps three stages (or all its units) when that lets two
    // CTAs share an SM; plans that stream several tiles keep the deep ring.
    if (s > 1 && ntl == 1 && !deep) {
        const int floor_st = std::min(3, nu);
        while (stages > floor_st &&
               plan_smem(fmt, p.bn, stages, fused, fused ? max_chunks : 0, splitbuf, nacc, partbuf) > kSmemLimit / 2 &&
               plan_smem(fmt, p.bn, floor_st, fused, fused ? max_chunks : 0, splitbuf, nacc, partbuf) <= kSmemLimit / 2)
            --stages;
    }
    p.fused = fused ? 1 : 0;
    // CTA pairs (fused plans with an even number of CTAs per K split): the
    // cluster grows to two neighbouring channel tiles per split, each
    // quantizing every other chunk of the shared slice into both CTAs'
    // shared memory (one store to each, one arrival on each CTA's barrier).
    p.qpair = (fused && pair_ok && p.grid_x % 2 == 0 && 2 * s <= kMaxSplits && max_chunks >= 2) ? 1 : 0;
    p.nacc = nacc;
    p.stages = stages;
    p.slots = p.fused ? max_chunks : 0;
    p.part_bytes = (int)partbuf;
    p.recv_bytes = (int)splitbuf;
    if (stages == 0) return p;
    // Two CTAs can share an SM when the shared memory allows it (a dependent
    // launch starting early); keep the tensor-memory allocation within half
    // of the SM's 512 columns then.
    p.smem_bytes = plan_smem(fmt, p.bn, p.stages, p.fused, p.slots, splitbuf, p.nacc, partbuf);
    int cols = p.nacc * p.bn + p.stages * sfc;
    if (p.smem_bytes <= kSmemLimit / 2) {
        while (cols > 256 && p.stages > 1) {
            --p.stages;
            cols = p.nacc * p.bn + p.stages * sfc;
        }
        p.smem_bytes = plan_smem(fmt, p.bn, p.stages, p.fused, p.slots, splitbuf, p.nacc, partbuf);
    }
    int alloc = 32;
    while (alloc < cols) alloc *= 2;
    p.tmem_cols = alloc;
    // more than half of the tensor memory: never two such CTAs on one SM
    // (the second one's allocation would wait for the first to finish)
    if (alloc > 256 && p.smem_bytes <= kSmemLimit / 2) p.smem_bytes = kSmemLimit / 2 + 1024;
    return p;
}

// Split count: minimise the chunks the busiest CTA streams, plus, for a split
// plan whose CTAs take several tiles, 1.5 x splits chunks per extra tile (the
// cross-CTA reduction of every tile holds the whole cluster: measured about
// 0.75 x splits us per tile against 0.4 us per streamed chunk); prefer fewer
// splits on a tie.  A split plan must keep a pipeline of at least four stages
// (three when its CTAs take one tile each and two of them share an SM), or
// all of its units, next to its split-K buffers.  A plan that could
// quantize inside the GEMM but does not fit it is charged 7 chunks for the
// separate quantizer launch and the operand's round trip.
static GemmPlan plan_impl(int fmt, bool fold, int M, int N, int K, int num_sms, bool allow_fused) {
    const int sms = num_sms > 0 ? num_sms : 148;
    const int chunks = (K + 255) / 256;
    GemmPlan best = plan_for_splits(fmt, fold, M, N, K, sms, 1, allow_fused);
    if (best.stages == 0) best.stages = 1;  // cannot happen for the supported tile shapes
    auto load_of = [&](const GemmPlan& p) {  // in half chunks
        const int tiles = p.n_tiles * p.b_tiles;
        const long ntl = (tiles + p.grid_x - 1) / p.grid_x;
        const long streamed = 2 * ntl * (long)((p.chunks + p.splits - 1) / p.splits);
        return streamed + (p.splits > 1 ? 3 * (ntl - 1) * p.splits : 0) + (allow_fused && !p.fused ? 14 : 0);
    };
    long best_load = load_of(best);
    auto ntl_of = [](const GemmPlan& p) {
        const int tiles = p.n_tiles * p.b_tiles;
        return (tiles + p.grid_x - 1) / p.grid_x;
    };
    for (int s = 2; s <= std::min(chunks, kMaxSplits); ++s) {
        const GemmPlan p = plan_for_splits(fmt, fold, M, N, K, sms, s, allow_fused);
        const int tiles = p.n_tiles * p.b_tiles;
        const int nu = ((tiles + p.grid_x - 1) / p.grid_x) * ((chunks + s - 1) / s);
        const bool capped = ntl_of(p) == 1 && p.smem_bytes <= kSmemLimit / 2;  // two CTAs per SM
        if (p.stages < std::min(capped ? 3 : 4, nu)) continue;
        const long load = load_of(p);
        if (load < best_load) {
            best = p;
            best_load = load;
        }
    }
    return best;
}

// The paired-CTA kernel (rs_gemm_pair.cu) is chosen only on request: on
// this GPU the single-CTA kernel is faster for every shape measured (the
// pair's stages land at about 52 GB/s per SM from L2 against about 81 GB/s
// for the single-CTA kernel's larger stages).
static int g_pair_gemm = 0;

GemmPlan make_gemm_plan_analytic(int fmt, bool fold, int M, int N, int K, int num_sms, bool allow_fused) {
    return plan_impl(fmt, fold, M, N, K, num_sms, allow_fused);
}

GemmPlan make_gemm_plan(int fmt, bool fold, int M, int N, int K, int num_sms, bool allow_fused) {
    GemmPlan p = plan_impl(fmt, fold, M, N, K, num_sms, allow_fused);
    Tactic t;
    if (num_sms > 0 && find_tactic(fmt, fold, M, N, K, num_sms, &t) && t.splits <= (K + 255) / 256) {
        const GemmPlan q =
            plan_for_splits(fmt, fold, M, N, K, num_sms, t.splits, allow_fused && t.fused, t.bn, t.fused == 2,
                            t.deep != 0);
        if (q.stages > 0) {
            p = q;
            p.tuned = 1;
        }
    }
    // Operands of at least two 256-row activation tiles with an even number
    // of channel tiles can run on the pair kernel, whose two SMs share one
    // 256 x 256 MMA and each stage half the activation bytes.
    p.pair = (g_pair_gemm && !p.fused && p.Rb >= 512 && p.n_tiles % 2 == 0) ? 1 : 0;
    return p;
}

void set_pair_gemm(int enable) { g_pair_gemm = enable ? 1 : 0; }

size_t plan_b_stage_bytes(const GemmPlan& p) { return b_stage_bytes(p.fmt, p.bn); }

size_t alpha_slot_offset(int fmt, bool compensated, int M, int K) {
    return align_up(operand_bytes(fmt, compensated ? 2 * M : M, K), 1024);
}

size_t workspace_bytes(int fmt, bool compensated, int M, int K) {
    return alpha_slot_offset(fmt, compensated, M, K) + 256;  // + the activation tensor scale
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

// Activation codes: [rows][K/2] bytes, box = 128 bytes (256 K) x box_rows,
// 128-byte swizzle (the image the K-major SW128 descriptor reads).
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
template <int FMT, int BN, bool FUSED>
static cudaError_t ensure_smem_attr() {
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(gemm_kernel<FMT, BN, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemLimit);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

bool multicast_eligible(const GemmPlan& p) {
    // (with one tile per CTA the pair's lock step measured slower)
    return sf_by_warps(p.bn, p.fused != 0) && p.splits == 1 && p.n_tiles % 2 == 0 && p.grid_x >= 2 &&
           p.n_tiles * p.b_tiles >= 2 * p.grid_x;
}

// The kernels with scale warps (TMA-fed, 256-row activation tiles).
static const void* scale_warp_kernel(int fmt) {
    return fmt == 0 ? (const void*)gemm_kernel<0, 256, false> : (const void*)gemm_kernel<1, 256, false>;
}

// Clusters of two CTAs of `func` that can be resident at once on the current
// device (0 when none), per device and shared-memory size.
static int pair_clusters_resident(const void* func, size_t smem, int threads) {
    static std::mutex mu;
    static int cache_dev[16] = {};
    static size_t cache_smem[16] = {};
    static const void* cache_fn[16] = {};
    static int cache_n[16] = {};
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < used; ++i)
            if (cache_dev[i] == dev && cache_smem[i] == smem && cache_fn[i] == func) return cache_n[i];
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2u, 1u, 1u);
    cfg.blockDim = dim3((unsigned)threads, 1u, 1u);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (used < 16) {
        cache_dev[used] = dev;
        cache_smem[used] = smem;
        cache_fn[used] = func;
        cache_n[used] = n;
        ++used;
    }
    return n;
}

template <int FMT, int BN, bool FUSED>
static cudaError_t launch_typed(const GemmPlan& p, const CUtensorMap& tb, const GemmArgs& args, cudaStream_t stream) {
    cudaError_t e = ensure_smem_attr<FMT, BN, FUSED>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)p.grid_x, 1u, (unsigned)p.splits);
    cfg.blockDim = dim3((unsigned)gemm_threads(BN, FUSED), 1, 1);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.splits > 1 || p.qpair || args.mcast) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (p.qpair || args.mcast) ? 2 : 1;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = (unsigned)p.splits;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<FMT, BN, FUSED>, tb, args);
}

#ifdef RS_TRACE
static uint64_t* g_trace = nullptr;
#endif

uint64_t* trace_buffer() {
#ifdef RS_TRACE
    return g_trace;
#else
    return nullptr;
#endif
}

cudaError_t launch_gemm(const GemmPlan& p, const GemmCall& c, cudaStream_t stream) {
    if (p.pair) {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
#ifdef RS_TRACE
        uint64_t* trace = g_trace;
#else
        uint64_t* trace = nullptr;
#endif
        return launch_gemm_pair(p.fmt, p.M, p.Rb, p.N, p.K, p.fold, c.xq, c.wq, c.alpha_x, c.alpha_w, c.y, c.out_f32,
                                c.err, trace, sms, stream);
    }
    // Scale-warp plans without split whose channel tiles pair up share each
    // activation tile between the two CTAs of a cluster (multicast), on a
    // persistent grid of the pair clusters that fit at once.  Prefill GEMM
    // (M = 4096, K = N = 8192): 123.8 -> 116.2 us W4A4, 229.6 -> 212.2 us
    // compensated.
    GemmPlan q = p;
    int mcast = 0;
    if (multicast_eligible(q)) {
        const int pairs = pair_clusters_resident(scale_warp_kernel(q.fmt), q.smem_bytes,
                                                 gemm_threads(q.bn, false));
        const int grid = std::min(q.grid_x / 2, pairs) * 2;
        if (grid >= 2) {
            q.grid_x = grid;
            mcast = 1;
        }
    }
    alignas(64) CUtensorMap tb;
    std::memset(&tb, 0, sizeof tb);
    if (!q.fused && !encode_codes_map(&tb, c.xq, q.Rb, q.K, mcast ? q.bn / 2 : q.bn)) return cudaErrorInvalidValue;
    GemmArgs a{};
    a.wq = static_cast<const uint8_t*>(c.wq);
    a.x = static_cast<const uint16_t*>(c.x);
    a.sfb = p.fused ? nullptr : static_cast<const uint8_t*>(c.xq) + operand_sf_offset(p.fmt, p.Rb, p.K);
    a.y = c.y;
    a.alpha_x = c.alpha_x;
    a.alpha_w = c.alpha_w;
    a.err = c.err;
#ifdef RS_TRACE
    a.trace = g_trace;
#else
    a.trace = nullptr;
#endif
    a.N = p.N;
    a.K = p.K;
    a.M = p.M;
    a.Rb = p.Rb;
    a.n_atoms_k = n_atoms_k_host(p.fmt, p.K);
    a.b_row_tiles = (p.Rb + 127) / 128;
    a.chunks = p.chunks;
    a.splits = p.splits;
    a.fold = p.fold;
    a.out_f32 = c.out_f32;
    a.stages = p.stages;
    a.slots = p.slots;
    a.n_tiles = p.n_tiles;
    a.b_tiles = p.b_tiles;
    a.nacc = p.nacc;
    a.recv_bytes = p.recv_bytes;
    a.tmem_cols = p.tmem_cols;
    a.part_bytes = p.part_bytes;
    a.dyn_alpha = c.dyn_alpha;
    a.qpair = p.fused ? p.qpair : 0;
    a.qdump = p.fused ? static_cast<uint8_t*>(c.qdump) : nullptr;
    a.mcast = mcast;
#define RS_CASE(F, B, FU)                                                      \
    if (q.fmt == F && q.bn == B && (q.fused != 0) == FU) return launch_typed<F, B, FU>(q, tb, a, stream);
    RS_CASE(0, 16, true) RS_CASE(0, 32, true) RS_CASE(1, 16, true) RS_CASE(1, 32, true)
    RS_CASE(0, 16, false) RS_CASE(0, 32, false) RS_CASE(0, 64, false) RS_CASE(0, 128, false) RS_CASE(0, 256, false)
    RS_CASE(1, 16, false) RS_CASE(1, 32, false) RS_CASE(1, 64, false) RS_CASE(1, 128, false) RS_CASE(1, 256, false)
#undef RS_CASE
    return cudaErrorInvalidValue;
}

}  // namespace rs

#ifdef RS_TRACE
// Trace builds only: set the device buffer (32 uint64 per CTA) that the next
// GEMM launches stamp (32 per CTA); NULL turns tracing off.
extern "C" __attribute__((visibility("default"))) void rs_debug_set_trace(void* buf) {
    rs::g_trace = static_cast<uint64_t*>(buf);
}
#endif
