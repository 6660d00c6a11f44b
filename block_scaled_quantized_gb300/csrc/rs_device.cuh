// Device-side building blocks for librs (sm_103a): FP4 / FP8 / E8M0 codecs,
// the scale-atom layout, and thin inline-PTX wrappers around mbarrier, TMA,
// and the tcgen05 tensor-memory / MMA instructions.
//
// Formats follow ResServe (arXiv 2611.08713) Sec. 2 and App. B.2 Eq. 8-10;
// the scale layout is the one the block-scaled tcgen05 MMA consumes after a
// 32x128b.warpx4 copy into tensor memory.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace rs {

// ------------------------------------------------------------- constants --

constexpr int kNvBlock = 16;          // NVFP4 elements per E4M3 scale
constexpr int kMxBlock = 32;          // MXFP4 elements per E8M0 scale
constexpr int kAtomRows = 128;        // rows per scale atom
constexpr int kAtomBlocks = 4;        // scale bytes per row per atom
constexpr int kAtomBytes = 512;       // bytes per scale atom
constexpr float kE2M1Max = 6.0f;      // App. B.2: largest E2M1 magnitude

// Device error word values (mirror rs_status).
constexpr uint32_t kErrInvalidArg = 1;
constexpr uint32_t kErrTimeout = 7;

__host__ __device__ constexpr int block_elems(int fmt) { return fmt == 0 ? kNvBlock : kMxBlock; }

// Elements of K covered by one scale atom (4 blocks).
__host__ __device__ constexpr int atom_k(int fmt) { return kAtomBlocks * block_elems(fmt); }

// Tiled weight operand: one block per (128 output channels, 256 K) holding
// the codes (128 rows x 128 bytes, 128-byte-swizzled shared-memory image)
// followed by the block's scale atoms.
constexpr int kWeightCodeBytes = 128 * 128;
__host__ __device__ constexpr int weight_atoms_per_block(int fmt) { return 256 / atom_k(fmt); }
__host__ __device__ constexpr uint32_t weight_block_bytes(int fmt) {
    return (uint32_t)kWeightCodeBytes + (uint32_t)weight_atoms_per_block(fmt) * (uint32_t)kAtomBytes;
}

// Byte offset of the scale of (row r, block b) inside the scale region of an
// operand whose atoms per row tile along K is n_atoms_k.
__host__ __device__ inline size_t sf_offset(int r, int b, int n_atoms_k) {
    size_t atom = (size_t)(r / kAtomRows) * n_atoms_k + (size_t)(b / kAtomBlocks);
    return atom * kAtomBytes + (size_t)(r % 32) * 16 + (size_t)((r / 32) % 4) * 4 + (b % 4);
}

// ------------------------------------------------------------------ codecs --

// E2M1 round-to-nearest-even with saturation at +-6 and the sign kept.  The
// seven thresholds are the midpoints of the grid {0,.5,1,1.5,2,3,4,6}; a tie
// resolves to the even code, hence the alternating > / >= comparisons.
__device__ __forceinline__ uint32_t e2m1_encode(float v) {
    const float a = fabsf(v);
    uint32_t idx = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                   (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
                   (uint32_t)(a > 5.0f);
    return idx | ((__float_as_uint(v) >> 28) & 8u);
}

// E2M1 code -> fp32 (exact).  Twice the magnitude is 0,1,2,3,4,6,8,12.
__device__ __forceinline__ float e2m1_decode(uint32_t c) {
    const uint32_t i = c & 7u;
    const uint32_t twice = i < 2u ? i : ((2u + (i & 1u)) << ((i >> 1) - 1u));
    const float m = (float)twice * 0.5f;
    return (c & 8u) ? -m : m;
}

// Eight fp32 values -> eight E2M1 codes (element e in bits 4e..4e+3) with the
// hardware conversion (round to nearest even, saturating to +-6, sign kept;
// identical to e2m1_encode on every input, including ties and signed zero).
__device__ __forceinline__ uint32_t e2m1_encode8(const float (&v)[8]) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// Eight E2M1 codes (as packed by e2m1_encode8) -> eight exact fp32 values.
__device__ __forceinline__ void e2m1_decode8(uint32_t codes, float (&v)[8]) {
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(codes));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 p = *reinterpret_cast<const __half2*>(&h[i]);
        v[2 * i] = __low2float(p);
        v[2 * i + 1] = __high2float(p);
    }
}

// 2^e as fp32 for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// E4M3 byte (sign 0, finite) -> fp32 (exact).
__device__ __forceinline__ float e4m3_decode(uint32_t b) {
    const uint32_t E = (b >> 3) & 15u, m = b & 7u;
    return E == 0 ? (float)m * exp2i(-9) : (float)(8u + m) * exp2i((int)E - 10);
}

// Non-negative fp32 -> E4M3 byte, round to nearest even, saturating to 448.
// The value is scaled by an exact power of two so that one E4M3 quantum
// becomes 1, rounded to an integer with rintf (ties to even), and re-encoded.
__device__ __forceinline__ uint32_t e4m3_encode_satfinite(float t) {
    if (!(t < 448.0f)) return 0x7Eu;
    const int e = (int)(__float_as_uint(t) >> 23) - 127;  // floor(log2 t); -127 for 0/subnormal
    const int qe = (e < -6 ? -6 : e) - 3;                  // log2 of the quantum
    const float n = rintf(t * exp2i(-qe));                  // exact scaling, RNE
    const uint32_t ni = (uint32_t)n;
    if (e < -6) return ni;                                 // subnormal; 8 -> 0x08 (2^-6)
    return ((uint32_t)(e + 7) << 3) + ni - 8u;             // 16 carries into the exponent
}

// Two fp32 products / differences in one packed instruction (mul/sub.rn.f32x2,
// each half rounded to nearest even like __fmul_rn / __fsub_rn).
__device__ __forceinline__ void fmul2_rn(float a0, float a1, float b0, float b1, float& r0, float& r1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rc, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void fsub2_rn(float a0, float a1, float b0, float b1, float& r0, float& r1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rc, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Hardware E4M3 conversions: cvt.rn.satfinite.e4m3x2.f32 (round to nearest
// even, finite inputs above 448 saturate to 448) and cvt.rn.f16x2.e4m3x2
// (exact).  On every non-negative finite float and every finite byte they
// agree with e4m3_encode_satfinite / e4m3_decode above.
// Two floats -> two bytes: `a` in bits 8-15, `b` in bits 0-7.
__device__ __forceinline__ uint32_t e4m3x2_encode_hw(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float e4m3_decode_hw(uint32_t byte) {
    uint32_t h2;
    const uint16_t b16 = (uint16_t)byte;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(b16));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// ------------------------------------------------------------ misc helpers --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One lane of the (converged) warp is elected.  Work issued by the elected
// lane inside a warp-wide loop keeps its operands warp-uniform, which the
// tensor-pipe issue of tcgen05.mma / tcgen05.cp needs to run at full rate.
__device__ __forceinline__ bool elect_one_sync() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .b32 r;\n\t.reg .pred p;\n\t"
        "elect.sync r|p, 0xffffffff;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// `count` arrivals at once (one thread standing for the blocks of its warp).
__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with cluster-scope acquire: for phases completed by arrivals
// from other CTAs of the cluster (mbar_arrive_remote).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Arrive on an mbarrier of another CTA of the cluster (address from
// map_dsmem), releasing this thread's prior shared-memory accesses at
// cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
// The same with an arrival count.
__device__ __forceinline__ void mbar_arrive_remote_cnt(uint32_t bar_cluster, uint32_t n) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(bar_cluster), "r"(n)
                 : "memory");
}

// Bounded wait for the phase with the given parity to complete.  Gives up
// after `limit_ns` of wall-clock time or as soon as *abort becomes non-zero;
// on a timeout it records kErrTimeout in the device error word and raises
// the CTA's abort flag so that the other roles stop too.  Returns true when
// the phase completed.
// With `cluster` the wait acquires at cluster scope.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t* abort, uint32_t* err,
                                                  uint64_t limit_ns = 1000000000ull, bool cluster = false) {
    auto try_once = [&]() { return cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (try_once()) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (try_once()) return true;
        if ((it & 63u) == 0u) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                *abort = 1u;
                if (err) atomicExch(err, kErrTimeout);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled TMA load into (CTA-local) shared memory, completion on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int x,
                                            int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// The same 2-D load multicast to the CTAs of `mask` in the cluster: the box
// lands at the same shared-memory offset in each, and each one's mbarrier at
// the offset of `bar` receives the completed bytes.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const void* tmap, uint32_t bar, int x, int y,
                                               uint16_t mask, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5, %6;" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar), "h"(mask), "l"(policy)
        : "memory");
}

// Bulk copy global -> shared multicast to the CTAs of `mask` (same offsets).
__device__ __forceinline__ void bulk_load_mc(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                             uint16_t mask, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4, %5;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "h"(mask), "l"(policy)
        : "memory");
}

// Non-tensor bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy
// (TMA, tcgen05.cp, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// The same for every state space (stores into other CTAs' shared memory).
__device__ __forceinline__ void fence_proxy_async_all() {
    asm volatile("fence.proxy.async;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05 --

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address >> 4 in
// bits 0-13, leading-dimension byte offset >> 4 in bits 16-29, stride
// byte offset >> 4 in bits 32-45, the fixed value 0b001 in bits 46-48,
// base offset 0, and the swizzle mode in bits 61-63 (0 none, 2 = 128-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)(swizzle & 7u) << 61;
    return d;
}

// K-major operand tile with 128-byte rows and the 128-byte swizzle: 8-row
// groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t addr) {
    return smem_desc(addr, 16, 1024, 2);
}

// Scale atom (32 rows x 16 bytes, contiguous, no swizzle) as the source of
// a 32x128b tcgen05.cp.
__device__ __forceinline__ uint64_t sf_atom_desc(uint32_t addr) { return smem_desc(addr, 0, 128, 0); }

// Copy one 512-byte scale atom from shared memory into 4 tensor-memory
// columns, replicated into all four 32-lane quarters.
__device__ __forceinline__ void tc_cp_sf_atom(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// Instruction descriptor of kind::mxf4nvf4 (dense, K = 64): A and B E2M1
// (format code 1) in K-major layout, N >> 3 in bits 17-22, scale type in bit
// 23 (0 = UE4M3, 1 = UE8M0), M >> 4 in bits 24-28, and the scale-factor byte
// selectors for B (bits 4-5) and A (bits 29-30).
__host__ __device__ constexpr uint32_t mxf4_idesc(int n, bool ue8m0, uint32_t sf_id) {
    return (sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((ue8m0 ? 1u : 0u) << 23) | ((uint32_t)(128 >> 4) << 24) | (sf_id << 29);
}

// One block-scaled MMA: D[128 x N] (+)= A[128 x 64] * B[N x 64]^T with UE4M3
// scales per 16 elements (NVFP4) ...
__device__ __forceinline__ void mma_nvfp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// ... or UE8M0 scales per 32 elements (MXFP4).
__device__ __forceinline__ void mma_mxfp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// Arrive on `bar` once all previously issued tcgen05 async operations of
// this thread have completed.
// Arrive on `bar` at the same offset in each CTA of `mask` once this
// thread's earlier tcgen05 operations are done.
__device__ __forceinline__ void tc_commit_mc(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 lanes x 32-bit, 16 consecutive columns -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32-bit, 32 consecutive columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 8 / 16 consecutive 32-bit columns of this warp's 32 tensor-memory
// lanes (thread l: lane l of the warp's quarter, register c: column taddr + c).
// Asynchronous: tmem_st_wait() before another thread may read the columns.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// N (8, 16 or 32) consecutive columns from registers.
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
    static_assert(N == 8 || N % 16 == 0, "8 or a multiple of 16 columns");
    if constexpr (N == 8) {
        tmem_st8(taddr, r);
    } else {
#pragma unroll
        for (int h = 0; h < N / 16; ++h)
            tmem_st16(taddr + (uint32_t)(16 * h), *reinterpret_cast<const uint32_t(*)[16]>(&r[16 * h]));
    }
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// --------------------------------------------------- clusters and DSMEM --

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Whole-cluster barrier; every thread of every CTA in the cluster executes
// it (warp-converged).  Release/acquire order shared-memory traffic.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_dsmem(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Bulk copy from this CTA's shared memory into another CTA's shared memory
// in the cluster, completing bytes on that CTA's mbarrier (both cluster
// addresses from map_dsmem); 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                                     uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst_cluster),
        "r"(src_cta), "r"(bytes), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until every committed bulk copy of this thread has finished reading
// its source.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_u8(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u8 [%0], %1;" ::"r"(addr), "h"((unsigned short)v) : "memory");
}
__device__ __forceinline__ void st_dsmem_v2(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st_dsmem_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Asynchronous 4-byte store into another CTA's shared memory (cluster
// address from map_dsmem), completing 4 bytes of transaction count on that
// CTA's mbarrier, whose waiters then see the value.
__device__ __forceinline__ void st_async_b32(uint32_t dst_cluster, uint32_t v, uint32_t bar_cluster) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(dst_cluster),
                 "r"(v), "r"(bar_cluster)
                 : "memory");
}

// Asynchronous 16-byte store into another CTA's shared memory (cluster
// addresses from map_dsmem, 16-byte aligned); completes 16 bytes of
// transaction count on that CTA's mbarrier, whose waiters then see the data.
__device__ __forceinline__ void st_async_v4(uint32_t dst_cluster, uint4 v, uint32_t bar_cluster) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     dst_cluster),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar_cluster)
                 : "memory");
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ------------------------------------------------------ named CTA barriers --

// Named barrier over `nthreads` threads (non-aligned form: callers may reach
// it from divergent paths within a warp).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------ trace build only --
// Built with -DRS_TRACE, kernels stamp the global timer at phase boundaries
// into a caller-provided buffer (32 slots per CTA); a normal build compiles
// the marks away.
#ifdef RS_TRACE
#define RS_TRACE_MARK(buf, slot)                                                              \
    do {                                                                                      \
        if (buf) {                                                                            \
            const size_t cta = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x; \
            (buf)[cta * 32 + (slot)] = rs::globaltimer_ns();                                  \
        }                                                                                     \
    } while (0)
#define RS_TRACE_VALUE(buf, slot, v)                                                          \
    do {                                                                                      \
        if (buf) {                                                                            \
            const size_t cta = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x; \
            (buf)[cta * 32 + (slot)] = (uint64_t)(v);                                         \
        }                                                                                     \
    } while (0)
#else
#define RS_TRACE_MARK(buf, slot) do { } while (0)
#define RS_TRACE_VALUE(buf, slot, v) do { } while (0)
#endif

// ---------------------------------------------- programmatic launch (PDL) --

__device__ __forceinline__ void pdl_wait_prior_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace rs
