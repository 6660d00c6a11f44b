// Internal host-side interfaces shared by the librs translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "rs.h"
#include "rs_device.cuh"

namespace rs {

// Layout of an rs operand (see include/rs.h): codes first, scale atoms at a
// 1024-byte aligned offset.
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int atom_k_host(int fmt) { return fmt == 0 ? 64 : 128; }
inline int n_atoms_k_host(int fmt, int K) { return (K + atom_k_host(fmt) - 1) / atom_k_host(fmt); }
inline size_t operand_sf_offset(int fmt, int rows, int K) {
    (void)fmt;
    return align_up((size_t)rows * (size_t)(K / 2), 1024);
}
inline size_t operand_sf_bytes(int fmt, int rows, int K) {
    return (size_t)((rows + 127) / 128) * (size_t)n_atoms_k_host(fmt, K) * 512;
}
inline size_t operand_bytes(int fmt, int rows, int K) {
    return operand_sf_offset(fmt, rows, K) + operand_sf_bytes(fmt, rows, K);
}

// Tiled weight operand (see rs_device.cuh): ceil(N/128) x ceil(K/256) blocks.
inline size_t weight_bytes(int fmt, int N, int K) {
    return (size_t)((N + 127) / 128) * (size_t)((K + 255) / 256) * weight_block_bytes(fmt);
}

// GEMM launch plan for one linear call.
struct GemmPlan {
    int fmt, fold;
    int M, N, K;
    int Rb;          // rows of the activation operand (M, or 2M when folded)
    int bn;          // MMA N: 16, 32, 64, 128 or 256
    int n_tiles;     // ceil(N / 128)
    int b_tiles;     // ceil(Rb / bn)
    int chunks;      // ceil(K / 256)
    int splits;      // K splits per output tile (= cluster size when > 1)
    int grid_x;      // persistent CTAs per K split; CTA x takes tiles x, x + grid_x, ...
    int nacc;        // accumulator buffers in tensor memory (2: epilogue overlaps the next tile)
    int part_bytes;  // split-K: partial buffer in shared memory
    int stages;      // pipeline depth
    int fused;       // quantize the activations inside the GEMM
    int slots;       // fused: activation chunks resident in shared memory
    int recv_bytes;  // split-K: one receive buffer in shared memory
    int tmem_cols;   // tensor-memory columns to allocate
    size_t smem_bytes;
    int pair;        // large operands: the paired-CTA kernel (rs_gemm_pair.cu) runs the call
    int tuned;       // 1: a measured tactic chose splits, fused and bn
    int qpair;       // fused: pairs of neighbouring CTAs (same K slice) quantize half of it each
};

constexpr int kMaxSplits = 8;   // portable thread-block cluster size

// Plan for a given SM count.  allow_fused: the caller passes bf16 input, so
// small-M plans may quantize inside the GEMM.  A measured tactic for the
// shape (below) takes precedence over the analytic choice when its plan fits.
GemmPlan make_gemm_plan(int fmt, bool fold, int M, int N, int K, int num_sms, bool allow_fused);
// Whether a plan shares each activation tile between the two CTAs of a
// cluster by multicast: 256-row activation tiles fed by TMA, no K split, an
// even number of channel tiles and at least two output tiles per CTA.  (A
// launch also needs two pair clusters resident at once, else it runs the
// plan without multicast.)
bool multicast_eligible(const GemmPlan& p);
// The analytic plan alone (what make_gemm_plan gives without a tactic).
GemmPlan make_gemm_plan_analytic(int fmt, bool fold, int M, int N, int K, int num_sms, bool allow_fused);

// Layout autotuning (ResServe Sec. 5.1, Fig. 3): a launch tactic measured for
// one linear shape on a GPU with num_sms SMs -- the K-split count, whether a
// bf16 input is quantized inside the GEMM, and the MMA width bn (at least
// the width the activation rows need; wider pads the operand with zero rows).
struct Tactic {
    int splits;  // 1..kMaxSplits
    int fused;   // 0: separate quantizer; 1: in the GEMM; 2: in the GEMM, shared by CTA pairs
    int bn;      // 16, 32, 64, 128 or 256
    int deep;    // 1: split plans keep their deepest weight ring (one CTA per SM)
};
// Install (replace) the tactic of (fmt, fold, M, N, K, num_sms); false on an
// out-of-range field.  Thread-safe.
bool set_tactic(int fmt, bool fold, int M, int N, int K, int num_sms, const Tactic& t);
// Remove every installed tactic, built-in ones included (builtin = false), or
// restore the built-in table (builtin = true).
void reset_tactics(bool builtin);
int tactic_count();
// The tactic for a call of M rows: the entry of the same format, fold, N, K
// and SM count with the smallest tuned row count >= M.
bool find_tactic(int fmt, bool fold, int M, int N, int K, int num_sms, Tactic* t);

// Workspace of a linear call given a bf16 input: the quantized activation
// operand when the plan quantizes in a separate kernel (sized for the worst
// case so that it does not depend on the device).
size_t workspace_bytes(int fmt, bool compensated, int M, int K);
// Workspace offset of the activation tensor scale a two-kernel plan computes
// when the caller passes no alpha_x.
size_t alpha_slot_offset(int fmt, bool compensated, int M, int K);

cudaError_t launch_tensor_scale(const void* x, int64_t n, float* alpha, uint32_t* err,
                                cudaStream_t stream, int num_sms);
// pdl: launch with programmatic stream serialization and let the dependent
// GEMM start (its weight prefetch) as soon as this kernel's own wait on the
// previous grid has returned.  Only for activations consumed by our GEMM.
cudaError_t launch_quantize(int fmt, bool paired, int rows, int K, const void* x, int64_t ldx,
                            const float* alpha, void* q_out, cudaStream_t stream, int num_sms, bool pdl);
// kext_k > 0: the extended weight [W | W[:, S]] of K-Ext (K_eff = K + K kext_k / 8
// columns; kext_mask: device bytes, one per group of 8 channels).
cudaError_t launch_quantize_weight(int fmt, int N, int K, const void* w, int64_t ldw, const float* alpha,
                                   void* wq_out, cudaStream_t stream, int num_sms, int kext_k = 0,
                                   const uint8_t* kext_mask = nullptr);
// K-Ext activation operand [X^ | R^_S] (rs operand layout, rows x K_eff), K % 256 == 0.
cudaError_t launch_quantize_kext(int fmt, int k, int rows, int K, const void* x, int64_t ldx, const float* alpha,
                                 const uint8_t* mask, void* q_out, cudaStream_t stream, int num_sms, bool pdl);
// Mean |x| of every channel over rows (the calibration score of Eq. 7).
cudaError_t launch_channel_mean_abs(const void* x, int rows, int K, int64_t ldx, float* score, cudaStream_t stream);

struct GemmCall {
    const void* x;         // fused plans: bf16 activations [M][K]
    const void* xq;        // other plans: activation operand (Rb rows)
    const void* wq;        // tiled weight operand
    const float* alpha_x;
    const float* alpha_w;
    void* y;
    int out_f32;
    uint32_t* err;
    int dyn_alpha;         // fused NVFP4 plans: compute the activation tensor scale in the GEMM
    void* qdump;           // fused plans, test hook: quantized slices out (null: off)
};
// Shared-memory bytes of one activation stage (codes + scale atoms) of a plan.
size_t plan_b_stage_bytes(const GemmPlan& p);
// Returns cudaErrorInvalidValue if a tensor map cannot be encoded.
cudaError_t launch_gemm(const GemmPlan& plan, const GemmCall& call, cudaStream_t stream);
// Trace builds: the buffer the kernels stamp (null otherwise).
uint64_t* trace_buffer();
// Route eligible large calls to the paired-CTA GEMM (off by default).
void set_pair_gemm(int enable);
// Paired-CTA GEMM on a quantized activation operand of Rb rows (Rb >= 256,
// an even number of 128-channel tiles).
cudaError_t launch_gemm_pair(int fmt, int M, int Rb, int N, int K, int fold, const void* xq, const void* wq,
                             const float* alpha_x, const float* alpha_w, void* y, int out_f32, uint32_t* err,
                             uint64_t* trace, int num_sms, cudaStream_t stream);

// Separate Fold of an expanded fp32 output of paired rows (z [2M][N] -> y [M][N]).
cudaError_t launch_fold_pairs(const float* z, void* y, int M, int N, int out_f32, cudaStream_t stream, int num_sms);

// Residue-compensated decode attention (rs_attn.cu).
struct AttnArgs {
    const uint16_t* q;        // bf16 query [B][Hq][D]: each CTA quantizes its group's rows (Alg. 1)
    const float* alpha_q;     // query tensor scale (device)
    const uint8_t* k_cache;   // [pages][Hkv] page blocks
    const uint8_t* v_cache;
    const int* block_table;   // [B][max_pages]
    const int* seq_lens;      // [B]
    float* part;              // [B][Hkv][splits][G][D + 2]: o, then m, l per head
    uint32_t* err;
    uint64_t* trace;          // trace builds only: 32 timer stamps per CTA
    int B, Hq, Hkv, D, max_pages, max_len, split_tokens, splits;
};

// Tokens per split of a ResAttn call, a multiple of the 128-token tile.
int resattn_split_tokens(int B, int Hkv, int D, int max_len, int num_sms);
cudaError_t launch_resattn(int D, const AttnArgs& a, void* out, int out_f32, cudaStream_t stream);

// Device error word of the current device.
uint32_t* device_error_word();
// RS_OK with the SM count and error word of the current device, or the
// status a call on it returns (RS_ERR_CUDA, RS_ERR_UNSUPPORTED).
rs_status current_device_status(int* num_sms, uint32_t** err);

}  // namespace rs
