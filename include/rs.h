/*
 * rs.h - C ABI of librs: residue-compensated block-scaled FP4 linear layers
 * for NVIDIA GB300 (sm_103a).
 *
 * The method is ResServe ("ResServe: Accurate and Efficient FP4 LLM Inference
 * with Residue Compensation", arXiv 2611.08713): activations X are quantized
 * to NVFP4 or MXFP4 at run time, the quantization residue R = X - QDQ(X) is
 * quantized to the same format, and a linear layer against offline-quantized
 * FP4 weights computes Y = X^ W^T + R^ W^T (Sec. 4.2 Eq. 1, full
 * compensation), with base and residue stacked as paired activation rows of
 * one block-scaled GEMM and folded on chip (Sec. 4.3 Eq. 2, Sec. 5.1).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers marked (device) are CUDA device pointers on the current device;
 *   the caller owns and allocates every buffer.  librs never allocates device
 *   memory and keeps no per-call state beyond a small host-side cache of
 *   device properties and kernel attributes.
 * - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *   stream) and is asynchronous.  Host-checkable errors are returned before
 *   anything is enqueued; a failed launch returns RS_ERR_CUDA.  Device-side
 *   problems (a bounded wait that ran out, a non-finite tensor amax) set a
 *   device error word that rs_get_device_error() reads.
 * - Every device pointer must be 16-byte aligned.  K must be a positive
 *   multiple of 32 (two E2M1 codes per byte, 16-byte row pitch of the code
 *   array).  Row counts may be 0 (nothing is enqueued) and need no padding.
 * - No exception crosses the ABI.
 *
 * Formats (Sec. 2, Fig. 1; App. B.2 Eq. 8-10)
 * -------------------------------------------
 *   RS_NVFP4: E2M1 codes, one E4M3 block scale per 16 elements along K and
 *             one fp32 tensor scale alpha (0, or finite and >= 2^-117; see
 *             rs_get_device_error).
 *   RS_MXFP4: E2M1 codes, one E8M0 block scale per 32 elements along K, no
 *             tensor scale (alpha pointers are ignored and may be NULL).
 *
 * Quantization rule (the one the oracle follows): per block, Max = max|x|,
 * s = fl(Max/6), NVFP4 scale byte = E4M3 round-to-nearest-even of fl(s/alpha)
 * saturated to 448 (0 when alpha == 0), s~ = fl(alpha * dec(byte)); MXFP4
 * scale = 2^e with e = floor(log2 Max) - 2 clamped to [-127, 127] (Max == 0
 * gives e = -127), byte = e + 127.  Elements: v = fl(x * fl(1/s~)) (NVFP4) or
 * fl(x * 2^-e) (MXFP4), code = E2M1 round-to-nearest-even with saturation at
 * +-6 and the sign kept.  x^ = fl(s~ * dec(code)); residue r = fl(x - x^),
 * quantized by the same rule with its own block scales and the same alpha.
 *
 * Device layout of a quantized operand ("rs operand", `rows` x K)
 * ---------------------------------------------------------------
 * One buffer of rs_operand_bytes(fmt, rows, K) bytes:
 *   [0, rows*K/2)          codes, row-major, row pitch K/2 bytes, element 2j
 *                          of a row in the low nibble of byte j.
 *   [sf_off, +sf_bytes)    block scales, sf_off = rs_operand_sf_offset().
 *                          Stored as 512-byte atoms.  An atom holds the scales
 *                          of 128 consecutive rows and 4 consecutive blocks
 *                          (64 elements of K for NVFP4, 128 for MXFP4).  The
 *                          atom for row tile t = r/128 and block group
 *                          g = b/4 is atom number t * ceil(K/(4*bs)) + g; the
 *                          byte for row r and block b within it is at
 *                          (r % 32) * 16 + ((r / 32) % 4) * 4 + (b % 4).
 *                          Rows are padded to a multiple of 128 and blocks to
 *                          a multiple of 4 with zero bytes.
 * This is the scale layout the tcgen05 block-scaled MMA reads from tensor
 * memory after a 32x128b.warpx4 copy, so the quantizer writes what the GEMM
 * reads and no reordering pass sits between them (App. B.2, Sec. 4.4).
 *
 * A paired operand (compensated input; the row-pair layout of Sec. 5.1 and
 * Fig. 5a) is an rs operand with 2*M rows: row 2j holds the base X^ of token
 * j and row 2j+1 its residue R^.
 *
 * Device layout of a quantized weight ("rs weight", W [N][K], offline)
 * --------------------------------------------------------------------
 * rs_weight_bytes(fmt, N, K) bytes made of ceil(N/128) x ceil(K/256) blocks,
 * block (t, c) at byte ((t * ceil(K/256)) + c) * B with B = 18432 (NVFP4) or
 * 17408 (MXFP4).  A block covers output channels [128t, 128t+128) and K
 * elements [256c, 256c+256):
 *   [0, 16384)     codes of the 128 channels, 128 bytes each (element 2j of
 *                  the block in the low nibble of byte j), stored as the
 *                  128-byte-swizzled image: byte j of channel r at
 *                  r*128 + ((j/16) XOR (r%8))*16 + j%16.
 *   [16384, B)     the block's scale atoms (4 for NVFP4, 2 for MXFP4), each
 *                  512 bytes laid out as in an rs operand (channel r, block b
 *                  of the atom at (r%32)*16 + ((r/32)%4)*4 + b).
 * Channels beyond N and elements beyond K hold zero codes and zero scales.
 * The GEMM streams one whole block per pipeline stage with a single bulk
 * copy of consecutive bytes.
 */
#ifndef RS_H
#define RS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RS_API __attribute__((visibility("default")))
#else
#define RS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *rs_stream_t; /* binary-compatible with cudaStream_t */

typedef enum {
    RS_OK = 0,
    RS_ERR_INVALID_ARG = 1,    /* bad enum, NULL pointer, negative size, ldx < K */
    RS_ERR_ALIGNMENT = 2,      /* pointer or row pitch not 16-byte aligned */
    RS_ERR_SHAPE = 3,          /* K not a positive multiple of 32, size limits */
    RS_ERR_UNSUPPORTED = 4,    /* no GPU with tcgen05 (sm_100 family) */
    RS_ERR_WORKSPACE = 5,      /* workspace NULL or smaller than rs_workspace_bytes() */
    RS_ERR_CUDA = 6,           /* a CUDA runtime/driver call or launch failed */
    RS_ERR_DEVICE_TIMEOUT = 7  /* a bounded device wait ran out (reported later) */
} rs_status;

typedef enum { RS_NVFP4 = 0, RS_MXFP4 = 1 } rs_format;
typedef enum { RS_OUT_BF16 = 0, RS_OUT_F32 = 1 } rs_out_dtype;

/* Human-readable name of a status code (static string, never NULL). */
RS_API const char *rs_status_string(rs_status s);

/* Library ABI version (incremented on incompatible changes). */
RS_API int rs_version(void);

/* ---- sizes (host only, no CUDA calls) ----------------------------------- */

/* Bytes of an rs operand of `rows` x K (layout above); 0 on invalid input. */
RS_API size_t rs_operand_bytes(rs_format fmt, int rows, int K);
/* Byte offset of the scale atoms inside an rs operand. */
RS_API size_t rs_operand_sf_offset(rs_format fmt, int rows, int K);
/* Activation operand sizes: `rows` tokens quantized alone (W4A4 input) or,
 * for rs_quantize_residue, pass rows = 2*M. */
RS_API size_t rs_act_bytes(rs_format fmt, int rows, int K);
/* Weight operand size, W [N][K] (nn.Linear layout), rs weight layout. */
RS_API size_t rs_weight_bytes(rs_format fmt, int N, int K);
/* Workspace that rs_linear_w4a4 / rs_linear_compensated need when given a
 * bf16 input: room for the quantized activation operand, which plans with
 * larger M produce in a separate quantizer kernel, and for the activation
 * tensor scale those plans compute when alpha_x is NULL (small-M plans
 * quantize inside the GEMM and leave the workspace untouched).  No initialisation is
 * needed; calls that share a workspace must be ordered (same stream). */
RS_API size_t rs_workspace_bytes(rs_format fmt, int M, int N, int K, int compensated);

/* Diagnostic, host only (no GPU needed): the launch plan that rs_linear_* of
 * this shape would use on a GPU with num_sms SMs.  x_in_call != 0: the call
 * passes bf16 X (small operands are then quantized inside the GEMM).  Writes
 * up to n_out ints to out (host), in this order: bn (MMA N: 16..256), n_tiles
 * (ceil(N/128)), b_tiles, chunks (ceil(K/256)), splits (K splits = cluster
 * size), grid_x (persistent CTAs per split), stages (weight ring depth),
 * fused (1: quantized inside the GEMM), slots, nacc (accumulator buffers),
 * tmem_cols, smem_bytes (dynamic shared memory per CTA), tuned (1: a
 * measured tactic below chose splits, fused and bn), mcast (1: the two CTAs
 * of a cluster share each 256-row activation tile by multicast, when two
 * such clusters fit at once on the GPU).  Returns the number written, or
 * minus an rs_status code on bad arguments. */
RS_API int rs_plan_linear(rs_format fmt, int compensated, int M, int N, int K, int num_sms, int x_in_call,
                          int *out, int n_out);

/* ---- layout autotuning (Sec. 5.1 "Layout Autotuning", Fig. 3) ------------ */

/* The paper picks a kernel layout per (M, N, K) by measurement.  Here a
 * tactic fixes, for one (fmt, compensated, M, N, K) on a GPU with num_sms
 * SMs: the K-split count (1..8, the cluster size); whether a bf16 input may
 * be quantized inside the GEMM (fused: 0 no, 1 yes, 2 yes with CTA pairs
 * sharing the quantization of a K slice; only plans whose activation tile
 * is at most 32 rows can); the MMA width bn (16, 32, 64, 128 or 256; a
 * width below what the activation rows need is raised to it, a wider one
 * pads the operand with zero rows); and deep (0/1: a split plan whose CTAs
 * take one output tile each keeps the deepest weight ring that fits, one
 * CTA per SM, instead of the 3-stage ring that lets two CTAs share an SM).
 * A linear call of M rows takes the
 * tactic of the same fmt, compensated, N, K and SM count with the smallest
 * tuned M' >= M; its plan replaces the analytic one when it fits the SM's
 * shared and tensor memory and splits <= ceil(K/256), else the analytic plan
 * stays.  Results agree with any other plan within the output tolerance
 * (the K-split order of the fp32 sums differs).  librs ships a table
 * measured on GB300 (152 SMs) by block_scaled_quantized_gb300/tune.py.
 * Host only, thread-safe; a change affects calls planned after it (not CUDA
 * graphs already captured).  RS_ERR_INVALID_ARG for a field out of range,
 * RS_ERR_SHAPE unless K % 32 == 0. */
RS_API rs_status rs_set_tactic(rs_format fmt, int compensated, int M, int N, int K, int num_sms, int splits,
                               int fused, int bn, int deep);
/* builtin != 0: restore the shipped table (dropping rs_set_tactic entries);
 * builtin == 0: remove every tactic, so that every call uses the analytic plan. */
RS_API rs_status rs_reset_tactics(int builtin);
/* Number of tactics installed (shipped ones included). */
RS_API int rs_tactic_count(void);

/* ---- tensor scale (App. B.2 Eq. 8) -------------------------------------- */

/* alpha = fl(amax / 2688) over n bf16 values (device); writes one float to
 * alpha_out (device).  A non-finite amax sets the device error word to
 * RS_ERR_INVALID_ARG.  The paper computes this scale offline or outside its
 * timed region (App. C.1); it is a separate call for that reason. */
RS_API rs_status rs_compute_tensor_scale(const void *x_bf16, int64_t n, float *alpha_out,
                                  rs_stream_t stream);

/* ---- quantizers (Sec. 4.4, App. B.2 Algorithm 1) ------------------------- */

/* Quantize bf16 rows x[rows][ldx] (device, first K columns used) into an rs
 * operand q_out (device, rs_operand_bytes(fmt, rows, K) bytes), the W4A4
 * activation input (Fig. 1c).  alpha (device, one float) is the NVFP4 tensor
 * scale; ignored for MXFP4. */
RS_API rs_status rs_quantize_fp4(rs_format fmt, int rows, int K, const void *x_bf16, int64_t ldx,
                          const float *alpha, void *q_out, rs_stream_t stream);

/* Offline weight quantization (Fig. 1c): W[N][ldw] (device, bf16, first K
 * columns) into the rs weight layout wq_out (device, rs_weight_bytes(fmt, N,
 * K) bytes), same quantization rule as the activations; alpha (device) is
 * the weight's NVFP4 tensor scale (ignored for MXFP4). */
RS_API rs_status rs_quantize_weight(rs_format fmt, int N, int K, const void *w_bf16, int64_t ldw,
                                    const float *alpha, void *wq_out, rs_stream_t stream);

/* Fused base + residue quantizer (Alg. 1; Sec. 4.4): one pass over x[M][ldx]
 * forms X^, the residue R = X - X^ in registers and R^, and writes the paired
 * rs operand with 2*M rows (row 2j = X^ of token j, row 2j+1 = R^ of token j)
 * to q_paired_out (device, rs_act_bytes(fmt, 2*M, K) bytes). */
RS_API rs_status rs_quantize_residue(rs_format fmt, int M, int K, const void *x_bf16, int64_t ldx,
                              const float *alpha, void *q_paired_out, rs_stream_t stream);

/* ---- linear layers (Sec. 4.3 Eq. 2, Sec. 5.1 Eq. 4) ----------------------- */

/* Uncompensated W4A4 linear (Fig. 1c): Y[M][N] = alpha_x alpha_w * X^ W^T.
 * Exactly one of x_bf16 (device, [M][K] contiguous, quantized inside the
 * call) and xq (device, rs operand with M rows) is non-NULL.  wq: rs weight
 * of W [N][K] from rs_quantize_weight.  alpha_w (device float) is required
 * for NVFP4.  alpha_x (device float) is the activation tensor scale; with
 * x_bf16 it may be NULL, and the call then uses this input's own scale
 * fl(amax(X)/2688) (App. B.2 Eq. 8, the value rs_compute_tensor_scale gives):
 * small-M plans find it inside the GEMM (each K-split CTA takes its slice's
 * amax and the cluster trades them), others compute it into the workspace
 * first.  A non-finite amax sets the device error word.  y (device): [M][N]
 * row-major, bf16 or fp32.
 * workspace (device): at least rs_workspace_bytes(fmt, M, N, K, 0) bytes when
 * x_bf16 is given; may be NULL with xq.
 *
 * The GEMM is launched with programmatic stream serialization: it may start
 * while the previous kernel in the stream is still running and begins
 * streaming wq before it waits for that kernel.  wq must therefore not be
 * written by a kernel that signals early completion (griddepcontrol
 * launch_dependents) right before this call; librs's own kernels that write
 * weights never do.  Inputs x / xq / alpha and the output y are touched only
 * after the previous kernel has completed. */
RS_API rs_status rs_linear_w4a4(rs_format fmt, int M, int N, int K,
                         const void *x_bf16, const void *xq, const float *alpha_x,
                         const void *wq, const float *alpha_w,
                         void *y, rs_out_dtype out_dtype,
                         void *workspace, size_t ws_bytes, rs_stream_t stream);

/* Fully compensated linear (M-Ext, Sec. 4.3 Eq. 2):
 *   Y[M][N] = alpha_x alpha_w * (X^ W^T + R^ W^T).
 * The GEMM runs in the swapped orientation Z^T = W^ [X^; R^]^T (Eq. 4) with
 * base and residue as adjacent accumulator columns, and each output is folded
 * (Y_j = Z_2j + Z_2j+1) in fp32 registers before the scale and the store, so
 * no expanded result leaves the SM.  Exactly one of x_bf16 (device, [M][K])
 * and xq_paired (device, paired rs operand, 2*M rows) is non-NULL. */
RS_API rs_status rs_linear_compensated(rs_format fmt, int M, int N, int K,
                                const void *x_bf16, const void *xq_paired, const float *alpha_x,
                                const void *wq, const float *alpha_w,
                                void *y, rs_out_dtype out_dtype,
                                void *workspace, size_t ws_bytes, rs_stream_t stream);

/* ---- selective prefill compensation, K-Ext (Sec. 5.3 Eq. 6, App. A Eq. 7) -- */

/* Selective compensation keeps the residues of k of every 8 consecutive
 * input channels (ratio rho = k / 8, k in {1, 2, 4, 8}; k = 8 is full
 * compensation) and appends them to the activation as extra reduction
 * columns, with the matching weight columns appended offline, so one GEMM
 * over K_eff = K + K k / 8 sums the base and the correction (Eq. 6):
 *   Y = alpha_x alpha_w [X^ | R^_S] [W^ | W^_S]^T.
 * Selection masks: one byte per group of 8 channels, bit t set when channel
 * 8g + t is compensated, exactly k bits per byte.  Extension element
 * g k + j holds the j-th selected channel of group g (increasing channel
 * order); the selected residues r = fl(x - x^) are quantized as their own
 * blocks of 16 (NVFP4) / 32 (MXFP4) extension elements with the base
 * operand's tensor scale.  The extended weight is [W | W[:, S]] quantized
 * as one tensor with alpha_w.  K must be a multiple of 256. */

/* K k / 8 (the number of extension columns), 0 for an unsupported K or k. */
RS_API int rs_kext_width(int K, int k);

/* Eq. 7 on the host: for each group of 8 channels, the k channels with the
 * largest calibration score (mean |x|); equal scores keep the lower channel.
 * score: host float[K]; mask: host uint8[K / 8]. */
RS_API rs_status rs_kext_select(int K, int k, const float *score, uint8_t *mask);

/* Calibration score of Eq. 7 on the device: score[c] = mean over the rows of
 * |x[r][c]| (fp32, rows summed in order).  x: bf16 [rows][ldx]. */
RS_API rs_status rs_channel_mean_abs(const void *x_bf16, int rows, int K, int64_t ldx, float *score,
                                     rs_stream_t stream);

/* Sizes: the extended activation operand (rs operand layout, rows x K_eff),
 * the extended weight (rs weight layout, N x K_eff), and the workspace of
 * rs_linear_kext given a bf16 input.  0 for unsupported arguments. */
RS_API size_t rs_kext_act_bytes(rs_format fmt, int rows, int K, int k);
RS_API size_t rs_kext_weight_bytes(rs_format fmt, int N, int K, int k);
RS_API size_t rs_kext_workspace_bytes(rs_format fmt, int M, int N, int K, int k);

/* Offline: the extended weight [W | W[:, S]] of W bf16 [N][K] (row pitch
 * ldw), quantized with alpha_w (NVFP4) into wq_out (device,
 * rs_kext_weight_bytes).  mask: device uint8[K / 8]. */
RS_API rs_status rs_quantize_weight_kext(rs_format fmt, int N, int K, int k, const void *w_bf16, int64_t ldw,
                                         const float *alpha_w, const uint8_t *mask, void *wq_out,
                                         rs_stream_t stream);

/* The extended activation operand [X^ | R^_S] of x bf16 [rows][ldx] (Sec. 5.3,
 * App. B.2 Alg. 1) into q_out (device, rs_kext_act_bytes).  A mask byte
 * without exactly k bits set sets the device error word. */
RS_API rs_status rs_quantize_kext(rs_format fmt, int rows, int K, int k, const void *x_bf16, int64_t ldx,
                                  const float *alpha, const uint8_t *mask, void *q_out, rs_stream_t stream);

/* Selective-compensation linear (Eq. 6): Y[M][N] = alpha_x alpha_w *
 * [X^ | R^_S] [W^ | W^_S]^T.  Exactly one of x_bf16 (device [M][K]; then mask
 * and a workspace of rs_kext_workspace_bytes are needed) and xq (an extended
 * operand from rs_quantize_kext) is non-NULL; wq_ext from
 * rs_quantize_weight_kext with the same mask.  alpha_x may be NULL with
 * x_bf16 (the input's own tensor scale, as for rs_linear_w4a4).  Other
 * arguments, alignment and errors as for rs_linear_w4a4. */
RS_API rs_status rs_linear_kext(rs_format fmt, int M, int N, int K, int k, const void *x_bf16, const void *xq,
                                const float *alpha_x, const uint8_t *mask, const void *wq_ext,
                                const float *alpha_w, void *y, rs_out_dtype out_dtype, void *workspace,
                                size_t ws_bytes, rs_stream_t stream);

/* ---- residue-compensated decode attention (ResAttn, Sec. 4.3, Sec. 5.2) -- */

/* Paged NVFP4 KV cache ("rs page"): the cache holds pages of 32 tokens; page
 * p of KV head h is the block of 32 * (D/2 + D/16) bytes at byte
 * (p * Hkv + h) * 32 * (D/2 + D/16): the E2M1 codes of its 32 tokens
 * [32][D/2] (token-major, element 2j of a token in the low nibble of byte
 * j), then their E4M3 block scales [32][D/16] (16-element blocks along the
 * head dimension, tensor scale 1.0).  block_table [B][max_pages] (int32)
 * lists the pages of each sequence in token order; token t of sequence b
 * lives in page block_table[b][t / 32] at row t % 32.  Unused entries of a
 * page are never read. */

/* Workspace of rs_resattn_decode: the partial outputs of the sequence splits
 * (fp32 o, m and l per split and query head; an upper bound for any device).
 * 0 for a shape rs_resattn_decode refuses. */
RS_API size_t rs_resattn_workspace_bytes(int B, int Hq, int Hkv, int D, int max_len);

/* Tokens per sequence split that rs_resattn_decode uses on a device with
 * num_sms SMs (a multiple of 128; host only; 0 for invalid arguments): the
 * (split, KV head, sequence) CTAs run in waves of two CTAs per SM at D = 128
 * and one at D = 256, and the split count minimises waves x (128-token
 * tiles per split + 1), the fewer splits on a tie. */
RS_API int rs_resattn_split_tokens(int B, int Hkv, int D, int max_len, int num_sms);

/* One decode step of ResAttn (Sec. 4.3 Eq. 3, Fig. 3; Sec. 5.2 "ResAttn
 * execution").  q_bf16 [B][Hq][D] (device, bf16) is quantized with Alg. 1
 * into base and residue rows with the tensor scale *alpha_q (device; e.g.
 * rs_compute_tensor_scale over Q) inside the attention kernel, each CTA its
 * own query group (a tensor scale outside the supported range is reported as
 * RS_ERR_INVALID_ARG by rs_get_device_error); query head g reads KV head
 * g / (Hq/Hkv).
 * Scores s = (<Q^, K^> + <R^, K^>) alpha_q / sqrt(D) are folded in fp32
 * before an online softmax over 128-token tiles; V goes from NVFP4 to E4M3
 * on chip; the softmax weights are rounded to E4M3 for PV with fp32
 * accumulation, and the normalizer sums the rounded weights; the sequence
 * splits are combined as O = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s.
 * out [B][Hq][D] (device) is bf16 or fp32; a sequence of length 0 gives 0.
 * seq_lens [B] (device, int32) must not exceed max_len <= 32 * max_pages: a
 * longer one is clamped to max_len and reported as RS_ERR_INVALID_ARG by
 * rs_get_device_error.  D is 128 or 256, Hq a multiple of Hkv with at most
 * 8 query heads per KV head.  Errors: RS_ERR_SHAPE (sizes), RS_ERR_INVALID_ARG
 * (NULL pointer, dtype), RS_ERR_ALIGNMENT (16 bytes for q, caches, out and
 * workspace; 4 for alpha_q, block_table, seq_lens), RS_ERR_WORKSPACE. */
RS_API rs_status rs_resattn_decode(int B, int Hq, int Hkv, int D, int max_pages, int max_len, const void *q_bf16,
                                   const float *alpha_q, const void *k_cache, const void *v_cache,
                                   const int *block_table, const int *seq_lens, void *out, rs_out_dtype out_dtype,
                                   void *workspace, size_t ws_bytes, rs_stream_t stream);

/* ---- alternative prefill GEMM (comparison) ------------------------------- */

/* enable != 0: linear calls whose activation operand has at least 512 rows
 * (after pairing) and an even number of 128-channel tiles, and that do not
 * quantize inside the GEMM, run on the paired-CTA kernel instead: two CTAs
 * of a cluster share one tcgen05.mma.cta_group::2 of 256 output channels x
 * 256 activation rows (the larger tile of ResServe Sec. 5.1), each staging
 * its own 128 weight channels and 128 activation rows.  Results are those
 * of the default kernel within the output tolerance.  It is off by default
 * because it is slower on GB300 (see the benchmark's prefill figures); the
 * switch is process-wide and not thread-safe, for tests and benchmarks. */
RS_API void rs_debug_pair_gemm(int enable);

/* ---- separate Fold (ablation of the on-chip Fold) ------------------------ */

/* y[j][n] = z[2j][n] + z[2j+1][n] for j < M, n < N (Sec. 4.3 Eq. 2, Fold):
 * the Fold as its own kernel over an expanded fp32 output z [2M][N]
 * (device, row-major) of paired activation rows, e.g. rs_linear_w4a4 run on a
 * paired operand of 2M rows with fp32 output.  y [M][N] (device) is bf16 or
 * fp32 per out_dtype; the sums are fp32, rounded once.  It exists to measure
 * what folding on chip saves (Sec. 5.1, Fig. 6b); the linear calls never use
 * it.  RS_ERR_INVALID_ARG for negative sizes, a NULL pointer or a bad dtype;
 * RS_ERR_ALIGNMENT unless z and y are 16-byte aligned. */
RS_API rs_status rs_fold_pairs(int M, int N, const float *z, void *y, rs_out_dtype out_dtype, rs_stream_t stream);

/* ---- compensated linear without any device allocation -------------------- */

/* Largest quantized operand rs_linear_compensated_noalloc accepts (4 MiB);
 * its fixed device array holds that plus 1280 bytes (alignment and the
 * tensor-scale slot).  Every GPU that loads librs holds the array until the
 * process exits. */
#define RS_NOALLOC_SCRATCH_BYTES (4u << 20)

/* The paper has no counterpart to this entry point: it exists for callers
 * that cannot allocate device memory, such as a plugin that another
 * framework hands only its input and output buffers, or a process whose
 * device footprint must stay fixed after start-up.
 *
 * The compensated layer of rs_linear_compensated for a bf16 input x_bf16
 * ([M][K], device, contiguous), with the quantized activations (the paired
 * base and residue operand, rs_act_bytes(fmt, 2*M, K) bytes) in a fixed
 * device array inside librs instead of a caller workspace.  It always runs
 * the two-kernel form (the paired quantizer, then the GEMM on its operand),
 * where rs_linear_compensated may quantize inside the GEMM; the outputs agree
 * within the output tolerance (max|dY| <= 1e-3 max|Y|), not bit for bit.
 * Nothing is allocated: no cudaMalloc, no cudaFree.
 *   - Operands larger than RS_NOALLOC_SCRATCH_BYTES are rejected with
 *     RS_ERR_WORKSPACE before anything is enqueued, with or without alpha_x
 *     (NVFP4, K = 4096: up to M = 904; rs_act_bytes(fmt, 2*M, K) gives the
 *     exact size).  The array also holds the tensor-scale slot that a call
 *     without alpha_x fills.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.
 *   - Every call shares the one array per device, which keeps the last
 *     call's contents; calls that overlap on the GPU (different streams
 *     without ordering between them) race on it.  Calls ordered on one
 *     stream are safe: each call rewrites every byte it later reads.
 * Other arguments, alignment rules and errors as for rs_linear_compensated. */
RS_API rs_status rs_linear_compensated_noalloc(rs_format fmt, int M, int N, int K, const void *x_bf16,
                                               const float *alpha_x, const void *wq, const float *alpha_w,
                                               void *y, rs_out_dtype out_dtype, rs_stream_t stream);

/* ---- device error word --------------------------------------------------- */

/* Diagnostic of failure detection (no GPU fault): launches one CTA that
 * waits on an mbarrier nothing arrives on, with the bounded wait the kernels
 * use and a limit of limit_ns (1 .. 1e9 ns); the wait runs out, sets the
 * device error word to RS_ERR_DEVICE_TIMEOUT (read and cleared by
 * rs_get_device_error) and the kernel exits normally, leaving the context
 * usable.  RS_ERR_INVALID_ARG for a limit outside that range. */
RS_API rs_status rs_debug_wait_probe(uint64_t limit_ns, rs_stream_t stream);

/* Synchronizes `stream`, then returns and clears the device error word of the
 * current device: RS_OK, RS_ERR_DEVICE_TIMEOUT (a kernel's bounded wait ran
 * out; its outputs are invalid and the workspace must be zero-filled again)
 * or RS_ERR_INVALID_ARG (a non-finite tensor amax, or an NVFP4 tensor scale
 * that is neither 0 nor a finite value of at least 2^-117, i.e. a tensor amax
 * below about 4e-32: block scales of such a tensor can be subnormal, their
 * reciprocals infinite, and the codes of those blocks are unspecified).
 * Returns RS_ERR_CUDA if the synchronization itself fails. */
RS_API rs_status rs_get_device_error(rs_stream_t stream);

/* Sync-free form of rs_get_device_error, for a serving loop that polls the
 * error word without stalling its stream (no operation of the paper: the
 * device error word is this library's failure reporting).  Enqueues on
 * `stream`, behind the work already there, one single-thread kernel that
 * writes the device error word of the current device to *out and clears it.
 * `out` (4-byte aligned) is device memory, or pinned host memory the device
 * can reach; its value is one of the codes rs_get_device_error returns and
 * is valid once the stream has passed this point (an event, a later
 * synchronization).  Nothing is synchronized inside the call.
 * RS_ERR_INVALID_ARG for NULL, RS_ERR_ALIGNMENT for a misaligned pointer. */
RS_API rs_status rs_get_device_error_async(uint32_t *out, rs_stream_t stream);

/* Test hook of the quantizing GEMM prologue (Sec. 4.4: Algorithm 1 of
 * App. B.2 fused into the GEMM for small M).  Runs exactly the call
 * rs_linear_compensated (compensated != 0) or rs_linear_w4a4 makes with a
 * bf16 input and, when its plan quantizes inside the GEMM, also copies every
 * CTA's quantized activation slice to `dump` (device), as the MMAs read it.
 * layout (host, 7 ints) receives: fused (0 separate quantizer, 1 in the GEMM,
 * 2 in the GEMM with CTA pairs sharing the slice; rs_set_tactic), bn (rows of the activation
 * tile), grid_x (CTAs per K split), splits, slots (chunk stages per CTA),
 * stage_bytes, chunks (256-element K chunks of the call).  The slice of the
 * CTA (x, split z) starts at byte (z * grid_x + x) * slots * stage_bytes;
 * its K chunks are the consecutive chunks c0 .. c0 + n - 1 of split z, where
 * the chunks are dealt out as evenly as possible, the first
 * (chunks % splits) splits taking one more.  Chunk i of the slice occupies
 * stage_bytes at offset i * stage_bytes: codes of bn rows x 128 bytes in the
 * 128-byte-swizzled image (row r, byte b at r * 128 + ((b / 16) ^ (r % 8))
 * * 16 + b % 16; paired rows 2j = base, 2j + 1 = residue of token j), then
 * one 512-byte scale atom per 4 blocks in the rs operand's atom layout.
 * With dump == NULL only layout is written.  RS_ERR_UNSUPPORTED when the plan
 * quantizes in a separate kernel; RS_ERR_WORKSPACE when dump_bytes is below
 * grid_x * splits * slots * stage_bytes. */
RS_API rs_status rs_debug_linear_dump(rs_format fmt, int compensated, int M, int N, int K, const void *x_bf16,
                                      const float *alpha_x, const void *wq, const float *alpha_w, void *y,
                                      rs_out_dtype out_dtype, void *workspace, size_t ws_bytes, void *dump,
                                      size_t dump_bytes, int *layout, rs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RS_H */
