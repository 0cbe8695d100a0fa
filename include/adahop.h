/*
 * adahop.h -- C ABI of the GB300 (sm_103a) AdaHOP MXFP4 linear layer.
 *
 * Method: AdaHOP, "Fast and Accurate Low-Precision Training via Outlier-Pattern-Aware
 * Rotation" (Kim, Khodamoradi, Denolf, Park; arXiv 2604.02525).  Each linear layer runs three
 * GEMMs (Fig. 5): Fwd Y = X.W^T, dgrad dX = G_Y.W, wgrad dW = G_Y^T.X.  Every operand is
 * classified once as Row-wise, Column-wise or None (abstract; Fig. 4: patterns are stable, so
 * calibration is one-time), and each GEMM's operand pattern pair selects
 *   IHT      -- block-32 Hadamard along the inner dimension on both operands, then MXFP4;
 *   OE-Left  -- the top-r rows (by FOID score) of one operand go to a BF16 path, the residual
 *               (those rows zeroed) gets IHT + MXFP4;
 *   OE-Right -- the same with columns;
 *   BF16     -- a plain BF16 GEMM;
 *   MXFP4    -- plain MXFP4 without the Hadamard (the pages' "MXFP4" baseline, Table 3).
 * The data path follows Fig. 9 and the appendix implementation notes: FOID -> IHT and
 * quantisation -> fused MXFP4 + BF16 GEMM -> fused scatter-add.
 *
 * Conventions for every entry point
 *   - All matrices are row-major.  bf16 tensors are passed as raw 16-bit patterns.
 *     X is M x K, W is N x K, G_Y is M x N, Y is M x N, dX is M x K, dW is N x K.
 *   - Pointers are DEVICE pointers unless stated; the caller owns every buffer.  The library
 *     allocates no device memory: scratch lives in the caller's workspace.
 *   - Every call is asynchronous on the given CUDA stream (NULL = legacy default stream)
 *     unless documented as synchronous.  Host-side argument errors return before any launch.
 *   - Shapes: M, N, K must be positive multiples of 128.  OE rank r: 0 <= r <= 256 and r <= the
 *     number of lines it is drawn from.  Device pointers must be 16-byte aligned and the
 *     workspace 256-byte aligned; otherwise ADAHOP_ERR_ALIGN.
 *   - Inputs must be finite; results for NaN/Inf inputs are unspecified.
 *   - A workspace of the linear calls must start with its first 16384 bytes zeroed: the status
 *     word lives there, with the completion counters of FOID and of the fused GEMM's stream-K
 *     tiles; every call that completes leaves them zero, so a workspace is reused as it is.
 *     A device-side failure (a bounded wait that ran out) is recorded in the status word;
 *     adahop_get_device_status() reports and clears it (after such a failure, zero the header
 *     again before reusing the workspace).
 */
#ifndef ADAHOP_H
#define ADAHOP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st *adahop_stream_t;

typedef enum {
  ADAHOP_OK = 0,
  ADAHOP_ERR_INVALID_ARG = 1,   /* null pointer, bad enum value, bad option */
  ADAHOP_ERR_SHAPE = 2,         /* dimension not a positive multiple of 128, bad rank */
  ADAHOP_ERR_ALIGN = 3,         /* pointer misaligned */
  ADAHOP_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (see adahop_last_cuda_error) */
  ADAHOP_ERR_TIMEOUT = 5,       /* a device-side bounded wait gave up */
  ADAHOP_ERR_UNSUPPORTED = 6,   /* device is not sm_103a / feature not built */
  ADAHOP_ERR_WORKSPACE = 7      /* workspace missing or smaller than adahop_workspace_size() */
} adahop_status;

/* Outlier pattern of one tensor (abstract; Table 1). */
typedef enum { ADAHOP_PAT_NONE = 0, ADAHOP_PAT_ROW = 1, ADAHOP_PAT_COL = 2 } adahop_pattern;

/* Per-GEMM strategy (Fig. 5), plus the plain-MXFP4 baseline of Table 3. */
typedef enum {
  ADAHOP_IHT = 0, ADAHOP_OE_LEFT = 1, ADAHOP_OE_RIGHT = 2, ADAHOP_BF16 = 3, ADAHOP_MXFP4 = 4
} adahop_strategy;

typedef enum { ADAHOP_OUT_BF16 = 0, ADAHOP_OUT_FP32 = 1 } adahop_out_dtype;

/* Calibration options.  tau: threshold on max/lower-median of the per-line mean squares
 * (default 8.0); probe_len must be 64 (FOID probe, appendix FOID paragraph); oe_rank r
 * (default 64, Fig. 10: rank 64 is the favourable trade-off). */
typedef struct {
  double tau;
  int probe_len;
  int oe_rank;
} adahop_options;

/* The calibration record.  x, w, gy: adahop_pattern.  fwd, dgrad, wgrad: adahop_strategy.
 * rho: the ratios behind the decision (row, col) for X, W, G_Y.  A caller may override any
 * field before passing the plan to the linear calls. */
typedef struct {
  int32_t x, w, gy;
  int32_t fwd, dgrad, wgrad;
  int32_t oe_rank;
  int32_t reserved;
  double rho[6];
} adahop_plan;

/* Fills *opt with the defaults (tau 8.0, probe 64, rank 64). */
void adahop_default_options(adahop_options *opt);

/* Plain-text name of a status code (static storage). */
const char *adahop_status_string(adahop_status st);

/* The last CUDA error string seen by this thread's calls (static storage; "" if none). */
const char *adahop_last_cuda_error(void);

/* Workspace bytes needed by adahop_linear_fwd / adahop_linear_bwd / adahop_calibrate for this
 * plan and shape (the maximum over the three GEMMs; the GEMMs of one bwd call reuse it in
 * stream order).  *bytes receives the size. */
adahop_status adahop_workspace_size(const adahop_plan *plan, int64_t M, int64_t N, int64_t K,
                                    size_t *bytes);

/* One-time pattern calibration (Fig. 4: patterns are stable, enabling one-time calibration).
 * For each of X (M x K), W (N x K) and G_Y (M x N; may be NULL -> None) it computes the mean
 * square of every row and column on the GPU, then on the host rho = max / lower-median per
 * axis; pattern = None if both rho < tau, else Column-wise if rho_col >= rho_row, else
 * Row-wise.  The strategy of each GEMM is looked up from its pattern pair:
 *   CN, NN -> IHT; RC, RN -> OE-Left; NC -> OE-Right; CC, RR, NR, CR -> BF16.
 * SYNCHRONOUS: waits for the stream (it copies the statistics to the host).  The workspace needs
 * at least 16384 + 4 x (max(M, N) + max(N, K)) + 256 bytes (adahop_workspace_size() is enough).
 * opt may be NULL (defaults). */
adahop_status adahop_calibrate(const void *X, const void *W, const void *GY, int64_t M,
                               int64_t N, int64_t K, const adahop_options *opt,
                               adahop_plan *plan_out, void *workspace, size_t ws_bytes,
                               adahop_stream_t stream);

/* Forward GEMM Y = X.W^T (M x N) with plan->fwd.  out_dtype selects bf16 or fp32 Y. */
adahop_status adahop_linear_fwd(const adahop_plan *plan, const void *X, const void *W,
                                int64_t M, int64_t N, int64_t K, void *Y, adahop_out_dtype out_dtype,
                                void *workspace, size_t ws_bytes, adahop_stream_t stream);

/* Backward GEMMs dX = G_Y.W (M x K) with plan->dgrad and dW = G_Y^T.X (N x K) with
 * plan->wgrad.  Either output may be NULL to skip that GEMM. */
adahop_status adahop_linear_bwd(const adahop_plan *plan, const void *GY, const void *X,
                                const void *W, int64_t M, int64_t N, int64_t K, void *dX,
                                void *dW, adahop_out_dtype out_dtype, void *workspace, size_t ws_bytes,
                                adahop_stream_t stream);

/* Saved context (AdaHOP appendix, IHT and Quantization: the forward pass saves quantised
 * operands for the backward pass).  The forward pass writes X quantised in the wgrad
 * orientation (lines = the K columns, blocks along M) and W in the dgrad orientation (lines =
 * the K columns, blocks along N), each with the zero mask and Hadamard setting that backward
 * GEMM applies, into a caller-owned device buffer; the backward pass then skips both
 * quantisations.  Results are bit-identical to adahop_linear_fwd / adahop_linear_bwd.  Where
 * the forward GEMM quantises the same tensor with the same mask and Hadamard setting, one pass
 * over it writes both orientations; otherwise the forward call runs the extra pass.  X and W
 * are still passed to the backward call: outlier extraction reads r of their lines in bf16.
 *
 * adahop_saved_size: *bytes receives the buffer size for this plan and shape (0 when both
 * backward GEMMs use the BF16 strategy).  Layout: X codes (K x M/2), X scales (tensor-core
 * layout), W codes (K x N/2), W scales, each part 256-byte aligned, present only when that
 * backward GEMM quantises. */
adahop_status adahop_saved_size(const adahop_plan *plan, int64_t M, int64_t N, int64_t K,
                                size_t *bytes);

/* adahop_linear_fwd plus the saved context.  saved: device, 256-byte aligned, >= saved_size
 * bytes (may be NULL only when that size is 0); ADAHOP_ERR_WORKSPACE if saved_bytes is short.
 * The buffer must stay untouched until the matching adahop_linear_bwd_saved has run. */
adahop_status adahop_linear_fwd_save(const adahop_plan *plan, const void *X, const void *W,
                                     int64_t M, int64_t N, int64_t K, void *Y, adahop_out_dtype out_dtype,
                                     void *saved, size_t saved_bytes, void *workspace,
                                     size_t ws_bytes, adahop_stream_t stream);

/* adahop_linear_bwd reading X / W's backward-orientation operands from the saved context
 * written by adahop_linear_fwd_save with the same plan, shape, X and W. */
adahop_status adahop_linear_bwd_saved(const adahop_plan *plan, const void *GY, const void *X,
                                      const void *W, const void *saved, size_t saved_bytes,
                                      int64_t M, int64_t N, int64_t K, void *dX, void *dW,
                                      adahop_out_dtype out_dtype, void *workspace, size_t ws_bytes,
                                      adahop_stream_t stream);

/* Waits for the stream, then reads (and clears) the workspace status word.
 * Returns ADAHOP_ERR_TIMEOUT if any kernel that used this workspace gave up a bounded wait. */
adahop_status adahop_get_device_status(void *workspace, adahop_stream_t stream);

/* Diagnostic of the failure path (no counterpart in the method): launches one kernel whose single
 * thread waits, through the bounded wait every kernel of this library uses, on a shared-memory
 * mbarrier that nothing arrives on.  The wait gives up after its limit (2 s), the kernel records
 * the timeout in the status word of `workspace` (its first 256 bytes; ws_bytes >= 256, 256-byte
 * aligned) and returns; no memory fault, trap or hang is involved, and the context stays usable.
 * Asynchronous: a later adahop_get_device_status() on this workspace returns ADAHOP_ERR_TIMEOUT
 * (and clears the word).  Host errors: ADAHOP_ERR_WORKSPACE (null or < 256 bytes),
 * ADAHOP_ERR_ALIGN, ADAHOP_ERR_CUDA (launch failure). */
adahop_status adahop_check_bounded_wait(void *workspace, size_t ws_bytes, adahop_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Stage entry points (each is one step of Fig. 9; the linear calls above chain them).
 * --------------------------------------------------------------------------------------- */

/* FOID, Fast Outlier Index Detection (Fig. 9 caption; appendix FOID paragraph).
 * T: rows x cols bf16.  axis 0: the lines are rows and the probe of row i is T[i, 0:64];
 * axis 1: the lines are columns and the probe of column j is T[0:64, j].
 * Score = float32 population variance of the probe (fixed pairwise summation tree, no FMA);
 * idx_out (device, int32[r]) receives the r best lines in ascending order, ties to the lower
 * index.  line_mask_out (device, may be NULL) receives a bitmap of ceil(lines/32) uint32 words
 * with the selected lines set.  One kernel launch: the CTA that finishes the per-chunk ranking
 * last merges the chunks.  Needs adahop_foid_workspace_size() bytes of workspace, 256-byte
 * aligned, whose first 256 bytes are zero at the first call (a completion counter; every call
 * leaves it zero again, so a workspace can be reused without clearing). */
adahop_status adahop_foid(const void *T, int64_t rows, int64_t cols, int axis, int r,
                          int32_t *idx_out, uint32_t *line_mask_out, void *workspace,
                          size_t ws_bytes, adahop_stream_t stream);
size_t adahop_foid_workspace_size(int64_t lines, int r);

/* FOID without a workspace.  The paper has no counterpart to this entry point: it exists for
 * callers that cannot allocate device memory -- code that is handed only its inputs and outputs
 * (a plug-in or callback inside another runtime that owns all device memory) or that must not
 * call cudaMalloc (it may synchronise the device and can fail at run time).  It computes exactly
 * what adahop_foid computes (same arguments and results, minus the workspace) and allocates
 * nothing: its scratch is a fixed 64.25 KB device array inside the library (a 256-byte counter
 * header and 8192 candidate keys), held by every GPU that loads the library until the process
 * exits.
 *   - Limit: ceil(lines / 2048) * r must be <= 8192 (e.g. r = 256 for up to 65536 lines);
 *     larger requests return ADAHOP_ERR_SHAPE before anything is launched.
 *   - The first call on a device looks up the array's device address (with that device
 *     current) and keeps it for that device's context; after a device reset (a new context) the
 *     next call looks it up again.  Under CUDA's lazy module loading that first lookup may load
 *     the library's device code and allocate its device globals (this array among them) at that
 *     moment, and may synchronise: make the first call on each device before any stream capture
 *     and at a point where that one-time set-up is acceptable.  Later calls allocate nothing.
 *   - All calls share the array and it keeps the last call's contents.  The one part that must
 *     start at zero, the counter, is zero when the library loads and every call leaves it zero;
 *     the candidate slots are written before they are read.  Calls whose kernels overlap on the
 *     GPU (e.g. on different streams) race on it and must be serialised by the caller. */
adahop_status adahop_foid_noalloc(const void *T, int64_t rows, int64_t cols, int axis, int r,
                                  int32_t *idx_out, uint32_t *line_mask_out,
                                  adahop_stream_t stream);

/* IHT + MXFP4 quantisation (appendix, IHT and Quantization: 1D FWHT with block size 32 on
 * the residual, then MXFP4 with 1D scaling).
 * T: rows x cols bf16.  inner_axis 1: quantise along the columns (output lines = rows,
 * J = cols); inner_axis 0: along the rows (output lines = cols, J = rows; the transposed
 * orientation used by the backward GEMMs).
 * zero_rows_mask / zero_cols_mask (device bitmaps over T's rows / cols, may be NULL): entries
 * in those rows/columns are set to +0 first (the OE residual, appendix FOID paragraph).
 * hadamard: 1 = apply the orthonormal Sylvester H32 per 32-block (butterflies 1..16 in
 * float32, then times the float32 nearest 1/sqrt(32)); 0 = plain MXFP4.
 * Per 32-block: E8M0 byte = clamp(floor(log2 amax) - 2 + 127, 0, 254) (0 for an all-zero
 * block); codes = nearest E2M1, ties to even, saturating; sign bit from the element.
 * codes: lines x J/2 bytes, J-contiguous, even element in the low nibble.
 * scales: scale_layout 0 = lines x J/32 bytes (canonical); 1 = the tensor-core layout (atoms
 * of 128 lines x 4 blocks, 512 bytes each, atom (l/128, b/4) at ((l/128)*(J/128) + b/4)*512,
 * byte (l%32)*16 + ((l%128)/32)*4 + b%4 inside). */
adahop_status adahop_quantize_mxfp4(const void *T, int64_t rows, int64_t cols, int inner_axis,
                                    int hadamard, const uint32_t *zero_rows_mask,
                                    const uint32_t *zero_cols_mask, uint8_t *codes,
                                    uint8_t *scales, int scale_layout, adahop_stream_t stream);

/* Both orientations of adahop_quantize_mxfp4 from one read of T (prep fusion): codes_rows /
 * scales_rows receive exactly what inner_axis 1 produces (lines = rows, J = cols), codes_cols /
 * scales_cols exactly what inner_axis 0 produces (lines = cols, J = rows), with the same masks,
 * Hadamard flag and scale layout.  The linear calls use it for G_Y when dgrad and wgrad need the
 * same residual, and adahop_linear_fwd_save for X and W when the forward GEMM and the saved
 * backward orientation share mask and Hadamard setting.  Traffic 2 + 2 x 0.53 bytes per element
 * instead of 2 x 2.53. */
adahop_status adahop_quantize_mxfp4_dual(const void *T, int64_t rows, int64_t cols, int hadamard,
                                         const uint32_t *zero_rows_mask,
                                         const uint32_t *zero_cols_mask, uint8_t *codes_rows,
                                         uint8_t *scales_rows, uint8_t *codes_cols,
                                         uint8_t *scales_cols, int scale_layout,
                                         adahop_stream_t stream);

/* Outlier slice gather for the BF16 path.  T: rows x cols bf16; idx: int32[r] (device).
 * mode 0: out[i, :] = T[idx[i], :]          (r x cols)
 * mode 1: out[p, i] = T[p, idx[i]]          (rows x r)
 * mode 2: out[q, i] = T[idx[i], q]          (cols x r)
 * mode 3: out[i, p] = T[p, idx[i]]          (r x rows) */
adahop_status adahop_gather(const void *T, int64_t rows, int64_t cols, const int32_t *idx,
                            int r, int mode, void *out, adahop_stream_t stream);

/* Fused MXFP4 (+ BF16 inner outlier) GEMM (appendix, Fused MXFP4+BF16 GEMM).
 * C (P x Q) = deq(A) . deq(B)^T + A_o . B_o^T, accumulated in float32 in tensor memory.
 * A: P x J MXFP4 (codes P x J/2, scales in layout 1), B: Q x J likewise.
 * A_o: P x r bf16 and B_o: Q x r bf16 (r-contiguous; both NULL or r = 0 for no outlier term;
 * r a multiple of 8).  C: bf16 or fp32 per out_dtype.  P, Q, J multiples of 128.
 * Workspace: at least 256 bytes (the status word).  With at least
 * adahop_gemm_mxfp4_workspace_size() bytes, whose first 16384 bytes are zero at the first call
 * (every call leaves them zero), the GEMM balances the tiles that a whole round over the SMs would
 * leave short (stream-K: their J stages are spread over all CTA pairs, partial sums added in a
 * fixed order); with less it runs whole tiles only.  Both give results within the same bound. */
adahop_status adahop_gemm_mxfp4(const uint8_t *a_codes, const uint8_t *a_scales,
                                const uint8_t *b_codes, const uint8_t *b_scales, int64_t P,
                                int64_t Q, int64_t J, const void *A_o, const void *B_o, int r,
                                void *C, adahop_out_dtype out_dtype, void *workspace, size_t ws_bytes,
                                adahop_stream_t stream);

/* Workspace bytes that let adahop_gemm_mxfp4 use stream-K (a zeroed 16 KB header and one
 * 256 x 256 float32 partial tile per CTA pair). */
size_t adahop_gemm_mxfp4_workspace_size(void);

/* BF16 GEMM C (P x Q) = A . B, float32 accumulation (Fig. 5's BF16 path; also the outlier
 * GEMM of outer OE).  a_kmajor 1: A stored P x J (J-contiguous); 0: stored J x P.
 * b_kmajor 1: B stored Q x J (i.e. B^T row-major); 0: stored J x Q.
 * With c_partial non-NULL, J is cut into `splits` (>= 1) ranges and the partial sums go to
 * c_partial[s] (fp32, splits x P x Q) instead of C (C may then be NULL; splits > 1 requires
 * c_partial).  P >= 1 (a multiple of 64 when A is
 * stored J x P); Q and J multiples of 64.  The workspace only carries the status word. */
adahop_status adahop_gemm_bf16(const void *A, int a_kmajor, const void *B, int b_kmajor,
                               int64_t P, int64_t Q, int64_t J, void *C, adahop_out_dtype out_dtype,
                               int splits, float *c_partial, void *workspace, size_t ws_bytes,
                               adahop_stream_t stream);

/* Outlier GEMM of outer OE with the scatter-add fused (appendix, Fused Scatter-Add: the outlier
 * product is added in place, without materialising it).  O = A . B with A and B stored as in
 * adahop_gemm_bf16 (a_kmajor / b_kmajor); then
 *   axis 0 (P = r):  C[idx[i], q] += O[i, q]   for i < r, q < Q  (Q = c_cols)
 *   axis 1 (Q = r):  C[p, idx[i]] += O[p, i]   for p < P, i < r  (P = c_rows)
 * C: c_rows x c_cols, bf16 or fp32 per out_dtype, read and written in place; each sum is formed
 * in float32 (the J range split over the CTAs of a cluster, partials summed in a fixed order),
 * added to C's value in float32 and rounded once to C's type.  Indices outside C are skipped.
 * One kernel launch.  1 <= r <= 256; J a multiple of 64; c_cols a multiple of 8; P (Q) a multiple
 * of 64 when A (B) is stored J-major.  The workspace only carries the status word (>= 256 bytes). */
adahop_status adahop_gemm_bf16_scatter_add(const void *A, int a_kmajor, const void *B, int b_kmajor, int64_t P,
                                           int64_t Q, int64_t J, void *C, int64_t c_rows, int64_t c_cols,
                                           adahop_out_dtype out_dtype, const int32_t *idx, int r, int axis, void *workspace,
                                           size_t ws_bytes, adahop_stream_t stream);

/* Fused scatter-add (appendix, Fused Scatter-Add): adds the outlier product in place.
 * partial: fp32, splits x r x Q (axis 0) or splits x P x r (axis 1), summed over splits.
 * axis 0: C[idx[i], q] += sum_s partial[s, i, q];  axis 1: C[p, idx[i]] += sum_s partial[s, p, i].
 * The sum is formed in float32 and rounded once to C's type. */
adahop_status adahop_scatter_add(void *C, int64_t P, int64_t Q, adahop_out_dtype out_dtype,
                                 const float *partial, int splits, const int32_t *idx, int r,
                                 int axis, adahop_stream_t stream);

/* Calibration statistics: row_ms[i] = mean_j T[i,j]^2, col_ms[j] = mean_i T[i,j]^2 (float32,
 * device).  Both outputs are overwritten. */
adahop_status adahop_calibration_stats(const void *T, int64_t rows, int64_t cols, float *row_ms,
                                       float *col_ms, adahop_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Peak probes (K8; no counterpart on the pages): the roofline denominators measured on the part.
 * --------------------------------------------------------------------------------------- */

/* Number of CTAs adahop_probe_mma_rate launches on the current device (one per SM); 0 if the
 * device is unusable. */
int adahop_probe_ctas(void);

/* Tensor-pipe rate probe.  One CTA per SM; in each, one elected lane issues `iters` groups of
 * four back-to-back tcgen05.mma instructions (cta_group::1, M = 128, N = n: 128 or 256) on operands that
 * stay in shared memory, all accumulating into one tensor-memory tile, then waits (bounded) for
 * them to finish.  kind: 0 = kind::f16 (bf16 x bf16, K = 16 per instruction); 1 = kind::mxf4,
 * scale_vec::2X; 2 = kind::mxf4nvf4, scale_vec::2X; 3 = kind::mxf4nvf4, scale_vec::4X (kinds 1-3:
 * E2M1 operands, UE8M0 scales, K = 64).  sf_copies = 1 adds, per group, the six scale-factor
 * copies (tcgen05.cp) the fused MXFP4 GEMM issues per 256-wide slice of J (kinds 1-3 only; with
 * n = 128 the B copies cover 128 rows: four copies per group).
 * Operand values are a fixed pattern; nothing but timing is produced.
 * out: device, 16-byte aligned, out_bytes >= 24 * adahop_probe_ctas(); CTA c writes
 * out[3c] = clock64 cycles of its loop, out[3c+1] / out[3c+2] = %globaltimer ns at its start /
 * end.  FLOP per group: 4 x 2 x 128 x n x K.  iters: 1 .. 2^20 (ERR_SHAPE otherwise).
 * workspace: >= 256 bytes, 256-byte aligned, first 256 bytes zeroed (status word; a wait that
 * ran out is reported by adahop_get_device_status).  Asynchronous on `stream`. */
adahop_status adahop_probe_mma_rate(int kind, int sf_copies, int n, int64_t iters, uint64_t *out, size_t out_bytes,
                                    void *workspace, size_t ws_bytes, adahop_stream_t stream);

/* Streaming copy probe: dst[0:bytes] = src[0:bytes] with 16-byte loads and stores (streaming
 * cache hints), grid sized to the SM count.  bytes a multiple of 16, pointers 16-byte aligned,
 * buffers must not overlap.  Time it on `stream` (2 x bytes of DRAM traffic per call).
 * src NULL: write-only stream instead, every 16-bit half-word of dst[0:bytes] set to 0x3F80
 * (bytes of DRAM writes per call; the denominator for store-bound kernels).  dst NULL:
 * ADAHOP_ERR_INVALID_ARG.  Asynchronous. */
adahop_status adahop_probe_copy(const void *src, void *dst, size_t bytes, adahop_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ADAHOP_H */
