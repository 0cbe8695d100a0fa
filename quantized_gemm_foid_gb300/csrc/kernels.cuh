// Launch interfaces of the sm_103a kernels (host dispatcher <-> kernel translation units).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace adahop {

// Byte offset of scale factor (line, 32-block blk) in the tensor-core scale layout: atoms of
// 128 lines x 4 blocks (512 bytes), atom (line/128, blk/4) at ((line/128)*(J/128) + blk/4)*512,
// and inside the atom byte (line%32)*16 + ((line%128)/32)*4 + blk%4.
template <class I>
__host__ __device__ __forceinline__ I tiled_sf_offset(I line, I blk, I J) {
  return ((line >> 7) * (J >> 7) + (blk >> 2)) * 512 + (line & 31) * 16 + ((line >> 5) & 3) * 4 +
         (blk & 3);
}

struct QuantArgs {
  const uint16_t *T;            // rows x cols bf16
  int64_t rows, cols;
  const uint32_t *zero_rows;    // bitmap over rows (may be null)
  const uint32_t *zero_cols;    // bitmap over cols (may be null)
  uint8_t *codes;
  uint8_t *scales;
  int hadamard;
  int scale_layout;             // 0 canonical, 1 tensor-core atoms
};
cudaError_t launch_quant(const QuantArgs &a, int inner_axis, int num_sms, cudaStream_t s);
// Both orientations in one pass: a.codes / a.scales receive the J = cols orientation (lines = rows),
// codes_cols / scales_cols the J = rows orientation (lines = cols); same masks and Hadamard flag.
cudaError_t launch_quant_dual(const QuantArgs &a, uint8_t *codes_cols, uint8_t *scales_cols, cudaStream_t s);

// FOID in one launch: stage 1 (per-chunk top-r of 256..2048 lines), then the last CTA to finish
// merges (ascending indices, bitmap).  scratch: foid_scratch_bytes() of candidates; counter: one
// uint32 that must be zero when the launch starts (the launch leaves it zero).
size_t foid_scratch_bytes(int64_t lines, int r);
cudaError_t launch_foid(const uint16_t *T, int64_t rows, int64_t cols, int axis, int r,
                        int32_t *idx_out, uint32_t *mask_out, void *scratch, uint32_t *counter, cudaStream_t s);

// FOID with its candidate keys in a fixed device array instead of caller scratch (see foid.cu).
int64_t foid_static_capacity();
cudaError_t launch_foid_noalloc(const uint16_t *T, int64_t rows, int64_t cols, int axis, int r,
                                int32_t *idx_out, uint32_t *mask_out, cudaStream_t s);

cudaError_t launch_gather(const uint16_t *T, int64_t rows, int64_t cols, const int32_t *idx, int r,
                          int mode, uint16_t *out, cudaStream_t s);
// Several gathers (modes of launch_gather) in one launch, each on its own range of CTAs.
struct GatherJob {
  const uint16_t *T;
  int64_t rows, cols;
  const int32_t *idx;
  int r;
  int mode;
  uint16_t *out;
  int r_out;   // modes 1 / 2: values per output line (>= r; entries r .. r_out - 1 are +0); 0 = r
};
constexpr int kMaxGatherJobs = 4;
cudaError_t launch_gathers(const GatherJob *jobs, int count, cudaStream_t s);

cudaError_t launch_scatter_add(void *C, int64_t P, int64_t Q, int out_dtype, const float *partial,
                               int splits, const int32_t *idx, int r, int axis, cudaStream_t s);

cudaError_t launch_bounded_wait_probe(uint32_t *status, cudaStream_t s);
cudaError_t launch_calib_stats(const uint16_t *T, int64_t rows, int64_t cols, float *row_ms,
                               float *col_ms, cudaStream_t s);

// K8 peak probes.  kind: 0 kind::f16, 1 kind::mxf4 (2X), 2 kind::mxf4nvf4 (2X), 3 kind::mxf4nvf4
// (4X); n: MMA width 128 or 256; `ctas` CTAs (one per SM) each write {loop cycles, start ns, end ns}
// to out[3 * cta ..].
cudaError_t launch_mma_rate_probe(int kind, int sf_copies, int n, int64_t iters, uint64_t *out, uint32_t *status,
                                  int ctas, cudaStream_t s);
cudaError_t launch_copy_probe(const void *src, void *dst, size_t bytes, int num_sms, cudaStream_t s);

// tcgen05 GEMM (K3 MXFP4 + inner BF16 tail, K5/K6 BF16).
struct GemmArgs {
  int64_t P, Q, J;            // C is P x Q; inner dimension J
  int kind;                   // 0 = MXFP4 (+ optional BF16 tail), 1 = BF16
  int a_mn_major, b_mn_major; // BF16 only: operand stored J-major (MN contiguous)
  const uint8_t *sfa, *sfb;   // MXFP4 scale factors (tensor-core layout; read through maps.sfa / sfb)
  int tail_stages;            // MXFP4: ceil(r / 64) stages of BF16 outlier MMAs
  void *C;
  int out_dtype;              // 0 bf16, 1 fp32
  int splits;                 // BF16: split-K count (>= 1)
  float *c_partial;           // non-null: fp32 partials (splits x P x Q) are written here, not C
  uint32_t *status;
  // kind 2 (BF16 outlier GEMM with the scatter-add fused): the product O (P x Q) is added into the
  // output C (c_rows x c_cols, out_dtype): scatter_axis 0: C[idx[i], q] += O[i, q] (P = r);
  // scatter_axis 1: C[p, idx[i]] += O[p, i] (Q = r).  `splits` CTAs of one cluster share a tile.
  const int32_t *scatter_idx;
  int scatter_axis;
  int64_t c_rows, c_cols;
  // kind 0: stream-K for the tiles a whole round cannot fill (sk != 0, set by launch_gemm when the
  // caller provides both buffers): float32 partial tiles of the contributing pairs (sk_partial,
  // kSkPartialBytesPerPair per pair, at most sk_max_pairs pairs) and kSkCountersPerTile counters per
  // stream-K tile (sk_counters, zero when the launch starts; the launch leaves them zero).
  int sk;
  float *sk_partial;
  uint32_t *sk_counters;
  int sk_max_pairs;
};
// Stream-K scratch of the fused MXFP4 GEMM: one 256 x 256 float32 partial tile per CTA pair, and
// 16 counters per stream-K tile (2 CTAs x 8 epilogue warps), at most kSkMaxTiles tiles.
constexpr size_t kSkPartialBytesPerPair = 256 * 256 * 4;
constexpr int kSkMaxTiles = 160;
constexpr int kSkCountersPerTile = 16;
// MXFP4: a / b are the E2M1 codes (128-byte rows, 128 rows per box), sfa / sfb the tensor-core
// scale atoms viewed as rows of 128 uint32 (one 512-byte atom per row, two atoms per box), ao / bo
// the BF16 outlier slices, c the output C (MXFP4 only: 32-row boxes of 32 bytes, 32-byte swizzle,
// written by TMA stores; unused when C is null).  BF16: a / b only.
struct GemmMaps {
  CUtensorMap a, b, ao, bo, sfa, sfb, c;
};
cudaError_t launch_gemm(const GemmArgs &g, const GemmMaps &maps, int num_sms, cudaStream_t s);
// Cluster size (split-K count) the fused outlier GEMM uses for a P x Q x J product.
int scatter_gemm_splits(int64_t P, int64_t Q, int64_t J, int num_sms);
size_t gemm_smem_bytes(int kind);
int gemm_tail_cols_per_stage();

}  // namespace adahop
