// K4 (fused scatter-add), the outlier-slice gathers of the BF16 path, K7 (calibration
// statistics), and the probe of the bounded-wait failure path.
//
// AdaHOP appendix implementation notes, "Fused Scatter-Add": the outlier product is added in
// place into the residual GEMM's result.  Here the (possibly split-K) float32 partials are
// summed in float32, added to C's current value in float32, and rounded once to C's type.
// Calibration (one-time; Fig. 4 shows the patterns are stable): per-row and per-column mean
// squares in float32, from one pass over the tensor.
#include "common.cuh"
#include "kernels.cuh"

namespace adahop {

namespace {

// ------------------------------------------------------------------------------- gathers
// Each mode is a device function over a virtual grid (block vb of vg, 256 threads) so that one
// launch can run several gathers side by side (gather_multi_kernel); `tile` is the caller's
// shared memory (256 x 72 uint16 at most).
constexpr int kGatherThreads = 256;
constexpr int kGatherTileElems = 256 * 72;

// mode 0: out[i, :] = T[idx[i], :]   (r x cols), 16-byte copies
__device__ void gather_rows(const uint16_t *__restrict__ T, int64_t rows, int64_t cols, const int32_t *__restrict__ idx,
                            int r, uint16_t *out, int64_t vb, int64_t vg) {
  const int64_t vec = cols >> 3;
  const int64_t total = static_cast<int64_t>(r) * vec;
  for (int64_t t = vb * kGatherThreads + threadIdx.x; t < total; t += vg * kGatherThreads) {
    const int64_t i = t / vec, v = t - i * vec;
    const int64_t src = idx[i];
    if (src < 0 || src >= rows) continue;        // indices come from FOID; never read outside T
    reinterpret_cast<uint4 *>(out + i * cols)[v] = __ldg(reinterpret_cast<const uint4 *>(T + src * cols) + v);
  }
}
// mode 1: out[p, i] = T[p, idx[i]]   (rows x r_out; columns r .. r_out - 1 are +0)
__device__ void gather_cols(const uint16_t *__restrict__ T, int64_t rows, int64_t cols, const int32_t *__restrict__ idx,
                            int r, int r_out, uint16_t *out, int64_t vb, int64_t vg) {
  const int64_t total = rows * r_out;
  for (int64_t t = vb * kGatherThreads + threadIdx.x; t < total; t += vg * kGatherThreads) {
    const int64_t p = t / r_out, i = t - p * r_out;
    const int64_t c = i < r ? idx[i] : -1;
    out[t] = (c >= 0 && c < cols) ? __ldg(T + p * cols + c) : static_cast<uint16_t>(0);
  }
}
// mode 2: out[q, i] = T[idx[i], q]   (cols x r_out; columns r .. r_out - 1 are +0): a 32-column x
// r_out tile through shared memory
__device__ void gather_rows_t(const uint16_t *__restrict__ T, int64_t rows, int64_t cols, const int32_t *__restrict__ idx,
                              int r, int r_out, uint16_t *out, int64_t vb, uint16_t *tile /* [256][34] */) {
  const int64_t q0 = vb * 32;
  for (int t = threadIdx.x; t < r_out * 32; t += kGatherThreads) {
    const int i = t >> 5, q = t & 31;
    const int64_t src = i < r ? idx[i] : -1;
    tile[i * 34 + q] = (src >= 0 && src < rows) ? __ldg(T + src * cols + q0 + q) : static_cast<uint16_t>(0);
  }
  __syncthreads();
  for (int t = threadIdx.x; t < r_out * 32; t += kGatherThreads) {
    const int q = t / r_out, i = t - q * r_out;
    out[(q0 + q) * r_out + i] = tile[i * 34 + q];
  }
}
// mode 2 when cols % 64 == 0 and r % 32 == 0: a CTA moves 64 columns x r selected rows with
// 16-byte loads into shared memory, then each thread writes r/4 contiguous values of one output
// row with 16-byte stores (column reads from the tile are conflict-free: consecutive lanes read
// consecutive columns of one row).
__device__ void gather_rows_t_vec(const uint16_t *__restrict__ T, int64_t rows, int64_t cols,
                                  const int32_t *__restrict__ idx, int r, uint16_t *out, int64_t vb,
                                  uint16_t *tile /* [256][72], 16-byte aligned */) {
  const int64_t q0 = vb * 64;
  for (int t = threadIdx.x; t < r * 8; t += kGatherThreads) {
    const int i = t >> 3, c = t & 7;
    const int64_t src = idx[i];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (src >= 0 && src < rows) v = __ldg(reinterpret_cast<const uint4 *>(T + src * cols + q0) + c);
    *reinterpret_cast<uint4 *>(&tile[i * 72 + 8 * c]) = v;
  }
  __syncthreads();
  const int q = threadIdx.x & 63, part = threadIdx.x >> 6;   // four parts of r/4 values
  const int rp = r >> 2;
  uint16_t *dst = out + (q0 + q) * r + part * rp;
  for (int i = 0; i < rp; i += 8) {
    const int ib = part * rp + i;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = static_cast<uint32_t>(tile[(ib + 2 * k) * 72 + q]) | (static_cast<uint32_t>(tile[(ib + 2 * k + 1) * 72 + q]) << 16);
    *reinterpret_cast<uint4 *>(dst + i) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
// mode 3: out[i, p] = T[p, idx[i]]   (r x rows)
__device__ void gather_cols_t(const uint16_t *__restrict__ T, int64_t rows, int64_t cols, const int32_t *__restrict__ idx,
                              int r, uint16_t *out, int64_t vb, int64_t vg) {
  const int64_t total = rows * r;
  for (int64_t t = vb * kGatherThreads + threadIdx.x; t < total; t += vg * kGatherThreads) {
    const int64_t i = t / rows, p = t - i * rows;
    const int64_t c = idx[i];
    out[t] = (c >= 0 && c < cols) ? __ldg(T + p * cols + c) : static_cast<uint16_t>(0);
  }
}

unsigned grid_for(int64_t work, int threads, int64_t cap = 8192) {
  int64_t b = (work + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > cap) b = cap;
  return static_cast<unsigned>(b);
}

// The mode-2 variant and the block count of one gather job (r_out already resolved).
bool rows_t_vec(const GatherJob &j) { return j.cols % 64 == 0 && j.r % 32 == 0 && j.r_out == j.r; }
int64_t gather_blocks(const GatherJob &j) {
  switch (j.mode) {
    case 0: return grid_for(j.r * (j.cols >> 3), kGatherThreads);
    case 1: return grid_for(j.rows * j.r_out, kGatherThreads);
    case 2: return rows_t_vec(j) ? j.cols / 64 : j.cols / 32;
    default: return grid_for(j.rows * j.r, kGatherThreads);
  }
}

__device__ __forceinline__ void gather_job(const GatherJob &j, int64_t vb, int64_t vg, uint16_t *tile) {
  switch (j.mode) {
    case 0: gather_rows(j.T, j.rows, j.cols, j.idx, j.r, j.out, vb, vg); break;
    case 1: gather_cols(j.T, j.rows, j.cols, j.idx, j.r, j.r_out, j.out, vb, vg); break;
    case 2:
      if (j.cols % 64 == 0 && j.r % 32 == 0 && j.r_out == j.r)
        gather_rows_t_vec(j.T, j.rows, j.cols, j.idx, j.r, j.out, vb, tile);
      else
        gather_rows_t(j.T, j.rows, j.cols, j.idx, j.r, j.r_out, j.out, vb, tile);
      break;
    default: gather_cols_t(j.T, j.rows, j.cols, j.idx, j.r, j.out, vb, vg); break;
  }
}

// Up to kMaxGatherJobs gathers in one launch: blocks [first[k], first[k + 1]) run job k.
struct GatherLaunch {
  GatherJob job[kMaxGatherJobs];
  int64_t first[kMaxGatherJobs + 1];
  int count;
};

__global__ void __launch_bounds__(kGatherThreads) gather_multi_kernel(const __grid_constant__ GatherLaunch g) {
  __shared__ __align__(16) uint16_t tile[kGatherTileElems];
  int k = 0;
  while (k + 1 < g.count && blockIdx.x >= g.first[k + 1]) ++k;
  gather_job(g.job[k], blockIdx.x - g.first[k], g.first[k + 1] - g.first[k], tile);
}

// ------------------------------------------------------------------------------- scatter-add
__device__ __forceinline__ float load_out(const float *p) { return *p; }
__device__ __forceinline__ float load_out(const uint16_t *p) { return bf16_bits_to_f32(*p); }
__device__ __forceinline__ void store_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_out(uint16_t *p, float v) {
  *p = static_cast<uint16_t>(f32_to_bf16_bits(v));
}

// axis 0: C[idx[i], q] += sum_s partial[s, i, q]
template <typename OutT>
__global__ void scatter_rows_kernel(OutT *C, int64_t P, int64_t Q, const float *__restrict__ partial,
                                    int splits, const int32_t *__restrict__ idx, int r) {
  const int64_t total = static_cast<int64_t>(r) * Q;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = t / Q, q = t - i * Q;
    float acc = 0.0f;
    const int64_t row = idx[i];
    if (row < 0 || row >= P) continue;           // never write outside C
    for (int s = 0; s < splits; ++s) acc += partial[s * total + t];
    OutT *dst = C + row * Q + q;
    store_out(dst, load_out(dst) + acc);
  }
}
// axis 1: C[p, idx[i]] += sum_s partial[s, p, i]
template <typename OutT>
__global__ void scatter_cols_kernel(OutT *C, int64_t P, int64_t Q, const float *__restrict__ partial,
                                    int splits, const int32_t *__restrict__ idx, int r) {
  const int64_t total = P * r;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = t / r, i = t - p * r;
    float acc = 0.0f;
    const int64_t col = idx[i];
    if (col < 0 || col >= Q) continue;           // never write outside C
    for (int s = 0; s < splits; ++s) acc += partial[s * total + t];
    OutT *dst = C + p * Q + col;
    store_out(dst, load_out(dst) + acc);
  }
}

// ------------------------------------------------------------------------------- calibration
// Block: 256 threads x 8 columns = 2048 columns; 64 rows per block.  Row sums are reduced per
// block and added atomically; column sums are accumulated over the 64 rows and added atomically.
constexpr int kCalRows = 64;
__global__ void __launch_bounds__(256) calib_stats_kernel(const uint16_t *__restrict__ T,
                                                          int64_t rows, int64_t cols,
                                                          float *row_sum, float *col_sum) {
  __shared__ float red[8];
  const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) * 8;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kCalRows;
  const bool active = c0 < cols;
  float colacc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int rr = 0; rr < kCalRows && r0 + rr < rows; ++rr) {
    float rs = 0.0f;
    if (active) {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(T + (r0 + rr) * cols + c0));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a = bf16_bits_to_f32(w[k] & 0xFFFFu), b = bf16_bits_to_f32(w[k] >> 16);
        colacc[2 * k] += a * a;
        colacc[2 * k + 1] += b * b;
        rs += a * a + b * b;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xFFFFFFFFu, rs, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = rs;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int k = 0; k < 8; ++k) t += red[k];
      atomicAdd(row_sum + r0 + rr, t);
    }
    __syncthreads();
  }
  if (active) {
#pragma unroll
    for (int k = 0; k < 8; ++k) atomicAdd(col_sum + c0 + k, colacc[k]);
  }
}
__global__ void scale_kernel(float *v, int64_t n, float s) {
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x)
    v[t] *= s;
}

// Failure-path probe: one thread waits, through the same bounded wait the GEMM kernels use, on
// an mbarrier that nothing ever arrives on.  The wait gives up after its limit (2 s of
// %globaltimer); the thread records the timeout in the status word and the kernel returns, so the
// context stays usable.
__global__ void bounded_wait_probe_kernel(uint32_t *status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) mbar_init(smem_u32(&bar), 1);
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, nullptr)) report_status(status, kStatusTimeout);
  __syncthreads();
}

}  // namespace

cudaError_t launch_gathers(const GatherJob *jobs, int count, cudaStream_t s) {
  if (count < 0 || count > kMaxGatherJobs) return cudaErrorInvalidValue;
  GatherLaunch g{};
  int64_t blocks = 0;
  for (int k = 0; k < count; ++k) {
    if (jobs[k].r == 0) continue;
    GatherJob j = jobs[k];
    if (j.r_out == 0 || (j.mode != 1 && j.mode != 2)) j.r_out = j.r;
    if (j.mode < 0 || j.mode > 3 || j.r > 256 || j.r_out < j.r || j.r_out > 256) return cudaErrorInvalidValue;
    g.job[g.count] = j;
    g.first[g.count] = blocks;
    blocks += gather_blocks(j);
    ++g.count;
  }
  if (g.count == 0) return cudaSuccess;
  g.first[g.count] = blocks;
  gather_multi_kernel<<<static_cast<unsigned>(blocks), kGatherThreads, 0, s>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t *T, int64_t rows, int64_t cols, const int32_t *idx, int r,
                          int mode, uint16_t *out, cudaStream_t s) {
  const GatherJob j{T, rows, cols, idx, r, mode, out, 0};
  return launch_gathers(&j, 1, s);
}

cudaError_t launch_scatter_add(void *C, int64_t P, int64_t Q, int out_dtype, const float *partial,
                               int splits, const int32_t *idx, int r, int axis, cudaStream_t s) {
  if (r == 0) return cudaSuccess;
  const int64_t work = axis == 0 ? r * Q : P * r;
  const unsigned g = grid_for(work, 256);
  if (axis == 0) {
    if (out_dtype == 1)
      scatter_rows_kernel<float><<<g, 256, 0, s>>>(static_cast<float *>(C), P, Q, partial, splits, idx, r);
    else
      scatter_rows_kernel<uint16_t><<<g, 256, 0, s>>>(static_cast<uint16_t *>(C), P, Q, partial, splits,
                                                      idx, r);
  } else {
    if (out_dtype == 1)
      scatter_cols_kernel<float><<<g, 256, 0, s>>>(static_cast<float *>(C), P, Q, partial, splits,
                                                   idx, r);
    else
      scatter_cols_kernel<uint16_t><<<g, 256, 0, s>>>(static_cast<uint16_t *>(C), P, Q, partial,
                                                      splits, idx, r);
  }
  return cudaGetLastError();
}

cudaError_t launch_bounded_wait_probe(uint32_t *status, cudaStream_t s) {
  bounded_wait_probe_kernel<<<1, 32, 0, s>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_calib_stats(const uint16_t *T, int64_t rows, int64_t cols, float *row_ms,
                               float *col_ms, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(row_ms, 0, rows * sizeof(float), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(col_ms, 0, cols * sizeof(float), s);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((cols + 2047) / 2048),
            static_cast<unsigned>((rows + kCalRows - 1) / kCalRows));
  calib_stats_kernel<<<grid, 256, 0, s>>>(T, rows, cols, row_ms, col_ms);
  scale_kernel<<<grid_for(rows, 256), 256, 0, s>>>(row_ms, rows, 1.0f / static_cast<float>(cols));
  scale_kernel<<<grid_for(cols, 256), 256, 0, s>>>(col_ms, cols, 1.0f / static_cast<float>(rows));
  return cudaGetLastError();
}

}  // namespace adahop
