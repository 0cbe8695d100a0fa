// K1: FOID, Fast Outlier Index Detection.
//
// AdaHOP, Fig. 9 caption and appendix FOID paragraph: the variance of the first 64 elements
// along each row (or column) ranks the lines, and the top-k lines are the outliers.
//
// Score of line l (float32, one fixed order, no fused multiply-add):
//   level 0: s[i] = x[i] + x[i+32], q[i] = x[i]^2 + x[i+32]^2            (i < 32)
//   level k: s[i] += s[i + 2^(5-k)], q[i] += q[i + 2^(5-k)]               (k = 1..5)
//   mean = s * (1/64); var = q * (1/64) - mean * mean; var <- +0 unless var > 0.
// Ranking key = (float bits of var) << 32 | (0xFFFFFFFF - l): larger variance first, and for
// equal variance the lower index first.  Keys are unique, so the top-r set is well defined.
//
// Stage 1 (grid): each CTA scores one chunk of 256..2048 lines (the smallest chunk that keeps
// at most 8192 candidates overall); every warp sorts 32 keys in registers (bitonic network over
// shuffles), then merge levels in shared memory keep the best r of each merged pair until one
// run remains, written out as the chunk's r candidates.  Stage 2 (one CTA): merge levels over
// the chunks' runs down to the global best r, then each selected line's position in ascending
// line order is its count of smaller selected lines.  A merge level is one pass: output i of the
// best keys of sorted runs A and B is max(A[a], B[i - a]), where a, the number of A's keys among
// the i best, comes from a binary search (A[m] belongs to the i best iff A[m] > B[i - m - 1]).
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace adahop {

namespace {

constexpr int kFoidThreads = 512;
constexpr int kFoidMaxChunk = 2048;         // lines per stage-1 CTA, at most
constexpr int kFoidMinChunk = 256;
constexpr int kFoidMergeMaxKeys = 8192;     // candidates written by stage 1, at most
// stage-2 shared memory: the candidates plus the first level's output (at most half of them + r)
constexpr int kFoidMergeSmemKeys = kFoidMergeMaxKeys + kFoidMergeMaxKeys / 2 + 256;

int pow2_at_least(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// Smallest chunk (many stage-1 CTAs) that keeps the candidate count within the merge's capacity.
int foid_chunk(int64_t lines, int r) {
  const int rr = r > 0 ? r : 1;
  for (int chunk = kFoidMinChunk; chunk < kFoidMaxChunk; chunk <<= 1) {
    if (chunk >= pow2_at_least(rr) && (lines + chunk - 1) / chunk * rr <= kFoidMergeMaxKeys) return chunk;
  }
  return kFoidMaxChunk;
}

__device__ __forceinline__ float bf(uint32_t b) { return __uint_as_float(b << 16); }

// Level 0 of the tree for the pair (a = x[i], b = x[i+32]).
__device__ __forceinline__ void level0(float a, float b, float &s, float &q) {
  s = __fadd_rn(a, b);
  q = __fadd_rn(__fmul_rn(a, a), __fmul_rn(b, b));
}

template <int AXIS>
__device__ __forceinline__ uint64_t foid_key(const uint16_t *__restrict__ T, int64_t cols,
                                             int64_t line) {
  float s[32], q[32];
  if (AXIS == 0) {
    const uint4 *p = reinterpret_cast<const uint4 *>(T + line * cols);
#pragma unroll
    for (int k = 0; k < 4; ++k) {           // chunk k holds x[8k..8k+7], chunk k+4 x[8k+32..]
      const uint4 lo = __ldg(p + k), hi = __ldg(p + k + 4);
      const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w}, wh[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        level0(bf(wl[j] & 0xFFFFu), bf(wh[j] & 0xFFFFu), s[8 * k + 2 * j], q[8 * k + 2 * j]);
        level0(bf(wl[j] >> 16), bf(wh[j] >> 16), s[8 * k + 2 * j + 1], q[8 * k + 2 * j + 1]);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float a = bf(__ldg(T + static_cast<int64_t>(i) * cols + line));
      const float b = bf(__ldg(T + static_cast<int64_t>(i + 32) * cols + line));
      level0(a, b, s[i], q[i]);
    }
  }
#pragma unroll
  for (int h = 16; h >= 1; h >>= 1) {
#pragma unroll
    for (int i = 0; i < h; ++i) {
      s[i] = __fadd_rn(s[i], s[i + h]);
      q[i] = __fadd_rn(q[i], q[i + h]);
    }
  }
  const float inv64 = 0.015625f;
  const float mean = __fmul_rn(s[0], inv64);
  float var = __fsub_rn(__fmul_rn(q[0], inv64), __fmul_rn(mean, mean));
  if (!(var > 0.0f)) var = 0.0f;
  return (static_cast<uint64_t>(__float_as_uint(var)) << 32) |
         static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(line));
}

// Sorts the warp's 32 keys (one per lane) descending across the lanes: lane i ends with the
// (i+1)-th largest.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t key) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, key, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      key = keep_max ? (key > other ? key : other) : (key < other ? key : other);
    }
  }
  return key;
}

// The (i+1)-th largest key of the union of A[0..la) and B[0..lb), both sorted descending, keys
// distinct, i < la + lb.
__device__ __forceinline__ uint64_t merge_at(const uint64_t *A, int la, const uint64_t *B, int lb, int i) {
  int lo = i - lb > 0 ? i - lb : 0;
  int hi = i < la ? i : la;
  while (lo < hi) {                          // a = number of A's keys among the i largest
    const int mid = (lo + hi) >> 1;
    if (A[mid] > B[i - mid - 1])
      lo = mid + 1;
    else
      hi = mid;
  }
  const int b = i - lo;
  if (lo >= la) return B[b];
  if (b >= lb) return A[lo];
  return A[lo] > B[b] ? A[lo] : B[b];
}

template <int AXIS>
__global__ void __launch_bounds__(kFoidThreads) foid_local_kernel(const uint16_t *__restrict__ T,
                                                                  int64_t rows, int64_t cols, int r,
                                                                  int chunk, uint64_t *cand) {
  __shared__ uint64_t keys[2][kFoidMaxChunk];
  const int64_t lines = AXIS == 0 ? rows : cols;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * chunk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  for (int r0 = 32 * warp; r0 < chunk; r0 += 32 * nwarps) {
    const int64_t line = base + r0 + lane;
    const uint64_t key = line < lines ? foid_key<AXIS>(T, cols, line) : 0ull;
    keys[0][r0 + lane] = warp_sort_desc(key);
  }
  __syncthreads();
  // chunk / 32 runs (a power of two) of equal length; keep the best min(2 len, r) of each pair
  int g = chunk >> 5, len = 32, src = 0;
  while (g > 1) {
    const int out = 2 * len < r ? 2 * len : r;
    const int pairs = g >> 1;
    for (int o = tid; o < pairs * out; o += blockDim.x) {
      const int p = o / out, i = o - p * out;
      const uint64_t *A = keys[src] + 2 * p * len;
      keys[src ^ 1][p * out + i] = merge_at(A, len, A + len, len, i);
    }
    __syncthreads();
    src ^= 1;
    g = pairs;
    len = out;
  }
  for (int i = tid; i < r; i += blockDim.x)
    cand[static_cast<int64_t>(blockIdx.x) * r + i] = i < len ? keys[src][i] : 0ull;
}

// runs x r candidates (each run sorted descending, r keys).
__global__ void __launch_bounds__(1024) foid_merge_kernel(const uint64_t *cand, int runs, int r, int64_t lines,
                                                          int32_t *idx_out, uint32_t *mask_out) {
  extern __shared__ uint64_t skeys[];
  __shared__ uint32_t sline[256];
  uint64_t *src = skeys, *dst = skeys + static_cast<int64_t>(runs) * r;
  const int tid = threadIdx.x;
  for (int i = tid; i < runs * r; i += blockDim.x) src[i] = cand[i];
  const int64_t words = (lines + 31) >> 5;
  if (mask_out) {
    for (int64_t w = tid; w < words; w += blockDim.x) mask_out[w] = 0u;
  }
  __syncthreads();
  if (r == 0) return;
  int g = runs;
  while (g > 1) {
    const int pairs = g >> 1;
    for (int o = tid; o < pairs * r; o += blockDim.x) {
      const int p = o / r, i = o - p * r;
      const uint64_t *A = src + static_cast<int64_t>(2 * p) * r;
      dst[o] = merge_at(A, r, A + r, r, i);
    }
    if (g & 1) {
      for (int i = tid; i < r; i += blockDim.x) dst[pairs * r + i] = src[(g - 1) * r + i];
    }
    __syncthreads();
    uint64_t *t = src;
    src = dst;
    dst = t;
    g = pairs + (g & 1);
  }
  // src[0..r) holds the best r keys; each line's rank among them in ascending line order
  for (int i = tid; i < r; i += blockDim.x) sline[i] = 0xFFFFFFFFu - static_cast<uint32_t>(src[i] & 0xFFFFFFFFull);
  __syncthreads();
  for (int i = tid; i < r; i += blockDim.x) {
    const uint32_t l = sline[i];
    int pos = 0;
    for (int j = 0; j < r; ++j) pos += sline[j] < l ? 1 : 0;
    idx_out[pos] = static_cast<int32_t>(l);
    if (mask_out) atomicOr(mask_out + (l >> 5), 1u << (l & 31));
  }
}

}  // namespace

size_t foid_scratch_bytes(int64_t lines, int r) {
  const int chunk = foid_chunk(lines, r);
  const int64_t chunks = (lines + chunk - 1) / chunk;
  return static_cast<size_t>(chunks * (r > 0 ? r : 1)) * sizeof(uint64_t);
}

cudaError_t launch_foid(const uint16_t *T, int64_t rows, int64_t cols, int axis, int r,
                        int32_t *idx_out, uint32_t *mask_out, void *scratch, cudaStream_t s) {
  const int64_t lines = axis == 0 ? rows : cols;
  if (r < 0 || r > 256) return cudaErrorInvalidValue;
  const int chunk = foid_chunk(lines, r);
  const int64_t chunks = (lines + chunk - 1) / chunk;
  if (chunks * r > kFoidMergeMaxKeys) return cudaErrorInvalidValue;
  uint64_t *cand = static_cast<uint64_t *>(scratch);
  if (r > 0) {
    const int threads = chunk < kFoidThreads ? chunk : kFoidThreads;
    if (axis == 0)
      foid_local_kernel<0><<<static_cast<unsigned>(chunks), threads, 0, s>>>(T, rows, cols, r, chunk, cand);
    else
      foid_local_kernel<1><<<static_cast<unsigned>(chunks), threads, 0, s>>>(T, rows, cols, r, chunk, cand);
  }
  const int runs = r > 0 ? static_cast<int>(chunks) : 0;
  const size_t smem = static_cast<size_t>(runs > 0 ? runs * r + (runs + 1) / 2 * r : 1) * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(foid_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kFoidMergeSmemKeys * static_cast<int>(sizeof(uint64_t)));
  if (e != cudaSuccess) return e;
  foid_merge_kernel<<<1, 1024, smem, s>>>(cand, runs, r, lines, idx_out, mask_out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// FOID for callers that cannot hand the library any scratch memory.
//
// Some callers only own their inputs and outputs: a plug-in or callback running inside another
// runtime that manages all device memory itself, or a code path that must not call cudaMalloc
// (it can synchronise the device and fail at run time).  For them the candidate keys of stage 1
// live in the fixed array below instead of a workspace.  It holds kFoidStaticKeys = 8192 keys
// (64 KB), the same ceiling the merge stage already has, on every GPU that loads the library,
// for the life of the process.  Stage 1 writes every slot that stage 2 reads, so nothing in it
// has to start at zero; it keeps whatever the last call wrote.  All calls share it: two calls
// whose kernels overlap on the GPU (e.g. on two streams) race on it.
// ---------------------------------------------------------------------------------------------
constexpr int kFoidStaticKeys = kFoidMergeMaxKeys;
static __device__ __align__(256) uint64_t g_foid_static_keys[kFoidStaticKeys];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_keys_mutex;
void *g_static_keys_addr[kMaxDevices] = {};   // device address of the array, per device

// The array's name is only a host-side stand-in; its device address comes from the runtime,
// looked up once per device with that device current.
cudaError_t static_keys_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_keys_mutex);
  if (!g_static_keys_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_foid_static_keys);
    if (e != cudaSuccess) return e;
    g_static_keys_addr[dev] = p;
  }
  *out = g_static_keys_addr[dev];
  return cudaSuccess;
}
}  // namespace

int64_t foid_static_capacity() { return kFoidStaticKeys; }

cudaError_t launch_foid_noalloc(const uint16_t *T, int64_t rows, int64_t cols, int axis, int r,
                                int32_t *idx_out, uint32_t *mask_out, cudaStream_t s) {
  void *keys = nullptr;
  cudaError_t e = static_keys_address(&keys);
  if (e != cudaSuccess) return e;
  return launch_foid(T, rows, cols, axis, r, idx_out, mask_out, keys, s);
}

}  // namespace adahop
