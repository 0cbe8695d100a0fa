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
// at most 8192 candidates overall), sorts their keys in shared memory (bitonic) and writes its
// best r.  Stage 2 (one CTA): reduces the sorted runs pairwise -- the element-wise maximum of a
// run and the reverse of its partner is a bitonic sequence holding exactly their best keys, which
// half-cleaner steps sort again -- then writes the best r indices in ascending order and the
// bitmap of selected lines.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace adahop {

namespace {

constexpr int kFoidThreads = 512;
constexpr int kFoidMaxChunk = 2048;         // lines per stage-1 CTA, at most
constexpr int kFoidMinChunk = 256;
constexpr int kFoidMergeMaxKeys = 8192;     // candidates written by stage 1, at most
constexpr int kFoidMergeSmemKeys = 16384;   // stage-2 shared memory (runs padded to a power of 2)

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

// In-place bitonic sort of n (power of two) keys in shared memory, descending.
__device__ void bitonic_sort_desc(uint64_t *keys, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = keys[i], b = keys[ixj];
          const bool up = (i & k) == 0;     // this run ends descending
          if (up ? (a < b) : (a > b)) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

template <int AXIS>
__global__ void __launch_bounds__(kFoidThreads) foid_local_kernel(const uint16_t *__restrict__ T,
                                                                  int64_t rows, int64_t cols, int r,
                                                                  int chunk, uint64_t *cand) {
  __shared__ uint64_t keys[kFoidMaxChunk];
  const int64_t lines = AXIS == 0 ? rows : cols;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * chunk;
  for (int local = threadIdx.x; local < chunk; local += blockDim.x) {
    const int64_t line = base + local;
    keys[local] = line < lines ? foid_key<AXIS>(T, cols, line) : 0ull;
  }
  __syncthreads();
  bitonic_sort_desc(keys, chunk);
  for (int i = threadIdx.x; i < r; i += blockDim.x) cand[static_cast<int64_t>(blockIdx.x) * r + i] = keys[i];
}

// ncand = runs * r candidates (each run sorted descending); runs are padded to rp2 in shared memory.
__global__ void __launch_bounds__(1024) foid_merge_kernel(const uint64_t *cand, int runs, int r, int rp2,
                                                          int64_t lines, int32_t *idx_out, uint32_t *mask_out) {
  extern __shared__ uint64_t skeys[];
  __shared__ uint32_t sidx[256];
  const int n = runs * rp2;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int run = i / rp2, k = i - run * rp2;
    skeys[i] = k < r ? cand[static_cast<int64_t>(run) * r + k] : 0ull;
  }
  const int64_t words = (lines + 31) >> 5;
  if (mask_out) {
    for (int64_t w = threadIdx.x; w < words; w += blockDim.x) mask_out[w] = 0u;
  }
  __syncthreads();
  if (r == 0) return;
  int g = runs;
  while (g > 1) {
    const int pairs = g >> 1;
    const int m = pairs * rp2;
    // max(run 2p, reverse(run 2p+1)) -> run p, staged through registers (at most 16 per thread)
    uint64_t tmp[kFoidMergeSmemKeys / 1024];
    int cnt = 0;
    for (int i = threadIdx.x; i < m; i += blockDim.x, ++cnt) {
      const int pr = i / rp2, k = i - pr * rp2;
      const uint64_t a = skeys[(2 * pr) * rp2 + k], b = skeys[(2 * pr + 1) * rp2 + (rp2 - 1 - k)];
      tmp[cnt] = a > b ? a : b;
    }
    uint64_t odd[kFoidMergeSmemKeys / 1024];
    int ocnt = 0;
    if (g & 1) {
      for (int k = threadIdx.x; k < rp2; k += blockDim.x, ++ocnt) odd[ocnt] = skeys[(g - 1) * rp2 + k];
    }
    __syncthreads();
    cnt = 0;
    for (int i = threadIdx.x; i < m; i += blockDim.x, ++cnt) skeys[i] = tmp[cnt];
    ocnt = 0;
    if (g & 1) {
      for (int k = threadIdx.x; k < rp2; k += blockDim.x, ++ocnt) skeys[pairs * rp2 + k] = odd[ocnt];
    }
    __syncthreads();
    // each merged run is bitonic: half-cleaner steps sort it descending
    for (int j = rp2 >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < m; i += blockDim.x) {
        if ((i & j) == 0) {
          const uint64_t a = skeys[i], b = skeys[i + j];
          if (a < b) {
            skeys[i] = b;
            skeys[i + j] = a;
          }
        }
      }
      __syncthreads();
    }
    g = pairs + (g & 1);
  }
  // the best r lines, then ascending order (pad with 0xFFFFFFFF)
  for (int i = threadIdx.x; i < rp2; i += blockDim.x)
    sidx[i] = i < r ? 0xFFFFFFFFu - static_cast<uint32_t>(skeys[i] & 0xFFFFFFFFull) : 0xFFFFFFFFu;
  __syncthreads();
  for (int k = 2; k <= rp2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < rp2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint32_t a = sidx[i], b = sidx[ixj];
          const bool up = (i & k) == 0;   // ascending run
          if (up ? (a > b) : (a < b)) {
            sidx[i] = b;
            sidx[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < r; i += blockDim.x) {
    const uint32_t l = sidx[i];
    idx_out[i] = static_cast<int32_t>(l);
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
  const int rp2 = pow2_at_least(r > 0 ? r : 1);
  uint64_t *cand = static_cast<uint64_t *>(scratch);
  if (r > 0) {
    const int threads = chunk < kFoidThreads ? chunk : kFoidThreads;
    if (axis == 0)
      foid_local_kernel<0><<<static_cast<unsigned>(chunks), threads, 0, s>>>(T, rows, cols, r, chunk, cand);
    else
      foid_local_kernel<1><<<static_cast<unsigned>(chunks), threads, 0, s>>>(T, rows, cols, r, chunk, cand);
  }
  const int runs = r > 0 ? static_cast<int>(chunks) : 0;
  const size_t smem = static_cast<size_t>(runs > 0 ? runs * rp2 : 1) * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(foid_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kFoidMergeSmemKeys * static_cast<int>(sizeof(uint64_t)));
  if (e != cudaSuccess) return e;
  foid_merge_kernel<<<1, 1024, smem, s>>>(cand, runs, r, rp2, lines, idx_out, mask_out);
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
