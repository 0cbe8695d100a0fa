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
// run remains, written out as the chunk's r candidates.  A merge level is one pass: output i of
// the best keys of sorted runs A and B is max(A[a], B[i - a]), where a, the number of A's keys
// among the i best, comes from a binary search (A[m] belongs to the i best iff A[m] > B[i - m - 1]).
// Stage 2, in the same launch: every stage-1 CTA writes its candidates and counts itself done on
// a counter; the CTA that finishes last (no CTA waits for another) merges all of them: each warp
// holds a run of the best keys in its registers and folds the chunks' runs into it with bitonic
// merges (shuffles, no shared-memory searches); a tree over the warps leaves the global best r in
// one warp, which sorts their lines ascending.  The last CTA then sets the counter back to zero,
// so it starts every call at zero.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace adahop {

namespace {

constexpr int kFoidThreads = 512;
constexpr int kFoidMaxChunk = 2048;         // lines per stage-1 CTA, at most
constexpr int kFoidMinChunk = 256;
constexpr int kFoidMergeMaxKeys = 8192;     // candidates written by stage 1, at most

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

template <int KPL>
__device__ void foid_finish(uint32_t *counter, uint64_t *sk, const uint64_t *cand, int runs, int r, int64_t lines,
                            int32_t *idx_out, uint32_t *mask_out);

// Stage 1 for column probes (strided loads): each warp scores 32 columns at a time and sorts them
// in registers, then merge levels in shared memory keep the best r of each merged pair until one
// run remains, written out as the chunk's r candidates; the last CTA to finish merges all chunks.
template <int KPL>
__global__ void __launch_bounds__(kFoidThreads) foid_local_cols_kernel(const uint16_t *__restrict__ T,
                                                                       int64_t rows, int64_t cols, int r,
                                                                       int chunk, uint64_t *cand, uint32_t *counter,
                                                                       int32_t *idx_out, uint32_t *mask_out) {
  __shared__ uint64_t keys[2][kFoidMaxChunk];
  const int64_t lines = cols;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * chunk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  for (int r0 = 32 * warp; r0 < chunk; r0 += 32 * nwarps) {
    const int64_t line = base + r0 + lane;
    const uint64_t key = line < lines ? foid_key<1>(T, cols, line) : 0ull;
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
  __syncthreads();                             // keys[] is reused by the merge below
  foid_finish<KPL>(counter, &keys[0][0], cand, static_cast<int>(gridDim.x), r, lines, idx_out, mask_out);
}

// ---------------------------------------------------------------------------------------------
// Warp-held runs.  A run of R = 32 KPL keys sits in one warp, KPL registers per lane,
// element e = 32 s + lane in register s, sorted descending.  Merging keeps the R largest of two
// runs: with B reversed, max(A[e], B[R - 1 - e]) is a bitonic sequence holding exactly the R
// largest keys of both (the first half-cleaner of a bitonic merge), and half-cleaners with
// strides R/2, ..., 1 sort it -- strides of 32 and more between a lane's registers, smaller ones
// across lanes by shuffles.  No shared-memory searches, no bank conflicts.
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ uint64_t kmax(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t kmin(uint64_t a, uint64_t b) { return a < b ? a : b; }

template <int KPL>
__device__ __forceinline__ void run_load(uint64_t (&k)[KPL], const uint64_t *src, int len, int lane) {
#pragma unroll
  for (int s = 0; s < KPL; ++s) {
    const int e = 32 * s + lane;
    k[s] = e < len ? src[e] : 0ull;           // 0 sorts below every real key
  }
}

template <int KPL>
__device__ __forceinline__ void run_merge(uint64_t (&a)[KPL], const uint64_t (&b)[KPL], int lane) {
#pragma unroll
  for (int s = 0; s < KPL; ++s) a[s] = kmax(a[s], __shfl_xor_sync(0xFFFFFFFFu, b[KPL - 1 - s], 31));
#pragma unroll
  for (int ks = KPL / 2; ks >= 1; ks >>= 1) {
#pragma unroll
    for (int s = 0; s < KPL; ++s) {
      if ((s & ks) == 0) {
        const uint64_t x = a[s], y = a[s | ks];
        a[s] = kmax(x, y);
        a[s | ks] = kmin(x, y);
      }
    }
  }
#pragma unroll
  for (int j = 16; j >= 1; j >>= 1) {
#pragma unroll
    for (int s = 0; s < KPL; ++s) {
      const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, a[s], j);
      a[s] = (lane & j) == 0 ? kmax(a[s], o) : kmin(a[s], o);
    }
  }
}

// Sorts the warp's R = 32 KPL values ascending (full bitonic network over registers and lanes).
template <int KPL>
__device__ __forceinline__ void warp_sort_asc(uint32_t (&v)[KPL], int lane) {
#pragma unroll
  for (int size = 2; size <= 32 * KPL; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32) {
        const int ks = stride >> 5;
#pragma unroll
        for (int s = 0; s < KPL; ++s) {
          if ((s & ks) == 0) {
            const bool up = ((32 * s + lane) & size) == 0;
            const uint32_t x = v[s], y = v[s | ks];
            v[s] = up ? min(x, y) : max(x, y);
            v[s | ks] = up ? max(x, y) : min(x, y);
          }
        }
      } else {
#pragma unroll
        for (int s = 0; s < KPL; ++s) {
          const bool up = ((32 * s + lane) & size) == 0;
          const uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, v[s], stride);
          v[s] = (((lane & stride) == 0) == up) ? min(v[s], o) : max(v[s], o);
        }
      }
    }
  }
}

// Stage 1 for row probes: each warp scores 32 rows at a time, sorts them across its lanes and
// folds them into the run of the R largest keys it holds; a tree over the warps through shared
// memory leaves the chunk's R largest in warp 0, whose first r go to `cand`.  (Column probes use
// foid_local_kernel<1>, whose strided probe loads leave no registers for the held runs.)
template <int KPL>
__global__ void __launch_bounds__(kFoidThreads, 1) foid_local_rows_kernel(const uint16_t *__restrict__ T,
                                                                       int64_t rows, int64_t cols, int r,
                                                                       int chunk, uint64_t *cand, uint32_t *counter,
                                                                       int32_t *idx_out, uint32_t *mask_out) {
  __shared__ uint64_t sk[kFoidThreads / 32][32 * KPL];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * chunk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  uint64_t top[KPL];
#pragma unroll
  for (int s = 0; s < KPL; ++s) top[s] = 0ull;
  for (int r0 = 32 * warp; r0 < chunk; r0 += 32 * nwarps) {
    const int64_t line = base + r0 + lane;
    uint64_t b[KPL];
    b[0] = warp_sort_desc(line < rows ? foid_key<0>(T, cols, line) : 0ull);
#pragma unroll
    for (int s = 1; s < KPL; ++s) b[s] = 0ull;
    run_merge<KPL>(top, b, lane);
  }
#pragma unroll
  for (int s = 0; s < KPL; ++s) sk[warp][32 * s + lane] = top[s];
  __syncthreads();
  for (int half = nwarps / 2; half >= 1; half >>= 1) {
    if (warp < half) {
      uint64_t b[KPL];
      run_load<KPL>(b, sk[warp + half], 32 * KPL, lane);
      run_merge<KPL>(top, b, lane);
#pragma unroll
      for (int s = 0; s < KPL; ++s) sk[warp][32 * s + lane] = top[s];
    }
    __syncthreads();
  }
  if (warp == 0) {
#pragma unroll
    for (int s = 0; s < KPL; ++s) {
      const int e = 32 * s + lane;
      if (e < r) cand[static_cast<int64_t>(blockIdx.x) * r + e] = top[s];
    }
  }
  __syncthreads();                             // sk[] is reused by the merge below
  foid_finish<KPL>(counter, &sk[0][0], cand, static_cast<int>(gridDim.x), r, rows, idx_out, mask_out);
}

// Stage 2: runs x r candidates (each run sorted descending, r keys) at `cand`, merged by the
// calling CTA (nwarps = blockDim / 32, a power of two; sk holds nwarps x 32 KPL keys).  Every warp
// folds its share of the runs into one run of the R largest, a tree over the warps through shared
// memory leaves the R largest in warp 0, whose first r are the selection; warp 0 then sorts their
// lines ascending, writes them and sets their bits in the line bitmap (cleared first by all
// threads).  The candidates are read from L2 (written by other CTAs of the same launch).
template <int KPL>
__device__ void foid_merge_cta(uint64_t *sk_flat, const uint64_t *cand, int runs, int r, int64_t lines,
                               int32_t *idx_out, uint32_t *mask_out) {
  uint64_t (*sk)[32 * KPL] = reinterpret_cast<uint64_t (*)[32 * KPL]>(sk_flat);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int64_t words = (lines + 31) >> 5;
  if (mask_out) {
    for (int64_t w = tid; w < words; w += blockDim.x) mask_out[w] = 0u;
  }
  if (r == 0) return;
  uint64_t top[KPL];
#pragma unroll
  for (int s = 0; s < KPL; ++s) top[s] = 0ull;
  // kFly runs' loads in flight per warp, then their merges: one round of L2 reads covers all 128
  // runs of a 32768-line probe (eight keys per lane at r = 256 would spill, so four there)
  constexpr int kFly = KPL >= 8 ? 4 : 8;
  for (int run0 = warp; run0 < runs; run0 += kFly * nwarps) {
    uint64_t b[kFly][KPL];
#pragma unroll
    for (int u = 0; u < kFly; ++u) {
      const int run = run0 + u * nwarps;
#pragma unroll
      for (int s = 0; s < KPL; ++s) {
        const int e = 32 * s + lane;
        b[u][s] = (run < runs && e < r) ? __ldcg(cand + static_cast<int64_t>(run) * r + e) : 0ull;
      }
    }
#pragma unroll
    for (int u = 0; u < kFly; ++u) run_merge<KPL>(top, b[u], lane);
  }
#pragma unroll
  for (int s = 0; s < KPL; ++s) sk[warp][32 * s + lane] = top[s];
  __syncthreads();                            // also orders the bitmap clearing before the bits below
  for (int half = nwarps / 2; half >= 1; half >>= 1) {
    if (warp < half) {
      uint64_t b[KPL];
      run_load<KPL>(b, sk[warp + half], 32 * KPL, lane);
      run_merge<KPL>(top, b, lane);
#pragma unroll
      for (int s = 0; s < KPL; ++s) sk[warp][32 * s + lane] = top[s];
    }
    __syncthreads();
  }
  if (warp == 0) {
    uint32_t ln[KPL];
#pragma unroll
    for (int s = 0; s < KPL; ++s) {
      const int e = 32 * s + lane;
      ln[s] = e < r ? 0xFFFFFFFFu - static_cast<uint32_t>(top[s] & 0xFFFFFFFFull) : 0xFFFFFFFFu;
    }
    warp_sort_asc<KPL>(ln, lane);
#pragma unroll
    for (int s = 0; s < KPL; ++s) {
      const int e = 32 * s + lane;
      if (e < r) {
        idx_out[e] = static_cast<int32_t>(ln[s]);
        if (mask_out && ln[s] < lines) atomicOr(mask_out + (ln[s] >> 5), 1u << (ln[s] & 31));
      }
    }
  }
}

// End of every stage-1 CTA: publish the candidates, count this CTA done; the CTA whose count
// completes the grid merges everything and resets the counter.  No CTA waits for another.
template <int KPL>
__device__ void foid_finish(uint32_t *counter, uint64_t *sk, const uint64_t *cand, int runs, int r, int64_t lines,
                            int32_t *idx_out, uint32_t *mask_out) {
  __shared__ int is_last;
  __threadfence();                           // this thread's candidates are visible before the count
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(counter, 1u) == gridDim.x - 1u;
  __syncthreads();
  if (!is_last) return;
  __threadfence();                           // the other CTAs' candidates are read after their counts
  foid_merge_cta<KPL>(sk, cand, runs, r, lines, idx_out, mask_out);
  if (threadIdx.x == 0) *counter = 0u;       // every call starts at zero
}

// r = 0: only the line bitmap is written (cleared).
__global__ void foid_clear_kernel(int64_t lines, uint32_t *mask_out) {
  const int64_t words = (lines + 31) >> 5;
  if (mask_out)
    for (int64_t w = threadIdx.x; w < words; w += blockDim.x) mask_out[w] = 0u;
}

}  // namespace

size_t foid_scratch_bytes(int64_t lines, int r) {
  const int chunk = foid_chunk(lines, r);
  const int64_t chunks = (lines + chunk - 1) / chunk;
  return static_cast<size_t>(chunks * (r > 0 ? r : 1)) * sizeof(uint64_t);
}

cudaError_t launch_foid(const uint16_t *T, int64_t rows, int64_t cols, int axis, int r,
                        int32_t *idx_out, uint32_t *mask_out, void *scratch, uint32_t *counter, cudaStream_t s) {
  const int64_t lines = axis == 0 ? rows : cols;
  if (r < 0 || r > 256) return cudaErrorInvalidValue;
  if (r == 0) {
    foid_clear_kernel<<<1, 256, 0, s>>>(lines, mask_out);
    return cudaGetLastError();
  }
  const int chunk = foid_chunk(lines, r);
  const int64_t chunks = (lines + chunk - 1) / chunk;
  if (chunks * r > kFoidMergeMaxKeys) return cudaErrorInvalidValue;
  uint64_t *cand = static_cast<uint64_t *>(scratch);
  const int threads = chunk < kFoidThreads ? chunk : kFoidThreads;
  const unsigned grid = static_cast<unsigned>(chunks);
#define ADAHOP_FOID_LAUNCH(KPL)                                                                             \
  do {                                                                                                      \
    if (axis == 1)                                                                                          \
      foid_local_cols_kernel<KPL><<<grid, threads, 0, s>>>(T, rows, cols, r, chunk, cand, counter, idx_out, \
                                                           mask_out);                                       \
    else                                                                                                    \
      foid_local_rows_kernel<KPL><<<grid, threads, 0, s>>>(T, rows, cols, r, chunk, cand, counter, idx_out, \
                                                           mask_out);                                       \
  } while (0)
  if (r <= 32)
    ADAHOP_FOID_LAUNCH(1);
  else if (r <= 64)
    ADAHOP_FOID_LAUNCH(2);
  else if (r <= 128)
    ADAHOP_FOID_LAUNCH(4);
  else
    ADAHOP_FOID_LAUNCH(8);
#undef ADAHOP_FOID_LAUNCH
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// FOID for callers that cannot hand the library any scratch memory.
//
// Some callers only own their inputs and outputs: a plug-in or callback running inside another
// runtime that manages all device memory itself, or a code path that must not call cudaMalloc
// (it can synchronise the device and fail at run time).  For them FOID's scratch lives in the
// fixed array below instead of a workspace: a 256-byte header holding the completion counter of
// the single launch, then kFoidStaticKeys = 8192 candidate keys (the ceiling the merge already
// has); 64.25 KB on every GPU that loads the library, for the life of the process.  Device
// globals start at zero and every call leaves the counter at zero again; stage 1 writes every
// candidate slot the merge reads, so nothing else has to start at zero, and the array keeps
// whatever the last call wrote.  All calls share it: two calls whose kernels overlap on the GPU
// (e.g. on two streams) race on it.
// ---------------------------------------------------------------------------------------------
constexpr int kFoidStaticKeys = kFoidMergeMaxKeys;
constexpr int kFoidStaticHeader = 32;            // uint64 words (256 bytes) before the keys
static __device__ __align__(256) uint64_t g_foid_static_keys[kFoidStaticHeader + kFoidStaticKeys];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_keys_mutex;
// Per device: the array's device address and the id of the context it was looked up in.  A
// device reset (cudaDeviceReset) destroys the context and with it the module holding the array;
// the next context gets a new id, so the address is looked up again rather than reused.
struct StaticKeys {
  void *addr = nullptr;
  unsigned long long ctx_id = 0;
};
StaticKeys g_static_keys[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Unique id of the calling thread's current context (driver entry points fetched once).
cudaError_t current_context_id(unsigned long long *id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  if (get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

// The array's name is only a host-side stand-in; its device address comes from the runtime,
// looked up with the device current, once per device and context.
cudaError_t static_keys_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long ctx_id = 0;
  // With no context current yet (nothing has touched this device on this thread), the lookup
  // below creates the device's primary context; its id is read after it.
  const bool have_ctx = current_context_id(&ctx_id) == cudaSuccess;
  std::lock_guard<std::mutex> lock(g_static_keys_mutex);
  StaticKeys &k = g_static_keys[dev];
  if (have_ctx && k.addr && k.ctx_id == ctx_id) {
    *out = k.addr;
    return cudaSuccess;
  }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_foid_static_keys);
  if (e != cudaSuccess) return e;
  if (!have_ctx) {
    e = current_context_id(&ctx_id);
    if (e != cudaSuccess) return e;
  }
  k.addr = p;
  k.ctx_id = ctx_id;
  *out = p;
  return cudaSuccess;
}
}  // namespace

int64_t foid_static_capacity() { return kFoidStaticKeys; }

cudaError_t launch_foid_noalloc(const uint16_t *T, int64_t rows, int64_t cols, int axis, int r,
                                int32_t *idx_out, uint32_t *mask_out, cudaStream_t s) {
  void *base = nullptr;
  cudaError_t e = static_keys_address(&base);
  if (e != cudaSuccess) return e;
  uint64_t *words = static_cast<uint64_t *>(base);
  return launch_foid(T, rows, cols, axis, r, idx_out, mask_out, words + kFoidStaticHeader,
                     reinterpret_cast<uint32_t *>(words), s);
}

}  // namespace adahop
