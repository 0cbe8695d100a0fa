// K8: peak probes, the roofline denominators measured on the part itself.
//
// mma_rate_kernel: one CTA per SM, one elected lane of one warp issuing tcgen05.mma instructions
// back to back (128 x 256 tiles, cta_group::1) on operands that stay resident in shared memory,
// accumulating into one tensor-memory tile, so the only limit is the tensor pipe (and, with the
// per-slice scale-factor copies switched on, the copies the fused MXFP4 GEMM issues per 256-wide
// J slice).  Each CTA reports the clock64 cycles of its loop and its %globaltimer start and end;
// the host turns them into FLOP per clock per SM (independent of the clock the part ran at) and
// FLOP/s over the whole launch.  Operand values are a fixed finite pattern and every scale byte
// is 127 (2^0): the results are discarded.
//
// copy_probe_kernel: a streaming 16-byte copy (the HBM read + write denominator);
// fill_probe_kernel: a streaming 16-byte fill (the write-only denominator).
#include "common.cuh"
#include "kernels.cuh"

namespace adahop {

namespace {

constexpr int kProbeThreads = 128;
constexpr uint32_t kProbeA = 0;                          // 128 rows x 128 bytes (SW128)
constexpr uint32_t kProbeB = 16384;                      // 256 rows x 128 bytes (SW128)
constexpr uint32_t kProbeSF = 49152;                     // six 512-byte scale atoms
constexpr uint32_t kProbeBytes = kProbeSF + 6 * 512;
// More than half of an SM's shared memory, so that no two probe CTAs share an SM (each also
// allocates all 512 tensor-memory columns).
constexpr size_t kProbeSmem = 160 * 1024;
constexpr uint32_t kProbeSfBase = 256;                   // scale slots above the accumulator
constexpr uint32_t kProbeSfSlotCols = 24;                // A: 2 atoms x 4 cols, B: 4 atoms x 4 cols
constexpr int kProbeSfSlots = 6;
static_assert(kProbeSfBase + kProbeSfSlots * kProbeSfSlotCols <= 512, "TMEM budget");

// Block-scaled MMAs of the two 4-bit kinds (E2M1 operands, UE8M0 scales); M x N x 64.
__device__ __forceinline__ void mma_mxf4nvf4_2x(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
__device__ __forceinline__ void mma_mxf4nvf4_4x(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// KIND: 0 = kind::f16 (bf16 x bf16, K = 16); 1 = kind::mxf4 scale_vec::2X; 2 = kind::mxf4nvf4
// scale_vec::2X; 3 = kind::mxf4nvf4 scale_vec::4X (both with UE8M0 scales; K = 64).  N: 256 or 128
// (with N = 128 each group's MMAs take half the time, so the issuing lane has half as long to
// issue the same group; SF_COPIES then copies one B atom per 128 B rows, as a 128-wide tile needs).
// out[3 * cta + 0..2] = loop cycles, start ns, end ns.
template <int KIND, bool SF_COPIES, int N>
__global__ void __launch_bounds__(kProbeThreads, 1)
    mma_rate_kernel(int64_t iters, uint64_t *out, uint32_t *status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ uint32_t tmem_slot;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // bf16 0x3C1A (~0.0094) / E2M1 nibbles 0xA, 0x1, 0xC, 0x3 (-1, 0.5, -2, 1.5); scales 2^0
  for (uint32_t off = 16u * threadIdx.x; off < kProbeBytes; off += 16u * kProbeThreads) {
    const uint32_t w = off >= kProbeSF ? 0x7F7F7F7Fu : 0x3C1A3C1Au;
    st_shared_v4(base + off, w, w, w, w);
  }
  fence_proxy_async_smem();                      // generic writes before the tensor core reads them
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done_bar), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // The whole warp runs the loop; one elected lane issues (as in the GEMM kernels).
    constexpr bool scaled = KIND != 0;
    if (scaled && elect_one()) {
      for (int slot = 0; slot < kProbeSfSlots; ++slot) {
        const uint32_t sf = tmem + kProbeSfBase + slot * kProbeSfSlotCols;
#pragma unroll
        for (int a = 0; a < 6; ++a)
          tmem_cp_32x128b_x4(sf + 4 * a, make_smem_desc(base + kProbeSF + 512 * a, 0, 128, kLayoutNone));
      }
    }
    __syncwarp();
    const uint64_t c0 = clock64();
    const uint64_t g0 = global_timer_ns();
    int slot = 0;
    for (int64_t it = 0; it < iters; ++it) {
      if (elect_one()) {
        const uint32_t sfa = tmem + kProbeSfBase + slot * kProbeSfSlotCols;
        const uint32_t sfb = sfa + 8;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if (scaled && SF_COPIES && (kk & 1) == 0) {
            const int ka = kk >> 1;
            tmem_cp_32x128b_x4(sfa + 4 * ka, make_smem_desc(base + kProbeSF + 512 * ka, 0, 128, kLayoutNone));
            tmem_cp_32x128b_x4(sfb + 8 * ka, make_smem_desc(base + kProbeSF + 1024 + 512 * ka, 0, 128, kLayoutNone));
            if constexpr (N == 256)
              tmem_cp_32x128b_x4(sfb + 8 * ka + 4,
                                 make_smem_desc(base + kProbeSF + 2048 + 512 * ka, 0, 128, kLayoutNone));
          }
          const uint64_t adesc = make_smem_desc(base + kProbeA + 32 * kk, 16, 1024, kLayoutSw128);
          const uint64_t bdesc = make_smem_desc(base + kProbeB + 32 * kk, 16, 1024, kLayoutSw128);
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          const uint32_t sa = sfa + 4 * (kk >> 1), sb = sfb + 8 * (kk >> 1);
          if constexpr (KIND == 0) {
            mma_bf16(tmem, adesc, bdesc, make_idesc_bf16(128, N, false, false), acc);
          } else if constexpr (KIND == 1) {
            mma_mxf4(tmem, adesc, bdesc, (kk & 1) ? make_idesc_mxf4(128, N, 2, 2) : make_idesc_mxf4(128, N, 0, 0),
                     sa, sb, acc);
          } else if constexpr (KIND == 2) {
            mma_mxf4nvf4_2x(tmem, adesc, bdesc,
                            (kk & 1) ? make_idesc_mxf4(128, N, 2, 2) : make_idesc_mxf4(128, N, 0, 0), sa, sb, acc);
          } else {
            mma_mxf4nvf4_4x(tmem, adesc, bdesc, make_idesc_mxf4(128, N, 0, 0), sa, sb, acc);
          }
        }
      }
      __syncwarp();
      if (++slot == kProbeSfSlots) slot = 0;
    }
    if (elect_one()) tc_commit(smem_u32(&done_bar));
    __syncwarp();
    const bool ok = mbar_wait(smem_u32(&done_bar), 0, nullptr);   // bounded: the queue drains in microseconds
    const uint64_t c1 = clock64();
    const uint64_t g1 = global_timer_ns();
    if (lane == 0) {
      if (!ok) report_status(status, kStatusTimeout);
      out[3 * blockIdx.x + 0] = c1 - c0;
      out[3 * blockIdx.x + 1] = g0;
      out[3 * blockIdx.x + 2] = g1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// Streaming copy: each thread moves four 16-byte words per iteration (loads first, then stores).
__global__ void __launch_bounds__(256) copy_probe_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                         int64_t n16) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride), c = __ldcs(src + i + 2 * stride),
                d = __ldcs(src + i + 3 * stride);
    __stcs(dst + i, a);
    __stcs(dst + i + stride, b);
    __stcs(dst + i + 2 * stride, c);
    __stcs(dst + i + 3 * stride, d);
  }
  for (; i < n16; i += stride) __stcs(dst + i, __ldcs(src + i));
}

// Streaming fill (write-only): the denominator of a kernel whose DRAM traffic is mostly stores.
__global__ void __launch_bounds__(256) fill_probe_kernel(uint4 *__restrict__ dst, int64_t n16) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uint32_t v = 0x3F803F80u;                     // a bf16 1.0 pair
  const uint4 w = make_uint4(v, v, v, v);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) __stcs(dst + i, w);
}

template <int KIND, bool SF_COPIES, int N>
cudaError_t launch_rate(int64_t iters, uint64_t *out, uint32_t *status, int ctas, cudaStream_t s) {
  auto *k = mma_rate_kernel<KIND, SF_COPIES, N>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kProbeSmem));
  if (e != cudaSuccess) return e;
  k<<<ctas, kProbeThreads, kProbeSmem, s>>>(iters, out, status);
  return cudaGetLastError();
}

template <int N>
cudaError_t launch_rate_n(int kind, int sf_copies, int64_t iters, uint64_t *out, uint32_t *status, int ctas,
                          cudaStream_t s) {
  switch (kind * 2 + (sf_copies ? 1 : 0)) {
    case 0: case 1: return launch_rate<0, false, N>(iters, out, status, ctas, s);
    case 2: return launch_rate<1, false, N>(iters, out, status, ctas, s);
    case 3: return launch_rate<1, true, N>(iters, out, status, ctas, s);
    case 4: return launch_rate<2, false, N>(iters, out, status, ctas, s);
    case 5: return launch_rate<2, true, N>(iters, out, status, ctas, s);
    case 6: return launch_rate<3, false, N>(iters, out, status, ctas, s);
    case 7: return launch_rate<3, true, N>(iters, out, status, ctas, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_mma_rate_probe(int kind, int sf_copies, int n, int64_t iters, uint64_t *out, uint32_t *status,
                                  int ctas, cudaStream_t s) {
  if (n == 128) return launch_rate_n<128>(kind, sf_copies, iters, out, status, ctas, s);
  if (n == 256) return launch_rate_n<256>(kind, sf_copies, iters, out, status, ctas, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_copy_probe(const void *src, void *dst, size_t bytes, int num_sms, cudaStream_t s) {
  const int64_t n16 = static_cast<int64_t>(bytes / 16);
  if (n16 == 0) return cudaSuccess;
  int64_t grid = static_cast<int64_t>(num_sms) * 8;
  const int64_t need = (n16 + 255) / 256;
  if (grid > need) grid = need;
  if (src)
    copy_probe_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(static_cast<const uint4 *>(src),
                                                                   static_cast<uint4 *>(dst), n16);
  else
    fill_probe_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(static_cast<uint4 *>(dst), n16);
  return cudaGetLastError();
}

}  // namespace adahop
