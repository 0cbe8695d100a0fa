// K3 / K5 / K6: persistent tcgen05 GEMM for sm_103a.
//
// AdaHOP appendix implementation notes, "Fused MXFP4+BF16 GEMM": the MXFP4 residual product and
// the BF16 outlier product are computed together (on CDNA4 with 64 x 64 tiles).  Here both are
// tcgen05 MMAs that accumulate into the SAME float32 tile in tensor memory:
//   kind 0 (MXFP4): for each 256-wide slice of J, four kind::mxf4.block_scale MMAs
//                   (128 x 256 x 64, E2M1 operands in shared memory, UE8M0 scale factors copied
//                   to tensor memory with tcgen05.cp), then ceil(r/64) stages of kind::f16 MMAs
//                   over the BF16 outlier slices A_o (P x r) and B_o (Q x r):
//                   C = deq(A) deq(B)^T + A_o B_o^T.
//                   Operand rows are 128 bytes (128-byte swizzle), 4 stages of 51 KB (a variant
//                   with 64-byte rows and 8 stages of 26 KB measured 11% slower).
//   kind 1 (BF16):  kind::f16 MMAs (128 x 256 x 16) over bf16 operands stored J-contiguous
//                   ("K-major") or MN-contiguous ("MN-major"); 128-byte rows (128-byte swizzle),
//                   4 stages of 48 KB; optional split-K into float32 partials (the outlier GEMM
//                   of outer OE, which has only r rows).
//
// Warp roles (320 threads): warp 0 = TMA producer (one elected lane), warp 1 = tensor-memory
// allocator + MMA issuer (one lane), warps 2..9 = epilogue (two warps per 32-lane quadrant, each
// draining 128 of the 256 accumulator columns).  Tensor memory holds the 128 x 256 float32
// accumulator (columns 0..255) and per-stage scale factors (columns 256..351).
// The epilogue copies the accumulator to registers and releases it before storing, so the next
// tile's MMAs overlap the stores.  Every wait is bounded (common.cuh); on expiry the kernel sets
// the status word, stops issuing work, drains what it issued, frees tensor memory and returns.
#include "common.cuh"
#include "kernels.cuh"

namespace adahop {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmemBase = 256;              // scale factors live above the accumulator
constexpr uint32_t kLayoutSw64 = 4;

template <int KIND>
struct Cfg;
template <>
struct Cfg<0> {                                    // MXFP4 (+ BF16 tail)
  static constexpr int kStages = 4;
  static constexpr int kBK = 256;                  // J elements per main-loop stage
  static constexpr uint32_t kRowBytes = 128;
  static constexpr uint32_t kABytes = BM * 128;    // 16 KB
  static constexpr uint32_t kBBytes = BN * 128;    // 32 KB
  static constexpr uint32_t kSFA = kABytes + kBBytes;      // 2 atoms (128 rows x 8 blocks)
  static constexpr uint32_t kSFB = kSFA + 1024;            // 4 atoms (256 rows x 8 blocks)
  static constexpr uint32_t kStageBytes = kSFB + 2048;     // 51 KB
  static constexpr uint32_t kLayout = kLayoutSw128;
  static constexpr uint32_t kSBO = 8 * 128;                // 8-row swizzle atom
  static constexpr uint32_t kSfCols = 24;                  // TMEM columns of scale factors per stage
};
template <>
struct Cfg<1> {                                    // BF16
  static constexpr int kStages = 4;
  static constexpr int kBK = 64;
  static constexpr uint32_t kRowBytes = 128;
  static constexpr uint32_t kABytes = BM * 128;    // 16 KB
  static constexpr uint32_t kBBytes = BN * 128;    // 32 KB
  static constexpr uint32_t kSFA = 0, kSFB = 0;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kLayout = kLayoutSw128;
  static constexpr uint32_t kSBO = 8 * 128;
  static constexpr uint32_t kSfCols = 0;
};
static_assert(Cfg<0>::kStageBytes % 1024 == 0, "stage layout");
static_assert(kSfTmemBase + Cfg<0>::kStages * Cfg<0>::kSfCols <= kTmemCols, "TMEM budget");

template <int KIND>
struct SmemCtl {
  uint64_t full[Cfg<KIND>::kStages];
  uint64_t empty[Cfg<KIND>::kStages];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct TileInfo {
  int64_t m0, n0;
  int split;
  int k_begin, k_end;        // stage range of the main loop
};

__device__ __forceinline__ TileInfo tile_info(const GemmArgs &g, int64_t tile, int64_t tiles_m,
                                              int64_t tiles_n, int num_k, bool n_fastest) {
  TileInfo t;
  const int64_t mn = tiles_m * tiles_n;
  t.split = static_cast<int>(tile / mn);
  const int64_t rem = tile - static_cast<int64_t>(t.split) * mn;
  int64_t mi, ni;
  if (n_fastest) {
    mi = rem / tiles_n;
    ni = rem - mi * tiles_n;
  } else {
    ni = rem / tiles_m;
    mi = rem - ni * tiles_m;
  }
  t.m0 = mi * BM;
  t.n0 = ni * BN;
  if (g.splits > 1) {
    const int per = (num_k + g.splits - 1) / g.splits;
    t.k_begin = t.split * per;
    t.k_end = min(num_k, t.k_begin + per);
  } else {
    t.k_begin = 0;
    t.k_end = num_k;
  }
  return t;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs g) {
  using C = Cfg<KIND>;
  constexpr bool mxf4 = KIND == 0;
  extern __shared__ uint8_t smem_raw[];
  __shared__ SmemCtl<KIND> ctl;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;   // swizzle atoms need alignment
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_k = static_cast<int>((g.J + C::kBK - 1) / C::kBK);
  const int tail = mxf4 ? g.tail_stages : 0;
  const int64_t tiles_m = (g.P + BM - 1) / BM;
  const int64_t tiles_n = (g.Q + BN - 1) / BN;
  const int64_t num_tiles = tiles_m * tiles_n * (g.splits > 1 ? g.splits : 1);
  // stream the larger operand once: n fastest keeps B resident while A is read once
  const bool n_fastest = g.P >= g.Q;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&ctl.full[s]), 1);
      mbar_init(smem_u32(&ctl.empty[s]), 1);
    }
    mbar_init(smem_u32(&ctl.acc_full), 1);
    mbar_init(smem_u32(&ctl.acc_empty), kEpiWarps);
    mbar_init(smem_u32(&ctl.drain), 1);
    ctl.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int *abort_flag = &ctl.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&maps.a);
      prefetch_tensormap(&maps.b);
      if (tail) {
        prefetch_tensormap(&maps.ao);
        prefetch_tensormap(&maps.bo);
      }
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int64_t atoms_per_rowblk = g.J >> 7;          // 4-block scale atoms along J
      const int64_t nblocks = (g.Q + 127) >> 7;
      for (int64_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const TileInfo t = tile_info(g, tile, tiles_m, tiles_n, num_k, n_fastest);
        const int nsteps = (t.k_end - t.k_begin) + tail;
        for (int step = 0; step < nsteps; ++step) {
          if (!mbar_wait(smem_u32(&ctl.empty[stage]), phase ^ 1u, abort_flag, 32)) {
            ok = false;
            break;
          }
          const uint32_t sA = smem_base + stage * C::kStageBytes;
          const uint32_t sB = sA + C::kABytes;
          const uint32_t full = smem_u32(&ctl.full[stage]);
          const int ks = t.k_begin + step;
          if (step < t.k_end - t.k_begin) {
            if (mxf4) {
              // 128 bytes of codes per row; two 4-block scale atoms per 128 rows (one when the
              // last slice of a J that is an odd multiple of 128 is half full)
              const bool half = (ks == num_k - 1) && ((g.J & 255) != 0);
              const uint32_t sf_chunk = half ? 512u : 1024u;
              mbar_arrive_expect_tx(full, C::kABytes + C::kBBytes + 3 * sf_chunk);
              tma_load_2d(sA, &maps.a, full, ks * 128, static_cast<int32_t>(t.m0));
              tma_load_2d(sB, &maps.b, full, ks * 128, static_cast<int32_t>(t.n0));
              const int64_t mb = t.m0 >> 7;
              const int64_t nb0 = t.n0 >> 7;
              const int64_t nb1 = (nb0 + 1 < nblocks) ? nb0 + 1 : nb0;   // ragged Q: reuse finite scales
              bulk_load(sA + C::kSFA, g.sfa + (mb * atoms_per_rowblk + 2 * ks) * 512, sf_chunk, full);
              bulk_load(sA + C::kSFB, g.sfb + (nb0 * atoms_per_rowblk + 2 * ks) * 512, sf_chunk, full);
              bulk_load(sA + C::kSFB + 1024, g.sfb + (nb1 * atoms_per_rowblk + 2 * ks) * 512, sf_chunk, full);
            } else {
              mbar_arrive_expect_tx(full, C::kABytes + C::kBBytes);
              const int32_t k0 = ks * 64;
              if (g.a_mn_major) {
                tma_load_2d(sA, &maps.a, full, static_cast<int32_t>(t.m0), k0);
                tma_load_2d(sA + 8192, &maps.a, full, static_cast<int32_t>(t.m0 + 64), k0);
              } else {
                tma_load_2d(sA, &maps.a, full, k0, static_cast<int32_t>(t.m0));
              }
              if (g.b_mn_major) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  tma_load_2d(sB + c * 8192, &maps.b, full, static_cast<int32_t>(t.n0 + 64 * c), k0);
              } else {
                tma_load_2d(sB, &maps.b, full, k0, static_cast<int32_t>(t.n0));
              }
            }
          } else {
            // BF16 outlier tail (kind 0): 64 of the r outlier columns (128 bytes) per stage
            const int32_t r0 = (step - (t.k_end - t.k_begin)) * 64;
            mbar_arrive_expect_tx(full, C::kABytes + C::kBBytes);
            tma_load_2d(sA, &maps.ao, full, r0, static_cast<int32_t>(t.m0));
            tma_load_2d(sB, &maps.bo, full, r0, static_cast<int32_t>(t.n0));
          }
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        report_status(g.status, kStatusTimeout);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint32_t idesc_bf16 =
          make_idesc_bf16(BM, BN, !mxf4 && g.a_mn_major != 0, !mxf4 && g.b_mn_major != 0);
      for (int64_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const TileInfo t = tile_info(g, tile, tiles_m, tiles_n, num_k, n_fastest);
        const int nmain = t.k_end - t.k_begin;
        const int nsteps = nmain + tail;
        if (!mbar_wait(smem_u32(&ctl.acc_empty), acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t accumulate = 0;
        for (int step = 0; step < nsteps; ++step) {
          if (!mbar_wait(smem_u32(&ctl.full[stage]), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_base + stage * C::kStageBytes;
          const uint32_t sB = sA + C::kABytes;
          if (mxf4 && step < nmain) {
            const uint32_t sfa_t = tmem + kSfTmemBase + stage * C::kSfCols;
            const uint32_t sfb_t = sfa_t + 8;
            const int ks = t.k_begin + step;
            const bool half = (ks == num_k - 1) && ((g.J & 255) != 0);
            const int katoms = half ? 1 : 2;
            for (int ka = 0; ka < katoms; ++ka) {
              // SF-A atom ka -> columns sfa + 4 ka; SF-B rows 0..127 -> sfb + 8 ka, 128..255 -> +4
              tmem_cp_32x128b_x4(sfa_t + 4 * ka, make_smem_desc(sA + C::kSFA + 512 * ka, 0, 128, kLayoutNone));
              tmem_cp_32x128b_x4(sfb_t + 8 * ka, make_smem_desc(sA + C::kSFB + 512 * ka, 0, 128, kLayoutNone));
              tmem_cp_32x128b_x4(sfb_t + 8 * ka + 4,
                                 make_smem_desc(sA + C::kSFB + 1024 + 512 * ka, 0, 128, kLayoutNone));
            }
            const int kk_end = half ? 2 : 4;
            for (int kk = 0; kk < kk_end; ++kk) {
              const uint64_t adesc = make_smem_desc(sA + 32 * kk, 16, C::kSBO, C::kLayout);
              const uint64_t bdesc = make_smem_desc(sB + 32 * kk, 16, C::kSBO, C::kLayout);
              const uint32_t sf_id = static_cast<uint32_t>(kk & 1) * 2u;
              mma_mxf4(tmem, adesc, bdesc, make_idesc_mxf4(BM, BN, sf_id, sf_id), sfa_t + 4 * (kk >> 1),
                       sfb_t + 8 * (kk >> 1), accumulate);
              accumulate = 1;
            }
          } else if (mxf4) {
            // BF16 outlier tail: four K=16 MMAs over 128-byte rows
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = make_smem_desc(sA + 32 * kk, 16, C::kSBO, C::kLayout);
              const uint64_t bdesc = make_smem_desc(sB + 32 * kk, 16, C::kSBO, C::kLayout);
              mma_bf16(tmem, adesc, bdesc, idesc_bf16, accumulate);
              accumulate = 1;
            }
          } else {
            // BF16 main loop: four K=16 MMAs over 128-byte rows (K-major) or 16-row groups (MN-major)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = g.a_mn_major ? make_smem_desc(sA + 2048 * kk, 8192, 1024, kLayoutSw128)
                                                  : make_smem_desc(sA + 32 * kk, 16, 1024, kLayoutSw128);
              const uint64_t bdesc = g.b_mn_major ? make_smem_desc(sB + 2048 * kk, 8192, 1024, kLayoutSw128)
                                                  : make_smem_desc(sB + 32 * kk, 16, 1024, kLayoutSw128);
              mma_bf16(tmem, adesc, bdesc, idesc_bf16, accumulate);
              accumulate = 1;
            }
          }
          tc_commit(smem_u32(&ctl.empty[stage]));      // frees the smem stage when MMAs finish
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&ctl.acc_full));            // accumulator ready for the epilogue
        acc_phase ^= 1u;
      }
      if (!ok) {
        *abort_flag = 1;
        report_status(g.status, kStatusTimeout);
      }
      // drain: wait (bounded) until every MMA / copy this thread issued has completed
      tc_commit(smem_u32(&ctl.drain));
      if (!mbar_wait(smem_u32(&ctl.drain), 0, nullptr)) report_status(g.status, kStatusTimeout);
    }
  } else {
    // ------------------------------------------------------------------ epilogue warps
    const int quad = warp & 3;                        // TMEM lanes 32*quad .. 32*quad+31
    const int half = (warp - 2) >> 2;                 // accumulator columns 128*half ..
    // Partial mode (split-K or not) is chosen by a non-null c_partial; with neither output the
    // tiles are computed but nothing is stored and the status word records the bad argument.
    const bool to_partial = g.c_partial != nullptr;
    const bool can_store = to_partial || g.C != nullptr;
    if (!can_store && threadIdx.x == 64) report_status(g.status, kStatusBadArg);
    uint32_t acc_phase = 0;
    for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const TileInfo t = tile_info(g, tile, tiles_m, tiles_n, num_k, n_fastest);
      bool ready = true;
      if (lane == 0) ready = mbar_wait(smem_u32(&ctl.acc_full), acc_phase, abort_flag, 128);
      ready = __shfl_sync(0xFFFFFFFFu, ready ? 1 : 0, 0) != 0;
      if (!ready) {
        if (lane == 0) {
          *abort_flag = 1;
          report_status(g.status, kStatusTimeout);
        }
        break;
      }
      tc_fence_after();
      uint32_t v[4][32];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * quad) << 16) + 128u * half;
#pragma unroll
      for (int j = 0; j < 4; ++j) tmem_ld_32x32b_x32(taddr + 32u * j, v[j]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl.acc_empty));
      acc_phase ^= 1u;

      const int64_t row = t.m0 + 32 * quad + lane;
      if (can_store && row < g.P) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t col = t.n0 + 128 * half + 32 * j;
          if (col >= g.Q) continue;
          const bool full = col + 32 <= g.Q;
          if (to_partial || g.out_dtype == 1) {
            float *dst = (to_partial ? g.c_partial + static_cast<int64_t>(t.split) * g.P * g.Q
                                     : static_cast<float *>(g.C)) +
                         row * g.Q + col;
            if (full) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                reinterpret_cast<float4 *>(dst)[q] =
                    make_float4(__uint_as_float(v[j][4 * q]), __uint_as_float(v[j][4 * q + 1]),
                                __uint_as_float(v[j][4 * q + 2]), __uint_as_float(v[j][4 * q + 3]));
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (col + e < g.Q) dst[e] = __uint_as_float(v[j][e]);
            }
          } else {
            uint16_t *dst = static_cast<uint16_t *>(g.C) + row * g.Q + col;
            if (full) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  w[e] = f32_to_bf16_bits(__uint_as_float(v[j][8 * q + 2 * e])) |
                         (f32_to_bf16_bits(__uint_as_float(v[j][8 * q + 2 * e + 1])) << 16);
                reinterpret_cast<uint4 *>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (col + e < g.Q)
                  dst[e] = static_cast<uint16_t>(f32_to_bf16_bits(__uint_as_float(v[j][e])));
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int KIND>
cudaError_t launch_kind(const GemmArgs &g, const GemmMaps &maps, int num_sms, cudaStream_t s) {
  const size_t smem = gemm_smem_bytes(KIND);
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((g.P + BM - 1) / BM) * ((g.Q + BN - 1) / BN) * (g.splits > 1 ? g.splits : 1);
  const unsigned grid = static_cast<unsigned>(tiles < num_sms ? tiles : num_sms);
  gemm_kernel<KIND><<<grid, kThreads, smem, s>>>(maps, g);
  return cudaGetLastError();
}

}  // namespace

size_t gemm_smem_bytes(int kind) {
  return kind == 0 ? Cfg<0>::kStages * Cfg<0>::kStageBytes + 1024 : Cfg<1>::kStages * Cfg<1>::kStageBytes + 1024;
}

int gemm_tail_cols_per_stage() { return 64; }

cudaError_t launch_gemm(const GemmArgs &g, const GemmMaps &maps, int num_sms, cudaStream_t s) {
  return g.kind == 0 ? launch_kind<0>(g, maps, num_sms, s) : launch_kind<1>(g, maps, num_sms, s);
}

}  // namespace adahop
