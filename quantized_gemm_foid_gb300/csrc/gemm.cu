// K3 / K5 / K6: persistent tcgen05 GEMMs for sm_103a.
//
// AdaHOP appendix implementation notes, "Fused MXFP4+BF16 GEMM": the MXFP4 residual product and
// the BF16 outlier product are computed together (on CDNA4 with 64 x 64 tiles).  Here both are
// tcgen05 MMAs that accumulate into the SAME float32 tile in tensor memory.
//
// kind 0 (MXFP4, K3) runs on CTA pairs (clusters of two CTAs on paired SMs, cta_group::2): a pair
// owns a 256 x 256 tile of C; each CTA holds its 128 rows of A and its 128-row half of B in
// shared memory, and one thread of the even CTA issues 256 x 256 x 64 kind::mxf4.block_scale
// MMAs that read both CTAs' operands and accumulate into both CTAs' tensor memory (each CTA keeps
// its own 128 x 256 float32 rows).  Per SM that is half the B bytes per FLOP of a single-CTA
// 128 x 256 tile.  For each 256-wide slice of J: four MXFP4 MMAs (UE8M0 scale factors copied to
// tensor memory with tcgen05.cp: each CTA supplies its own 128 rows of A scales and all 256 rows
// of B scales), then ceil(r/64) stages of kind::f16 MMAs over the BF16 outlier slices A_o (P x r)
// and B_o (Q x r): C = deq(A) deq(B)^T + A_o B_o^T.  Operand rows are 128 bytes (128-byte
// swizzle); 6 stages of 35 KB per CTA.  Every TMA load of either CTA is counted on the even CTA's
// stage barrier, the MMA commits release the stage in both CTAs, and the odd CTA's epilogue warps
// release the accumulator on the even CTA's barrier.
//
// kind 1 (BF16, K5 / K6) runs on single CTAs: kind::f16 MMAs (128 x 256 x 16) over bf16
// operands stored J-contiguous ("K-major") or MN-contiguous ("MN-major"); 128-byte rows
// (128-byte swizzle), 4 stages of 48 KB; optional split-K into float32 partials (the outlier GEMM
// of outer OE, which has only r rows).
//
// Warp roles (320 threads per CTA): warp 0 = TMA producer (one lane), warp 1 = tensor-memory
// allocator + MMA issuer (one lane; in a pair only the even CTA's issues), warps 2..9 =
// epilogue (two warps per 32-lane quadrant, each draining 128 of the 256 accumulator columns).
// Tensor memory holds the 128 x 256 float32 accumulator (columns 0..255) and per-stage scale
// factors above it.  The epilogue copies the accumulator to registers and releases it before
// storing, so the next tile's MMAs overlap the stores.  In the MXFP4 kernel the stores go through
// shared memory: each epilogue warp converts 32 rows x 32 bytes of C into a 1 KB swizzled box
// and writes it with a TMA bulk store, which turns one-row-per-lane global stores into whole
// box writes (the J = 1024 shapes are bound by this store stream).  The MXFP4 kernel is launched
// with programmatic dependent launch: barrier set-up and the tensor-memory allocation run while
// the previous kernel on the stream finishes (its 212 KB of shared memory keep it off any SM that
// still holds another GEMM's CTA), and pdl_enter() waits for that kernel before the first global
// access.  Every mbarrier wait is bounded
// (common.cuh); on expiry the kernel sets the status word, stops issuing work, drains what it
// issued, frees tensor memory and returns.
#include "common.cuh"
#include "kernels.cuh"

namespace adahop {

namespace {

constexpr int BN = 256;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmemBase = 256;              // scale factors live above the accumulator

// ------------------------------------------------------------------ kind 0: MXFP4 on CTA pairs
// STAGES: main-loop pipeline depth; EPI_BUFS: 1 KB TMA-store staging buffers per epilogue warp.
// Long inner dimensions keep six stages and one buffer; short ones (J <= 2048, a tile's main loop
// is a handful of stages) are bound by the stream of output stores, so they trade stages for
// stores in flight.
template <int STAGES, int EPI_BUFS>
struct PairCfgT {
  static constexpr int kBM = 256;                  // rows of C per pair (128 per CTA)
  static constexpr int kStages = STAGES;
  static constexpr int kBK = 256;                  // J elements per main-loop stage
  static constexpr uint32_t kABytes = 128 * 128;   // this CTA's 128 rows x 128 bytes of codes
  static constexpr uint32_t kBBytes = 128 * 128;   // this CTA's 128 of the 256 B rows
  static constexpr uint32_t kSFA = kABytes + kBBytes;      // 2 atoms: this CTA's 128 rows x 8 blocks
  static constexpr uint32_t kSFB = kSFA + 1024;            // 4 atoms: all 256 B rows x 8 blocks
  static constexpr uint32_t kStageBytes = kSFB + 2048;     // 35 KB
  static constexpr uint32_t kSfCols = 24;                  // TMEM columns of scale factors per stage
  // bytes counted on the even CTA's stage barrier: both CTAs' loads (TMA counts whole boxes)
  static constexpr uint32_t kTxMain = 2 * kStageBytes;
  static constexpr uint32_t kTxTail = 2 * (kABytes + kBBytes);
  // epilogue staging: per epilogue warp kEpiBufs buffers of 32 rows x 32 bytes (TMA store boxes)
  static constexpr int kEpiBufs = EPI_BUFS;
  static constexpr uint32_t kEpiBufBytes = 1024;
  static constexpr uint32_t kEpiOffset = kStages * kStageBytes;
  static constexpr uint32_t kSmemBytes = kEpiOffset + kEpiWarps * kEpiBufs * kEpiBufBytes;
  static_assert(kEpiOffset % 1024 == 0, "epilogue buffers need the swizzle alignment");
  static_assert(kStageBytes % 1024 == 0, "stage layout");
  static_assert(kSfTmemBase + kStages * kSfCols <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes + 1024 <= 227 * 1024, "shared memory per CTA");
};
using PairCfg = PairCfgT<6, 1>;          // J > 2048
using PairCfgShortJ = PairCfgT<4, 8>;    // J <= 2048
constexpr int64_t kShortJ = 2048;

// ------------------------------------------------------------------ kind 1: BF16 on single CTAs
struct Bf16Cfg {
  static constexpr int kBM = 128;
  static constexpr int kStages = 4;
  static constexpr int kBK = 64;
  static constexpr uint32_t kABytes = 128 * 128;   // 16 KB
  static constexpr uint32_t kBBytes = BN * 128;    // 32 KB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
};

// kind 2 (the outlier GEMM with the fused scatter-add): 128 x 128 tiles, so that a product with
// few output tiles still spreads over many clusters of few CTAs (a wave of clusters must fit the
// GPU at once; clusters of 8 fit only 15 times on a 152-SM part).
struct ScatterCfg {
  static constexpr int kBM = 128;
  static constexpr int kBN = 128;
  static constexpr int kStages = 6;
  static constexpr int kBK = 64;
  static constexpr uint32_t kABytes = 128 * 128;   // 16 KB
  static constexpr uint32_t kBBytes = kBN * 128;   // 16 KB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 128;
  static constexpr uint32_t kPartialRowBytes = kBN * 4 + 16;   // padded: conflict-free 16-byte row writes
  static_assert(kBM * kPartialRowBytes <= kStages * kStageBytes, "the partial tile must fit the stage buffers");
};

template <int STAGES>
struct SmemCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
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
                                              int64_t tiles_n, int num_k, bool n_fastest, int bm) {
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
  t.m0 = mi * bm;
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

// Stores 32 accumulator columns (col .. col+31, clipped at Q) of one row of C, or of the split's
// float32 partials.
__device__ __forceinline__ void store_row32(const GemmArgs &g, bool to_partial, int split, int64_t row,
                                            int64_t col, const uint32_t (&v)[32]) {
  const bool full = col + 32 <= g.Q;
  if (to_partial || g.out_dtype == 1) {
    float *dst = (to_partial ? g.c_partial + static_cast<int64_t>(split) * g.P * g.Q
                             : static_cast<float *>(g.C)) +
                 row * g.Q + col;
    if (full) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4 *>(dst)[q] =
            make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                        __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (col + e < g.Q) dst[e] = __uint_as_float(v[e]);
    }
  } else {
    uint16_t *dst = static_cast<uint16_t *>(g.C) + row * g.Q + col;
    if (full) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = f32_to_bf16_bits(__uint_as_float(v[8 * q + 2 * e])) |
                 (f32_to_bf16_bits(__uint_as_float(v[8 * q + 2 * e + 1])) << 16);
        reinterpret_cast<uint4 *>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (col + e < g.Q) dst[e] = static_cast<uint16_t>(f32_to_bf16_bits(__uint_as_float(v[e])));
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Work of one CTA pair of the MXFP4 kernel.  Whole tiles go round robin over the pairs; when the
// last round would leave pairs idle (sk), the tiles of the last two rounds are cut into their
// `nsteps` J stages instead, and the stages spread evenly over all pairs (stream-K).  Each pair
// walks its share of stages from the end: a tile cut between pairs is first worked on by the pairs
// that hold its first stages (contributors: they leave float32 partial tiles and count their
// stages on the tile's counter) and last by the pair that holds its final stage (the finisher: it
// waits for the count, adds the partials, stores C and clears the counter).  A pair holds at most
// one contributing part (the end of its share, done first) and one finishing part (the start of
// its share, done last), so no contributor ever waits, and the finisher's wait ends as soon as the
// other pairs have done their first stream-K part.
// ---------------------------------------------------------------------------------------------
enum : int { kItemFull = 0, kItemContrib = 1, kItemFinish = 2 };

struct WorkItem {
  int64_t tile;        // tile index (n- or m-fastest order, see tile_info)
  int kb, ke;          // J stages [kb, ke) of the tile
  int role;
};

struct WorkSched {
  int64_t dp_tiles;    // whole tiles, round robin
  int64_t np;
  int32_t sk_units;    // stream-K stages over all pairs (the host enables stream-K only below 2^31)
  int32_t nsteps;
  // first stream-K stage of pair p
  __device__ __forceinline__ int32_t lo(int64_t p) const {
    return static_cast<int32_t>(p * static_cast<int64_t>(sk_units) / np);
  }
  // the pair whose share holds stage x: the largest p with lo(p) <= x
  __device__ __forceinline__ int64_t owner(int32_t x) const {
    return (static_cast<int64_t>(x + 1) * np + sk_units - 1) / sk_units - 1;
  }
};

struct WorkIter {
  int64_t next_dp;
  int32_t u_lo, u_hi;
  int32_t t;           // stream-K tile holding stage u_hi - 1 (kept, not divided out per item)
};

__device__ __forceinline__ WorkSched make_sched(int64_t num_tiles, int nsteps, int64_t np, bool sk) {
  WorkSched s;
  s.np = np;
  s.nsteps = nsteps;
  const int64_t rounds = num_tiles / np;
  s.dp_tiles = !sk ? num_tiles : (rounds >= 1 ? (rounds - 1) * np : 0);
  s.sk_units = static_cast<int32_t>((num_tiles - s.dp_tiles) * nsteps);
  return s;
}

__device__ __forceinline__ WorkIter make_iter(const WorkSched &s, int64_t pair) {
  WorkIter it{pair, s.lo(pair), s.lo(pair + 1), 0};
  it.t = it.u_hi > it.u_lo ? (it.u_hi - 1) / s.nsteps : 0;
  return it;
}

template <bool SK>
__device__ __forceinline__ bool next_item(const WorkSched &s, WorkIter &it, WorkItem &w) {
  if (it.next_dp < s.dp_tiles) {
    w = WorkItem{it.next_dp, 0, s.nsteps, kItemFull};
    it.next_dp += s.np;
    return true;
  }
  if constexpr (!SK) return false;
  if (it.u_hi <= it.u_lo) return false;
  const int32_t base = it.t * s.nsteps;
  const int32_t lo = it.u_lo > base ? it.u_lo : base;
  w.tile = s.dp_tiles + it.t;
  w.kb = lo - base;
  w.ke = it.u_hi - base;
  w.role = (w.kb == 0 && w.ke == s.nsteps) ? kItemFull : (w.ke == s.nsteps ? kItemFinish : kItemContrib);
  it.u_hi = lo;
  --it.t;
  return true;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait for a stream-K counter to reach `target` (false if it ran out or *abort was set).
__device__ __forceinline__ bool wait_count(const uint32_t *cnt, uint32_t target, const volatile int *abort) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (ld_acquire_u32(cnt) >= target) return true;
    if ((i & 15u) == 0) {
      if (abort && *abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    __nanosleep(64);
  }
}

// Stream-K exchange: every epilogue warp of a contributing CTA writes the 32 rows x 128 columns of
// the partial tile it holds (16-byte piece c = 32 half + 8 j + q of row r at float4 c * 128 + r,
// so a warp's stores cover 512 contiguous bytes) and counts itself on its own counter; the same
// warp of the finishing CTA waits for the count, then reads the same pieces.  No barrier spans
// warps, so a warp that gives up a wait never leaves another one waiting on it.
__device__ __forceinline__ uint32_t *sk_counter(const GemmArgs &g, int64_t sk_tile, uint32_t rank, int ew) {
  return g.sk_counters + sk_tile * kSkCountersPerTile + rank * kEpiWarps + ew;
}
__device__ __forceinline__ float4 *sk_slot(const GemmArgs &g, int64_t pair, uint32_t rank) {
  return reinterpret_cast<float4 *>(g.sk_partial) + (pair * 2 + rank) * (64 * 128);
}

// =============================================================================================
// kind 0: MXFP4 (+ BF16 outlier tail), CTA pairs
// =============================================================================================
template <class C, bool SK>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxf4_pair_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ SmemCtl<C::kStages> ctl;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;   // same offset in both CTAs
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();           // 0: issues the MMAs; 1: its peer
  const uint32_t peer = rank ^ 1u;
  const int64_t pair = blockIdx.x >> 1;
  const int64_t num_pairs = gridDim.x >> 1;
  const int num_k = static_cast<int>((g.J + C::kBK - 1) / C::kBK);
  const int tail = g.tail_stages;
  const int64_t tiles_m = (g.P + C::kBM - 1) / C::kBM;
  const int64_t tiles_n = (g.Q + BN - 1) / BN;
  const int64_t num_tiles = tiles_m * tiles_n;
  const bool n_fastest = g.P >= g.Q;                 // stream the larger operand once
  const WorkSched sched = make_sched(num_tiles, num_k + tail, num_pairs, SK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&ctl.full[s]), 1);          // the even CTA's producer + both CTAs' bytes
      mbar_init(smem_u32(&ctl.empty[s]), 1);         // one multicast MMA commit
    }
    mbar_init(smem_u32(&ctl.acc_full), 1);
    mbar_init(smem_u32(&ctl.acc_empty), 2 * kEpiWarps);   // epilogue warps of both CTAs
    mbar_init(smem_u32(&ctl.drain), 1);
    ctl.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&ctl.tmem_base), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();                                // barriers of both CTAs initialised
  tc_fence_after();
  pdl_enter();                                       // the set-up above overlaps the previous kernel's tail
  const uint32_t tmem = ctl.tmem_base;
  volatile int *abort_flag = &ctl.abort_flag;
  const uint32_t peer_abort = cluster_map(smem_u32(&ctl.abort_flag), peer);

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    // The whole warp runs the loop (warp-uniform operands; every lane waits on the barriers and
    // the warp agrees on each outcome); one elected lane issues.
    if (elect_one()) {
      prefetch_tensormap(&maps.a);
      prefetch_tensormap(&maps.b);
      prefetch_tensormap(&maps.sfa);
      prefetch_tensormap(&maps.sfb);
      if (tail) {
        prefetch_tensormap(&maps.ao);
        prefetch_tensormap(&maps.bo);
      }
    }
    __syncwarp();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const int32_t atoms_per_rowblk = static_cast<int32_t>(g.J >> 7);   // 4-block scale atoms along J
    const int64_t nblocks = (g.Q + 127) >> 7;
    WorkIter it = make_iter(sched, pair);
    WorkItem w;
    while (ok && next_item<SK>(sched, it, w)) {
      const TileInfo t = tile_info(g, w.tile, tiles_m, tiles_n, num_k, n_fastest, C::kBM);
      const int32_t my_m0 = static_cast<int32_t>(t.m0 + 128 * rank);
      const int32_t my_n0 = static_cast<int32_t>(t.n0 + 128 * rank);
      const int32_t mb = my_m0 >> 7;
      const int32_t nb0 = static_cast<int32_t>(t.n0 >> 7);
      const int32_t nb1 = (nb0 + 1 < nblocks) ? nb0 + 1 : nb0;   // ragged Q: reuse finite scales
      for (int step = w.kb; step < w.ke; ++step) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctl.empty[stage]), phase ^ 1u, abort_flag, 32))) {
          ok = false;
          break;
        }
        const uint32_t sA = smem_base + stage * C::kStageBytes;
        const uint32_t sB = sA + C::kABytes;
        const uint32_t full_own = smem_u32(&ctl.full[stage]);
        const uint32_t full = cluster_map(full_own, 0);          // the even CTA's barrier
        if (elect_one()) {
          if (step < num_k) {
            if (rank == 0) mbar_arrive_expect_tx(full_own, C::kTxMain);
            tma_load_2d_pair(sA, &maps.a, full, step * 128, my_m0);
            tma_load_2d_pair(sB, &maps.b, full, step * 128, my_n0);
            // scale atoms: two per 128 rows per stage (the second is unused when the last slice
            // of a J that is an odd multiple of 128 is half full; rows past P read zeros)
            tma_load_2d_pair(sA + C::kSFA, &maps.sfa, full, 0, mb * atoms_per_rowblk + 2 * step);
            tma_load_2d_pair(sA + C::kSFB, &maps.sfb, full, 0, nb0 * atoms_per_rowblk + 2 * step);
            tma_load_2d_pair(sA + C::kSFB + 1024, &maps.sfb, full, 0, nb1 * atoms_per_rowblk + 2 * step);
          } else {
            // BF16 outlier tail: 64 of the r outlier columns (128 bytes) per stage
            const int32_t r0 = (step - num_k) * 64;
            if (rank == 0) mbar_arrive_expect_tx(full_own, C::kTxTail);
            tma_load_2d_pair(sA, &maps.ao, full, r0, my_m0);
            tma_load_2d_pair(sB, &maps.bo, full, r0, my_n0);
          }
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      // a CTA that gives up tells its peer too, so that neither waits out the full limit
      *abort_flag = 1;
      st_cluster_u32(peer_abort, 1u);
      report_status(g.status, kStatusTimeout);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    // The whole warp runs the loop; one elected lane issues the copies, MMAs and commits.
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      constexpr uint32_t idesc_bf16 = make_idesc_bf16(C::kBM, BN, false, false);
      // shared-memory descriptors of stage 0; a stage's are these plus its offset in the 16-byte
      // address field
      const uint64_t a0 = make_smem_desc(smem_base, 16, 1024, kLayoutSw128);
      const uint64_t b0 = make_smem_desc(smem_base + C::kABytes, 16, 1024, kLayoutSw128);
      const uint64_t sfa0 = make_smem_desc(smem_base + C::kSFA, 0, 128, kLayoutNone);
      const uint64_t sfb0 = make_smem_desc(smem_base + C::kSFB, 0, 128, kLayoutNone);
      WorkIter it = make_iter(sched, pair);
      WorkItem w;
      while (ok && next_item<SK>(sched, it, w)) {
        // The item's first stage, peeled from the loop: its scale copies go to their own
        // tensor-memory columns while the epilogue still drains the accumulator, and only its
        // MMAs wait for the drain.
        {
          const int step = w.kb;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctl.full[stage]), phase, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t soff = (static_cast<uint32_t>(stage) * C::kStageBytes) >> 4;
          const uint32_t sfa_t = tmem + kSfTmemBase + stage * C::kSfCols;
          const uint32_t sfb_t = sfa_t + 8;
          const bool half = (step == num_k - 1) && ((g.J & 255) != 0);
          if (step < num_k && elect_one()) {
#pragma unroll
            for (uint32_t ka = 0; ka < 2; ++ka) {
              if (ka == 1 && half) break;
              tmem_cp_32x128b_x4_pair(sfa_t + 4 * ka, desc_add(sfa0, soff + 32 * ka));
              tmem_cp_32x128b_x4_pair(sfb_t + 8 * ka, desc_add(sfb0, soff + 32 * ka));
              tmem_cp_32x128b_x4_pair(sfb_t + 8 * ka + 4, desc_add(sfb0, soff + 64 + 32 * ka));
            }
          }
          __syncwarp();
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctl.acc_empty), acc_phase ^ 1u, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            if (step < num_k) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                if (kk == 2 && half) break;
                constexpr uint32_t idesc0 = make_idesc_mxf4(C::kBM, BN, 0, 0);
                constexpr uint32_t idesc2 = make_idesc_mxf4(C::kBM, BN, 2, 2);
                mma_mxf4_pair(tmem, desc_add(a0, soff + 2 * kk), desc_add(b0, soff + 2 * kk),
                              (kk & 1) ? idesc2 : idesc0, sfa_t + 4 * (kk >> 1), sfb_t + 8 * (kk >> 1),
                              kk > 0 ? 1u : 0u);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16_pair(tmem, desc_add(a0, soff + 2 * kk), desc_add(b0, soff + 2 * kk), idesc_bf16,
                              kk > 0 ? 1u : 0u);
            }
            tc_commit_pair(smem_u32(&ctl.empty[stage]), 0x3);
          }
          __syncwarp();
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        for (int step = w.kb + 1; step < w.ke; ++step) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctl.full[stage]), phase, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t soff = (static_cast<uint32_t>(stage) * C::kStageBytes) >> 4;
          if (elect_one()) {
            if (step < num_k) {
              const uint32_t sfa_t = tmem + kSfTmemBase + stage * C::kSfCols;
              const uint32_t sfb_t = sfa_t + 8;
              const bool half = (step == num_k - 1) && ((g.J & 255) != 0);
              // Scale factors go to tensor memory just ahead of the two MMAs that read them (SF-A
              // atom ka -> columns sfa + 4 ka; SF-B rows 0..127 -> sfb + 8 ka, 128..255 -> +4):
              // interleaved with the MMAs, the copies cost the tensor pipe less than in one group.
              // The last slice of a J that is an odd multiple of 128 holds one scale atom and two
              // MMAs.
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                if (kk == 2 && half) break;
                if ((kk & 1) == 0) {
                  const uint32_t ka = static_cast<uint32_t>(kk >> 1);
                  tmem_cp_32x128b_x4_pair(sfa_t + 4 * ka, desc_add(sfa0, soff + 32 * ka));
                  tmem_cp_32x128b_x4_pair(sfb_t + 8 * ka, desc_add(sfb0, soff + 32 * ka));
                  tmem_cp_32x128b_x4_pair(sfb_t + 8 * ka + 4, desc_add(sfb0, soff + 64 + 32 * ka));
                }
                const uint64_t adesc = desc_add(a0, soff + 2 * kk);
                const uint64_t bdesc = desc_add(b0, soff + 2 * kk);
                constexpr uint32_t idesc0 = make_idesc_mxf4(C::kBM, BN, 0, 0);
                constexpr uint32_t idesc2 = make_idesc_mxf4(C::kBM, BN, 2, 2);
                mma_mxf4_pair(tmem, adesc, bdesc, (kk & 1) ? idesc2 : idesc0, sfa_t + 4 * (kk >> 1),
                              sfb_t + 8 * (kk >> 1), (step > w.kb || kk > 0) ? 1u : 0u);
              }
            } else {
              // BF16 outlier tail: four K=16 MMAs over 128-byte rows (the first of a stream-K part
              // that starts with a tail stage overwrites the accumulator)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16_pair(tmem, desc_add(a0, soff + 2 * kk), desc_add(b0, soff + 2 * kk), idesc_bf16,
                              (step > w.kb || kk > 0) ? 1u : 0u);
            }
            tc_commit_pair(smem_u32(&ctl.empty[stage]), 0x3);   // frees the stage in both CTAs
          }
          __syncwarp();
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) tc_commit_pair(smem_u32(&ctl.acc_full), 0x3);   // both accumulators ready
        __syncwarp();
        acc_phase ^= 1u;
      }
      if (!ok && lane == 0) {
        *abort_flag = 1;
        st_cluster_u32(peer_abort, 1u);
        report_status(g.status, kStatusTimeout);
      }
      // drain: wait (bounded) until every MMA / copy this warp issued has completed
      if (elect_one()) tc_commit_pair(smem_u32(&ctl.drain), 0x1);
      __syncwarp();
      if (!mbar_wait(smem_u32(&ctl.drain), 0, nullptr) && lane == 0) report_status(g.status, kStatusTimeout);
    }
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;                        // TMEM lanes 32*quad .. 32*quad+31
    const int half = (warp - 2) >> 2;                 // accumulator columns 128*half ..
    const uint32_t acc_empty = cluster_map(smem_u32(&ctl.acc_empty), 0);
    const bool can_store = g.C != nullptr;
    if (!can_store && threadIdx.x == 64) report_status(g.status, kStatusBadArg);
    const uint32_t epi_buf = smem_base + C::kEpiOffset + static_cast<uint32_t>(warp - 2) * C::kEpiBufs * C::kEpiBufBytes;
    uint32_t epi_seq = 0;
    uint32_t acc_phase = 0;
    if (lane == 0 && can_store) prefetch_tensormap(&maps.c);
    const int ew = warp - 2;                           // epilogue warp 0..7
    const int row_in_cta = 32 * quad + lane;
    WorkIter it = make_iter(sched, pair);
    WorkItem w;
    while (next_item<SK>(sched, it, w)) {
      const TileInfo t = tile_info(g, w.tile, tiles_m, tiles_n, num_k, n_fastest, C::kBM);
      bool ready = true;
      // polled without back-off: this wait sits on the accumulator hand-off between tiles
      if (lane == 0) ready = mbar_wait(smem_u32(&ctl.acc_full), acc_phase, abort_flag);
      ready = __shfl_sync(0xFFFFFFFFu, ready ? 1 : 0, 0) != 0;
      if (!ready) {
        if (lane == 0) {
          *abort_flag = 1;
          st_cluster_u32(peer_abort, 1u);
          report_status(g.status, kStatusTimeout);
        }
        break;
      }
      tc_fence_after();
      uint32_t v[128];                               // columns 128 half .. 128 half + 127 of this lane's row
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * quad) << 16) + 128u * half;
#pragma unroll
      for (int j = 0; j < 4; ++j) tmem_ld_32x32b_x32(taddr + 32u * j, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * j));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty);
      acc_phase ^= 1u;

      if (SK && w.role == kItemContrib) {
        // this pair's share of the tile's J stages: hand the partial sums to the finisher
        float4 *slot = sk_slot(g, pair, rank);
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            slot[(32 * half + 8 * j + q) * 128 + row_in_cta] =
                make_float4(__uint_as_float(v[32 * j + 4 * q]), __uint_as_float(v[32 * j + 4 * q + 1]),
                            __uint_as_float(v[32 * j + 4 * q + 2]), __uint_as_float(v[32 * j + 4 * q + 3]));
        __threadfence();                             // the partial is visible before the count
        __syncwarp();
        if (lane == 0) atomicAdd(sk_counter(g, w.tile - sched.dp_tiles, rank, ew), 1u);
        continue;
      }
      if (SK && w.role == kItemFinish) {
        // the pairs before this one that hold the tile's earlier stages (each holds one part)
        const int64_t sk_tile = w.tile - sched.dp_tiles;
        const uint32_t n_contrib =
            static_cast<uint32_t>(pair - sched.owner(static_cast<int32_t>(sk_tile) * sched.nsteps));
        uint32_t *cnt = sk_counter(g, sk_tile, rank, ew);
        bool got = true;
        if (lane == 0) got = wait_count(cnt, n_contrib, abort_flag);
        got = __shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) != 0;
        if (!got) {
          if (lane == 0) {
            *abort_flag = 1;
            st_cluster_u32(peer_abort, 1u);
            report_status(g.status, kStatusTimeout);
          }
          break;
        }
        // add the partials in a fixed order (the nearest pair first): same sums on every run
        for (uint32_t k = 0; k < n_contrib; ++k) {
          const float4 *slot = sk_slot(g, pair - 1 - static_cast<int64_t>(k), rank);
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 o = __ldcg(slot + (32 * half + 8 * j + q) * 128 + row_in_cta);
              const int e = 32 * j + 4 * q;
              v[e] = __float_as_uint(__uint_as_float(v[e]) + o.x);
              v[e + 1] = __float_as_uint(__uint_as_float(v[e + 1]) + o.y);
              v[e + 2] = __float_as_uint(__uint_as_float(v[e + 2]) + o.z);
              v[e + 3] = __float_as_uint(__uint_as_float(v[e + 3]) + o.w);
            }
        }
        __syncwarp();
        if (lane == 0) *cnt = 0u;                    // read by this warp only: clear it for the next launch
      }

      // Stores through shared memory: each 32-row x 32-byte box (16 bf16 or 8 fp32 columns) is
      // written by the warp into its staging buffer, lane i filling row i with the 32-byte swizzle
      // (16-byte piece p at p ^ ((i >> 2) & 1): no bank conflicts), then stored by one TMA bulk
      // copy that runs while the warp converts the next box.
      const int32_t row0 = static_cast<int32_t>(t.m0 + 128 * rank + 32 * quad);   // 32 rows, all in or all out
      if (can_store && row0 < g.P) {
        const bool f32 = g.out_dtype == 1;
        const int nbox = f32 ? 16 : 8;
        const uint32_t sw = (static_cast<uint32_t>(lane) >> 2) & 1u;
#pragma unroll
        for (int bx = 0; bx < 16; ++bx) {
          if (bx >= nbox) break;
          const int32_t col = static_cast<int32_t>(t.n0 + 128 * half) + (f32 ? 8 : 16) * bx;
          if (col >= g.Q) break;                   // Q is a multiple of 128: whole boxes only
          uint32_t w[2][4];
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            if (f32) {
              const int e = 8 * bx + 4 * p;
#pragma unroll
              for (int k = 0; k < 4; ++k) w[p][k] = v[e + k];
            } else {
              const int e = 16 * bx + 8 * p;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                w[p][k] = pack_bf16x2_rn(__uint_as_float(v[e + 2 * k]), __uint_as_float(v[e + 2 * k + 1]));
            }
          }
          const uint32_t buf = epi_buf + (epi_seq % C::kEpiBufs) * C::kEpiBufBytes;
          ++epi_seq;
          if (lane == 0) bulk_wait_group_read<C::kEpiBufs - 1>();   // this buffer's last box has left it
          __syncwarp();
#pragma unroll
          for (int p = 0; p < 2; ++p)
            st_shared_v4(buf + 32u * lane + 16u * (static_cast<uint32_t>(p) ^ sw), w[p][0], w[p][1], w[p][2], w[p][3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&maps.c, buf, col, row0);
            bulk_commit_group();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();             // staging buffers stay live until read
  }

  // neither CTA frees tensor memory or exits while its peer may still signal it
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  // After the barrier both CTAs read the same flag (a thread that gives up sets its own CTA's
  // and its peer's before arriving), so the second barrier is taken by both or by neither.
  if (*abort_flag) {
    if (threadIdx.x == 0) settle_inflight_loads();
    cluster_sync_all();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

// =============================================================================================
// kind 1: BF16, single CTAs
// =============================================================================================
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs g) {
  using C = Bf16Cfg;
  extern __shared__ uint8_t smem_raw[];
  __shared__ SmemCtl<C::kStages> ctl;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;   // swizzle atoms need alignment
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_k = static_cast<int>((g.J + C::kBK - 1) / C::kBK);
  const int64_t tiles_m = (g.P + C::kBM - 1) / C::kBM;
  const int64_t tiles_n = (g.Q + BN - 1) / BN;
  const int64_t num_tiles = tiles_m * tiles_n * (g.splits > 1 ? g.splits : 1);
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
    // Whole-warp loops with one elected issuing lane keep every operand warp-uniform.
    if (elect_one()) {
      prefetch_tensormap(&maps.a);
      prefetch_tensormap(&maps.b);
    }
    __syncwarp();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      const TileInfo t = tile_info(g, tile, tiles_m, tiles_n, num_k, n_fastest, C::kBM);
      for (int ks = t.k_begin; ks < t.k_end; ++ks) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctl.empty[stage]), phase ^ 1u, abort_flag, 32))) {
          ok = false;
          break;
        }
        const uint32_t sA = smem_base + stage * C::kStageBytes;
        const uint32_t sB = sA + C::kABytes;
        const uint32_t full = smem_u32(&ctl.full[stage]);
        if (elect_one()) {
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
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report_status(g.status, kStatusTimeout);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const uint32_t idesc = make_idesc_bf16(C::kBM, BN, g.a_mn_major != 0, g.b_mn_major != 0);
    for (int64_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      const TileInfo t = tile_info(g, tile, tiles_m, tiles_n, num_k, n_fastest, C::kBM);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctl.acc_empty), acc_phase ^ 1u, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int ks = t.k_begin; ks < t.k_end; ++ks) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctl.full[stage]), phase, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sA = smem_base + stage * C::kStageBytes;
        const uint32_t sB = sA + C::kABytes;
        if (elect_one()) {
          // four K=16 MMAs over 128-byte rows (K-major) or 16-row groups (MN-major)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = g.a_mn_major ? make_smem_desc(sA + 2048 * kk, 8192, 1024, kLayoutSw128)
                                                : make_smem_desc(sA + 32 * kk, 16, 1024, kLayoutSw128);
            const uint64_t bdesc = g.b_mn_major ? make_smem_desc(sB + 2048 * kk, 8192, 1024, kLayoutSw128)
                                                : make_smem_desc(sB + 32 * kk, 16, 1024, kLayoutSw128);
            mma_bf16(tmem, adesc, bdesc, idesc, (ks > t.k_begin || kk > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&ctl.empty[stage]));      // frees the smem stage when MMAs finish
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) tc_commit(smem_u32(&ctl.acc_full));   // accumulator ready for the epilogue
      __syncwarp();
      acc_phase ^= 1u;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report_status(g.status, kStatusTimeout);
    }
    // drain: wait (bounded) until every MMA this warp issued has completed
    if (elect_one()) tc_commit(smem_u32(&ctl.drain));
    __syncwarp();
    if (!mbar_wait(smem_u32(&ctl.drain), 0, nullptr) && lane == 0) report_status(g.status, kStatusTimeout);
  } else {
    // ------------------------------------------------------------------ epilogue warps
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    // Partial mode (split-K or not) is chosen by a non-null c_partial; with neither output the
    // tiles are computed but nothing is stored and the status word records the bad argument.
    const bool to_partial = g.c_partial != nullptr;
    const bool can_store = to_partial || g.C != nullptr;
    if (!can_store && threadIdx.x == 64) report_status(g.status, kStatusBadArg);
    uint32_t acc_phase = 0;
    for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const TileInfo t = tile_info(g, tile, tiles_m, tiles_n, num_k, n_fastest, C::kBM);
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
      if (t.k_end <= t.k_begin) {            // a split with no K range contributes zeros
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 32; ++e) v[j][e] = 0u;
      }

      const int64_t row = t.m0 + 32 * quad + lane;
      if (can_store && row < g.P) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t col = t.n0 + 128 * half + 32 * j;
          if (col < g.Q) store_row32(g, to_partial, t.split, row, col, v[j]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {                                 // the same value for every thread after the barrier
    if (threadIdx.x == 0) settle_inflight_loads();
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// =============================================================================================
// kind 2: BF16 outlier GEMM of outer OE with the scatter-add fused (appendix, Fused Scatter-Add:
// the outlier product is added in place, with no intermediate result written out).  The product
// has only r rows (or columns), so its J range is split over the S CTAs of a cluster (S = 1, 2, 4
// or 8; one (tile, J range) per CTA).  Each CTA leaves its float32 partial tile in its own shared
// memory; after a cluster barrier CTA k sums rows [k 128/S, (k+1) 128/S) of the tile over the S
// partials in rank order (through distributed shared memory), adds the sum to C's current value
// in float32 and rounds once to C's type: C[idx[i], q] += O[i, q] (axis 0) or C[p, idx[i]] +=
// O[p, i] (axis 1).  A second cluster barrier keeps every partial alive until all are read.
// =============================================================================================

__device__ __forceinline__ void scatter_add4(const GemmArgs &g, int64_t row, int64_t col, const float4 &o) {
  const float add[4] = {o.x, o.y, o.z, o.w};
  if (g.scatter_axis == 0) {
    const int64_t dst = g.scatter_idx[row];
    if (dst < 0 || dst >= g.c_rows || col + 4 > g.c_cols) return;   // never write outside C
    if (g.out_dtype == 1) {
      float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(g.C) + dst * g.c_cols + col);
      float4 c = *p;
      c.x += add[0]; c.y += add[1]; c.z += add[2]; c.w += add[3];
      *p = c;
    } else {
      uint2 *p = reinterpret_cast<uint2 *>(static_cast<uint16_t *>(g.C) + dst * g.c_cols + col);
      const uint2 c = *p;
      const uint32_t w0 = pack_bf16x2_rn(bf16_bits_to_f32(c.x & 0xFFFFu) + add[0], bf16_bits_to_f32(c.x >> 16) + add[1]);
      const uint32_t w1 = pack_bf16x2_rn(bf16_bits_to_f32(c.y & 0xFFFFu) + add[2], bf16_bits_to_f32(c.y >> 16) + add[3]);
      *p = make_uint2(w0, w1);
    }
  } else {
    if (row >= g.c_rows) return;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (col + e >= g.Q) break;
      const int64_t dst = g.scatter_idx[col + e];
      if (dst < 0 || dst >= g.c_cols) continue;
      if (g.out_dtype == 1) {
        float *p = static_cast<float *>(g.C) + row * g.c_cols + dst;
        *p = *p + add[e];
      } else {
        uint16_t *p = static_cast<uint16_t *>(g.C) + row * g.c_cols + dst;
        *p = static_cast<uint16_t>(f32_to_bf16_bits(bf16_bits_to_f32(*p) + add[e]));
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_scatter_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs g) {
  using C = ScatterCfg;
  extern __shared__ uint8_t smem_raw[];
  __shared__ SmemCtl<C::kStages> ctl;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;   // swizzle atoms need alignment
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t split = cluster_ctarank();
  const uint32_t nsplit = cluster_nctarank();
  const int64_t tile = blockIdx.x / nsplit;
  const int num_k = static_cast<int>((g.J + C::kBK - 1) / C::kBK);
  const int64_t tiles_n = (g.Q + C::kBN - 1) / C::kBN;
  const int64_t m0 = (tile / tiles_n) * C::kBM, n0 = (tile % tiles_n) * C::kBN;
  const int per = (num_k + static_cast<int>(nsplit) - 1) / static_cast<int>(nsplit);
  const int k_begin = min(num_k, static_cast<int>(split) * per);
  const int k_end = min(num_k, k_begin + per);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&ctl.full[s]), 1);
      mbar_init(smem_u32(&ctl.empty[s]), 1);
    }
    mbar_init(smem_u32(&ctl.acc_full), 1);
    mbar_init(smem_u32(&ctl.drain), 1);
    ctl.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int *abort_flag = &ctl.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (elect_one()) {
      prefetch_tensormap(&maps.a);
      prefetch_tensormap(&maps.b);
    }
    __syncwarp();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int ks = k_begin; ks < k_end; ++ks) {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctl.empty[stage]), phase ^ 1u, abort_flag, 32))) {
        ok = false;
        break;
      }
      const uint32_t sA = smem_base + stage * C::kStageBytes;
      const uint32_t sB = sA + C::kABytes;
      const uint32_t full = smem_u32(&ctl.full[stage]);
      if (elect_one()) {
        mbar_arrive_expect_tx(full, C::kABytes + C::kBBytes);
        const int32_t k0 = ks * 64;
        if (g.a_mn_major) {
          tma_load_2d(sA, &maps.a, full, static_cast<int32_t>(m0), k0);
          tma_load_2d(sA + 8192, &maps.a, full, static_cast<int32_t>(m0 + 64), k0);
        } else {
          tma_load_2d(sA, &maps.a, full, k0, static_cast<int32_t>(m0));
        }
        if (g.b_mn_major) {
#pragma unroll
          for (int c = 0; c < C::kBN / 64; ++c)
            tma_load_2d(sB + c * 8192, &maps.b, full, static_cast<int32_t>(n0 + 64 * c), k0);
        } else {
          tma_load_2d(sB, &maps.b, full, k0, static_cast<int32_t>(n0));
        }
      }
      __syncwarp();
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report_status(g.status, kStatusTimeout);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const uint32_t idesc = make_idesc_bf16(C::kBM, C::kBN, g.a_mn_major != 0, g.b_mn_major != 0);
    for (int ks = k_begin; ks < k_end; ++ks) {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctl.full[stage]), phase, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sA = smem_base + stage * C::kStageBytes;
      const uint32_t sB = sA + C::kABytes;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t adesc = g.a_mn_major ? make_smem_desc(sA + 2048 * kk, 8192, 1024, kLayoutSw128)
                                              : make_smem_desc(sA + 32 * kk, 16, 1024, kLayoutSw128);
          const uint64_t bdesc = g.b_mn_major ? make_smem_desc(sB + 2048 * kk, 8192, 1024, kLayoutSw128)
                                              : make_smem_desc(sB + 32 * kk, 16, 1024, kLayoutSw128);
          mma_bf16(tmem, adesc, bdesc, idesc, (ks > k_begin || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&ctl.empty[stage]));
      }
      __syncwarp();
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (ok && elect_one()) tc_commit(smem_u32(&ctl.acc_full));   // the partial is in tensor memory
    __syncwarp();
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report_status(g.status, kStatusTimeout);
    }
    if (elect_one()) tc_commit(smem_u32(&ctl.drain));
    __syncwarp();
    if (!mbar_wait(smem_u32(&ctl.drain), 0, nullptr) && lane == 0) report_status(g.status, kStatusTimeout);
  } else {
    // ------------------------------------------------------------------ partial -> shared memory
    // The pipeline is drained once the accumulator is ready (every MMA, hence every operand load,
    // has completed), so the stage buffers hold the partial tile: 128 rows of 128 floats.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    bool ready = true;
    if (k_end > k_begin) {
      if (lane == 0) ready = mbar_wait(smem_u32(&ctl.acc_full), 0, abort_flag, 128);
      ready = __shfl_sync(0xFFFFFFFFu, ready ? 1 : 0, 0) != 0;
    }
    if (!ready) {
      if (lane == 0) {
        *abort_flag = 1;
        report_status(g.status, kStatusTimeout);
      }
    } else {
      tc_fence_after();
      const uint32_t row_addr = smem_base + static_cast<uint32_t>(32 * quad + lane) * C::kPartialRowBytes;
#pragma unroll
      for (int j = 0; j < C::kBN / 64; ++j) {                 // this warp's half: BN / 2 columns
        uint32_t v[32];
        if (k_end > k_begin) {
          tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * quad) << 16) + (C::kBN / 2) * half + 32u * j, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;             // an empty J range adds zeros
        }
        const uint32_t a = row_addr + ((C::kBN / 2) * half + 32u * j) * 4u;
#pragma unroll
        for (int q = 0; q < 8; ++q) st_shared_v4(a + 16u * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
  }

  // every partial of the cluster is in shared memory (or its CTA gave up)
  tc_fence_before();
  cluster_sync_all();
  if (warp >= 2) {
    bool any_abort = false;
    for (uint32_t k = 0; k < nsplit; ++k) any_abort |= ld_cluster_u32(cluster_map(smem_u32(&ctl.abort_flag), k)) != 0;
    if (!any_abort) {
      const int te = threadIdx.x - 64;                        // 256 reducing threads
      const int rows_per = C::kBM / static_cast<int>(nsplit);
      const int items = rows_per * (C::kBN / 4);
      for (int it = te; it < items; it += kEpiWarps * 32) {
        const int rr = static_cast<int>(split) * rows_per + it / (C::kBN / 4);
        const int c4 = it % (C::kBN / 4);
        const int64_t row = m0 + rr, col = n0 + 4 * c4;
        if (row >= g.P || col >= g.Q) continue;
        const uint32_t off = smem_base + static_cast<uint32_t>(rr) * C::kPartialRowBytes + 16u * c4;
        float4 acc = ld_cluster_v4(cluster_map(off, 0));
        for (uint32_t k = 1; k < nsplit; ++k) {
          const float4 o = ld_cluster_v4(cluster_map(off, k));
          acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
        }
        scatter_add4(g, row, col, acc);
      }
    }
  }
  cluster_sync_all();                                 // no CTA leaves while its partial may be read
  if (*abort_flag) {
    if (threadIdx.x == 0) settle_inflight_loads();
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// attr must hold two entries: the cluster shape and programmatic dependent launch (pdl_enter).
cudaLaunchConfig_t pair_launch_config(cudaLaunchAttribute *attr, unsigned grid, size_t smem, cudaStream_t s) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// Co-resident CTA pairs of the MXFP4 kernel (configuration C) on the current device (its
// persistent grid), cached per device.
template <class C>
int pair_capacity(int num_sms) {
  constexpr int kMaxDevices = 64;
  static int cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return num_sms / 2;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg =
      pair_launch_config(attr, static_cast<unsigned>(num_sms & ~1), C::kSmemBytes + 1024, 0);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, gemm_mxf4_pair_kernel<C, false>, &cfg) != cudaSuccess ||
      clusters <= 0) {
    (void)cudaGetLastError();
    clusters = num_sms / 2;
  }
  cached[dev] = clusters;
  return clusters;
}

template <class C>
cudaError_t launch_mxf4_cfg(const GemmArgs &g0, const GemmMaps &maps, int num_sms, cudaStream_t s) {
  const size_t smem = C::kSmemBytes + 1024;
  GemmArgs g = g0;
  const int64_t tiles = ((g.P + C::kBM - 1) / C::kBM) * ((g.Q + BN - 1) / BN);
  const int64_t cap = pair_capacity<C>(num_sms);
  int64_t pairs = tiles < cap ? tiles : cap;
  // Stream-K where it measured faster: at least two whole rounds of tiles, a last round that
  // would leave over 3% of the pairs idle, and a long J (the wgrad shapes with few tiles).  With
  // fewer rounds, or a short J, splitting tiles across pairs loses more to operand reuse in L2
  // (pairs no longer stream the same J slices of shared operand rows together) than it gains.
  g.sk = 0;
  if (g.sk_partial && g.sk_counters && cap <= g.sk_max_pairs && g.J >= 16384) {
    const int64_t rounds = (tiles + cap - 1) / cap;
    const int64_t dp = tiles / cap >= 1 ? (tiles / cap - 1) * cap : 0;
    const int64_t nsteps = (g.J + C::kBK - 1) / C::kBK + g.tail_stages;
    const int64_t units = (tiles - dp) * nsteps;
    const bool short_round = tiles < 97 * rounds * cap / 100;
    // every pair needs at least one stage (the finisher counts the pairs before it as contributors)
    if (tiles >= 2 * cap && short_round && tiles - dp <= kSkMaxTiles && units >= cap &&
        units < (int64_t(1) << 31)) {
      g.sk = 1;
      pairs = cap;
    }
  }
  auto *kernel = g.sk ? gemm_mxf4_pair_kernel<C, true> : gemm_mxf4_pair_kernel<C, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_launch_config(attr, static_cast<unsigned>(2 * pairs), smem, s);
  e = cudaLaunchKernelEx(&cfg, kernel, maps, g);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_mxf4(const GemmArgs &g, const GemmMaps &maps, int num_sms, cudaStream_t s) {
  return g.J <= kShortJ ? launch_mxf4_cfg<PairCfgShortJ>(g, maps, num_sms, s)
                        : launch_mxf4_cfg<PairCfg>(g, maps, num_sms, s);
}

cudaError_t launch_bf16(const GemmArgs &g, const GemmMaps &maps, int num_sms, cudaStream_t s) {
  const size_t smem = gemm_smem_bytes(1);
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((g.P + Bf16Cfg::kBM - 1) / Bf16Cfg::kBM) * ((g.Q + BN - 1) / BN) *
                        (g.splits > 1 ? g.splits : 1);
  const unsigned grid = static_cast<unsigned>(tiles < num_sms ? tiles : num_sms);
  gemm_bf16_kernel<<<grid, kThreads, smem, s>>>(maps, g);
  return cudaGetLastError();
}

size_t scatter_smem_bytes() { return ScatterCfg::kStages * ScatterCfg::kStageBytes + 1024; }

cudaLaunchConfig_t scatter_launch_config(cudaLaunchAttribute *attr, unsigned grid, int splits, cudaStream_t s) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = scatter_smem_bytes();
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of `splits` CTAs of the outlier GEMM that fit the current device at once (cached per
// device and size).
int64_t scatter_cluster_capacity(int splits) {
  constexpr int kMaxDevices = 64;
  static int64_t cached[kMaxDevices][4] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  const int slot = splits == 1 ? 0 : splits == 2 ? 1 : splits == 4 ? 2 : 3;
  if (cached[dev][slot] > 0) return cached[dev][slot];
  if (cudaFuncSetAttribute(gemm_bf16_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(scatter_smem_bytes())) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = scatter_launch_config(attr, static_cast<unsigned>(splits * 8), splits, 0);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, gemm_bf16_scatter_kernel, &cfg) != cudaSuccess || clusters <= 0) {
    (void)cudaGetLastError();
    return 0;
  }
  cached[dev][slot] = clusters;
  return clusters;
}

// The J split (cluster size): the largest of 8, 4, 2 that keeps at least four 64-wide J stages
// per CTA, no more CTAs than SMs, and every cluster resident in one wave; else 1.
int scatter_splits(int64_t P, int64_t Q, int64_t J, int num_sms) {
  const int64_t tiles = ((P + ScatterCfg::kBM - 1) / ScatterCfg::kBM) * ((Q + ScatterCfg::kBN - 1) / ScatterCfg::kBN);
  const int64_t k_stages = (J + ScatterCfg::kBK - 1) / ScatterCfg::kBK;
  for (int s = 8; s >= 2; s >>= 1)
    if (tiles * s <= num_sms && k_stages >= 4 * s && tiles <= scatter_cluster_capacity(s)) return s;
  return 1;
}

cudaError_t launch_bf16_scatter(const GemmArgs &g, const GemmMaps &maps, int num_sms, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(scatter_smem_bytes()));
  if (e != cudaSuccess) return e;
  const int splits = scatter_splits(g.P, g.Q, g.J, num_sms);
  const int64_t tiles = ((g.P + ScatterCfg::kBM - 1) / ScatterCfg::kBM) * ((g.Q + ScatterCfg::kBN - 1) / ScatterCfg::kBN);
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = scatter_launch_config(attr, static_cast<unsigned>(tiles * splits), splits, s);
  e = cudaLaunchKernelEx(&cfg, gemm_bf16_scatter_kernel, maps, g);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int scatter_gemm_splits(int64_t P, int64_t Q, int64_t J, int num_sms) { return scatter_splits(P, Q, J, num_sms); }

size_t gemm_smem_bytes(int kind) {
  return kind == 0 ? (PairCfg::kSmemBytes > PairCfgShortJ::kSmemBytes ? PairCfg::kSmemBytes : PairCfgShortJ::kSmemBytes) + 1024
                   : Bf16Cfg::kStages * Bf16Cfg::kStageBytes + 1024;
}

int gemm_tail_cols_per_stage() { return 64; }

cudaError_t launch_gemm(const GemmArgs &g, const GemmMaps &maps, int num_sms, cudaStream_t s) {
  if (g.kind == 0) return launch_mxf4(g, maps, num_sms, s);
  if (g.kind == 2) return launch_bf16_scatter(g, maps, num_sms, s);
  return launch_bf16(g, maps, num_sms, s);
}

}  // namespace adahop
