// Host side of the C ABI (include/adahop.h): argument validation, workspace carving, TMA tensor
// maps, and the launch sequence of each strategy (AdaHOP Fig. 5 and Fig. 9: FOID -> IHT and
// quantisation -> fused MXFP4 + BF16 GEMM -> fused scatter-add).
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/adahop.h"
#include "common.cuh"
#include "kernels.cuh"

using namespace adahop;

namespace {

thread_local char g_last_cuda_error[256] = "";

adahop_status cuda_fail(cudaError_t e, const char *what) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", what, cudaGetErrorString(e));
  return ADAHOP_ERR_CUDA;
}
#define CUDA_TRY(expr, what)                           \
  do {                                                 \
    cudaError_t _e = (expr);                           \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)
#define ST_TRY(expr)                \
  do {                              \
    adahop_status _s = (expr);      \
    if (_s != ADAHOP_OK) return _s; \
  } while (0)

// ------------------------------------------------------------------------- device facts
struct DeviceInfo {
  int num_sms = 0;
  bool supported = false;
};
DeviceInfo g_devices[64];
std::mutex g_dev_mutex;

adahop_status device_info(DeviceInfo *out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= 64) return ADAHOP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo &d = g_devices[dev];
  if (d.num_sms == 0) {
    int major = 0, minor = 0, sms = 0;
    CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "cc major");
    CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "cc minor");
    CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "sm count");
    d.num_sms = sms;
    d.supported = (major == 10 && minor == 3);
  }
  *out = d;
  return d.supported ? ADAHOP_OK : ADAHOP_ERR_UNSUPPORTED;
}

// ------------------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

adahop_status get_encoder(EncodeTiledFn *fn) {
  static EncodeTiledFn cached = nullptr;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!cached) return cuda_fail(err == cudaSuccess ? cudaErrorNotSupported : err, "cuTensorMapEncodeTiled lookup");
  *fn = cached;
  return ADAHOP_OK;
}

// 2D tiled map over a row-major matrix: `inner` elements per row (contiguous), `outer` rows.
adahop_status make_map(CUtensorMap *map, CUtensorMapDataType dt, size_t elem_bytes, const void *base,
                       uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                       CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc;
  ST_TRY(get_encoder(&enc));
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * elem_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "cuTensorMapEncodeTiled failed (%d)",
                  static_cast<int>(r));
    return ADAHOP_ERR_CUDA;
  }
  return ADAHOP_OK;
}

// ------------------------------------------------------------------------- validation
bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
// the GEMMs carry tile coordinates in int32 (TMA coordinates are signed 32-bit)
bool dim_ok(int64_t d) { return d > 0 && d % 128 == 0 && d < (int64_t(1) << 31); }

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
int round8(int r) { return (r + 7) & ~7; }

// The zeroed header every workspace starts with (zero at the first call; every call that
// completes leaves it zero): the status word at offset 0, FOID's completion counter at 64, and
// the fused GEMM's stream-K counters from 1024.
constexpr size_t kHeaderBytes = 16384;
constexpr size_t kFoidCounterOffset = 64;
constexpr size_t kSkCounterOffset = 1024;
static_assert(kSkCounterOffset + sizeof(uint32_t) * kSkMaxTiles * kSkCountersPerTile <= kHeaderBytes, "header layout");
constexpr int kSkMaxPairs = 80;   // stream-K partial slots: one per CTA pair (>= 76 pairs on 152 SMs)

// ------------------------------------------------------------------------- workspace layout
// One GEMM's scratch.  The region sizes are upper bounds over all strategies.
struct GemmWs {
  size_t status, foid, idx, mask, a_codes, a_sf, b_codes, b_sf, ao, bo, gath, partial, sk, total;
};

constexpr int kMaxRank = 256;
constexpr int kSizingSms = 160;   // upper bound on the SM count used to size split-K partials

int choose_splits(int64_t tiles, int64_t k_stages, int num_sms) {
  int s = static_cast<int>(std::max<int64_t>(1, num_sms / std::max<int64_t>(1, tiles)));
  s = static_cast<int>(std::min<int64_t>(s, std::max<int64_t>(1, k_stages / 4)));
  return std::max(1, std::min(s, 16));
}

// `lines` bounds the number of lines FOID ranks (the largest of M, N, K for a linear layer), so
// the status / FOID / index / mask prefix is laid out identically for the three GEMMs of a layer.
GemmWs gemm_ws(int64_t P, int64_t Q, int64_t J, int r, int num_sms, int64_t lines) {
  GemmWs w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const int rr = std::max(r, 1);
  w.status = take(kHeaderBytes);
  w.foid = take(foid_scratch_bytes(lines, rr));
  w.idx = take(sizeof(int32_t) * kMaxRank);
  w.mask = take(sizeof(uint32_t) * ((lines + 31) / 32));
  w.a_codes = take(static_cast<size_t>(P * J / 2));
  w.a_sf = take(static_cast<size_t>(P * J / 32));
  w.b_codes = take(static_cast<size_t>(Q * J / 2));
  w.b_sf = take(static_cast<size_t>(Q * J / 32));
  w.ao = take(static_cast<size_t>(P) * round8(rr) * 2);
  w.bo = take(static_cast<size_t>(Q) * round8(rr) * 2);
  w.gath = take(static_cast<size_t>(rr) * J * 2);
  // outlier GEMM partials: rows case r x Q per split, cols case P x r per split
  const int64_t k_stages = (J + 63) / 64;
  const int s_rows = choose_splits((Q + 255) / 256, k_stages, num_sms);
  const int s_cols = choose_splits((P + 127) / 128, k_stages, num_sms);
  const size_t part = std::max(static_cast<size_t>(s_rows) * rr * Q, static_cast<size_t>(s_cols) * P * rr);
  w.partial = take(part * sizeof(float));
  w.sk = take(kSkPartialBytesPerPair * kSkMaxPairs);
  w.total = off;
  return w;
}

struct GemmShape {
  int64_t P, Q, J;
};
GemmShape shape_of(int gemm, int64_t M, int64_t N, int64_t K) {
  switch (gemm) {
    case 0: return {M, N, K};   // Y = X W^T
    case 1: return {M, K, N};   // dX = G_Y W
    default: return {N, K, M};  // dW = G_Y^T X
  }
}

// ------------------------------------------------------------------------- one GEMM
enum { T_X = 0, T_W = 1, T_GY = 2 };
struct Tensor {
  const uint16_t *p;
  int64_t rows, cols;
};

// Which tensor is the A-source / B-source of each GEMM, and how A / B^T are stored.
struct GemmRoles {
  int a_src, b_src;
  int a_inner_axis, b_inner_axis;   // quantisation orientation of the stored tensor
  int a_kmajor, b_kmajor;           // BF16 operand majorness as stored
};
GemmRoles roles_of(int gemm) {
  switch (gemm) {
    case 0: return {T_X, T_W, 1, 1, 1, 1};
    case 1: return {T_GY, T_W, 1, 0, 1, 0};
    default: return {T_GY, T_X, 0, 0, 0, 0};
  }
}
// Role of a source tensor's line axis in a GEMM: 'P' (rows of C), 'Q' (columns of C) or 'J'
// (the inner dimension).
char axis_role(int gemm, int tensor, int axis /*0 rows, 1 cols*/) {
  static const char table[3][3][2] = {
      /* fwd   */ {{'P', 'J'}, {'Q', 'J'}, {'?', '?'}},
      /* dgrad */ {{'?', '?'}, {'J', 'Q'}, {'P', 'J'}},
      /* wgrad */ {{'J', 'Q'}, {'?', '?'}, {'J', 'P'}},
  };
  return table[gemm][tensor][axis];
}

struct OeChoice {
  int tensor = -1, axis = 0;
  char role = 0;
};
// OE-Left extracts rows of the Row-wise operand (the A-source when none or both are Row-wise);
// OE-Right extracts columns of the Column-wise operand (the B-source when none or both are).
OeChoice oe_choice(int gemm, int strategy, const int pats[3]) {
  const GemmRoles ro = roles_of(gemm);
  OeChoice c;
  if (strategy == ADAHOP_OE_LEFT) {
    const bool ra = pats[ro.a_src] == ADAHOP_PAT_ROW, rb = pats[ro.b_src] == ADAHOP_PAT_ROW;
    c.tensor = (ra != rb) ? (ra ? ro.a_src : ro.b_src) : ro.a_src;
    c.axis = 0;
  } else if (strategy == ADAHOP_OE_RIGHT) {
    const bool ca = pats[ro.a_src] == ADAHOP_PAT_COL, cb = pats[ro.b_src] == ADAHOP_PAT_COL;
    c.tensor = (ca != cb) ? (ca ? ro.a_src : ro.b_src) : ro.b_src;
    c.axis = 1;
  } else {
    return c;
  }
  c.role = axis_role(gemm, c.tensor, c.axis);
  return c;
}

struct Ctx {
  cudaStream_t s;
  uint8_t *ws;
  GemmWs lay;
  int num_sms;
  bool sk = false;     // the workspace carries the fused GEMM's stream-K scratch (lay.sk, the header counters)
  uint32_t *status() const { return reinterpret_cast<uint32_t *>(ws + lay.status); }
  uint32_t *foid_counter() const { return reinterpret_cast<uint32_t *>(ws + lay.status + kFoidCounterOffset); }
};
// Context of a linear call: its workspace layout always includes the stream-K scratch.
Ctx linear_ctx(cudaStream_t s, void *workspace, const GemmWs &lay, int num_sms) {
  Ctx cx{s, static_cast<uint8_t *>(workspace), lay, num_sms};
  cx.sk = true;
  return cx;
}

adahop_status bf16_gemm(const Ctx &cx, const void *A, int a_kmajor, const void *B, int b_kmajor,
                        int64_t P, int64_t Q, int64_t J, void *C, int out_dtype, int splits,
                        float *partial) {
  if (!partial && !C) return ADAHOP_ERR_INVALID_ARG;
  GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (a_kmajor)
    ST_TRY(make_map(&maps.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, J, P, 64, 128));
  else
    ST_TRY(make_map(&maps.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, P, J, 64, 64));
  if (b_kmajor)
    ST_TRY(make_map(&maps.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, J, Q, 64, 256));
  else
    ST_TRY(make_map(&maps.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, Q, J, 64, 64));
  maps.ao = maps.a;
  maps.bo = maps.b;
  GemmArgs g{};
  g.P = P; g.Q = Q; g.J = J;
  g.kind = 1;
  g.a_mn_major = !a_kmajor;
  g.b_mn_major = !b_kmajor;
  g.C = C;
  g.out_dtype = out_dtype;
  g.splits = splits;
  g.c_partial = partial;
  g.status = cx.status();
  CUDA_TRY(launch_gemm(g, maps, cx.num_sms, cx.s), "bf16 gemm launch");
  return ADAHOP_OK;
}

// Outer-OE outlier product with the scatter-add fused: C[idx, :] += A . B (axis 0, P = r) or
// C[:, idx] += A . B (axis 1, Q = r); C is c_rows x c_cols.  One launch (a cluster split-K GEMM).
adahop_status bf16_scatter_gemm(const Ctx &cx, const void *A, int a_kmajor, const void *B, int b_kmajor, int64_t P,
                                int64_t Q, int64_t J, void *C, int64_t c_rows, int64_t c_cols, int out_dtype,
                                const int32_t *idx, int axis) {
  GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (a_kmajor)
    ST_TRY(make_map(&maps.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, J, P, 64, 128));
  else
    ST_TRY(make_map(&maps.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, P, J, 64, 64));
  // 128 x 128 output tiles: B boxes of 128 rows (K-major) or two 64-column boxes (MN-major)
  if (b_kmajor)
    ST_TRY(make_map(&maps.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, J, Q, 64, 128));
  else
    ST_TRY(make_map(&maps.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, Q, J, 64, 64));
  maps.ao = maps.a;
  maps.bo = maps.b;
  GemmArgs g{};
  g.P = P; g.Q = Q; g.J = J;
  g.kind = 2;
  g.a_mn_major = !a_kmajor;
  g.b_mn_major = !b_kmajor;
  g.C = C;
  g.out_dtype = out_dtype;
  g.splits = 1;
  g.status = cx.status();
  g.scatter_idx = idx;
  g.scatter_axis = axis;
  g.c_rows = c_rows;
  g.c_cols = c_cols;
  CUDA_TRY(launch_gemm(g, maps, cx.num_sms, cx.s), "bf16 outlier gemm (scatter-add) launch");
  return ADAHOP_OK;
}

adahop_status mxf4_gemm(const Ctx &cx, const uint8_t *ac, const uint8_t *asf, const uint8_t *bc,
                        const uint8_t *bsf, int64_t P, int64_t Q, int64_t J, const void *Ao,
                        const void *Bo, int r, void *C, int out_dtype) {
  GemmMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  // 128-byte rows (256 E2M1 codes, or 64 bf16 outlier columns) with the 128-byte swizzle; each
  // CTA of a pair loads 128 rows of A and 128 rows of B
  ST_TRY(make_map(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ac, J / 2, P, 128, 128));
  ST_TRY(make_map(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, bc, J / 2, Q, 128, 128));
  // scale atoms (512 bytes = 128 uint32 each), two consecutive atoms per load
  ST_TRY(make_map(&maps.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, asf, 128, (P / 128) * (J / 128), 128, 2,
                  CU_TENSOR_MAP_SWIZZLE_NONE));
  ST_TRY(make_map(&maps.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, bsf, 128, (Q / 128) * (J / 128), 128, 2,
                  CU_TENSOR_MAP_SWIZZLE_NONE));
  if (r > 0) {
    ST_TRY(make_map(&maps.ao, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Ao, r, P, 64, 128));
    ST_TRY(make_map(&maps.bo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Bo, r, Q, 64, 128));
  } else {
    maps.ao = maps.a;
    maps.bo = maps.b;
  }
  // C is written by TMA stores of 32 rows x 32 bytes (16 bf16 or 8 fp32 columns), 32-byte swizzle
  if (C) {
    if (out_dtype == 1)
      ST_TRY(make_map(&maps.c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, Q, P, 8, 32, CU_TENSOR_MAP_SWIZZLE_32B));
    else
      ST_TRY(make_map(&maps.c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, Q, P, 16, 32, CU_TENSOR_MAP_SWIZZLE_32B));
  }
  GemmArgs g{};
  g.P = P; g.Q = Q; g.J = J;
  g.kind = 0;
  g.sfa = asf;
  g.sfb = bsf;
  g.tail_stages = (r + 63) / 64;
  g.C = C;
  g.out_dtype = out_dtype;
  g.splits = 1;
  g.status = cx.status();
  if (cx.sk) {
    g.sk_partial = reinterpret_cast<float *>(cx.ws + cx.lay.sk);
    g.sk_counters = reinterpret_cast<uint32_t *>(cx.ws + cx.lay.status + kSkCounterOffset);
    g.sk_max_pairs = kSkMaxPairs;
  }
  CUDA_TRY(launch_gemm(g, maps, cx.num_sms, cx.s), "mxfp4 gemm launch");
  return ADAHOP_OK;
}

// FOID result shared between the two backward GEMMs when they extract the same lines.
struct FoidCache {
  int tensor = -1, axis = -1, r = -1;
};

// A operand already quantised (codes + tensor-core scales) by the dual-orientation pass.
struct PreA {
  uint8_t *codes, *sf;
};

// Outlier slices of one GEMM already gathered (one launch for both backward GEMMs): ao / bo
// for inner OE, gath for outer OE.
struct PreGath {
  uint16_t *ao, *bo, *gath;
};

// The gathers one OE GEMM needs (0, 1 or 2 jobs) into ao / bo / gath; returns the job count.
int oe_gather_jobs(int gemm, const OeChoice &oe, const Tensor t[3], const int32_t *idx, int r, const PreGath &dst,
                   GatherJob *jobs) {
  const GemmRoles ro = roles_of(gemm);
  const Tensor &ta = t[ro.a_src];
  const Tensor &tb = t[ro.b_src];
  if (oe.role == 'J') {
    // r8 columns per slice line, the last r8 - r of them +0 (they add nothing to the product): the
    // fused GEMM loads slices whose rows are a multiple of 16 bytes
    jobs[0] = GatherJob{ta.p, ta.rows, ta.cols, idx, r, ro.a_inner_axis == 1 ? 1 : 2, dst.ao, round8(r)};
    jobs[1] = GatherJob{tb.p, tb.rows, tb.cols, idx, r, ro.b_inner_axis == 1 ? 1 : 2, dst.bo, round8(r)};
    return 2;
  }
  if (oe.role == 'P') {
    jobs[0] = GatherJob{ta.p, ta.rows, ta.cols, idx, r, ro.a_inner_axis == 1 ? 0 : 3, dst.gath, 0};
    return 1;
  }
  jobs[0] = GatherJob{tb.p, tb.rows, tb.cols, idx, r, ro.b_inner_axis == 1 ? 0 : 3, dst.gath, 0};
  return 1;
}

// pre_a / pre_b: operand already quantised in this GEMM's orientation (codes + tensor-core
// scales), so its quantisation is skipped.  alt_a / alt_b: the operand is quantised by the
// dual-orientation pass, which also writes its other orientation (J = the stored rows) there;
// only valid where the GEMM quantises the stored tensor along its columns (inner axis 1).
adahop_status run_gemm(const Ctx &cx, int gemm, int strategy, int r, const Tensor t[3],
                       const int pats[3], void *C, int out_dtype, FoidCache *fc,
                       const PreA *pre_a = nullptr, const PreA *pre_b = nullptr,
                       const PreA *alt_a = nullptr, const PreA *alt_b = nullptr,
                       const PreGath *pre_g = nullptr) {
  const GemmShape sh = shape_of(gemm, t[T_X].rows, t[T_W].rows, t[T_X].cols);
  const GemmRoles ro = roles_of(gemm);
  const Tensor &ta = t[ro.a_src];
  const Tensor &tb = t[ro.b_src];
  uint8_t *ws = cx.ws;
  if (strategy == ADAHOP_BF16) {
    // A as stored: fwd/dgrad P x J (K-major); wgrad J x P.  B as stored: fwd Q x J; else J x Q.
    return bf16_gemm(cx, ta.p, ro.a_kmajor, tb.p, ro.b_kmajor, sh.P, sh.Q, sh.J, C, out_dtype, 1,
                     nullptr);
  }
  const int hadamard = strategy != ADAHOP_MXFP4;
  OeChoice oe;
  if ((strategy == ADAHOP_OE_LEFT || strategy == ADAHOP_OE_RIGHT) && r > 0) oe = oe_choice(gemm, strategy, pats);
  int32_t *idx = reinterpret_cast<int32_t *>(ws + cx.lay.idx);
  uint32_t *mask = reinterpret_cast<uint32_t *>(ws + cx.lay.mask);
  if (oe.tensor >= 0) {
    const Tensor &src = t[oe.tensor];
    const bool cached = fc && fc->tensor == oe.tensor && fc->axis == oe.axis && fc->r == r;
    if (!cached) {
      CUDA_TRY(launch_foid(src.p, src.rows, src.cols, oe.axis, r, idx, mask, ws + cx.lay.foid, cx.foid_counter(), cx.s),
               "foid");
      if (fc) *fc = FoidCache{oe.tensor, oe.axis, r};
    }
  }
  // quantise A (stored tensor ta, orientation a_inner_axis) and B^T (tb, b_inner_axis)
  uint8_t *ac = pre_a ? pre_a->codes : ws + cx.lay.a_codes;
  uint8_t *asf = pre_a ? pre_a->sf : ws + cx.lay.a_sf;
  uint8_t *bc = pre_b ? pre_b->codes : ws + cx.lay.b_codes;
  uint8_t *bsf = pre_b ? pre_b->sf : ws + cx.lay.b_sf;
  if ((alt_a && ro.a_inner_axis != 1) || (alt_b && ro.b_inner_axis != 1)) return ADAHOP_ERR_INVALID_ARG;
  {
    QuantArgs q{};
    q.hadamard = hadamard;
    q.scale_layout = 1;
    if (!pre_a) {
      q.T = ta.p; q.rows = ta.rows; q.cols = ta.cols;
      q.zero_rows = (oe.tensor == ro.a_src && oe.axis == 0) ? mask : nullptr;
      q.zero_cols = (oe.tensor == ro.a_src && oe.axis == 1) ? mask : nullptr;
      q.codes = ac; q.scales = asf;
      if (alt_a)
        CUDA_TRY(launch_quant_dual(q, alt_a->codes, alt_a->sf, cx.s), "quantise A (both orientations)");
      else
        CUDA_TRY(launch_quant(q, ro.a_inner_axis, cx.num_sms, cx.s), "quantise A");
    }
    if (!pre_b) {
      q.T = tb.p; q.rows = tb.rows; q.cols = tb.cols;
      q.zero_rows = (oe.tensor == ro.b_src && oe.axis == 0) ? mask : nullptr;
      q.zero_cols = (oe.tensor == ro.b_src && oe.axis == 1) ? mask : nullptr;
      q.codes = bc; q.scales = bsf;
      if (alt_b)
        CUDA_TRY(launch_quant_dual(q, alt_b->codes, alt_b->sf, cx.s), "quantise B (both orientations)");
      else
        CUDA_TRY(launch_quant(q, ro.b_inner_axis, cx.num_sms, cx.s), "quantise B");
    }
  }
  if (oe.tensor < 0) return mxf4_gemm(cx, ac, asf, bc, bsf, sh.P, sh.Q, sh.J, nullptr, nullptr, 0, C, out_dtype);

  const PreGath own{reinterpret_cast<uint16_t *>(ws + cx.lay.ao), reinterpret_cast<uint16_t *>(ws + cx.lay.bo),
                    reinterpret_cast<uint16_t *>(ws + cx.lay.gath)};
  const PreGath &g = pre_g ? *pre_g : own;
  if (!pre_g) {
    // one launch for this GEMM's outlier slices (A_o and B_o, or the outer lines)
    GatherJob jobs[2];
    const int n = oe_gather_jobs(gemm, oe, t, idx, r, own, jobs);
    CUDA_TRY(launch_gathers(jobs, n, cx.s), "gather outlier slices");
  }
  if (oe.role == 'J') {
    // inner: A_o[p, i] = A[p, idx[i]], B_o[q, i] = B^T[q, idx[i]] from the original bf16 values
    return mxf4_gemm(cx, ac, asf, bc, bsf, sh.P, sh.Q, sh.J, g.ao, g.bo, round8(r), C, out_dtype);
  }
  ST_TRY(mxf4_gemm(cx, ac, asf, bc, bsf, sh.P, sh.Q, sh.J, nullptr, nullptr, 0, C, out_dtype));
  if (oe.role == 'P')   // outer rows: C[idx, :] += A[idx, :] . B  (r x Q)
    return bf16_scatter_gemm(cx, g.gath, 1, tb.p, ro.b_kmajor, r, sh.Q, sh.J, C, sh.P, sh.Q, out_dtype, idx, 0);
  // outer cols: C[:, idx] += A . B[:, idx]  (P x r)
  return bf16_scatter_gemm(cx, ta.p, ro.a_kmajor, g.gath, 1, sh.P, r, sh.J, C, sh.P, sh.Q, out_dtype, idx, 1);
}

adahop_status check_plan(const adahop_plan *plan) {
  if (!plan) return ADAHOP_ERR_INVALID_ARG;
  const int pats[3] = {plan->x, plan->w, plan->gy};
  for (int p : pats)
    if (p < 0 || p > 2) return ADAHOP_ERR_INVALID_ARG;
  const int strats[3] = {plan->fwd, plan->dgrad, plan->wgrad};
  for (int s : strats)
    if (s < 0 || s > 4) return ADAHOP_ERR_INVALID_ARG;
  if (plan->oe_rank < 0 || plan->oe_rank > kMaxRank) return ADAHOP_ERR_SHAPE;
  return ADAHOP_OK;
}

adahop_status check_shapes(int64_t M, int64_t N, int64_t K) {
  if (!dim_ok(M) || !dim_ok(N) || !dim_ok(K)) return ADAHOP_ERR_SHAPE;
  return ADAHOP_OK;
}

// Region for G_Y's second orientation written by the dual-orientation pass of a backward call:
// it follows the larger of the dgrad / wgrad layouts.
size_t bwd_alt_offset(int64_t M, int64_t N, int64_t K, int r) {
  const int64_t lines = std::max(std::max(M, N), K);
  const GemmShape shd = shape_of(1, M, N, K), shw = shape_of(2, M, N, K);
  return align256(std::max(gemm_ws(shd.P, shd.Q, shd.J, r, kSizingSms, lines).total,
                           gemm_ws(shw.P, shw.Q, shw.J, r, kSizingSms, lines).total));
}

// Region for the outlier slices both backward GEMMs gather in one launch: after G_Y's second
// orientation; per GEMM (P + Q + J) x r bf16 (A_o P x r, B_o Q x r, outer lines r x J).
size_t bwd_gath_offset(int64_t M, int64_t N, int64_t K, int r) {
  return bwd_alt_offset(M, N, K, r) + align256(static_cast<size_t>(M * N / 2)) + align256(static_cast<size_t>(M * N / 32));
}
struct BwdGath {
  size_t ao[2], bo[2], gath[2];   // offsets for dgrad, wgrad
  size_t end;
  PreGath at(uint8_t *ws, int k) const {
    return PreGath{reinterpret_cast<uint16_t *>(ws + ao[k]), reinterpret_cast<uint16_t *>(ws + bo[k]),
                   reinterpret_cast<uint16_t *>(ws + gath[k])};
  }
};
BwdGath bwd_gath_layout(int64_t M, int64_t N, int64_t K, int r) {
  BwdGath b{};
  size_t off = bwd_gath_offset(M, N, K, r);
  const size_t rr = static_cast<size_t>(round8(std::max(r, 1)));
  for (int k = 0; k < 2; ++k) {
    const GemmShape sh = shape_of(k + 1, M, N, K);
    b.ao[k] = off;
    off += align256(static_cast<size_t>(sh.P) * rr * 2);
    b.bo[k] = off;
    off += align256(static_cast<size_t>(sh.Q) * rr * 2);
    b.gath[k] = off;
    off += align256(static_cast<size_t>(sh.J) * rr * 2);
  }
  b.end = off;
  return b;
}

size_t linear_ws_bytes(int64_t M, int64_t N, int64_t K, int r) {
  size_t b = 0;
  const int64_t lines = std::max(std::max(M, N), K);
  for (int g = 0; g < 3; ++g) {
    const GemmShape sh = shape_of(g, M, N, K);
    b = std::max(b, gemm_ws(sh.P, sh.Q, sh.J, r, kSizingSms, lines).total);
  }
  b = std::max(b, bwd_gath_layout(M, N, K, r).end);
  // calibration statistics: rows + cols floats of the largest tensor
  b = std::max(b, align256(kHeaderBytes + sizeof(float) * static_cast<size_t>(std::max(M, N) + std::max(N, K)) + 256));
  return b;
}

double lower_median_ratio(const std::vector<float> &v) {
  float top = 0.0f;
  for (float x : v) top = std::max(top, x);
  std::vector<float> w(v);
  const size_t k = (w.size() - 1) / 2;
  std::nth_element(w.begin(), w.begin() + k, w.end());
  const double med = w[k];
  if (med > 0) return static_cast<double>(top) / med;
  return top == 0.0f ? 1.0 : 1e300;
}

adahop_status calibrate_one(const void *T, int64_t rows, int64_t cols, double tau, uint8_t *ws,
                            cudaStream_t s, int *pattern, double *rho_row, double *rho_col) {
  float *row_ms = reinterpret_cast<float *>(ws + kHeaderBytes);
  float *col_ms = row_ms + rows;
  CUDA_TRY(launch_calib_stats(static_cast<const uint16_t *>(T), rows, cols, row_ms, col_ms, s), "calibration stats");
  std::vector<float> hr(rows), hc(cols);
  CUDA_TRY(cudaMemcpyAsync(hr.data(), row_ms, rows * sizeof(float), cudaMemcpyDeviceToHost, s), "stats copy");
  CUDA_TRY(cudaMemcpyAsync(hc.data(), col_ms, cols * sizeof(float), cudaMemcpyDeviceToHost, s), "stats copy");
  CUDA_TRY(cudaStreamSynchronize(s), "stream sync");
  *rho_row = lower_median_ratio(hr);
  *rho_col = lower_median_ratio(hc);
  if (std::max(*rho_row, *rho_col) < tau)
    *pattern = ADAHOP_PAT_NONE;
  else
    *pattern = (*rho_col >= *rho_row) ? ADAHOP_PAT_COL : ADAHOP_PAT_ROW;
  return ADAHOP_OK;
}

int strategy_for_pair(int pa, int pb) {
  if (pa == ADAHOP_PAT_COL && pb == ADAHOP_PAT_NONE) return ADAHOP_IHT;
  if (pa == ADAHOP_PAT_NONE && pb == ADAHOP_PAT_NONE) return ADAHOP_IHT;
  if (pa == ADAHOP_PAT_ROW && (pb == ADAHOP_PAT_COL || pb == ADAHOP_PAT_NONE)) return ADAHOP_OE_LEFT;
  if (pa == ADAHOP_PAT_NONE && pb == ADAHOP_PAT_COL) return ADAHOP_OE_RIGHT;
  return ADAHOP_BF16;
}

adahop_status linear_common(const adahop_plan *plan, int64_t M, int64_t N, int64_t K, void *workspace,
                            size_t ws_bytes, DeviceInfo *di) {
  ST_TRY(check_plan(plan));
  ST_TRY(check_shapes(M, N, K));
  if (!workspace) return ADAHOP_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return ADAHOP_ERR_ALIGN;
  if (ws_bytes < linear_ws_bytes(M, N, K, plan->oe_rank)) return ADAHOP_ERR_WORKSPACE;
  // FOID draws r lines from M, N or K
  if (plan->oe_rank > std::min(std::min(M, N), K)) return ADAHOP_ERR_SHAPE;
  ST_TRY(device_info(di));
  return ADAHOP_OK;
}

// Saved context (AdaHOP appendix, IHT and Quantization: the forward pass saves quantised
// operands for the backward pass).  X quantised in the wgrad orientation (lines = K columns,
// J = M) and W in the dgrad orientation (lines = K columns, J = N), codes then tensor-core scales,
// each present only when that backward GEMM quantises (strategy other than BF16).
struct SavedLayout {
  bool has_x = false, has_w = false;
  size_t x_codes = 0, x_sf = 0, w_codes = 0, w_sf = 0, total = 0;
};
SavedLayout saved_layout(const adahop_plan *plan, int64_t M, int64_t N, int64_t K) {
  SavedLayout l;
  l.has_x = plan->wgrad != ADAHOP_BF16;
  l.has_w = plan->dgrad != ADAHOP_BF16;
  size_t off = 0;
  if (l.has_x) {
    l.x_codes = off;
    off += align256(static_cast<size_t>(K * M / 2));
    l.x_sf = off;
    off += align256(static_cast<size_t>(K * M / 32));
  }
  if (l.has_w) {
    l.w_codes = off;
    off += align256(static_cast<size_t>(K * N / 2));
    l.w_sf = off;
    off += align256(static_cast<size_t>(K * N / 32));
  }
  l.total = off;
  return l;
}

// The lines a backward GEMM zeroes in a stored tensor before quantising it: -1 none, else the
// axis (0 rows, 1 columns) of the tensor whose FOID lines are zeroed.
int zero_axis(int gemm, int strategy, int r, const int pats[3], int tensor) {
  if (r <= 0 || (strategy != ADAHOP_OE_LEFT && strategy != ADAHOP_OE_RIGHT)) return -1;
  const OeChoice c = oe_choice(gemm, strategy, pats);
  return c.tensor == tensor ? c.axis : -1;
}

// Quantises one stored tensor into a saved orientation on its own (when the forward pass cannot
// write it from its own quantisation): FOID on the tensor if the backward GEMM zeroes its lines,
// then the quantiser along the stored rows (inner axis 0).
adahop_status quantise_saved(const Ctx &cx, const Tensor &src, int zaxis, int r, int hadamard, uint8_t *codes,
                             uint8_t *sf) {
  uint32_t *mask = reinterpret_cast<uint32_t *>(cx.ws + cx.lay.mask);
  if (zaxis >= 0)
    CUDA_TRY(launch_foid(src.p, src.rows, src.cols, zaxis, r, reinterpret_cast<int32_t *>(cx.ws + cx.lay.idx), mask,
                         cx.ws + cx.lay.foid, cx.foid_counter(), cx.s),
             "foid");
  QuantArgs q{};
  q.T = src.p; q.rows = src.rows; q.cols = src.cols;
  q.zero_rows = zaxis == 0 ? mask : nullptr;
  q.zero_cols = zaxis == 1 ? mask : nullptr;
  q.codes = codes; q.scales = sf;
  q.hadamard = hadamard;
  q.scale_layout = 1;
  CUDA_TRY(launch_quant(q, 0, cx.num_sms, cx.s), "quantise saved operand");
  return ADAHOP_OK;
}

// Backward pass; `saved` (may be null) holds X / W already quantised in the backward orientations.
adahop_status linear_bwd_impl(const adahop_plan *plan, const void *GY, const void *X, const void *W, int64_t M,
                              int64_t N, int64_t K, void *dX, void *dW, int out_dtype, void *workspace,
                              size_t ws_bytes, cudaStream_t s, const uint8_t *saved) {
  DeviceInfo di;
  ST_TRY(linear_common(plan, M, N, K, workspace, ws_bytes, &di));
  const Tensor t[3] = {{static_cast<const uint16_t *>(X), M, K},
                       {static_cast<const uint16_t *>(W), N, K},
                       {static_cast<const uint16_t *>(GY), M, N}};
  const int pats[3] = {plan->x, plan->w, plan->gy};
  // dgrad and wgrad reuse the workspace in stream order.  Their layouts share the FOID / index /
  // mask prefix, so when both extract the same lines (e.g. Row-wise G_Y: outer rows for dgrad,
  // inner rows for wgrad) FOID runs once.
  const int64_t lines = std::max(std::max(M, N), K);
  const GemmShape shd = shape_of(1, M, N, K), shw = shape_of(2, M, N, K);
  const GemmWs ld = gemm_ws(shd.P, shd.Q, shd.J, plan->oe_rank, kSizingSms, lines);
  const GemmWs lw = gemm_ws(shw.P, shw.Q, shw.J, plan->oe_rank, kSizingSms, lines);
  FoidCache fc;
  const bool share = ld.idx == lw.idx && ld.mask == lw.mask;
  // Prep fusion: when both GEMMs quantise G_Y (dgrad along N, wgrad along M) with the same
  // Hadamard setting and the same outlier mask, one pass over G_Y writes both orientations.
  PreA pre_d{}, pre_w{};
  bool dual = false;
  if (dX && dW && share) {
    const int sd = plan->dgrad, sw = plan->wgrad, r = plan->oe_rank;
    const bool quant_d = sd != ADAHOP_BF16, quant_w = sw != ADAHOP_BF16;
    const int gmask_d = zero_axis(1, sd, r, pats, T_GY), gmask_w = zero_axis(2, sw, r, pats, T_GY);
    dual = quant_d && quant_w && ((sd == ADAHOP_MXFP4) == (sw == ADAHOP_MXFP4)) && gmask_d == gmask_w;
    if (dual) {
      uint8_t *ws = static_cast<uint8_t *>(workspace);
      uint32_t *mask = reinterpret_cast<uint32_t *>(ws + ld.mask);
      if (gmask_d >= 0) {
        CUDA_TRY(launch_foid(t[T_GY].p, M, N, gmask_d, r, reinterpret_cast<int32_t *>(ws + ld.idx), mask,
                             ws + ld.foid, reinterpret_cast<uint32_t *>(ws + kFoidCounterOffset), s),
                 "foid");
        fc = FoidCache{T_GY, gmask_d, r};
      }
      const size_t alt = bwd_alt_offset(M, N, K, r);
      pre_d = PreA{ws + ld.a_codes, ws + ld.a_sf};
      pre_w = PreA{ws + alt, ws + alt + align256(static_cast<size_t>(M * N / 2))};
      QuantArgs q{};
      q.T = t[T_GY].p; q.rows = M; q.cols = N;
      q.zero_rows = gmask_d == 0 ? mask : nullptr;
      q.zero_cols = gmask_d == 1 ? mask : nullptr;
      q.codes = pre_d.codes; q.scales = pre_d.sf;
      q.hadamard = sd != ADAHOP_MXFP4;
      q.scale_layout = 1;
      CUDA_TRY(launch_quant_dual(q, pre_w.codes, pre_w.sf, s), "quantise G_Y (both orientations)");
    }
  }
  // Outlier slices of both GEMMs in one launch, when both extract the lines the shared FOID found
  // (each GEMM's own gathers otherwise).
  PreGath pg[2]{};
  bool pre_gath[2] = {false, false};
  if (fc.tensor >= 0) {
    const BwdGath bl = bwd_gath_layout(M, N, K, plan->oe_rank);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int32_t *idx = reinterpret_cast<const int32_t *>(ws + ld.idx);
    GatherJob jobs[4];
    int n = 0;
    const int strat[2] = {plan->dgrad, plan->wgrad};
    void *const outs[2] = {dX, dW};
    for (int k = 0; k < 2; ++k) {
      if (!outs[k] || (strat[k] != ADAHOP_OE_LEFT && strat[k] != ADAHOP_OE_RIGHT) || plan->oe_rank <= 0) continue;
      const OeChoice oe = oe_choice(k + 1, strat[k], pats);
      if (oe.tensor != fc.tensor || oe.axis != fc.axis) continue;
      pg[k] = bl.at(ws, k);
      pre_gath[k] = true;
      n += oe_gather_jobs(k + 1, oe, t, idx, plan->oe_rank, pg[k], jobs + n);
    }
    CUDA_TRY(launch_gathers(jobs, n, s), "gather outlier slices (both backward GEMMs)");
  }
  const SavedLayout sl = saved ? saved_layout(plan, M, N, K) : SavedLayout{};
  uint8_t *sv = const_cast<uint8_t *>(saved);
  const PreA saved_w{sv + sl.w_codes, sv + sl.w_sf}, saved_x{sv + sl.x_codes, sv + sl.x_sf};
  if (dX) {
    const Ctx cx = linear_ctx(s, workspace, ld, di.num_sms);
    ST_TRY(run_gemm(cx, 1, plan->dgrad, plan->oe_rank, t, pats, dX, out_dtype, share ? &fc : nullptr,
                    dual ? &pre_d : nullptr, sl.has_w ? &saved_w : nullptr, nullptr, nullptr,
                    pre_gath[0] ? &pg[0] : nullptr));
  }
  if (dW) {
    const Ctx cx = linear_ctx(s, workspace, lw, di.num_sms);
    ST_TRY(run_gemm(cx, 2, plan->wgrad, plan->oe_rank, t, pats, dW, out_dtype, share ? &fc : nullptr,
                    dual ? &pre_w : nullptr, sl.has_x ? &saved_x : nullptr, nullptr, nullptr,
                    pre_gath[1] ? &pg[1] : nullptr));
  }
  return ADAHOP_OK;
}

}  // namespace

// =====================================================================================
extern "C" {

void adahop_default_options(adahop_options *opt) {
  if (!opt) return;
  opt->tau = 8.0;
  opt->probe_len = 64;
  opt->oe_rank = 64;
}

const char *adahop_status_string(adahop_status st) {
  switch (st) {
    case ADAHOP_OK: return "ok";
    case ADAHOP_ERR_INVALID_ARG: return "invalid argument";
    case ADAHOP_ERR_SHAPE: return "unsupported shape";
    case ADAHOP_ERR_ALIGN: return "misaligned pointer";
    case ADAHOP_ERR_CUDA: return "CUDA error";
    case ADAHOP_ERR_TIMEOUT: return "device wait timed out";
    case ADAHOP_ERR_UNSUPPORTED: return "unsupported device or feature";
    case ADAHOP_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char *adahop_last_cuda_error(void) { return g_last_cuda_error; }

adahop_status adahop_workspace_size(const adahop_plan *plan, int64_t M, int64_t N, int64_t K, size_t *bytes) {
  if (!bytes) return ADAHOP_ERR_INVALID_ARG;
  ST_TRY(check_plan(plan));
  ST_TRY(check_shapes(M, N, K));
  *bytes = linear_ws_bytes(M, N, K, plan->oe_rank);
  return ADAHOP_OK;
}

adahop_status adahop_calibrate(const void *X, const void *W, const void *GY, int64_t M, int64_t N, int64_t K,
                               const adahop_options *opt, adahop_plan *plan_out, void *workspace,
                               size_t ws_bytes, adahop_stream_t stream) {
  if (!X || !W || !plan_out || !workspace) return ADAHOP_ERR_INVALID_ARG;
  adahop_options o;
  adahop_default_options(&o);
  if (opt) o = *opt;
  if (!(o.tau > 0) || o.probe_len != 64 || o.oe_rank < 0 || o.oe_rank > kMaxRank)
    return ADAHOP_ERR_INVALID_ARG;
  ST_TRY(check_shapes(M, N, K));
  if (!aligned(X, 16) || !aligned(W, 16) || (GY && !aligned(GY, 16)) || !aligned(workspace, 256))
    return ADAHOP_ERR_ALIGN;
  const size_t need = align256(kHeaderBytes + sizeof(float) * static_cast<size_t>(std::max(M, N) + std::max(N, K)) + 256);
  if (ws_bytes < need) return ADAHOP_ERR_WORKSPACE;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  adahop_plan p{};
  int px, pw, pg = ADAHOP_PAT_NONE;
  ST_TRY(calibrate_one(X, M, K, o.tau, ws, s, &px, &p.rho[0], &p.rho[1]));
  ST_TRY(calibrate_one(W, N, K, o.tau, ws, s, &pw, &p.rho[2], &p.rho[3]));
  if (GY) ST_TRY(calibrate_one(GY, M, N, o.tau, ws, s, &pg, &p.rho[4], &p.rho[5]));
  p.x = px; p.w = pw; p.gy = pg;
  p.fwd = strategy_for_pair(px, pw);
  p.dgrad = strategy_for_pair(pg, pw);
  p.wgrad = strategy_for_pair(pg, px);
  p.oe_rank = o.oe_rank;
  *plan_out = p;
  return ADAHOP_OK;
}

adahop_status adahop_linear_fwd(const adahop_plan *plan, const void *X, const void *W, int64_t M, int64_t N,
                                int64_t K, void *Y, adahop_out_dtype out_dtype, void *workspace, size_t ws_bytes,
                                adahop_stream_t stream) {
  if (!X || !W || !Y) return ADAHOP_ERR_INVALID_ARG;
  if (out_dtype != ADAHOP_OUT_BF16 && out_dtype != ADAHOP_OUT_FP32) return ADAHOP_ERR_INVALID_ARG;
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(Y, 16)) return ADAHOP_ERR_ALIGN;
  DeviceInfo di;
  ST_TRY(linear_common(plan, M, N, K, workspace, ws_bytes, &di));
  const GemmShape sh = shape_of(0, M, N, K);
  const Ctx cx = linear_ctx(reinterpret_cast<cudaStream_t>(stream), workspace,
                            gemm_ws(sh.P, sh.Q, sh.J, plan->oe_rank, kSizingSms, std::max(std::max(M, N), K)), di.num_sms);
  const Tensor t[3] = {{static_cast<const uint16_t *>(X), M, K}, {static_cast<const uint16_t *>(W), N, K}, {nullptr, M, N}};
  const int pats[3] = {plan->x, plan->w, plan->gy};
  return run_gemm(cx, 0, plan->fwd, plan->oe_rank, t, pats, Y, out_dtype, nullptr);
}

adahop_status adahop_linear_bwd(const adahop_plan *plan, const void *GY, const void *X, const void *W, int64_t M,
                                int64_t N, int64_t K, void *dX, void *dW, adahop_out_dtype out_dtype, void *workspace,
                                size_t ws_bytes, adahop_stream_t stream) {
  if (!GY || !X || !W || (!dX && !dW)) return ADAHOP_ERR_INVALID_ARG;
  if (out_dtype != ADAHOP_OUT_BF16 && out_dtype != ADAHOP_OUT_FP32) return ADAHOP_ERR_INVALID_ARG;
  if (!aligned(GY, 16) || !aligned(X, 16) || !aligned(W, 16) || (dX && !aligned(dX, 16)) || (dW && !aligned(dW, 16)))
    return ADAHOP_ERR_ALIGN;
  return linear_bwd_impl(plan, GY, X, W, M, N, K, dX, dW, out_dtype, workspace, ws_bytes,
                         reinterpret_cast<cudaStream_t>(stream), nullptr);
}

adahop_status adahop_saved_size(const adahop_plan *plan, int64_t M, int64_t N, int64_t K, size_t *bytes) {
  if (!bytes) return ADAHOP_ERR_INVALID_ARG;
  ST_TRY(check_plan(plan));
  ST_TRY(check_shapes(M, N, K));
  *bytes = saved_layout(plan, M, N, K).total;
  return ADAHOP_OK;
}

adahop_status adahop_linear_fwd_save(const adahop_plan *plan, const void *X, const void *W, int64_t M, int64_t N,
                                     int64_t K, void *Y, adahop_out_dtype out_dtype, void *saved, size_t saved_bytes,
                                     void *workspace, size_t ws_bytes, adahop_stream_t stream) {
  if (!X || !W || !Y) return ADAHOP_ERR_INVALID_ARG;
  if (out_dtype != ADAHOP_OUT_BF16 && out_dtype != ADAHOP_OUT_FP32) return ADAHOP_ERR_INVALID_ARG;
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(Y, 16)) return ADAHOP_ERR_ALIGN;
  DeviceInfo di;
  ST_TRY(linear_common(plan, M, N, K, workspace, ws_bytes, &di));
  const SavedLayout sl = saved_layout(plan, M, N, K);
  if (sl.total > 0 && !saved) return ADAHOP_ERR_INVALID_ARG;
  if (saved && !aligned(saved, 256)) return ADAHOP_ERR_ALIGN;
  if (saved_bytes < sl.total) return ADAHOP_ERR_WORKSPACE;
  const GemmShape sh = shape_of(0, M, N, K);
  const Ctx cx = linear_ctx(reinterpret_cast<cudaStream_t>(stream), workspace,
                            gemm_ws(sh.P, sh.Q, sh.J, plan->oe_rank, kSizingSms, std::max(std::max(M, N), K)), di.num_sms);
  const Tensor t[3] = {{static_cast<const uint16_t *>(X), M, K}, {static_cast<const uint16_t *>(W), N, K}, {nullptr, M, N}};
  const int pats[3] = {plan->x, plan->w, plan->gy};
  const int r = plan->oe_rank;
  uint8_t *sv = static_cast<uint8_t *>(saved);
  const PreA save_x{sv + sl.x_codes, sv + sl.x_sf}, save_w{sv + sl.w_codes, sv + sl.w_sf};
  // X (wgrad's B) and W (dgrad's B) need, in the backward orientation, the zero mask and Hadamard
  // setting of that backward GEMM.  Where those equal the forward GEMM's, the forward
  // quantisation writes both orientations in one pass.
  const int zx_f = zero_axis(0, plan->fwd, r, pats, T_X), zw_f = zero_axis(0, plan->fwd, r, pats, T_W);
  const int zx_b = zero_axis(2, plan->wgrad, r, pats, T_X), zw_b = zero_axis(1, plan->dgrad, r, pats, T_W);
  const bool fwd_quant = plan->fwd != ADAHOP_BF16;
  const bool had_f = plan->fwd != ADAHOP_MXFP4;
  const bool dual_x = sl.has_x && fwd_quant && zx_f == zx_b && had_f == (plan->wgrad != ADAHOP_MXFP4);
  const bool dual_w = sl.has_w && fwd_quant && zw_f == zw_b && had_f == (plan->dgrad != ADAHOP_MXFP4);
  ST_TRY(run_gemm(cx, 0, plan->fwd, r, t, pats, Y, out_dtype, nullptr, nullptr, nullptr, dual_x ? &save_x : nullptr,
                  dual_w ? &save_w : nullptr));
  if (sl.has_x && !dual_x)
    ST_TRY(quantise_saved(cx, t[T_X], zx_b, r, plan->wgrad != ADAHOP_MXFP4, save_x.codes, save_x.sf));
  if (sl.has_w && !dual_w)
    ST_TRY(quantise_saved(cx, t[T_W], zw_b, r, plan->dgrad != ADAHOP_MXFP4, save_w.codes, save_w.sf));
  return ADAHOP_OK;
}

adahop_status adahop_linear_bwd_saved(const adahop_plan *plan, const void *GY, const void *X, const void *W,
                                      const void *saved, size_t saved_bytes, int64_t M, int64_t N, int64_t K,
                                      void *dX, void *dW, adahop_out_dtype out_dtype, void *workspace, size_t ws_bytes,
                                      adahop_stream_t stream) {
  if (!GY || !X || !W || (!dX && !dW)) return ADAHOP_ERR_INVALID_ARG;
  if (out_dtype != ADAHOP_OUT_BF16 && out_dtype != ADAHOP_OUT_FP32) return ADAHOP_ERR_INVALID_ARG;
  if (!aligned(GY, 16) || !aligned(X, 16) || !aligned(W, 16) || (dX && !aligned(dX, 16)) || (dW && !aligned(dW, 16)))
    return ADAHOP_ERR_ALIGN;
  ST_TRY(check_plan(plan));
  ST_TRY(check_shapes(M, N, K));
  const SavedLayout sl = saved_layout(plan, M, N, K);
  if (sl.total > 0 && !saved) return ADAHOP_ERR_INVALID_ARG;
  if (saved && !aligned(saved, 256)) return ADAHOP_ERR_ALIGN;
  if (saved_bytes < sl.total) return ADAHOP_ERR_WORKSPACE;
  static const uint8_t kNone = 0;
  return linear_bwd_impl(plan, GY, X, W, M, N, K, dX, dW, out_dtype, workspace, ws_bytes,
                         reinterpret_cast<cudaStream_t>(stream),
                         saved ? static_cast<const uint8_t *>(saved) : &kNone);
}

adahop_status adahop_get_device_status(void *workspace, adahop_stream_t stream) {
  if (!workspace) return ADAHOP_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  CUDA_TRY(cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s), "status copy");
  CUDA_TRY(cudaStreamSynchronize(s), "stream sync");
  if (word != 0) CUDA_TRY(cudaMemsetAsync(workspace, 0, sizeof(word), s), "status clear");
  if (word & kStatusTimeout) return ADAHOP_ERR_TIMEOUT;
  if (word & kStatusBadArg) return ADAHOP_ERR_INVALID_ARG;
  return ADAHOP_OK;
}

adahop_status adahop_check_bounded_wait(void *workspace, size_t ws_bytes, adahop_stream_t stream) {
  if (!workspace) return ADAHOP_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return ADAHOP_ERR_ALIGN;
  if (ws_bytes < 256) return ADAHOP_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CUDA_TRY(launch_bounded_wait_probe(static_cast<uint32_t *>(workspace), s), "bounded-wait probe launch");
  return ADAHOP_OK;
}

int adahop_probe_ctas(void) {
  DeviceInfo di;
  if (device_info(&di) != ADAHOP_OK) return 0;
  return di.num_sms;
}

adahop_status adahop_probe_mma_rate(int kind, int sf_copies, int n, int64_t iters, uint64_t *out, size_t out_bytes,
                                    void *workspace, size_t ws_bytes, adahop_stream_t stream) {
  if (!out || !workspace || kind < 0 || kind > 3 || (sf_copies != 0 && sf_copies != 1) || (n != 128 && n != 256))
    return ADAHOP_ERR_INVALID_ARG;
  if (iters < 1 || iters > (int64_t(1) << 20)) return ADAHOP_ERR_SHAPE;
  if (!aligned(out, 16) || !aligned(workspace, 256)) return ADAHOP_ERR_ALIGN;
  if (ws_bytes < 256) return ADAHOP_ERR_WORKSPACE;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  if (out_bytes < 3 * sizeof(uint64_t) * static_cast<size_t>(di.num_sms)) return ADAHOP_ERR_WORKSPACE;
  CUDA_TRY(launch_mma_rate_probe(kind, sf_copies, n, iters, out, static_cast<uint32_t *>(workspace), di.num_sms,
                                 reinterpret_cast<cudaStream_t>(stream)),
           "mma rate probe launch");
  return ADAHOP_OK;
}

adahop_status adahop_probe_copy(const void *src, void *dst, size_t bytes, adahop_stream_t stream) {
  if (!dst) return ADAHOP_ERR_INVALID_ARG;
  if (bytes % 16) return ADAHOP_ERR_SHAPE;
  if ((src && !aligned(src, 16)) || !aligned(dst, 16)) return ADAHOP_ERR_ALIGN;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  CUDA_TRY(launch_copy_probe(src, dst, bytes, di.num_sms, reinterpret_cast<cudaStream_t>(stream)), "copy probe launch");
  return ADAHOP_OK;
}

// adahop_foid's workspace: a 256-byte header (the completion counter; zero at the first call,
// left zero by every call) and then the stage-1 candidates.
size_t adahop_foid_workspace_size(int64_t lines, int r) {
  return 256 + align256(foid_scratch_bytes(lines, r));
}

adahop_status adahop_foid(const void *T, int64_t rows, int64_t cols, int axis, int r, int32_t *idx_out,
                          uint32_t *line_mask_out, void *workspace, size_t ws_bytes, adahop_stream_t stream) {
  if (!T || (!idx_out && r > 0) || !workspace || (axis != 0 && axis != 1)) return ADAHOP_ERR_INVALID_ARG;
  if (rows < 64 || cols < 64 || (axis == 0 && cols % 8)) return ADAHOP_ERR_SHAPE;
  const int64_t lines = axis == 0 ? rows : cols;
  if (r < 0 || r > kMaxRank || r > lines) return ADAHOP_ERR_SHAPE;
  if ((lines + 2047) / 2048 * static_cast<int64_t>(r) > 8192) return ADAHOP_ERR_SHAPE;
  if (!aligned(T, 16) || !aligned(workspace, 256)) return ADAHOP_ERR_ALIGN;
  if (ws_bytes < adahop_foid_workspace_size(lines, r)) return ADAHOP_ERR_WORKSPACE;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  CUDA_TRY(launch_foid(static_cast<const uint16_t *>(T), rows, cols, axis, r, idx_out, line_mask_out,
                       static_cast<uint8_t *>(workspace) + 256, static_cast<uint32_t *>(workspace),
                       reinterpret_cast<cudaStream_t>(stream)),
           "foid");
  return ADAHOP_OK;
}

adahop_status adahop_foid_noalloc(const void *T, int64_t rows, int64_t cols, int axis, int r, int32_t *idx_out,
                                  uint32_t *line_mask_out, adahop_stream_t stream) {
  if (!T || (!idx_out && r > 0) || (axis != 0 && axis != 1)) return ADAHOP_ERR_INVALID_ARG;
  if (rows < 64 || cols < 64 || (axis == 0 && cols % 8)) return ADAHOP_ERR_SHAPE;
  const int64_t lines = axis == 0 ? rows : cols;
  if (r < 0 || r > kMaxRank || r > lines) return ADAHOP_ERR_SHAPE;
  // the candidates of stage 1 must fit the fixed device array
  if ((lines + 2047) / 2048 * static_cast<int64_t>(r) > foid_static_capacity()) return ADAHOP_ERR_SHAPE;
  if (!aligned(T, 16)) return ADAHOP_ERR_ALIGN;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  CUDA_TRY(launch_foid_noalloc(static_cast<const uint16_t *>(T), rows, cols, axis, r, idx_out, line_mask_out,
                               reinterpret_cast<cudaStream_t>(stream)),
           "foid (no workspace)");
  return ADAHOP_OK;
}

adahop_status adahop_quantize_mxfp4(const void *T, int64_t rows, int64_t cols, int inner_axis, int hadamard,
                                    const uint32_t *zero_rows_mask, const uint32_t *zero_cols_mask, uint8_t *codes,
                                    uint8_t *scales, int scale_layout, adahop_stream_t stream) {
  if (!T || !codes || !scales || (inner_axis != 0 && inner_axis != 1) || (hadamard != 0 && hadamard != 1) ||
      (scale_layout != 0 && scale_layout != 1))
    return ADAHOP_ERR_INVALID_ARG;
  if (!dim_ok(rows) || !dim_ok(cols)) return ADAHOP_ERR_SHAPE;
  if (!aligned(T, 16) || !aligned(codes, 16) || !aligned(scales, 16)) return ADAHOP_ERR_ALIGN;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  QuantArgs q{};
  q.T = static_cast<const uint16_t *>(T);
  q.rows = rows; q.cols = cols;
  q.zero_rows = zero_rows_mask; q.zero_cols = zero_cols_mask;
  q.codes = codes; q.scales = scales; q.hadamard = hadamard; q.scale_layout = scale_layout;
  CUDA_TRY(launch_quant(q, inner_axis, di.num_sms, reinterpret_cast<cudaStream_t>(stream)), "quantise");
  return ADAHOP_OK;
}

adahop_status adahop_quantize_mxfp4_dual(const void *T, int64_t rows, int64_t cols, int hadamard,
                                         const uint32_t *zero_rows_mask, const uint32_t *zero_cols_mask,
                                         uint8_t *codes_rows, uint8_t *scales_rows, uint8_t *codes_cols,
                                         uint8_t *scales_cols, int scale_layout, adahop_stream_t stream) {
  if (!T || !codes_rows || !scales_rows || !codes_cols || !scales_cols || (hadamard != 0 && hadamard != 1) ||
      (scale_layout != 0 && scale_layout != 1))
    return ADAHOP_ERR_INVALID_ARG;
  if (!dim_ok(rows) || !dim_ok(cols)) return ADAHOP_ERR_SHAPE;
  if (!aligned(T, 16) || !aligned(codes_rows, 16) || !aligned(scales_rows, 16) || !aligned(codes_cols, 16) ||
      !aligned(scales_cols, 16))
    return ADAHOP_ERR_ALIGN;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  QuantArgs q{};
  q.T = static_cast<const uint16_t *>(T);
  q.rows = rows; q.cols = cols;
  q.zero_rows = zero_rows_mask; q.zero_cols = zero_cols_mask;
  q.codes = codes_rows; q.scales = scales_rows; q.hadamard = hadamard; q.scale_layout = scale_layout;
  CUDA_TRY(launch_quant_dual(q, codes_cols, scales_cols, reinterpret_cast<cudaStream_t>(stream)), "quantise (dual)");
  return ADAHOP_OK;
}

adahop_status adahop_gather(const void *T, int64_t rows, int64_t cols, const int32_t *idx, int r, int mode,
                            void *out, adahop_stream_t stream) {
  if (!T || !out || (!idx && r > 0) || mode < 0 || mode > 3) return ADAHOP_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || cols % 32 || r < 0 || r > kMaxRank) return ADAHOP_ERR_SHAPE;
  if (!aligned(T, 16) || !aligned(out, 16)) return ADAHOP_ERR_ALIGN;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  CUDA_TRY(launch_gather(static_cast<const uint16_t *>(T), rows, cols, idx, r, mode, static_cast<uint16_t *>(out),
                         reinterpret_cast<cudaStream_t>(stream)),
           "gather");
  return ADAHOP_OK;
}

size_t adahop_gemm_mxfp4_workspace_size(void) {
  return kHeaderBytes + kSkPartialBytesPerPair * static_cast<size_t>(kSkMaxPairs);
}

adahop_status adahop_gemm_mxfp4(const uint8_t *a_codes, const uint8_t *a_scales, const uint8_t *b_codes,
                                const uint8_t *b_scales, int64_t P, int64_t Q, int64_t J, const void *A_o,
                                const void *B_o, int r, void *C, adahop_out_dtype out_dtype, void *workspace, size_t ws_bytes,
                                adahop_stream_t stream) {
  if (!a_codes || !a_scales || !b_codes || !b_scales || !C || !workspace) return ADAHOP_ERR_INVALID_ARG;
  if (out_dtype != 0 && out_dtype != 1) return ADAHOP_ERR_INVALID_ARG;
  if (!dim_ok(P) || !dim_ok(Q) || !dim_ok(J)) return ADAHOP_ERR_SHAPE;
  if (r < 0 || r > kMaxRank || r % 8 || (r > 0 && (!A_o || !B_o))) return ADAHOP_ERR_SHAPE;
  if (!aligned(a_codes, 16) || !aligned(b_codes, 16) || !aligned(a_scales, 16) || !aligned(b_scales, 16) ||
      !aligned(C, 16) || (A_o && !aligned(A_o, 16)) || (B_o && !aligned(B_o, 16)) || !aligned(workspace, 256))
    return ADAHOP_ERR_ALIGN;
  if (ws_bytes < 256) return ADAHOP_ERR_WORKSPACE;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  Ctx cx{reinterpret_cast<cudaStream_t>(stream), static_cast<uint8_t *>(workspace), GemmWs{}, di.num_sms};
  if (ws_bytes >= adahop_gemm_mxfp4_workspace_size()) {   // room for the stream-K scratch after the header
    cx.lay.sk = kHeaderBytes;
    cx.sk = true;
  }
  return mxf4_gemm(cx, a_codes, a_scales, b_codes, b_scales, P, Q, J, A_o, B_o, r, C, out_dtype);
}

adahop_status adahop_gemm_bf16(const void *A, int a_kmajor, const void *B, int b_kmajor, int64_t P, int64_t Q,
                               int64_t J, void *C, adahop_out_dtype out_dtype, int splits, float *c_partial, void *workspace,
                               size_t ws_bytes, adahop_stream_t stream) {
  if (!A || !B || !workspace || (a_kmajor != 0 && a_kmajor != 1) || (b_kmajor != 0 && b_kmajor != 1))
    return ADAHOP_ERR_INVALID_ARG;
  if (splits < 1 || splits > 64 || (splits > 1 && !c_partial) || (!c_partial && !C)) return ADAHOP_ERR_INVALID_ARG;
  if (out_dtype != 0 && out_dtype != 1) return ADAHOP_ERR_INVALID_ARG;
  if (P <= 0 || Q <= 0 || J <= 0 || Q % 64 || J % 64) return ADAHOP_ERR_SHAPE;
  if (!a_kmajor && P % 64) return ADAHOP_ERR_SHAPE;
  if (!aligned(A, 16) || !aligned(B, 16) || (C && !aligned(C, 16)) || (c_partial && !aligned(c_partial, 16)) ||
      !aligned(workspace, 256))
    return ADAHOP_ERR_ALIGN;
  if (ws_bytes < 256) return ADAHOP_ERR_WORKSPACE;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  Ctx cx{reinterpret_cast<cudaStream_t>(stream), static_cast<uint8_t *>(workspace), GemmWs{}, di.num_sms};
  return bf16_gemm(cx, A, a_kmajor, B, b_kmajor, P, Q, J, C, out_dtype, splits, c_partial);
}

adahop_status adahop_gemm_bf16_scatter_add(const void *A, int a_kmajor, const void *B, int b_kmajor, int64_t P,
                                           int64_t Q, int64_t J, void *C, int64_t c_rows, int64_t c_cols,
                                           adahop_out_dtype out_dtype, const int32_t *idx, int r, int axis, void *workspace,
                                           size_t ws_bytes, adahop_stream_t stream) {
  if (!A || !B || !C || !workspace || (!idx && r > 0) || (a_kmajor != 0 && a_kmajor != 1) ||
      (b_kmajor != 0 && b_kmajor != 1) || (axis != 0 && axis != 1) || (out_dtype != 0 && out_dtype != 1))
    return ADAHOP_ERR_INVALID_ARG;
  if (r < 1 || r > kMaxRank || (axis == 0 ? P != r : Q != r)) return ADAHOP_ERR_SHAPE;
  if (P <= 0 || Q <= 0 || J <= 0 || J % 64 || c_cols % 8 || c_rows <= 0 || c_cols <= 0) return ADAHOP_ERR_SHAPE;
  if (axis == 0 && Q != c_cols) return ADAHOP_ERR_SHAPE;
  if (axis == 1 && P != c_rows) return ADAHOP_ERR_SHAPE;
  if (a_kmajor ? false : P % 64) return ADAHOP_ERR_SHAPE;
  if (b_kmajor ? false : Q % 64) return ADAHOP_ERR_SHAPE;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(workspace, 256)) return ADAHOP_ERR_ALIGN;
  if (ws_bytes < 256) return ADAHOP_ERR_WORKSPACE;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  Ctx cx{reinterpret_cast<cudaStream_t>(stream), static_cast<uint8_t *>(workspace), GemmWs{}, di.num_sms};
  return bf16_scatter_gemm(cx, A, a_kmajor, B, b_kmajor, P, Q, J, C, c_rows, c_cols, out_dtype, idx, axis);
}

adahop_status adahop_scatter_add(void *C, int64_t P, int64_t Q, adahop_out_dtype out_dtype, const float *partial, int splits,
                                 const int32_t *idx, int r, int axis, adahop_stream_t stream) {
  if (!C || !partial || (!idx && r > 0) || (axis != 0 && axis != 1) || splits < 1) return ADAHOP_ERR_INVALID_ARG;
  if (out_dtype != 0 && out_dtype != 1) return ADAHOP_ERR_INVALID_ARG;
  if (P <= 0 || Q <= 0 || r < 0 || r > kMaxRank) return ADAHOP_ERR_SHAPE;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  CUDA_TRY(launch_scatter_add(C, P, Q, out_dtype, partial, splits, idx, r, axis, reinterpret_cast<cudaStream_t>(stream)),
           "scatter-add");
  return ADAHOP_OK;
}

adahop_status adahop_calibration_stats(const void *T, int64_t rows, int64_t cols, float *row_ms, float *col_ms,
                                       adahop_stream_t stream) {
  if (!T || !row_ms || !col_ms) return ADAHOP_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || cols % 8) return ADAHOP_ERR_SHAPE;
  if (!aligned(T, 16)) return ADAHOP_ERR_ALIGN;
  DeviceInfo di;
  ST_TRY(device_info(&di));
  CUDA_TRY(launch_calib_stats(static_cast<const uint16_t *>(T), rows, cols, row_ms, col_ms,
                              reinterpret_cast<cudaStream_t>(stream)),
           "calibration stats");
  return ADAHOP_OK;
}

}  // extern "C"
