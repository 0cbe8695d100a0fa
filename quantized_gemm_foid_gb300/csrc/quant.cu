// K2: outlier-residual zeroing + Inner Hadamard Transform + MXFP4 quantisation.
//
// AdaHOP appendix implementation notes, "IHT and Quantization": the residual tensor (outlier
// lines zeroed, per the FOID paragraph) gets a 1D fast Walsh-Hadamard transform with block
// size 32 along the GEMM's inner dimension, then MXFP4 quantisation with one scale per 32
// elements along that same dimension.
//
// Arithmetic (identical, operation for operation, to the definition it implements):
//   * bf16 -> float32 widening; zeroed lines become +0;
//   * butterflies with stride 1, 2, 4, 8, 16: (a, b) -> (a + b, a - b), each rounded to
//     float32; then x * c with c = float32 nearest 1/sqrt(32) (0x3E3504F3);
//   * amax = max |x| over the block; E8M0 byte = clamp(floor(log2 amax) - 2 + 127, 0, 254),
//     floor(log2) read from the exponent bits (subnormals via the leading mantissa bit);
//   * v = |x| * 2^(127 - byte) (exact power-of-two scaling); the E2M1 magnitude index is
//     counted from the midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 with ties to the even
//     index (strict > before odd indices, >= before even ones); values above 5 saturate to 6;
//   * sign bit = the element's sign bit; an all-zero block stores byte 0 and codes 0.
// Two orientations:
//   rows kernel: J = columns (J-contiguous input); 4 threads per 32-block, 8 elements each,
//                the strides 8 and 16 of the butterfly across lanes via warp shuffles;
//   cols kernel: J = rows (the transposed orientation); a 128 x 128 tile is staged in shared
//                memory and every thread transforms two 32-blocks of one column in registers.
#include "common.cuh"
#include "kernels.cuh"

namespace adahop {

namespace {

constexpr uint32_t kInvSqrt32Bits = 0x3E3504F3u;

__device__ __forceinline__ float inv_sqrt32() { return __uint_as_float(kInvSqrt32Bits); }

__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const uint32_t ex = b >> 23;                 // amax >= 0: sign bit clear
  int e;
  if (ex == 0) {
    const uint32_t man = b & 0x7FFFFFu;
    if (man == 0) return 0u;
    e = (31 - __clz(static_cast<int>(man))) - 149;
  } else {
    e = static_cast<int>(ex) - 127;
  }
  const int byte = e - 2 + 127;
  return static_cast<uint32_t>(byte < 0 ? 0 : (byte > 254 ? 254 : byte));
}

// 2^(127 - byte) as a float; byte <= 252 for any finite float32 amax, so this is normal.
__device__ __forceinline__ float mx_inv_scale(uint32_t byte) {
  return __uint_as_float((254u - byte) << 23);
}

__device__ __forceinline__ uint32_t e2m1_code(float x, float inv_s) {
  const float v = __fmul_rn(fabsf(x), inv_s);
  const uint32_t m = static_cast<uint32_t>(v > 0.25f) + static_cast<uint32_t>(v >= 0.75f) +
                     static_cast<uint32_t>(v > 1.25f) + static_cast<uint32_t>(v >= 1.75f) +
                     static_cast<uint32_t>(v > 2.5f) + static_cast<uint32_t>(v >= 3.5f) +
                     static_cast<uint32_t>(v > 5.0f);
  return m | ((__float_as_uint(x) >> 28) & 8u);
}

__device__ __forceinline__ void butterfly(float &a, float &b) {
  const float s = __fadd_rn(a, b);
  const float d = __fsub_rn(a, b);
  a = s;
  b = d;
}

// In-thread butterflies with stride H over N consecutive elements (N a multiple of 2H).
template <int N, int H>
__device__ __forceinline__ void butterfly_stage(float (&x)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if ((i & H) == 0) butterfly(x[i], x[i + H]);
  }
}

__device__ __forceinline__ void unpack8(const uint4 &raw, float (&x)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = bf16_bits_to_f32(w[k] & 0xFFFFu);
    x[2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
  }
}

__device__ __forceinline__ void store_scale(uint8_t *scales, int layout, int64_t line, int64_t blk,
                                            int64_t J, uint32_t byte) {
  const int64_t off = layout == 0 ? line * (J >> 5) + blk : tiled_sf_offset(line, blk, J);
  scales[off] = static_cast<uint8_t>(byte);
}

// ---------------------------------------------------------------------------------------------
// rows kernel: lines = rows of T, J = cols.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void quant_rows_chunk(const QuantArgs &a, int64_t chunk, uint4 raw,
                                                 uint32_t gmask, int sub) {
  const int64_t J = a.cols;
  const int64_t cpr = J >> 3;                  // 8-element chunks per row
  const int64_t row = chunk / cpr;
  const int64_t col0 = (chunk - row * cpr) << 3;
  float x[8];
  unpack8(raw, x);
  bool zero_all = false;
  if (a.zero_rows) zero_all = (a.zero_rows[row >> 5] >> (row & 31)) & 1u;
  uint32_t zc = 0;
  if (a.zero_cols) zc = (a.zero_cols[col0 >> 5] >> (col0 & 31)) & 0xFFu;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (zero_all || ((zc >> i) & 1u)) x[i] = 0.0f;
  }
  if (a.hadamard) {
    butterfly_stage<8, 1>(x);
    butterfly_stage<8, 2>(x);
    butterfly_stage<8, 4>(x);
    // stride 8: partner lane sub ^ 1; the lower element keeps a + b, the upper b' = a - b
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float y = __shfl_xor_sync(gmask, x[i], 1);
      x[i] = (sub & 1) ? __fsub_rn(y, x[i]) : __fadd_rn(x[i], y);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float y = __shfl_xor_sync(gmask, x[i], 2);
      x[i] = (sub & 2) ? __fsub_rn(y, x[i]) : __fadd_rn(x[i], y);
    }
    const float c = inv_sqrt32();
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(x[i], c);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 2));
  const uint32_t byte = mx_scale_byte(amax);
  uint32_t word = 0;
  if (amax > 0.0f) {
    const float inv_s = mx_inv_scale(byte);
#pragma unroll
    for (int i = 0; i < 8; ++i) word |= e2m1_code(x[i], inv_s) << (4 * i);
  }
  *reinterpret_cast<uint32_t *>(a.codes + row * (J >> 1) + (col0 >> 1)) = word;
  if (sub == 0) store_scale(a.scales, a.scale_layout, row, col0 >> 5, J, byte);
}

__global__ void __launch_bounds__(256) quant_rows_kernel(QuantArgs a) {
  const int64_t total = a.rows * (a.cols >> 3);
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;
  const uint32_t gmask = 0xFu << (lane & ~3);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint4 *src = reinterpret_cast<const uint4 *>(a.T);
  // Two independent chunks in flight per thread.  The four lanes of one 32-block always take
  // the same branch: their chunk indices are 4q..4q+3, and total and stride are multiples of 4.
  for (; c + stride < total; c += 2 * stride) {
    const uint4 r0 = __ldg(src + c);
    const uint4 r1 = __ldg(src + c + stride);
    quant_rows_chunk(a, c, r0, gmask, sub);
    quant_rows_chunk(a, c + stride, r1, gmask, sub);
  }
  if (c < total) quant_rows_chunk(a, c, __ldg(src + c), gmask, sub);
}

// ---------------------------------------------------------------------------------------------
// cols kernel: lines = columns of T, J = rows.  Tile 128 rows x 128 cols, 256 threads.
// ---------------------------------------------------------------------------------------------
constexpr int kColTile = 128;

__global__ void __launch_bounds__(256) quant_cols_kernel(QuantArgs a) {
  __shared__ __align__(16) uint16_t tile[kColTile][kColTile];
  const int64_t R = a.rows, C = a.cols;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kColTile;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kColTile;
  const int tid = threadIdx.x;
  // load 128 x 128 bf16: 2048 chunks of 16 B, 16 per row
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int chunk = tid + 256 * k;
    const int row = chunk >> 4, cc = (chunk & 15) << 3;
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.T + (r0 + row) * C + c0 + cc));
    *reinterpret_cast<uint4 *>(&tile[row][cc]) = v;
  }
  __syncthreads();
  const int c = tid & 127;
  const int half = tid >> 7;                    // rows [64*half, 64*half + 64)
  const int64_t line = c0 + c;
  bool zero_line = false;
  if (a.zero_cols) zero_line = (a.zero_cols[line >> 5] >> (line & 31)) & 1u;
  uint32_t codes_out[8];
  uint32_t bytes_out[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const int rb = 64 * half + 32 * b;          // first row of this block inside the tile
    uint32_t zr = 0;
    if (a.zero_rows) zr = a.zero_rows[(r0 + rb) >> 5];
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float v = bf16_bits_to_f32(tile[rb + i][c]);
      x[i] = (zero_line || ((zr >> i) & 1u)) ? 0.0f : v;
    }
    if (a.hadamard) {
      butterfly_stage<32, 1>(x);
      butterfly_stage<32, 2>(x);
      butterfly_stage<32, 4>(x);
      butterfly_stage<32, 8>(x);
      butterfly_stage<32, 16>(x);
      const float cst = inv_sqrt32();
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = __fmul_rn(x[i], cst);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const uint32_t byte = mx_scale_byte(amax);
    bytes_out[b] = byte;
    const float inv_s = mx_inv_scale(byte);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t word = 0;
      if (amax > 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) word |= e2m1_code(x[8 * w + i], inv_s) << (4 * i);
      }
      codes_out[4 * b + w] = word;
    }
  }
  uint4 *dst = reinterpret_cast<uint4 *>(a.codes + line * (R >> 1) + ((r0 + 64 * half) >> 1));
  dst[0] = make_uint4(codes_out[0], codes_out[1], codes_out[2], codes_out[3]);
  dst[1] = make_uint4(codes_out[4], codes_out[5], codes_out[6], codes_out[7]);
  const int64_t blk = (r0 + 64 * half) >> 5;    // even
  const int64_t off = a.scale_layout == 0 ? line * (R >> 5) + blk : tiled_sf_offset(line, blk, R);
  *reinterpret_cast<uint16_t *>(a.scales + off) =
      static_cast<uint16_t>(bytes_out[0] | (bytes_out[1] << 8));
}

}  // namespace

cudaError_t launch_quant(const QuantArgs &a, int inner_axis, int num_sms, cudaStream_t s) {
  if (inner_axis == 1) {
    const int64_t total = a.rows * (a.cols >> 3);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8 * 2;   // ~2 waves of 8 CTAs/SM
    if (blocks > 2 * cap) blocks = 2 * cap;
    quant_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  } else {
    dim3 grid(static_cast<unsigned>(a.cols / kColTile), static_cast<unsigned>(a.rows / kColTile));
    quant_cols_kernel<<<grid, 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace adahop
