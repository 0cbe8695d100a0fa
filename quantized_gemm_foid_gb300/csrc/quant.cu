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
//   * v = x * 2^(127 - byte) (exact power-of-two scaling, |v| < 8); the E2M1 code is v rounded
//     to the nearest E2M1 value, ties to the even code, saturating at 6, sign from v (so -0 and
//     negative values that round to zero give 0x8) -- exactly what cvt.rn.satfinite.e2m1x2.f32
//     computes, two elements per instruction;
//   * an all-zero block stores byte 0 and codes 0.
// The transform and scaling run on packed float32 pairs (add/sub/mul.rn.f32x2, each lane rounded
// as the scalar instruction), which halves the float32 instruction count of the butterflies; at
// HBM rate the two-orientation pass is otherwise bound by float32 issue, not by memory.
// Work distribution (2 B read + 0.53 B written per element and orientation):
//   rows kernel: J = columns.  Each thread takes two 32-blocks of a grid-stride sequence and
//                transforms them side by side in the two float32 lanes: 16-byte loads, all five
//                butterfly stages in registers, 16-byte code stores (a warp's blocks are
//                contiguous, so it stores 512 contiguous bytes).
//   cols kernel: J = rows (the transposed orientation).  A 64 x 128 tile is staged in shared
//                memory; each thread reads a column pair as 32-bit words and transforms one
//                32-row block of both columns side by side in the two lanes; the two threads of
//                a column pair hold its two 32-row blocks, so their code stores fill whole
//                32-byte sectors.
//   dual kernel: both orientations from one staged 64 x 128 tile (described at the kernel).
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

// Eight scaled elements -> eight E2M1 codes, element i in bits 4i..4i+3.
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                           float v5, float v6, float v7) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return out;
}

// Two float32 lanes in one 64-bit register: the packed add / sub / mul instructions round each
// lane exactly like the scalar float32 instruction (round to nearest even, no flush to zero).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Quantises two 32-blocks side by side: p[i] holds element i of block A in its low lane and
// element i of block B in its high lane (zeroed lines already +0).  Per block: optional
// orthonormal block-32 Sylvester Hadamard (butterflies with stride 1, 2, 4, 8, 16, each
// (a, b) -> (a + b, a - b) rounded to float32, then * c), E8M0 scale from the block amax, E2M1
// codes; byte_a / byte_b receive the scale bytes, codes_a / codes_b 16 code bytes (element i in
// nibble i).  An all-zero block gives byte 0 and codes 0.
//
// Every lane sees the same operands in the same order as the scalar definition, so the results
// are identical to it.  Scaling: with y the transformed block, the definition computes
// v = RN(RN(y c) s), s = 2^(127 - byte), and amax = max |RN(y c)| = RN(max |y| c) (rounding is
// monotonic and odd).  Where 2^-100 <= amax <= 2^100, c s is an exact normal float32 and
// RN(y (c s)) equals RN(RN(y c) s) for every y with |y c| >= 2^-126 (power-of-two scaling of
// normal floats is exact and commutes with rounding); smaller |y c| give |v| <= 2^-24 either way,
// i.e. a signed zero code.  So one multiply replaces two there; elsewhere both are done (the
// other lane is multiplied by 1, which is exact).
__device__ __forceinline__ void quantize32x2(uint64_t (&p)[32], int hadamard, uint4 &codes_a, uint4 &codes_b,
                                             uint32_t &byte_a, uint32_t &byte_b) {
  if (hadamard) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if ((i & h) == 0) {
          const uint64_t u = p[i], w = p[i + h];
          p[i] = add2(u, w);
          p[i + h] = sub2(u, w);
        }
      }
    }
  }
  float amax_a = 0.0f, amax_b = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float lo, hi;
    unpack2(p[i], lo, hi);
    amax_a = fmaxf(amax_a, fabsf(lo));
    amax_b = fmaxf(amax_b, fabsf(hi));
  }
  const float c = inv_sqrt32();
  if (hadamard) {
    amax_a = __fmul_rn(amax_a, c);
    amax_b = __fmul_rn(amax_b, c);
  }
  byte_a = mx_scale_byte(amax_a);
  byte_b = mx_scale_byte(amax_b);
  const float s_a = mx_inv_scale(byte_a), s_b = mx_inv_scale(byte_b);
  const bool fast_a = amax_a >= 0x1p-100f && amax_a <= 0x1p100f;
  const bool fast_b = amax_b >= 0x1p-100f && amax_b <= 0x1p100f;
  float m_a = s_a, m_b = s_b;
  if (hadamard) {
    if (!fast_a || !fast_b) {
      const uint64_t pre = pack2(fast_a ? 1.0f : c, fast_b ? 1.0f : c);
#pragma unroll
      for (int i = 0; i < 32; ++i) p[i] = mul2(p[i], pre);
    }
    if (fast_a) m_a = __fmul_rn(c, s_a);
    if (fast_b) m_b = __fmul_rn(c, s_b);
  }
  const uint64_t mm = pack2(m_a, m_b);
  float va[32], vb[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) unpack2(mul2(p[i], mm), va[i], vb[i]);
  if (amax_a > 0.0f) {
    codes_a.x = e2m1x8(va[0], va[1], va[2], va[3], va[4], va[5], va[6], va[7]);
    codes_a.y = e2m1x8(va[8], va[9], va[10], va[11], va[12], va[13], va[14], va[15]);
    codes_a.z = e2m1x8(va[16], va[17], va[18], va[19], va[20], va[21], va[22], va[23]);
    codes_a.w = e2m1x8(va[24], va[25], va[26], va[27], va[28], va[29], va[30], va[31]);
  } else {
    codes_a = make_uint4(0u, 0u, 0u, 0u);
  }
  if (amax_b > 0.0f) {
    codes_b.x = e2m1x8(vb[0], vb[1], vb[2], vb[3], vb[4], vb[5], vb[6], vb[7]);
    codes_b.y = e2m1x8(vb[8], vb[9], vb[10], vb[11], vb[12], vb[13], vb[14], vb[15]);
    codes_b.z = e2m1x8(vb[16], vb[17], vb[18], vb[19], vb[20], vb[21], vb[22], vb[23]);
    codes_b.w = e2m1x8(vb[24], vb[25], vb[26], vb[27], vb[28], vb[29], vb[30], vb[31]);
  } else {
    codes_b = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Zeroes the elements of a block whose bit is set in zmask (element i <-> bit i).
__device__ __forceinline__ void apply_zero_mask(float (&x)[32], uint32_t zmask) {
  if (zmask) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if ((zmask >> i) & 1u) x[i] = 0.0f;
  }
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// bf16 pair word -> packed (low element, high element) as float32.
__device__ __forceinline__ uint64_t unpack_bf16x2(uint32_t w) {
  return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// The bf16 in half H (0 = low, 1 = high) of a pair word, widened exactly to float32.
template <int H>
__device__ __forceinline__ float widen_bf16(uint32_t w) {
  return __uint_as_float(H == 0 ? (w << 16) : (w & 0xFFFF0000u));
}

// Stride-1 butterfly (a, b) -> (RN(a + b), RN(a - b)) with a the bf16 in half H of w, read by the
// mixed-precision add / sub (a widened exactly inside the instruction, then one float32
// rounding: the same result as widening a first), b already float32.  Returns (a + b, a - b).
template <int H>
__device__ __forceinline__ uint64_t bfly1_bf16(uint32_t w, float b) {
  float s, d;
  if (H == 0)
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, l, %3;\n\t}"
        : "=f"(s), "=f"(d) : "r"(w), "f"(b));
  else
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, h, %3;\n\tsub.rn.f32.bf16 %1, h, %3;\n\t}"
        : "=f"(s), "=f"(d) : "r"(w), "f"(b));
  return pack2(s, d);
}

// Quantises one 32-block held as 16 packed registers of adjacent elements, p[j] = (x_{2j},
// x_{2j+1}) (zeroed lines already +0) -- the order of a row of bf16 pairs, so unpacking and the
// final E2M1 conversion need no register shuffling.  Optional orthonormal block-32 Sylvester
// Hadamard: the caller has already applied the stride-1 butterflies (the two lanes of each
// register, taken straight from the bf16 pairs by bfly1_bf16); strides 2, 4, 8, 16 pair p[j]
// with p[j + h/2] two lanes at a time; every lane sees the same operands in the same order as the
// scalar definition, so the results are identical.  Then E8M0 scale from the block amax and E2M1
// codes; returns the scale byte and writes 16 code bytes (element i in nibble i).  An all-zero
// block gives byte 0 and codes 0.
//
// Scaling: with y the transformed block, the definition computes v = RN(RN(y c) s),
// s = 2^(127 - byte), and amax = max |RN(y c)| = RN(max |y| c) (rounding is monotonic and odd).
// Where 2^-100 <= amax <= 2^100, c s is an exact normal float32 and RN(y (c s)) equals
// RN(RN(y c) s) for every y with |y c| >= 2^-126 (power-of-two scaling of normal floats is
// exact and commutes with rounding); smaller |y c| give |v| <= 2^-24 either way, i.e. a signed
// zero code.  So one multiply replaces two there; elsewhere both are done.
__device__ __forceinline__ uint32_t quantize32(uint64_t (&p)[16], int hadamard, uint4 &codes) {
  if (hadamard) {
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if ((j & h) == 0) {
          const uint64_t u = p[j], w = p[j + h];
          p[j] = add2(u, w);
          p[j + h] = sub2(u, w);
        }
      }
    }
  }
  float amax = 0.0f;
  if (hadamard) {
    // last stage (element stride 16); max(|u + w|, |u - w|) = |u| + |w| exactly, and rounding is
    // monotonic and odd, so the block amax is the largest RN(|u| + |w|) over the pairs
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint64_t u = p[j], w = p[j + 8];
      float u0, u1, w0, w1;
      unpack2(u, u0, u1);
      unpack2(w, w0, w1);
      amax = max3(amax, __fadd_rn(fabsf(u0), fabsf(w0)), __fadd_rn(fabsf(u1), fabsf(w1)));
      p[j] = add2(u, w);
      p[j + 8] = sub2(u, w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float lo, hi;
      unpack2(p[j], lo, hi);
      amax = max3(amax, fabsf(lo), fabsf(hi));
    }
  }
  const float c = inv_sqrt32();
  if (hadamard) amax = __fmul_rn(amax, c);
  const uint32_t byte = mx_scale_byte(amax);
  if (!(amax > 0.0f)) {
    codes = make_uint4(0u, 0u, 0u, 0u);
    return byte;
  }
  const float s = mx_inv_scale(byte);
  const bool fast = amax >= 0x1p-100f && amax <= 0x1p100f;
  if (hadamard && !fast) {
    const uint64_t cc = pack2(c, c);
#pragma unroll
    for (int j = 0; j < 16; ++j) p[j] = mul2(p[j], cc);
  }
  const float m = (hadamard && fast) ? __fmul_rn(c, s) : s;
  const uint64_t mm = pack2(m, m);
  float v[32];
#pragma unroll
  for (int j = 0; j < 16; ++j) unpack2(mul2(p[j], mm), v[2 * j], v[2 * j + 1]);
  codes.x = e2m1x8(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
  codes.y = e2m1x8(v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]);
  codes.z = e2m1x8(v[16], v[17], v[18], v[19], v[20], v[21], v[22], v[23]);
  codes.w = e2m1x8(v[24], v[25], v[26], v[27], v[28], v[29], v[30], v[31]);
  return byte;
}

// Scale-byte offset in either layout, in the index type I of the launch.  The cols and dual
// kernels are instantiated for I = int32_t (tensors of fewer than 2^31 elements, so that every
// offset fits) and int64_t: they are bound by instruction issue, and 64-bit address arithmetic
// costs two or more instructions per operation (32-bit offsets: cols 222 -> 209 us, dual 308 ->
// 290 us on a 32768 x 14336 tensor).  The rows kernel keeps 64-bit indices.
template <class I>
__device__ __forceinline__ I sf_offset(int layout, I line, I blk, I J) {
  return layout == 0 ? line * (J >> 5) + blk : tiled_sf_offset<I>(line, blk, J);
}

// ---------------------------------------------------------------------------------------------
// rows kernel: lines = rows of T, J = cols; each thread transforms two 32-blocks (b and
// b + stride of the grid-stride loop) side by side.
// ---------------------------------------------------------------------------------------------
template <class I>
__device__ __forceinline__ void load_row_block(const QuantArgs &a, I blkid, const uint4 (&raw)[4], float (&x)[32]) {
  const I bpr = static_cast<I>(a.cols >> 5);   // 32-blocks per row
  const I row = blkid / bpr;
  const I blk = blkid - row * bpr;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[8 * k + 2 * j] = bf16_bits_to_f32(w[j] & 0xFFFFu);
      x[8 * k + 2 * j + 1] = bf16_bits_to_f32(w[j] >> 16);
    }
  }
  uint32_t zmask = 0;
  if (a.zero_rows && ((a.zero_rows[row >> 5] >> (row & 31)) & 1u)) zmask = 0xFFFFFFFFu;
  if (a.zero_cols) zmask |= a.zero_cols[blk];          // bits of columns 32*blk .. 32*blk+31
  apply_zero_mask(x, zmask);
}

template <class I>
__device__ __forceinline__ void store_row_block(const QuantArgs &a, I blkid, const uint4 &codes, uint32_t byte) {
  const I J = static_cast<I>(a.cols);
  const I bpr = J >> 5;
  const I row = blkid / bpr;
  const I blk = blkid - row * bpr;
  *reinterpret_cast<uint4 *>(a.codes + row * (J >> 1) + (blk << 4)) = codes;
  a.scales[sf_offset<I>(a.scale_layout, row, blk, J)] = static_cast<uint8_t>(byte);
}

// Blocks ba and bb (bb == ba: one block).
template <class I>
__device__ __forceinline__ void quant_rows_pair(const QuantArgs &a, I ba, const uint4 (&ra)[4], I bb,
                                                const uint4 (&rb)[4]) {
  uint64_t p[32];
  {
    float xa[32], xb[32];
    load_row_block(a, ba, ra, xa);
    load_row_block(a, bb, rb, xb);
#pragma unroll
    for (int i = 0; i < 32; ++i) p[i] = pack2(xa[i], xb[i]);
  }
  uint4 ca, cb;
  uint32_t ya, yb;
  quantize32x2(p, a.hadamard, ca, cb, ya, yb);
  store_row_block(a, ba, ca, ya);
  if (bb != ba) store_row_block(a, bb, cb, yb);
}

template <class I>
__global__ void __launch_bounds__(256, 2) quant_rows_kernel(QuantArgs a) {
  const I total = static_cast<I>(a.rows * (a.cols >> 5));
  const I stride = static_cast<I>(gridDim.x) * static_cast<I>(blockDim.x);
  I b = static_cast<I>(blockIdx.x) * static_cast<I>(blockDim.x) + static_cast<I>(threadIdx.x);
  const uint4 *src = reinterpret_cast<const uint4 *>(a.T);
  // two blocks (128 bytes) in flight per thread
  for (; b + stride < total; b += 2 * stride) {
    uint4 r0[4], r1[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) r0[k] = __ldg(src + 4 * b + k);
#pragma unroll
    for (int k = 0; k < 4; ++k) r1[k] = __ldg(src + 4 * (b + stride) + k);
    quant_rows_pair(a, b, r0, b + stride, r1);
  }
  if (b < total) {
    uint4 r0[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) r0[k] = __ldg(src + 4 * b + k);
    quant_rows_pair(a, b, r0, b, r0);
  }
}

// ---------------------------------------------------------------------------------------------
// Shared by the cols and dual kernels: a 64 x 128 tile of bf16 pairs in shared memory, and the
// column-orientation pass over it (J = rows): thread t takes the column pair
// (2 (t % 64), 2 (t % 64) + 1) and the 32-row block t / 64, both columns side by side.  Small
// tiles let six CTAs share an SM, so that some load while others compute.
// ---------------------------------------------------------------------------------------------
constexpr int kColTile = 128;                     // columns per tile
constexpr int kTileRows = 64;                     // rows per tile (two 32-row blocks)
constexpr int kTileThreads = 128;

// 16 bytes global -> shared without passing through registers (cp.async, L1 bypassed); the
// copies a thread issued complete at cp_async_wait_all().
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

template <int PITCH, class I>
__device__ __forceinline__ void load_tile(const QuantArgs &a, I r0, I c0, uint32_t (*tile)[PITCH]) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int k = 0; k < 8; ++k) {                   // 1024 chunks of 16 B, 16 per tile row
    const int chunk = tid + kTileThreads * k;
    const int row = chunk >> 4, cc = (chunk & 15) << 2;   // cc in 32-bit words
    // rows 32..63 rotated by 16 words: the column pass's lane pairs read the same word of rows
    // r and r + 32, which would otherwise share a bank
    cp_async16(&tile[row][(cc + ((row >> 5) << 4)) & 63],
               reinterpret_cast<const uint4 *>(a.T + (r0 + row) * static_cast<I>(a.cols) + c0) + (chunk & 15));
  }
  cp_async_wait_all();
}

template <int PITCH, class I>
__device__ __forceinline__ void quant_tile_cols(const QuantArgs &a, I r0, I c0, const uint32_t (*tile)[PITCH],
                                                uint8_t *codes, uint8_t *scales) {
  const I R = static_cast<I>(a.rows);
  const int tid = threadIdx.x;
  // lane pairs take the two 32-row blocks of one column pair, so each line's two adjacent 16-byte
  // code blocks leave in one full 32-byte sector
  const int cp = tid >> 1;                        // column pair
  const int rb = tid & 1;                         // 32-row block inside the tile
  const int pw = (cp + 16 * rb) & 63;             // its staged word (rows 32..63 rotated)
  const I blk = (r0 >> 5) + rb;
  const I line0 = c0 + 2 * cp;
  uint32_t zr = 0;
  if (a.zero_rows) zr = a.zero_rows[(r0 + 32 * rb) >> 5];
  uint32_t z0 = zr, z1 = zr;
  if (a.zero_cols) {
    const uint32_t zc = a.zero_cols[line0 >> 5];
    if ((zc >> (line0 & 31)) & 1u) z0 = 0xFFFFFFFFu;
    if ((zc >> ((line0 + 1) & 31)) & 1u) z1 = 0xFFFFFFFFu;
  }
  uint64_t p[32];
  {
    float x0[32], x1[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t w = tile[32 * rb + i][pw];
      x0[i] = bf16_bits_to_f32(w & 0xFFFFu);
      x1[i] = bf16_bits_to_f32(w >> 16);
    }
    apply_zero_mask(x0, z0);
    apply_zero_mask(x1, z1);
#pragma unroll
    for (int i = 0; i < 32; ++i) p[i] = pack2(x0[i], x1[i]);
  }
  uint4 c0c, c1c;
  uint32_t y0, y1;
  quantize32x2(p, a.hadamard, c0c, c1c, y0, y1);
  *reinterpret_cast<uint4 *>(codes + line0 * (R >> 1) + (blk << 4)) = c0c;
  *reinterpret_cast<uint4 *>(codes + (line0 + 1) * (R >> 1) + (blk << 4)) = c1c;
  scales[sf_offset<I>(a.scale_layout, line0, blk, R)] = static_cast<uint8_t>(y0);
  scales[sf_offset<I>(a.scale_layout, line0 + 1, blk, R)] = static_cast<uint8_t>(y1);
}

// cols kernel: lines = columns of T, J = rows.
template <class I>
__global__ void __launch_bounds__(kTileThreads, 6) quant_cols_kernel(QuantArgs a) {
  __shared__ __align__(16) uint32_t tile[kTileRows][kColTile / 2];   // bf16 pairs
  const I r0 = static_cast<I>(blockIdx.y) * kTileRows;
  const I c0 = static_cast<I>(blockIdx.x) * kColTile;
  load_tile<kColTile / 2, I>(a, r0, c0, tile);
  __syncthreads();
  quant_tile_cols<kColTile / 2, I>(a, r0, c0, tile, a.codes, a.scales);
}

// ---------------------------------------------------------------------------------------------
// dual kernel: both orientations of one tensor from a single read (prep fusion).  Tile 64 rows x
// 128 cols staged in shared memory with 4-word row padding and rows 32..63 rotated by 16 words
// (conflict-free row reads and column-pair reads), 128 threads, eight CTAs per SM (64 registers:
// the kernel is bound by instruction issue, and more resident warps hide its latencies better
// than six did); each thread quantises two 32-blocks along the tile's rows (J = cols) and one
// 32-row block of each column of a column pair (J = rows).  Lanes are paired so that every
// 16-byte code store has its neighbour in the same 32-byte sector from the adjacent lane.  Same
// arithmetic as the two kernels above.
// ---------------------------------------------------------------------------------------------
constexpr int kDualPitch = kColTile / 2 + 4;     // 32-bit words per staged row

// Staged position of word w (0..63) of tile row `row`: rows 32..63 are rotated by 16 words, so
// that the column pass, whose lane pairs read the same word of rows r and r + 32, hits 32
// distinct banks (with the 4-word row padding alone those two rows share banks).
__device__ __forceinline__ int dual_word(int row, int w) { return (w + ((row >> 5) << 4)) & 63; }

// One 32-row block of column 2 cp + H of the staged tile (rows row0 .. row0 + 31; cp here is
// the staged word, dual_word(row0, pair)) as packed pairs
// of consecutive rows, rows whose bit is set in zmask zeroed (ZM); with the transform (HAD), the
// stride-1 butterflies already applied (bfly1_bf16 on the even row's half word).
template <int H, bool ZM, bool HAD>
__device__ __forceinline__ void dual_col_block(const uint32_t (*tile)[kDualPitch], int row0, int cp, uint32_t zmask,
                                               uint64_t (&p)[16]) {
  constexpr uint32_t kHalf = H ? 0xFFFF0000u : 0x0000FFFFu;   // this column's half of each word
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    uint32_t w0 = tile[row0 + 2 * j][cp], w1 = tile[row0 + 2 * j + 1][cp];
    if (ZM) {
      if ((zmask >> (2 * j)) & 1u) w0 &= ~kHalf;
      if ((zmask >> (2 * j + 1)) & 1u) w1 &= ~kHalf;
    }
    p[j] = HAD ? bfly1_bf16<H>(w0, widen_bf16<H>(w1)) : pack2(widen_bf16<H>(w0), widen_bf16<H>(w1));
  }
}

template <int H>
__device__ __forceinline__ void dual_col_load(const uint32_t (*tile)[kDualPitch], int row0, int cp, uint32_t zmask,
                                              int hadamard, uint64_t (&p)[16]) {
  if (hadamard) {
    if (zmask) dual_col_block<H, true, true>(tile, row0, cp, zmask, p);
    else dual_col_block<H, false, true>(tile, row0, cp, zmask, p);
  } else {
    if (zmask) dual_col_block<H, true, false>(tile, row0, cp, zmask, p);
    else dual_col_block<H, false, false>(tile, row0, cp, zmask, p);
  }
}

// I: index type of the offsets (int32_t when the tensor has fewer than 2^31 elements, so that
// every offset below fits; int64_t otherwise).  32-bit offsets take 6% off the kernel's time: it
// is bound by instruction issue, and 64-bit address arithmetic costs two or more instructions
// per operation.
template <class I>
__global__ void __launch_bounds__(kTileThreads, 8) quant_dual_kernel(QuantArgs a, uint8_t *codes_c, uint8_t *scales_c) {
  __shared__ __align__(16) uint32_t tile[kTileRows][kDualPitch];
  const I R = static_cast<I>(a.rows), C = static_cast<I>(a.cols);
  const I r0 = static_cast<I>(blockIdx.y) * kTileRows;
  const I c0 = static_cast<I>(blockIdx.x) * kColTile;
  const int tid = threadIdx.x;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int chunk = tid + kTileThreads * k;
    const int row = chunk >> 4, cc = (chunk & 15) << 2;
    cp_async16(&tile[row][dual_word(row, cc)], reinterpret_cast<const uint4 *>(a.T + (r0 + row) * C + c0) + (chunk & 15));
  }
  cp_async_wait_all();
  __syncthreads();
  // (1) along the rows: row tid / 2, blocks (tid % 2) and (tid % 2) + 2 of the tile; the two
  // threads of a row store adjacent 16-byte code blocks (one full 32-byte sector) and read
  // disjoint banks
  {
    const int rr = tid >> 1;
    const int rot = (rr >> 5) << 4;
    const I row = r0 + rr;
    const bool zrow = a.zero_rows && ((a.zero_rows[row >> 5] >> (row & 31)) & 1u);
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
      const int bl = (tid & 1) + 2 * b;                // 32-column block inside the tile
      const I blk = (c0 >> 5) + bl;
      uint32_t zmask = zrow ? 0xFFFFFFFFu : 0u;
      if (a.zero_cols) zmask |= a.zero_cols[blk];
      uint32_t u[16];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint4 v = *reinterpret_cast<const uint4 *>(&tile[rr][(16 * bl + 4 * w + rot) & 63]);
        u[4 * w] = v.x;
        u[4 * w + 1] = v.y;
        u[4 * w + 2] = v.z;
        u[4 * w + 3] = v.w;
      }
      if (zmask) {                                    // word j holds elements 2j (low) and 2j + 1
#pragma unroll
        for (int j = 0; j < 16; ++j)
          u[j] &= ~((((zmask >> (2 * j)) & 1u) ? 0xFFFFu : 0u) | (((zmask >> (2 * j + 1)) & 1u) ? 0xFFFF0000u : 0u));
      }
      uint64_t p[16];
      if (a.hadamard) {
#pragma unroll
        for (int j = 0; j < 16; ++j) p[j] = bfly1_bf16<0>(u[j], widen_bf16<1>(u[j]));
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) p[j] = unpack_bf16x2(u[j]);
      }
      uint4 codes;
      const uint32_t byte = quantize32(p, a.hadamard, codes);
      *reinterpret_cast<uint4 *>(a.codes + row * (C >> 1) + (blk << 4)) = codes;
      a.scales[sf_offset<I>(a.scale_layout, row, blk, C)] = static_cast<uint8_t>(byte);
    }
  }
  // (2) along the columns: column pair tid / 2, 32-row block tid % 2; the two threads of a column
  // store its two adjacent 16-byte code blocks (one full sector) and adjacent scale bytes
  {
    const int cp = tid >> 1;
    const int rb = tid & 1;
    const int pw = dual_word(32 * rb, cp);             // staged word of the column pair
    const I blk = (r0 >> 5) + rb;
    uint32_t zr = 0;
    if (a.zero_rows) zr = a.zero_rows[(r0 + 32 * rb) >> 5];
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      const I line = c0 + 2 * cp + h;
      uint32_t zmask = zr;
      if (a.zero_cols && ((a.zero_cols[line >> 5] >> (line & 31)) & 1u)) zmask = 0xFFFFFFFFu;
      uint64_t p[16];
      if (h) dual_col_load<1>(tile, 32 * rb, pw, zmask, a.hadamard, p);
      else dual_col_load<0>(tile, 32 * rb, pw, zmask, a.hadamard, p);
      uint4 codes;
      const uint32_t byte = quantize32(p, a.hadamard, codes);
      *reinterpret_cast<uint4 *>(codes_c + line * (R >> 1) + (blk << 4)) = codes;
      scales_c[sf_offset<I>(a.scale_layout, line, blk, R)] = static_cast<uint8_t>(byte);
    }
  }
}

}  // namespace

cudaError_t launch_quant_dual(const QuantArgs &a, uint8_t *codes_cols, uint8_t *scales_cols, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(a.cols / kColTile), static_cast<unsigned>(a.rows / kTileRows));
  if (a.rows * a.cols < (int64_t(1) << 31))
    quant_dual_kernel<int32_t><<<grid, kTileThreads, 0, s>>>(a, codes_cols, scales_cols);
  else
    quant_dual_kernel<int64_t><<<grid, kTileThreads, 0, s>>>(a, codes_cols, scales_cols);
  return cudaGetLastError();
}

cudaError_t launch_quant(const QuantArgs &a, int inner_axis, int num_sms, cudaStream_t s) {
  const bool small = a.rows * a.cols < (int64_t(1) << 31);   // every offset fits in 32 bits
  if (inner_axis == 1) {
    const int64_t total = a.rows * (a.cols >> 5);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    // (64-bit block indices here: the 32-bit instantiation measured 13% slower on this kernel)
    quant_rows_kernel<int64_t><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  } else {
    dim3 grid(static_cast<unsigned>(a.cols / kColTile), static_cast<unsigned>(a.rows / kTileRows));
    if (small)
      quant_cols_kernel<int32_t><<<grid, kTileThreads, 0, s>>>(a);
    else
      quant_cols_kernel<int64_t><<<grid, kTileThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace adahop
