// k3moe_device.cuh -- device-side helpers shared by the layer's kernels:
// bf16 conversions, the on-device MXFP4 tile format and its two decoders,
// and small warp utilities.
//
// MXFP4 (kimi-k3-mlx README, "Tiers"; K3_ARTIFACT_AUDIT section 4.3): each
// weight is an e2m1 code (bit 3 sign, bits 2..1 exponent with bias 1, bit 0
// mantissa, exponent 0 = subnormal 0.5*m) and every 32 consecutive weights
// along the input dimension share an e8m0 scale 2^(S-127).  In the
// checkpoint, byte i of a row holds element 2i in its low nibble.
//
// On-device tile format ("MXFP4 tile", 4352 bytes): 128 rows x 64 input
// columns of one matrix.
//   bytes [0, 4096): 256 chunks of 16 bytes; chunk (c, r) at (c*128 + r)*16
//     holds row r, input columns [32c, 32c+32) (one scale group).  Within a
//     chunk, 32-bit word j covers columns 8j..8j+7 of the group: its low
//     16 bits hold the nibbles of columns 8j+0, +2, +4, +6 (bits 0-3, 4-7,
//     8-11, 12-15) and its high 16 bits those of columns 8j+1, +3, +5, +7.
//   bytes [4096, 4352): row r's two scale bytes at 4096 + 2r (group 0) and
//     4096 + 2r + 1 (group 1).
// Consecutive threads reading chunk c of consecutive rows touch consecutive
// 16-byte words (coalesced loads, conflict-free shared-memory reads), and
// each 32-bit word decodes into four bf16x2 words of consecutive columns
// with shifts and masks only (decoder 1), or byte by byte with the
// hardware e2m1 converter (decoder 2).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace k3 {

constexpr int kTileRows = 128;
constexpr int kTileCols = 64;
constexpr int kTilePackedBytes = kTileRows * kTileCols / 2;  // 4096
constexpr int kTileBytes = kTilePackedBytes + kTileRows * 2;  // 4352

// ---------------------------------------------------------------- bf16
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// float -> bf16 bits, round to nearest even (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint16_t r;
  asm("{ .reg .b16 t; cvt.rn.bf16.f32 t, %1; mov.b16 %0, t; }" : "=h"(r) : "f"(f));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// ---------------------------------------------------------------- tile format
// Re-layout of one 32-bit tile word from the four checkpoint bytes that hold
// columns 8j..8j+7 (byte b: column 8j+2b in the low nibble, 8j+2b+1 high).
__host__ __device__ __forceinline__ uint32_t tile_word_from_checkpoint(uint32_t b0, uint32_t b1, uint32_t b2,
                                                                       uint32_t b3) {
  uint32_t lo = (b0 & 0xFu) | ((b1 & 0xFu) << 4) | ((b2 & 0xFu) << 8) | ((b3 & 0xFu) << 12);
  uint32_t hi = (b0 >> 4) | ((b1 >> 4) << 4) | ((b2 >> 4) << 8) | ((b3 >> 4) << 12);
  return lo | (hi << 16);
}

// ---------------------------------------------------------------- decoder 1
// Tile word -> four bf16x2 words holding columns (0,1), (2,3), (4,5), (6,7)
// of the word, each value equal to e2m1 * 2^-126: the three magnitude bits
// land on the low exponent bits and the top mantissa bit of a bf16 whose
// exponent bias then contributes 2^-126 (code 1, the e2m1 subnormal 0.5,
// becomes the bf16 subnormal 2^-127).
__device__ __forceinline__ void tile_word_to_bf16x2_raw(uint32_t q, uint32_t o[4]) {
  const uint32_t M = 0x01C001C0u, S = 0x80008000u;
  o[0] = ((q << 6) & M) | ((q << 12) & S);
  o[1] = ((q << 2) & M) | ((q << 8) & S);
  o[2] = ((q >> 2) & M) | ((q << 4) & S);
  o[3] = ((q >> 6) & M) | (q & S);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// bf16x2 multipliers that turn the raw decoder-1 values into
// e2m1 * 2^(S-127).  The raw value carries 2^-126, so the total factor is
// 2^(S-1): one bf16 multiply when S <= 128 (2^(S-1) is a bf16 normal),
// otherwise 2^126 first (exact e2m1) and then 2^(S-127).  Every product is
// exact whenever the result is a bf16 value (scale bytes 0..252); larger
// scales overflow by IEEE rules.  S = 255 (NaN) gives NaN.
struct ScaleMul {
  uint32_t first, second;  // second == 0 means "no second multiply"
};
__device__ __forceinline__ ScaleMul scale_multipliers(uint32_t S) {
  ScaleMul m;
  if (S == 255u) {
    m.first = 0x7FC07FC0u;
    m.second = 0u;
  } else if (S <= 128u) {
    uint32_t e = (S + 126u) << 7;  // bf16 bits of 2^(S-1)
    m.first = e | (e << 16);
    m.second = 0u;
  } else {
    m.first = 0x7E807E80u;  // 2^126
    uint32_t e = S << 7;    // 2^(S-127), S in 129..254
    m.second = e | (e << 16);
  }
  return m;
}

// Exact bf16 values of the 8 columns of one tile word.
__device__ __forceinline__ void tile_word_to_bf16(uint32_t q, const ScaleMul& m, uint32_t o[4]) {
  tile_word_to_bf16x2_raw(q, o);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    o[p] = bf16x2_mul(o[p], m.first);
    if (m.second) o[p] = bf16x2_mul(o[p], m.second);
  }
}

// ---------------------------------------------------------------- decoder 2
// One byte of a tile word -> two e2m1 values (unscaled) as f16x2 with the
// hardware converter; f16 holds every e2m1 value exactly.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "r"(byte));
  return r;
}
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h2) {
  float lo, hi;
  asm("{ .reg .f16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b; }"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
  return make_float2(lo, hi);
}

// The e8m0 scale as an fp32 factor (0 -> the fp32 subnormal 2^-127,
// 255 -> NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t S) {
  if (S == 0u) return __uint_as_float(0x00400000u);
  if (S == 255u) return __uint_as_float(0x7FC00000u);
  return __uint_as_float(S << 23);
}

// Decoder 2 writes, for byte b of a tile word, the columns below (the
// hardware converter puts the low nibble in the low half):
//   byte 0 -> columns (0, 2), byte 1 -> (4, 6), byte 2 -> (1, 3), byte 3 -> (5, 7).
// Kernels that use decoder 2 stage their activations in this order, so that
// value i of the decoded stream multiplies activation i of the staged stream.
__host__ __device__ __forceinline__ int dec2_column_of(int i) {  // i in 0..7 -> column
  // stream order: b0.lo b0.hi b1.lo b1.hi b2.lo b2.hi b3.lo b3.hi
  const int col[8] = {0, 2, 4, 6, 1, 3, 5, 7};
  return col[i];
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
  return ((unsigned long long)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float2 unpack_f32x2(unsigned long long v) {
  return make_float2(__uint_as_float((uint32_t)v), __uint_as_float((uint32_t)(v >> 32)));
}

}  // namespace k3
