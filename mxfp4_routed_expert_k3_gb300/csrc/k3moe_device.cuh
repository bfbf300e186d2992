// k3moe_device.cuh -- device-side helpers shared by the layer's kernels:
// bf16 conversions, the on-device MXFP4 tile format and its decoder, and
// small warp utilities.
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
//     holds row r, input columns [32c, 32c+32) (one scale group); 32-bit
//     word j of the chunk holds columns 8j..8j+7.
//   bytes [4096, 4352): row r's two scale bytes at 4096 + 2r (group 0) and
//     4096 + 2r + 1 (group 1).
// Inside a word the 8 codes are split into sign bit s_i and 3-bit
// magnitude m_i (column i of the word) and placed so that the bf16x2 word of
// columns (2p, 2p+1) is one or two shifts and masks away:
//   m0 @6..8  s0 @15  m1 @22..24 s1 @31        (columns 0,1: already in place)
//   m2 @9..11 s2 @14  m3 @25..27 s3 @30        (>>3 for m, <<1 for s)
//   m4 @0..2  s4 @12  m5 @16..18 s5 @28        (<<6 for m, <<3 for s)
//   m6 @3..5  s6 @13  m7 @19..21 s7 @29        (<<3 for m, <<2 for s)
// Consecutive threads reading chunk c of consecutive rows touch consecutive
// 16-byte words (coalesced loads, conflict-free shared-memory reads).  The
// tile keeps 4.25 bits per weight, like the checkpoint.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include <utility>

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
// One tile word from the four checkpoint bytes holding columns 8j..8j+7
// (byte b: column 8j+2b in the low nibble, 8j+2b+1 in the high nibble).
__host__ __device__ __forceinline__ uint32_t tile_word_from_checkpoint(uint32_t b0, uint32_t b1, uint32_t b2,
                                                                       uint32_t b3) {
  const uint32_t n[8] = {b0 & 0xFu, b0 >> 4, b1 & 0xFu, b1 >> 4, b2 & 0xFu, b2 >> 4, b3 & 0xFu, b3 >> 4};
  const int mpos[8] = {6, 22, 9, 25, 0, 16, 3, 19};
  const int spos[8] = {15, 31, 14, 30, 12, 28, 13, 29};
  uint32_t q = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) q |= ((n[i] & 7u) << mpos[i]) | ((n[i] >> 3) << spos[i]);
  return q;
}

// Tile word -> four bf16x2 words holding columns (0,1), (2,3), (4,5), (6,7),
// each value equal to e2m1 * 2^-126: the three magnitude bits land on the
// low exponent bits and the top mantissa bit of a bf16 whose exponent bias
// then contributes 2^-126 (code 1, the e2m1 subnormal 0.5, becomes the bf16
// subnormal 2^-127).  12 integer operations per 8 weights.
__device__ __forceinline__ void tile_word_to_bf16x2_raw(uint32_t q, uint32_t o[4]) {
  const uint32_t M = 0x01C001C0u, S = 0x80008000u;
  const uint32_t q3 = q << 3;
  o[0] = q & (M | S);
  o[1] = ((q >> 3) & M) | ((q << 1) & S);
  o[2] = ((q << 6) & M) | (q3 & S);
  o[3] = (q3 & M) | ((q << 2) & S);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// bf16x2 multipliers that turn the raw values into e2m1 * 2^(S-127).  The
// raw value carries 2^-126, so the total factor is 2^(S-1): one bf16
// multiply when S <= 128 (2^(S-1) is a bf16 normal), otherwise 2^126 first
// (exact e2m1) and then 2^(S-127).  Every product is exact whenever the
// result is a bf16 value (scale bytes 0..252); larger scales overflow by
// IEEE rules.  S = 255 (NaN) gives NaN.
struct ScaleMul {
  uint32_t first, second;  // second == 0 means "no second multiply"
};
__device__ __forceinline__ ScaleMul scale_multipliers(uint32_t S) {
  ScaleMul m;
  if (S == 255u) {
    m.first = 0x7FC07FC0u;
    m.second = 0u;
  } else if (S <= 128u) {
    const uint32_t e = (S + 126u) << 7;  // bf16 bits of 2^(S-1)
    m.first = e | (e << 16);
    m.second = 0u;
  } else {
    m.first = 0x7E807E80u;  // 2^126
    const uint32_t e = S << 7;  // 2^(S-127), S in 129..254
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

// One scale group (a 16-byte chunk, 32 columns) to 16 bf16x2 words, with a
// single branch on the scale: scale bytes up to 128 (all practical weight
// scales) take one multiply per pair.
__device__ __forceinline__ void group_to_bf16(const uint4& c, uint32_t S, uint32_t v[16]) {
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
  if (S <= 128u) {
    const uint32_t e = (S + 126u) << 7;
    const uint32_t mul = e | (e << 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      tile_word_to_bf16x2_raw(words[q], v + 4 * q);
#pragma unroll
      for (int p = 0; p < 4; ++p) v[4 * q + p] = bf16x2_mul(v[4 * q + p], mul);
    }
  } else {
    const ScaleMul m = scale_multipliers(S);
#pragma unroll
    for (int q = 0; q < 4; ++q) tile_word_to_bf16(words[q], m, v + 4 * q);
  }
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
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

// ------------------------------------------------------------------ programmatic dependent launch
// The kernels of a forward after the first are launched with programmatic
// stream serialization, so a kernel's launch and its CTAs' start overlap the
// tail of its predecessor.  pdl_trigger() lets the next kernel launch;
// pdl_wait() blocks until the preceding kernel has completed and its memory
// is visible.  Every CTA of such a kernel calls pdl_wait() before its first
// access to a buffer that another kernel writes or reads, before any early
// exit (so that a kernel never completes ahead of its predecessor, which
// makes the wait cover every earlier kernel) and before allocating TMEM (an
// early-launched CTA holding columns while it waits could starve a CTA of
// the kernel it waits for).  Only static data (weights) may be touched
// before it.  Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialization (see pdl_wait above).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace k3
