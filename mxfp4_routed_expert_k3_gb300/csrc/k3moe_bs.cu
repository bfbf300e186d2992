// k3moe_bs.cu -- MXFP4 expert GEMMs on the block-scaled tensor cores.
//
// tcgen05.mma with block scaling multiplies two MX operands with one UE8M0
// scale per 32 elements of K on each side and accumulates in fp32:
//   D[m, n] += sum_k (a[m, k] 2^(SA[m, k/32]-127)) (b[n, k] 2^(SB[n, k/32]-127)).
// A is an expert weight exactly as the checkpoint stores it (e2m1 nibbles,
// low nibble first; e8m0 scale per 32 along the input dimension: kimi-k3-mlx
// README, "Tiers"; K3_ARTIFACT_AUDIT section 4.3), so no CUDA-core work
// touches the weights: TMA moves the packed nibbles into shared memory and
// the scales go to tensor memory with tcgen05.cp.
//
// B carries the bf16 activations (latent rows, then h) as block-scaled
// terms with per-32 scales, all terms of a tile stacked into one operand:
//  * prefill tiles (kind::mxf8f6f4, e2m1 A in the 16-byte-slot layout
//    16U4_ALIGN16B): two e4m3 terms, x = q0 2^(S0-127) + q1 2^(S1-127),
//      S0 = max(E - 7, 0) for the block's largest biased bf16 exponent E, so
//           |x| 2^(127-S0) < 2^8 (inside e4m3's range), q0 = RN_e4m3 of that;
//      S1 = max(S0 - 4, 0), q1 = RN_e4m3((x 2^(127-S0) - q0) 2^(S0-S1)).
//    The first term keeps the top 4 significant bits, the remainder has at
//    most 4 more, so the split is exact for every element within 2^13 of
//    its block's largest magnitude; smaller elements keep an absolute error
//    below 2^(S0-127-13).
//  * decode tiles (kind::mxf4, e2m1 A dense with the 64-byte swizzle): six
//    e2m1 terms (see the split below).
//
// Tile scheme: M = 128 weight rows, N = terms x tile rows (one tile of an
// expert's slots: 16 rows at decode, 88 at prefill).  Warp 0 issues the
// copies, warp 1 the MMAs, the remaining warps run the epilogue.  Every wait
// is bounded (status bit + shared abort flag, as in the bf16 kernels).
#include <cuda.h>

#include <algorithm>

#include "k3moe_bs.h"
#include "k3moe_device.cuh"
#include "k3moe_tc.cuh"

namespace k3 {

namespace {

constexpr int kQM = 128;   // weight rows per tile (MMA M)
constexpr int kQK = 128;   // input columns per stage
constexpr int kAtom = 512; // scale bytes per 128 rows x 128 columns
enum BsMode { BS_GATEUP = 0, BS_DOWN = 1 };

// Position of the scale of row r (0..127), group g (0..3) inside an atom:
// 32 rows of 16 bytes; row r % 32 holds the 4 groups of rows r%32, +32,
// +64, +96 in turn.  tcgen05.cp 32x128b.warpx4 puts the 16 bytes of row i
// in TMEM lane i of every lane quarter (4 columns), and the MMA of lane
// quarter q reads column q, byte g (the scale-factor id).
__host__ __device__ __forceinline__ int atom_index(int r, int g) { return (r & 31) * 16 + (r >> 5) * 4 + g; }

// ------------------------------------------------------------------ scales
__global__ void scale_atoms_kernel(const uint8_t* __restrict__ in, int ne, int rows, int cols, int n_mat, int mat,
                                   uint8_t* __restrict__ out) {
  const int G = cols / 32, MT = rows / kQM, KC = cols / kQK;
  const long long total = (long long)ne * rows * G;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int g = (int)(i % G);
    const long long er = i / G;
    const int row = (int)(er % rows);
    const int e = (int)(er / rows);
    const size_t atom = (((size_t)e * MT + row / kQM) * KC + g / 4) * n_mat + mat;
    out[atom * kAtom + atom_index(row % kQM, g % 4)] = in[i];
  }
}

// Packed nibbles [ne][rows][cols/2] -> boxes [ne][rows/128][cols/128][n_mat][128 rows][64 bytes]
// (mat selects the slot), so that every 128 x 128 tile is one contiguous
// 8 KB block and the gate and up tiles of one (row tile, column chunk) are
// adjacent.  Bytes are moved unchanged, 16 at a time.
__global__ void e2m1_boxes_kernel(const uint8_t* __restrict__ in, int ne, int rows, int cols, int n_mat, int mat,
                                  uint8_t* __restrict__ out) {
  const int rb = cols / 2 / 16;  // 16-byte vectors per row
  const int MT = rows / kQM, KC = cols / kQK;
  const long long total = (long long)ne * rows * rb;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int v = (int)(i % rb);
    const long long er = i / rb;
    const int row = (int)(er % rows);
    const int e = (int)(er / rows);
    const size_t box = (((size_t)e * MT + row / kQM) * KC + v / 4) * n_mat + mat;
    reinterpret_cast<uint4*>(out)[(box * kQM + row % kQM) * 4 + (v & 3)] = reinterpret_cast<const uint4*>(in)[i];
  }
}

// ------------------------------------------------------------------ two-term e4m3 split
__device__ __forceinline__ float exp2i(int n) { return __uint_as_float((uint32_t)(n + 127) << 23); }  // |n| <= 126
__device__ __forceinline__ uint32_t to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}
__device__ __forceinline__ float from_e4m3(uint32_t q) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)q));
  float f;
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.f32.f16 %0, lo; }" : "=f"(f) : "r"(h2));
  return f;
}
__device__ __forceinline__ uint32_t term0_scale(uint32_t emax) { return emax >= 255u ? 255u : (uint32_t)max((int)emax - 7, 0); }
__device__ __forceinline__ uint32_t term1_scale(uint32_t s0) { return s0 >= 255u ? 255u : (uint32_t)max((int)s0 - 4, 0); }
// q0 | q1 << 8 for one element (a block with Inf/NaN gets scale 255: NaN)
__device__ __forceinline__ uint32_t split_e4m3(float x, uint32_t s0, uint32_t s1) {
  if (s0 == 255u) return 0u;
  const float xs = x * exp2i(127 - (int)s0);
  const uint32_t q0 = to_e4m3(xs);
  const float r = (xs - from_e4m3(q0)) * exp2i((int)s0 - (int)s1);
  return q0 | (to_e4m3(r) << 8);
}

// ------------------------------------------------------------------ e2m1 term split
// Decode-size tiles carry each activation as kFp4Terms e2m1 terms with their
// own UE8M0 scale per 32-column group: term t quantises what the earlier
// terms left, x = sum_t q_t * 2^(S_t - 127).  The scale puts the group's
// largest remaining magnitude in (3, 6] (6 is the largest e2m1 value), so
// each term shrinks the group's largest residual at least 3x; on the layer's
// activations six terms leave an RMS error near 1e-7 of theirs (four leave
// 1e-4: enough for the layer's output, not for the per-step checks that
// hold h and o to one bf16 ulp and 2e-5).  2^n for n in [-127, 127]
// (2^-127 is subnormal).
constexpr int kFp4Terms = 6;
__device__ __forceinline__ float exp2_any(int n) {
  return n >= -126 ? __uint_as_float((uint32_t)(n + 127) << 23) : __uint_as_float(0x00400000u);
}
// UE8M0 byte of the group whose largest magnitude has the float bits mb
// (255 for Inf/NaN: the MMA then yields NaN).
__device__ __forceinline__ uint32_t e2m1_scale_byte(uint32_t mb) {
  const uint32_t eb = (mb >> 23) & 0xFFu;
  if (eb == 0xFFu) return 255u;
  const int S = (int)eb - 129 + ((mb & 0x7FFFFFu) > 0x400000u ? 1 : 0);  // m 2^e <= 6 * 2^S
  return (uint32_t)(max(S, -127) + 127);
}
// Two e2m1 codes in one byte: lo in bits 0..3, hi in bits 4..7 (round to
// nearest even, saturating at 6).
__device__ __forceinline__ uint32_t to_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// The two values of an e2m1x2 byte (lo nibble -> .x).
__device__ __forceinline__ float2 from_e2m1x2(uint32_t b) {
  uint32_t h2;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(b));
  float lo, hi;
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h; }" : "=f"(lo), "=f"(hi) : "r"(h2));
  return make_float2(lo, hi);
}

// Byte of operand row R's scales (group g added by the caller) among the
// activation atoms of one chunk: rows 0..127 in the first 512-byte atom,
// 128..255 in the second, each at (R%32)*16 + ((R%128)/32)*4 -- row R is
// read from TMEM lane R%32 of column R/32 once the atoms sit in consecutive
// 4-column groups.
__device__ __forceinline__ int act_atom_byte(int R) { return (R >> 7) * kAtom + (R & 31) * 16 + ((R & 127) >> 5) * 4; }
// Term t of row n of a tile of `stack` rows: the terms of a tile form one
// MMA operand, term t of row n being operand row t*stack + n.
__device__ __forceinline__ int act_scale_byte(int t, int n, int stack) { return act_atom_byte(t * stack + n); }

// Slot-ordered rows: dst row s = src row (perm ? perm[s] / K : s), written
// as terms q[C/128][t][rows_max][128]; the scales go to the tile atoms
// sf[tile][C/128][2][512] at act_scale_byte(t, n, stack) + g for row n of
// the tile (slot_tile[s] = tile << 8 | n).  With slot_of the rows are
// tokens instead, each split once and written to its K slots.  A half
// warp covers 128 columns per chunk (8 per lane, 4 lanes per scale group)
// and four chunks of one slot per pass, their loads issued together; the
// loop runs per warp so that both halves always meet at the shuffles.
constexpr int kQuantChunks = 4;
__global__ void quant_rows_kernel(const uint16_t* __restrict__ src, const int* __restrict__ perm, int K, int rows,
                                  const int* __restrict__ rows_dev, int C, int rows_max,
                                  const int* __restrict__ slot_tile, int stack, uint8_t* __restrict__ q,
                                  uint8_t* __restrict__ sf, const int* __restrict__ slot_of,
                                  int* __restrict__ sched) {
  pdl_trigger();
  pdl_wait();
  if (sched && blockIdx.x == 0 && threadIdx.x == 0) sched[0] = sched[1] = 0;  // the expert kernels' item counters
  // slot_of: rows are tokens, each split once and written to its K slots
  // slot_of[t * K + k] (those below *rows_dev with an expert shard)
  const int slot_lim = (slot_of && rows_dev) ? *rows_dev : 0x7FFFFFFF;
  if (rows_dev && !slot_of) rows = min(rows, *rows_dev);  // an expert shard: its own slots only
  const int hl = threadIdx.x & 15, half = (threadIdx.x >> 4) & 1;
  const int KC = C / kQK;
  const int KG = (KC + kQuantChunks - 1) / kQuantChunks;  // chunk groups per row
  const long long nwork = (long long)rows * KG;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long wi = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; 2 * wi < nwork; wi += nwarps) {
    const long long i = 2 * wi + half;
    const bool valid = i < nwork;
    const int s = valid ? (int)(i / KG) : 0, kg = valid ? (int)(i - (long long)s * KG) : 0;
    uint4 v[kQuantChunks];
    int tn = 0;
    if (valid) {
      const int t = perm ? perm[s] / K : s;
      tn = slot_of ? 0 : slot_tile[s];
#pragma unroll
      for (int c = 0; c < kQuantChunks; ++c) {
        const int kc = kg * kQuantChunks + c;
        v[c] = kc < KC ? *reinterpret_cast<const uint4*>(src + (size_t)t * C + kc * kQK + hl * 8)
                       : make_uint4(0u, 0u, 0u, 0u);
      }
    } else {
#pragma unroll
      for (int c = 0; c < kQuantChunks; ++c) v[c] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int c = 0; c < kQuantChunks; ++c) {
      const int kc = kg * kQuantChunks + c;
      const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
      uint32_t e = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) e = max(e, max((w[j] >> 7) & 0xFFu, (w[j] >> 23) & 0xFFu));
      e = max(e, __shfl_xor_sync(0xFFFFFFFFu, e, 1));
      e = max(e, __shfl_xor_sync(0xFFFFFFFFu, e, 2));
      const uint32_t s0 = term0_scale(e), s1 = term1_scale(s0);
      uint32_t a0 = 0, a1 = 0, b0 = 0, b1 = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = split_e4m3(__uint_as_float(w[j] << 16), s0, s1);
        const uint32_t hi = split_e4m3(__uint_as_float(w[j] & 0xFFFF0000u), s0, s1);
        const uint32_t p0 = (lo & 0xFFu) | ((hi & 0xFFu) << 8), p1 = (lo >> 8) | (hi & 0xFF00u);
        if (j < 2) {
          a0 |= p0 << (16 * j);
          a1 |= p1 << (16 * j);
        } else {
          b0 |= p0 << (16 * (j - 2));
          b1 |= p1 << (16 * (j - 2));
        }
      }
      // the four groups' scales of this (slot, chunk) are adjacent bytes of
      // the atom: gather them to lane 0 of the half warp, one 4-byte store per term
      const uint32_t base_lane = threadIdx.x & 16;
      uint32_t w0 = 0, w1 = 0;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        w0 |= __shfl_sync(0xFFFFFFFFu, s0, base_lane + 4 * g) << (8 * g);
        w1 |= __shfl_sync(0xFFFFFFFFu, s1, base_lane + 4 * g) << (8 * g);
      }
      if (!valid || kc >= KC) continue;
      for (int k = 0; k < (slot_of ? K : 1); ++k) {
        const int sl = slot_of ? slot_of[(size_t)s * K + k] : s;
        if (sl >= slot_lim) continue;
        const size_t r0 = (size_t)kc * 2 * rows_max + sl;
        *reinterpret_cast<uint2*>(q + r0 * kQK + hl * 8) = make_uint2(a0, b0);
        *reinterpret_cast<uint2*>(q + (r0 + rows_max) * kQK + hl * 8) = make_uint2(a1, b1);
        if (hl == 0) {
          const int tk = slot_of ? slot_tile[sl] : tn;
          const int n = tk & 0xFF;
          uint8_t* atom = sf + (((size_t)(tk >> 8) * KC + kc) * 2) * kAtom;
          *reinterpret_cast<uint32_t*>(atom + act_scale_byte(0, n, stack)) = w0;
          *reinterpret_cast<uint32_t*>(atom + act_scale_byte(1, n, stack)) = w1;
        }
      }
    }
  }
}

// The same for decode-size tiles (`stack` rows): kFp4Terms e2m1 terms
// q[C/128][kFp4Terms][rows_max][64] (two codes per byte, low nibble first)
// and their scales at act_scale_byte(t, n, stack) + g of the tile's first
// atom, for every slot of the token (slot_of[t * K + k], those below
// *rows_dev with an expert shard).  One CTA per (token, 16 chunks): each
// half warp of the first 256 threads splits one 128-column chunk (8
// columns per lane, 4 lanes per scale group) into shared memory; then each
// of the 384 threads owns one 16-byte piece (chunk, term, quarter of the
// 64-byte row) and stores it for every slot of the token (K <= 32).
constexpr int kTokChunks = 16;
constexpr int kTokThreads = kTokChunks * kFp4Terms * 4;
__global__ void __launch_bounds__(kTokThreads) quant_tok_fp4_kernel(const uint16_t* __restrict__ src, int K, int C,
                                                            const int* __restrict__ rows_dev, int rows_max,
                                                            const int* __restrict__ slot_tile, int stack,
                                                            uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                            const int* __restrict__ slot_of,
                                                            int* __restrict__ sched) {
  __shared__ __align__(16) uint32_t wq[kTokChunks][kFp4Terms][16];  // term words: [chunk][term][lane]
  __shared__ uint32_t wsc[kTokChunks][kFp4Terms];                   // the chunk's four scale bytes per term
  __shared__ int s_sl[32], s_tk[32];
  pdl_trigger();
  pdl_wait();
  if (sched && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    sched[0] = sched[1] = 0;  // the expert kernels' item counters
  const int t = blockIdx.x, kc0 = blockIdx.y * kTokChunks;
  const int KC = C / kQK, nc = min(kTokChunks, KC - kc0);
  const int slot_lim = rows_dev ? *rows_dev : 0x7FFFFFFF;
  if (threadIdx.x < K) {
    const int sl = slot_of[(size_t)t * K + threadIdx.x];
    s_sl[threadIdx.x] = sl;
    s_tk[threadIdx.x] = sl < slot_lim ? slot_tile[sl] : 0;
  }
  const int hw = threadIdx.x >> 4, hl = threadIdx.x & 15;
  const uint32_t base_lane = threadIdx.x & 16;
  const int kc = kc0 + hw;
  // (warps past the first eight only store)
  if (threadIdx.x < 256) {
    const uint4 v = hw < nc ? *reinterpret_cast<const uint4*>(src + (size_t)t * C + kc * kQK + hl * 8)
                            : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float x[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(w[j] << 16);
      x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
#pragma unroll
    for (int tt = 0; tt < kFp4Terms; ++tt) {
      uint32_t mb = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) mb = max(mb, __float_as_uint(fabsf(x[j])));
      mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
      mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
      const uint32_t sb = e2m1_scale_byte(mb);
      uint32_t word = 0;
      if (sb == 255u) {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = 0.f;
      } else {
        const float inv = exp2_any(127 - (int)sb), scl = exp2_any((int)sb - 127);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t b = to_e2m1x2(x[2 * j + 1] * inv, x[2 * j] * inv);
          const float2 d = from_e2m1x2(b);
          x[2 * j] = fmaf(-d.x, scl, x[2 * j]);
          x[2 * j + 1] = fmaf(-d.y, scl, x[2 * j + 1]);
          word |= b << (8 * j);
        }
      }
      // the four groups' scale bytes of this chunk and term, gathered in one word
      uint32_t ws = 0;
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) ws |= __shfl_sync(0xFFFFFFFFu, sb, base_lane + 4 * g4) << (8 * g4);
      if (hw < nc) {
        wq[hw][tt][hl] = word;
        if (hl == 0) wsc[hw][tt] = ws;
      }
    }
  }
  __syncthreads();
  // this thread's piece: chunk c, term tt, bytes 16 part .. 16 part + 15 of the 64-byte row
  const int part = threadIdx.x & 3, tt = (threadIdx.x >> 2) % kFp4Terms, c = threadIdx.x / (4 * kFp4Terms);
  if (c >= nc) return;
  const uint4 piece = *reinterpret_cast<const uint4*>(&wq[c][tt][part * 4]);
  uint8_t* qrow = q + ((size_t)(kc0 + c) * kFp4Terms + tt) * rows_max * 64 + part * 16;
  for (int k = 0; k < K; ++k) {
    const int sl = s_sl[k];
    if (sl < slot_lim) *reinterpret_cast<uint4*>(qrow + (size_t)sl * 64) = piece;
  }
  // the scale words: (chunk c, term tt) of every slot, at the slot's tile atom
  if (part == 0) {
    const uint32_t sw = wsc[c][tt];
    for (int k = 0; k < K; ++k) {
      if (s_sl[k] >= slot_lim) continue;
      const int tk = s_tk[k];
      uint8_t* atom = sf + (((size_t)(tk >> 8) * KC + kc0 + c) * 2) * kAtom;
      *reinterpret_cast<uint32_t*>(atom + act_atom_byte(tt * stack + (tk & 0xFF))) = sw;
    }
  }
}

// ------------------------------------------------------------------ tcgen05 block-scaled pieces
// Shared-memory descriptor of a 32-row x 16-byte scale block (no swizzle,
// 8-row core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)(128u >> 4) << 32) |
         ((uint64_t)1u << 46);
}
__device__ __forceinline__ void tc_cp_scales(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
// Instruction descriptor: kind::mxf8f6f4, A e2m1, B e4m3, both K-major,
// UE8M0 scales, M = 128, N = n (16 or 32), scale-factor ids (byte of the
// scale column).
__device__ __forceinline__ uint32_t bs_idesc(uint32_t sfa_id, uint32_t sfb_id, uint32_t n) {
  return (sfb_id << 4) | (5u << 7) | (0u << 10) | ((n >> 3) << 17) | (1u << 23) | ((uint32_t)(kQM >> 4) << 24) |
         (sfa_id << 29);
}
__device__ __forceinline__ void umma_bs(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %6, 0; "
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(
          d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

// kind::mxf4: A and B e2m1 (type code 1), UE8M0 scales per 32 columns
// (two per row and MMA, K = 64), M = 128, N = n.
__device__ __forceinline__ uint32_t fp4_idesc(uint32_t sfa_id, uint32_t sfb_id, uint32_t n) {
  return (sfb_id << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | (1u << 23) | ((uint32_t)(kQM >> 4) << 24) |
         (sfa_id << 29);
}
__device__ __forceinline__ void umma_fp4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %6, 0; "
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Per stage four copies: the e2m1 tiles (GATEUP: gate and up of one
// 128-column chunk; DOWN: kNK consecutive chunks, or at prefill one chunk of
// two row blocks -- two copies), all activation terms of
// the stage's chunks (one 4-D box), the weight scale atoms and the
// activation scale atoms (bulk copies).  Few large copies per stage keep the
// HBM stream going.  NQ is the tile height:
//   16 (T <= 128): kind::mxf4, six e2m1 activation terms (N = 96), two CTAs
//      per SM with four (gate/up) or three (down) stages; the kernel
//      streams weights;
//    8 (T <= 8, where no expert has more than 8 slots): the same with
//      N = 48; the smaller stages leave room for five (gate/up) or four
//      (down) stages per CTA and two gate/up accumulator buffers;
//   88 (larger batches): kind::mxf8f6f4, two e4m3 terms (N = 176); one
//      CTA per SM with four stages and two accumulators (gate and up, or
//      two row blocks of down: 352 TMEM columns).
template <int MODE, int NQ>
struct BsCfg {
  static constexpr bool kBig = NQ > 32;
  // All activation terms go into one MMA: B rows [term 0 of the NQ tokens;
  // term 1 of the same tokens; ...], N = terms * NQ, and the epilogue adds
  // accumulator columns t * NQ + j.  A block-scaled MMA instruction takes
  // about the same tensor-pipe time for any N up to 192 (measured: 152
  // cycles for kind::mxf8f6f4, 168 for kind::mxf4, one after another on
  // one accumulator), so one MMA per k step and matrix, N as large as the
  // tile allows.
  // Prefill: the two stacked accumulators (2 x 176 columns) need more than
  // a CTA's share of a two-CTA split, so one CTA per SM owns all 512
  // columns, with a deeper ring and two epilogue warpgroups.  Down takes
  // two row blocks of the expert's down matrix per item, two accumulators
  // sharing the stage's activation terms as gate and up do: eight MMAs per
  // stage, where one row block gave four and the issuing thread's per-stage
  // overhead left the pipe idle (one CTA per SM: 4.0 ms; two CTAs of one
  // row block each: 3.1 ms, at T = 8192).  Decode kernels run two CTAs per SM.
  static constexpr bool kWide = kBig;
  static constexpr int kRB = (kBig && MODE == BS_DOWN) ? 2 : 1;  // row blocks per item
  // Decode tiles use tcgen05.mma kind::mxf4: the e2m1 weights sit in shared
  // memory as stored (64-byte rows, half the room of the 16-byte-slot
  // layout kind::mxf8f6f4 reads), so a CTA keeps four stages in flight; the
  // activations are kFp4Terms e2m1 terms (N = 6 * 16 = 96).  Prefill tiles
  // keep kind::mxf8f6f4 with two e4m3 terms (N = 176: more terms would not
  // fit an MMA of N <= 256).
  static constexpr bool kFp4 = !kBig;
  static constexpr int kTerms = kFp4 ? kFp4Terms : 2;
  static constexpr int kRowB = kFp4 ? 64 : 128;  // shared-memory bytes per operand row of a 128-column chunk
  static constexpr int kCtas = kWide ? 1 : 2;                               // CTAs per SM
  static constexpr int kEpiWarps = kWide ? 8 : 4;                           // epilogue warps
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kMats = (MODE == BS_GATEUP) ? 2 : 1;                 // matrices in the weight tensor
  static constexpr int kNumA = kMats * kRB;                                 // accumulators
  static constexpr int kNK = (MODE == BS_GATEUP || kBig) ? 1 : 2;           // 128-column chunks per stage
  static constexpr int kNA = (MODE == BS_GATEUP || kRB == 2) ? 2 : kNK;     // e2m1 tiles per stage
  // tiles per weight copy, adjacent in memory: gate and up, or decode
  // down's kNK consecutive chunks; prefill down's two row blocks are KC
  // tiles apart (two copies)
  static constexpr int kABox = kRB == 2 ? 1 : kNA;
  // one e2m1 tile: dense, or in 16-byte slots (8 data + 8 padding bytes per 16 codes)
  static constexpr int kA = kQM * kRowB;
  static constexpr int kATx = kQM * kQK / 2;  // bytes a tile's copy brings (the packed codes)
  static constexpr int kB = NQ * kRowB;       // one activation term of one chunk
  static constexpr int kOffB = kNA * kA;
  static constexpr int kOffSfa = kOffB + kTerms * kNK * kB;
  static constexpr int kOffSfb = kOffSfa + kNA * kAtom;
  static constexpr int kStageBytes = (kOffSfb + 2 * kNK * kAtom + 1023) / 1024 * 1024;
  static constexpr int kStages = kWide ? 4 : !kFp4 ? 2 : MODE == BS_GATEUP ? (NQ <= 8 ? 5 : 4) : (NQ <= 8 ? 4 : 3);
  // accumulator buffers: one where the stacked accumulators fill the CTA's
  // columns (the epilogue then releases the buffer as soon as it has read it)
  static constexpr int kDBuf = (kBig || (MODE == BS_GATEUP && NQ > 8)) ? 1 : 2;
  static constexpr int kAccW = kTerms * NQ;  // accumulator columns (MMA N)
  static constexpr int kAccStride = (kWide || kFp4) ? kAccW : 128;          // TMEM columns between matrices
  static constexpr int kBufStride = kNumA * kAccStride;                     // TMEM columns between buffers
  static constexpr int kSfBase = (kDBuf - 1) * kBufStride + (kNumA - 1) * kAccStride + kAccW;
  // weight atoms, then the activation atoms: one per chunk holding both
  // terms' rows (stacked), else one per chunk and term
  static constexpr int kSfbAtoms = (kTerms * NQ + 127) / 128;
  static constexpr int kSfCols = 4 * kNA + 4 * kSfbAtoms * kNK;
  static constexpr int kTmemCols = kWide ? 512 : 256;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
  static_assert(kSfBase % 4 == 0 && kSfBase + kStages * kSfCols <= kTmemCols, "TMEM budget");
  static_assert((kNumA == 1 || kAccW <= kAccStride) && kAccW % 16 == 0 && kAccW <= 256, "accumulator width");
  static_assert(kCtas * kTmemCols <= 512, "TMEM per SM");
  static_assert(kB % (8 * kRowB) == 0 && kA % 1024 == 0, "operand blocks must keep their swizzle atoms aligned");
  static_assert(kCtas * (kSmem + 1024) <= 233472, "shared memory per SM");
};

struct BsParams {
  const uint8_t* sfa;  // weight scale atoms
  const uint8_t* sfb;  // activation scale atoms [tile][KC][2][512]
  int MT, KC, KS;      // weight row tiles, 128-column chunks, stages per item
  const int4* tiles;   // {expert, first slot, rows, rows rounded up to 16}
  const int* count;
  int ld_out;          // GATEUP: I, DOWN: L
  int rows_max;        // slot rows of the activation-term planes
  uint16_t* h;         // GATEUP outputs: h (bf16), its terms and scale atoms
  uint8_t* hq;
  uint8_t* hsf;
  float* o;            // DOWN output
  float beta, beta_lin;
  unsigned* status;
  uint64_t limit_ns;
  int withhold_item;   // test hook: the stage of this work item's first k step gets no copies (-1: none)
  // Work distribution: CTA b takes item b first, then the next unclaimed
  // item from this counter (zero when the kernel starts); NULL: items b,
  // b + gridDim.x, ...
  int* next_item;
  // K split (decode tiles): each (tile, row block) is n_split work items over
  // consecutive ranges of the K steps; with n_split > 1 the epilogue writes
  // fp32 partial sums (GATEUP: gate to part_a, up to part_b; DOWN: o to
  // part_a), [n_split][rows_max][ld_out], and a later kernel adds them in
  // part order
  int n_split;
  int part_rows;       // rows of a part plane (the slots: T * K)
  float* part_a;
  float* part_b;
};

// Work item -> (tile, row block, K part) and the part's K-step range.
struct BsItem {
  int ti, mt, part, k0, k1;
};
__device__ __forceinline__ BsItem bs_item(const BsParams& p, int item) {
  BsItem it;
  const int per_tile = p.MT * p.n_split;
  it.ti = item / per_tile;
  const int rem = item - it.ti * per_tile;
  it.mt = rem / p.n_split;
  it.part = rem - it.mt * p.n_split;
  it.k0 = it.part * p.KS / p.n_split;
  it.k1 = (it.part + 1) * p.KS / p.n_split;
  return it;
}

template <int MODE, int NQ>
__global__ void __launch_bounds__(BsCfg<MODE, NQ>::kThreads, BsCfg<MODE, NQ>::kCtas)
    bs_stream_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                     const BsParams p) {
  using C = BsCfg<MODE, NQ>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  // bars: full[S], free[S], dfull[2], dempty[2], drain
  constexpr int NB = 2 * C::kStages + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NB);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // the work item of each ring stage (copy thread -> MMA thread) and of
  // each accumulator buffer (MMA thread -> epilogue); -1 ends the work
  volatile int* stage_item = reinterpret_cast<volatile int*>(tmem_slot + 2);
  volatile int* acc_item = stage_item + C::kStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_trigger();
  pdl_wait();
  const int n_items = *p.count * p.MT * p.n_split;
  if ((int)blockIdx.x >= n_items) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) {
      const bool is_empty = i >= 2 * C::kStages + 2 && i < 2 * C::kStages + 4;
      // dfull: the MMAs' commit and the MMA thread's own arrival (which
      // publishes the buffer's item id)
      const bool is_dfull = i >= 2 * C::kStages && i < 2 * C::kStages + 2;
      mbar_init(smem_u32(bars + i), is_empty ? 32u * C::kEpiWarps : is_dfull ? 2u : 1u);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Guard g{abort_flag, p.status, p.limit_ns};
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto sfree = [&](int s) { return smem_u32(bars + C::kStages + s); };
  auto dfull = [&](int b) { return smem_u32(bars + 2 * C::kStages + b); };
  auto dempty = [&](int b) { return smem_u32(bars + 2 * C::kStages + 2 + b); };
  const uint32_t drain = smem_u32(bars + 2 * C::kStages + 4);
  auto stage = [&](int s) { return smem + (size_t)s * C::kStageBytes; };

  if (warp == 0) {
    // ================= copies
    if (lane == 0) {
      int kg = 0, issued = 0;
      bool ok = true;
      // The next item is claimed two K steps before the current one ends
      // and its tile entry read on the last step, so that the stage after
      // the item's last has its copies ready (a claim and a dependent read
      // at the boundary would leave a stage of the ring empty meanwhile;
      // the copy thread waits for a free stage at those points anyway).
      int4 next_tile = make_int4(0, 0, 0, 0);
      bool have_tile = false;
      for (int item = blockIdx.x, next = -1; item < n_items && ok;) {
        const BsItem bi = bs_item(p, item);
        const int ti = bi.ti, mt = bi.mt;
        const int4 tile = have_tile ? next_tile : p.tiles[ti];
        have_tile = false;
        // (expert, first row block of the item) chunk 0
        const size_t tile0 = ((size_t)tile.x * p.MT * C::kRB + (size_t)mt * C::kRB) * p.KC;
        for (int ks = bi.k0; ks < bi.k1; ++ks, ++kg) {
          const int s = kg % C::kStages, u = kg / C::kStages;
          if (u > 0 && !mbar_wait(sfree(s), (u - 1) & 1, g, 1u)) {
            ok = false;
            break;
          }
          if (ks == max(bi.k0, bi.k1 - 2))
            next = p.next_item ? (int)gridDim.x + atomicAdd(p.next_item, 1) : item + (int)gridDim.x;
          if (ks == bi.k1 - 1 && next < n_items) {
            next_tile = p.tiles[bs_item(p, next).ti];
            have_tile = true;
          }
          const int kc0 = ks * C::kNK;
          const int nk = min(C::kNK, p.KC - kc0);
          // GATEUP: tiles / atoms (kc, gate), (kc, up); DOWN: (kc0) .. (kc0 + kNK - 1),
          // or at prefill (row block, kc) and (row block + 1, kc), KC tiles apart
          const int n_sfa = (MODE == BS_GATEUP || C::kRB == 2) ? 2 : nk;
          const size_t first = (MODE == BS_GATEUP) ? (tile0 + kc0) * 2 : tile0 + kc0;
          stage_item[s] = item;  // published by the arrival below
          if (item == p.withhold_item && ks == bi.k0) {
            // test hook: this stage's full barrier never completes, so the
            // MMA issuer's bounded wait runs out and the CTA aborts
            ++issued;
            continue;
          }
          const uint32_t st = smem_u32(stage(s));
          // the e2m1 copies count their packed bytes; boxes past the end of a
          // tensor are zero-filled and counted in full
          mbar_expect_tx(full(s), (uint32_t)(C::kNA * C::kATx + C::kTerms * C::kNK * C::kB + n_sfa * kAtom +
                                             2 * nk * kAtom));
          if (C::kRB == 2) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              tma_load_3d(st + j * C::kA, &map_a, full(s), 0, 0, (int)(first + (size_t)j * p.KC));
              bulk_load(st + C::kOffSfa + j * kAtom, p.sfa + (first + (size_t)j * p.KC) * kAtom, kAtom, full(s));
            }
          } else {
            tma_load_3d(st, &map_a, full(s), 0, 0, (int)first);
            bulk_load(st + C::kOffSfa, p.sfa + first * kAtom, n_sfa * kAtom, full(s));
          }
          tma_load_4d(st + C::kOffB, &map_b, full(s), 0, tile.y, 0, kc0);
          bulk_load(st + C::kOffSfb, p.sfb + ((size_t)ti * p.KC + kc0) * 2 * kAtom, 2 * nk * kAtom, full(s));
          ++issued;
        }
        item = next;
      }
      if (ok) {
        // the end of the work: a stage without copies whose item is -1
        const int s = kg % C::kStages, u = kg / C::kStages;
        if (u == 0 || mbar_wait(sfree(s), (u - 1) & 1, g, 1u)) {
          stage_item[s] = -1;
          mbar_arrive(full(s));
        }
      }
      if (*abort_flag) {
        for (int k = max(0, issued - C::kStages); k < issued; ++k) {
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(full(k % C::kStages), (k / C::kStages) & 1))
            if (global_ns() - t0 > p.limit_ns) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issue
    // Descriptors are formed once: the start-address field of a shared-memory
    // descriptor is (address >> 4) in its low bits, so every operand of every
    // stage is base + (offset >> 4) with compile-time offsets (the stage ring
    // ends below 256 KB, so the 14-bit field never carries).
    if (lane == 0) {
      const uint32_t st0 = smem_u32(stage(0));
      const uint64_t a_base = C::kFp4 ? umma_desc_sw64(st0) : umma_desc_sw128(st0);
      const uint64_t b_base = C::kFp4 ? umma_desc_sw64(st0 + C::kOffB) : umma_desc_sw128(st0 + C::kOffB);
      const uint64_t sfa_base = sf_desc(st0 + C::kOffSfa);
      const uint64_t sfb_base = sf_desc(st0 + C::kOffSfb);
      int kg = 0, it = 0;
      bool ok = true;
      for (;; ++it) {
        // the item's first stage names it
        if (!mbar_wait(full(kg % C::kStages), (kg / C::kStages) & 1, g, 4u)) {
          ok = false;
          break;
        }
        const int item = stage_item[kg % C::kStages];
        const int buf = (C::kDBuf == 2) ? (it & 1) : 0;
        const int use = (C::kDBuf == 2) ? (it >> 1) : it;  // earlier uses of this buffer
        if (use > 0 && !mbar_wait(dempty(buf), (use - 1) & 1, g, 2u)) {
          ok = false;
          break;
        }
        if (item < 0) {
          // no more work: the end goes on to the epilogue
          acc_item[buf] = -1;
          mbar_arrive(dfull(buf));
          mbar_arrive(dfull(buf));
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + buf * C::kBufStride;
        const uint32_t n = (uint32_t)C::kAccW;  // MMA N: every term of the tile's NQ rows
        const BsItem bi = bs_item(p, item);
        for (int ks = bi.k0; ks < bi.k1; ++ks, ++kg) {
          const int s = kg % C::kStages;
          if (ks > bi.k0 && !mbar_wait(full(s), (kg / C::kStages) & 1, g, 4u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nk = min(C::kNK, p.KC - ks * C::kNK);
          const uint64_t so = (uint64_t)((uint32_t)(s * C::kStageBytes) >> 4);
          const uint64_t a_d = a_base + so, b_d = b_base + so;
          const uint32_t sfc = tmem + C::kSfBase + s * C::kSfCols;
#pragma unroll
          for (int j = 0; j < C::kNA; ++j)
            if (MODE == BS_GATEUP || C::kRB == 2 || j < nk) tc_cp_scales(sfc + 4 * j, sfa_base + so + (j * kAtom >> 4));
          // activation atoms in smem: [chunk][term][512] (stacked: term slot 0 holds both)
#pragma unroll
          for (int c = 0; c < C::kNK; ++c)
#pragma unroll
            for (int t = 0; t < C::kSfbAtoms; ++t)
              if (c < nk)
                tc_cp_scales(sfc + 4 * C::kNA + 4 * (c * C::kSfbAtoms + t), sfb_base + so + ((c * 2 + t) * kAtom >> 4));
          const uint32_t first = ks > bi.k0 ? 1u : 0u;
          if constexpr (C::kFp4) {
            // kind::mxf4: K = 64 per MMA (32 bytes of each 64-byte row), two
            // scale bytes per row and MMA (scale ids 0 and 2)
#pragma unroll
            for (int c = 0; c < C::kNK; ++c) {
              if (c >= nk) break;
#pragma unroll
              for (int kb = 0; kb < kQK / 64; ++kb)
#pragma unroll
                for (int a = 0; a < C::kNumA; ++a) {
                  const int ablk = C::kNumA == 2 ? a : c;
                  umma_fp4(d0 + a * C::kAccStride, a_d + ((ablk * C::kA + kb * 32) >> 4),
                           b_d + ((c * C::kTerms * C::kB + kb * 32) >> 4), fp4_idesc(2 * kb, 2 * kb, n),
                           sfc + 4 * ablk, sfc + 4 * C::kNA + 4 * c, (c | kb) ? 1u : first);
                }
            }
          } else
#pragma unroll
          for (int c = 0; c < C::kNK; ++c) {
            if (c >= nk) break;
#pragma unroll
            for (int kb = 0; kb < kQK / 32; ++kb)
#pragma unroll
              for (int a = 0; a < C::kNumA; ++a) {
                // B blocks of the 4-D box are [chunk][term]: a chunk's terms
                // are one terms*NQ-row operand
                const int ablk = C::kNumA == 2 ? a : c;
                umma_bs(d0 + a * C::kAccStride, a_d + ((ablk * C::kA + kb * 32) >> 4),
                        b_d + ((c * C::kTerms * C::kB + kb * 32) >> 4), bs_idesc(kb, kb, n), sfc + 4 * ablk,
                        sfc + 4 * C::kNA + 4 * c * C::kSfbAtoms, (c | kb) ? 1u : first);
              }
          }
          umma_commit(sfree(s));
        }
        if (!ok) break;
        acc_item[buf] = item;
        mbar_arrive(dfull(buf));
        umma_commit(dfull(buf));
      }
      if (!ok) {
        // MMAs already issued must finish before TMEM is released
        umma_commit(drain);
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(drain, 0))
          if (global_ns() - t0 > p.limit_ns) break;
      }
    }
    __syncwarp();
  } else {
    // ================= epilogue (warps 2..: lane quarter warp % 4; warpgroup
    // wg takes every kEpiWarps/4-th group of 32 token columns)
    const int quarter = warp & 3;
    const int wg = (warp - 2) >> 2;
    constexpr int kWG = C::kEpiWarps / 4;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    for (int it = 0;; ++it) {
      const int buf = (C::kDBuf == 2) ? (it & 1) : 0;
      const int use = (C::kDBuf == 2) ? (it >> 1) : it;
      if (!mbar_wait(dfull(buf), use & 1, g, 8u)) break;
      tc_fence_after();
      const int item = acc_item[buf];
      if (item < 0) break;
      const BsItem bi = bs_item(p, item);
      const int ti = bi.ti, mt = bi.mt;
      const int4 tile = p.tiles[ti];
      const int m = mt * C::kRB * kQM + r;  // output row (of the item's first row block)
      const uint32_t dbase = lane_base + buf * C::kBufStride;
      // Token columns per group: 32, or NQ for decode tiles, whose terms'
      // columns (term t of token j in column t*NQ + j) fit one or two
      // 32-column loads.  Stacked, token j's partial sums are added here.
      constexpr bool kPair = !C::kBig;
      constexpr int JW = kPair ? NQ : 32;
      static_assert(!kPair || ((NQ == 16 || NQ == 8) && C::kTerms == 6), "decode accumulator layout");
      auto load_acc = [&](uint32_t base, int j0, float* v) {
        if constexpr (kPair && NQ == 8) {
          // 16-column block b holds terms 2b and 2b + 1 of the 8 tokens (every
          // load starts at a multiple of its width; the accumulators are 48
          // columns apart); added in the pairs the 16-row tiles use
          float a[16], b[16], c[16];
          tmem_ld16(base, a);
          tmem_ld16(base + 16, b);
          tmem_ld16(base + 32, c);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = (a[j] + a[j + 8]) + (b[j] + b[j + 8]) + (c[j] + c[j + 8]);
        } else if (kPair) {
          // 32-column block b holds terms 2b and 2b + 1 of the NQ tokens
          tmem_ld32(base, v);
#pragma unroll
          for (int j = 0; j < JW; ++j) v[j] += v[j + JW];
#pragma unroll
          for (int b = 1; b < C::kTerms / 2; ++b) {
            float w2[32];
            tmem_ld32(base + 32 * b, w2);
#pragma unroll
            for (int j = 0; j < JW; ++j) v[j] += w2[j] + w2[j + JW];
          }
        } else {
          float w2[32];
          tmem_ld32(base + j0, v);
          tmem_ld32(base + NQ + j0, w2);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] += w2[j];
        }
      };
      // Prefill tiles: the sums of a warpgroup's consecutive tokens (term 0
      // in columns c, term 1 in NQ + c) go to registers, then the
      // accumulator is released before any store.  Warpgroup wg takes
      // tokens [wg * TPW, wg * TPW + n_wg): TPW = the tokens per warpgroup
      // rounded up to a multiple of 8 (the TMEM loads' width), the last
      // warpgroup the rest.
      constexpr int TPW = ((NQ + kWG - 1) / kWG + 7) / 8 * 8;
      const int n_wg = min(TPW, NQ - wg * TPW);
      static_assert(!C::kBig || (NQ % 8 == 0 && (kWG - 1) * TPW < NQ), "token split");
      auto load_sum = [&](uint32_t col, float* v) {
        float t[8];
#pragma unroll
        for (int c = 0; c < TPW; c += 32) {
          if (c + 32 <= TPW && c + 32 <= n_wg)
            tmem_ld32(col + c, v + c);
          else
#pragma unroll
            for (int c8 = c; c8 < TPW && c8 < c + 32; c8 += 8)
              if (c8 < n_wg) tmem_ld8(col + c8, v + c8);
        }
#pragma unroll
        for (int c8 = 0; c8 < TPW; c8 += 8) {
          if (c8 >= n_wg) break;
          tmem_ld8(col + NQ + c8, t);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[c8 + i] += t[i];
        }
      };
      if (!C::kBig && p.n_split > 1) {
        // a K part: fp32 partial sums of the tile's tokens, [part][slot][row]
#pragma unroll 1
        for (int j0 = JW * wg; j0 < NQ; j0 += JW * kWG) {
          float acc[32], up[32];
          load_acc(dbase, j0, acc);
          if (MODE == BS_GATEUP) load_acc(dbase + C::kAccStride, j0, up);
          if (j0 + JW * kWG >= NQ) {
            tc_fence_before();
            mbar_arrive(dempty(buf));
          }
#pragma unroll
          for (int j = 0; j < JW; ++j) {
            if (j0 + j < tile.z) {
              const size_t at = ((size_t)bi.part * p.part_rows + tile.y + j0 + j) * p.ld_out + m;
              p.part_a[at] = acc[j];
              if (MODE == BS_GATEUP) p.part_b[at] = up[j];
            }
          }
        }
      } else if (MODE == BS_GATEUP) {
        // h as bf16 and as the block-scaled terms (and scale atoms) of the down
        // GEMM's B operand, laid out for the down kernel's tiles
        constexpr int kHStack = NQ;  // the down kernel's tiles have the same height
        constexpr bool kHFp4 = BsCfg<BS_DOWN, NQ>::kFp4;
        constexpr int kHTerms = BsCfg<BS_DOWN, NQ>::kTerms;
        const int KCo = p.ld_out / kQK;
        const size_t rb0 = (size_t)((m >> 7) * 2) * p.rows_max, rb1 = rb0 + p.rows_max;  // [KC][2][rows_max]
        const int grp = (m >> 5) & 3;
        uint8_t* atoms = p.hsf + (((size_t)ti * KCo + (m >> 7)) * 2) * kAtom + grp;
        if constexpr (C::kBig) {
          // Each warpgroup takes its consecutive tokens: all their
          // gate and up sums go to registers and the accumulators back to
          // the MMA at once, so the epilogue math overlaps the next item.
          const int t_lo = wg * TPW;
          float gs[TPW], us[TPW];
          load_sum(dbase + t_lo, gs);
          load_sum(dbase + C::kAccStride + t_lo, us);
          tc_fence_before();
          mbar_arrive(dempty(buf));
          uint32_t my_sc[(TPW + 31) / 32] = {};  // lane l keeps the scales of tokens t_lo + 32 i + l
#pragma unroll
          for (int j = 0; j < TPW; ++j) {
            const int jj = t_lo + j;
            if (jj < tile.z) {
              const size_t row = (size_t)(tile.y + jj);
              const uint16_t hb = f32_to_bf16(situ_fast(gs[j], us[j], p.beta, p.beta_lin));
              p.h[row * p.ld_out + m] = hb;
              const uint32_t emax = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(hb >> 7) & 0xFFu);
              const uint32_t s0 = term0_scale(emax), s1 = term1_scale(s0);
              const uint32_t q = split_e4m3(bf16_to_f32(hb), s0, s1);
              p.hq[(rb0 + row) * kQK + (m & 127)] = (uint8_t)q;
              p.hq[(rb1 + row) * kQK + (m & 127)] = (uint8_t)(q >> 8);
              if (lane == (j & 31)) my_sc[j >> 5] = s0 | (s1 << 8);
            }
          }
#pragma unroll
          for (int i = 0; i < (TPW + 31) / 32; ++i) {
            const int jl = 32 * i + lane, jj = t_lo + jl;
            if (jl < TPW && jj < tile.z) {
              atoms[act_scale_byte(0, jj, kHStack)] = (uint8_t)my_sc[i];
              atoms[act_scale_byte(1, jj, kHStack)] = (uint8_t)(my_sc[i] >> 8);
            }
          }
        } else
#pragma unroll 1
        for (int j0 = JW * wg; j0 < NQ; j0 += JW * kWG) {
          float acc[32], up[32];
          load_acc(dbase, j0, acc);
          load_acc(dbase + C::kAccStride, j0, up);
          if (j0 + JW * kWG >= NQ) {
            tc_fence_before();
            mbar_arrive(dempty(buf));
          }
          unsigned long long my_sc = 0;  // lane l keeps the scales of token j0 + l (term t in byte t)
#pragma unroll
          for (int j = 0; j < JW; ++j) {
            const int jj = j0 + j;
            if (jj < tile.z) {
              const size_t row = (size_t)(tile.y + jj);
              const uint16_t hb = f32_to_bf16(situ_fast(acc[j], up[j], p.beta, p.beta_lin));
              p.h[row * p.ld_out + m] = hb;
              if constexpr (kHFp4) {
                // kHTerms e2m1 terms, [KC][kHTerms][rows_max][64]: lane pairs share a byte
                float rr = bf16_to_f32(hb);
                uint32_t qn = 0;
                unsigned long long sc = 0;
#pragma unroll
                for (int t = 0; t < kHTerms; ++t) {
                  const uint32_t sb = e2m1_scale_byte(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(rr))));
                  uint32_t qb = 0;
                  if (sb != 255u) {
                    qb = to_e2m1x2(0.f, rr * exp2_any(127 - (int)sb)) & 0xFu;
                    rr = fmaf(-from_e2m1x2(qb).x, exp2_any((int)sb - 127), rr);
                  } else {
                    rr = 0.f;
                  }
                  qn |= qb << (4 * t);
                  sc |= (unsigned long long)sb << (8 * t);
                }
                const uint32_t qo = __shfl_down_sync(0xFFFFFFFFu, qn, 1);
                if (!(lane & 1)) {
#pragma unroll
                  for (int t = 0; t < kHTerms; ++t)
                    p.hq[(((size_t)(m >> 7) * kHTerms + t) * p.rows_max + row) * 64 + ((m & 127) >> 1)] =
                        (uint8_t)(((qn >> (4 * t)) & 0xFu) | (((qo >> (4 * t)) & 0xFu) << 4));
                }
                if (lane == j) my_sc = sc;
              } else {
                const uint32_t emax = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(hb >> 7) & 0xFFu);
                const uint32_t s0 = term0_scale(emax), s1 = term1_scale(s0);
                const uint32_t q = split_e4m3(bf16_to_f32(hb), s0, s1);
                p.hq[(rb0 + row) * kQK + (m & 127)] = (uint8_t)q;
                p.hq[(rb1 + row) * kQK + (m & 127)] = (uint8_t)(q >> 8);
                if (lane == j) my_sc = s0 | (s1 << 8);
              }
            }
          }
          // lane l stores the scale bytes of token j0 + l (one byte of the
          // group's word per warp and term)
          const int jj = j0 + lane;
          if (lane < JW && jj < tile.z) {
#pragma unroll
            for (int t = 0; t < kHTerms; ++t) atoms[act_scale_byte(t, jj, kHStack)] = (uint8_t)(my_sc >> (8 * t));
          }
        }
      } else if constexpr (C::kBig) {
        // o of the warpgroup's tokens for both row blocks to registers, the
        // accumulators released, then the stores
        static_assert(MODE == BS_GATEUP || (C::kRB == 2 && C::kNumA == 2), "prefill down: two row blocks per item");
        const int t_lo = wg * TPW;
        float o0[TPW], o1[TPW];
        load_sum(dbase + t_lo, o0);
        load_sum(dbase + C::kAccStride + t_lo, o1);
        tc_fence_before();
        mbar_arrive(dempty(buf));
#pragma unroll
        for (int j = 0; j < TPW; ++j) {
          if (t_lo + j < tile.z) {
            float* orow = p.o + (size_t)(tile.y + t_lo + j) * p.ld_out;
            orow[m] = o0[j];
            orow[m + kQM] = o1[j];
          }
        }
      } else {
#pragma unroll 1
        for (int j0 = JW * wg; j0 < NQ; j0 += JW * kWG) {
          float acc[32];
          load_acc(dbase, j0, acc);
          if (j0 + JW * kWG >= NQ) {
            tc_fence_before();
            mbar_arrive(dempty(buf));
          }
#pragma unroll
          for (int j = 0; j < JW; ++j)
            if (j0 + j < tile.z) p.o[(size_t)(tile.y + j0 + j) * p.ld_out + m] = acc[j];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

// ------------------------------------------------------------------ second bank at decode sizes
// Experts of the second bank hold 2-bit affine weights: in every 64-column
// group g of row r, w = s[r, g] q + b[r, g] with q in {0, 1, 2, 3} and bf16
// s, b (kimi-k3-mlx README, "REAP expert pruning": graded mode).  So
//   sum_k w[r, k] x[k] = sum_g ( s[r, g] D[r, g] + b[r, g] X[g] ),
//   D[r, g] = sum_{k in g} q[r, k] x[k],  X[g] = sum_{k in g} x[k].
// q is exact in e2m1 (0, 1, 2, 3 are e2m1 values 0b0000, 0b0010, 0b0100,
// 0b0101), so D is one kind::mxf4 MMA per group (K = 64, the weight scale
// bytes all 127 = 1.0) against the same six-term activation operand the
// first bank's decode tiles use; the epilogue adds the terms' columns and
// applies s and b per group in fp32.  Per 128-column stage: the token terms
// (one 4-D box), the stage's 2-bit tiles (one bulk copy) and the tile's
// activation scale atom.  Warps of their own expand the codes to e2m1
// nibbles in shared memory (64-byte swizzle, the layout the MMA reads; one
// thread per weight row, two chunks in flight), one thread issues the
// MMAs, and four warps (one TMEM lane quarter each, both matrices) run the
// per-group epilogue.  Each group's accumulator alternates between two
// TMEM buffers, so the epilogue of one group overlaps the MMA of the next,
// and expansion, MMAs and epilogue all run at once (with the expansion and
// the epilogue on the same warps, their instruction latencies added up).
constexpr int kB2Tile = 2560;  // one 2-bit tile: 128 rows x 64 codes (16 B a row), then 128 bf16 scales and biases
template <bool GU>
struct B2Cfg {
  static constexpr int kNumMat = GU ? 2 : 1;
  static constexpr int kN = kFp4Terms * kBsDecodeRows;               // MMA N: six terms x 16 rows
  static constexpr int kB = kFp4Terms * kBsDecodeRows * 64;          // activation terms of one chunk
  static constexpr int kSrc = kNumMat * 2 * kB2Tile;                 // the chunk's two groups of 2-bit tiles
  static constexpr int kStage = (kB + kAtom + kSrc + 1023) / 1024 * 1024;
  static constexpr int kRing = GU ? 6 : 7;
  static constexpr int kDec = kNumMat * kQM * 64;                    // e2m1 tiles of one chunk
  static constexpr int kCtas = GU ? 1 : 2;
  static constexpr int kEpiThreads = 128;                            // one weight row (TMEM lane) each
  static constexpr int kExpThreads = 128;                            // one row (every matrix) each
  static constexpr int kXsFloats = kBsDecodeRows * 64;               // the item's per-group row sums (K/64 <= 64)
  static constexpr int kSmem = kRing * kStage + 2 * kDec + kAtom + 4 * kXsFloats + 1024 + 512;
  // TMEM: accumulators (matrix, buffer) at (m * 2 + buf) * kN, the weight
  // scale atom, one activation atom per ring stage
  static constexpr int kSfa = kNumMat * 2 * kN;
  static constexpr int kTmemCols = GU ? 512 : 256;
  static constexpr int kThreads = 64 + kEpiThreads + kExpThreads;   // copies, MMA, epilogue, expand
  static_assert(kSfa + 4 + 4 * kRing <= kTmemCols, "TMEM budget");
  static_assert(kCtas * (kSmem + 1024) <= 233472, "shared memory per SM");
  static_assert(kN % 16 == 0 && kN <= 256, "MMA N");
};

struct B2Params {
  const uint8_t* a_tiles;  // 2-bit tiles [expert][MT][K/64][mats][2560]
  int expert_base;         // weight index of a tile = its expert id - expert_base
  int MT, KC;              // row blocks of 128, chunks of 128 columns
  const int4* tiles;       // tile list; the second bank takes [*begin, *count)
  const int* count;
  const int* begin;
  const uint8_t* sfb;      // activation scale atoms [tile][KC][2][512]
  // per-group sums of the activation rows: GU: xsum [T][K/64] by token
  // (slot -> token through perm / K); DOWN: hsum [slots][K/32] by slot, the
  // two 32-row halves of a group added in order
  const float* xsum;
  const int* perm;
  int K;                   // top-k (slot -> token)
  const float* hsum_in;
  // outputs: GU: h (bf16), its e2m1 terms hq [I/128][6][rows][64] and atoms
  // hsf (the down GEMM's operand), hsum [slots][I/32]; DOWN: o (fp32)
  uint16_t* h;
  uint8_t* hq;
  uint8_t* hsf;
  float* hsum;
  float* o;
  int ld_out, rows_max;
  float beta, beta_lin;
  unsigned* status;
  uint64_t limit_ns;
};

// Sixteen 2-bit codes of a 32-bit word (four per byte, low bits first) ->
// sixteen e2m1 nibbles (low nibble first; codes 0..7 in .x), q -> 2q - [q == 3].
// Byte j of a holds codes 4j, 4j+1 as nibbles, byte j of b codes 4j+2,
// 4j+3; the byte permutes interleave them into code order.
__device__ __forceinline__ uint2 codes_to_e2m1(uint32_t w) {
  const uint32_t a = (w & 0x03030303u) | ((w << 2) & 0x30303030u);
  const uint32_t b = ((w >> 4) & 0x03030303u) | ((w >> 2) & 0x30303030u);
  const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(a, b, 0x7362);
  return make_uint2((t0 << 1) - (t0 & (t0 >> 1) & 0x11111111u), (t1 << 1) - (t1 & (t1 >> 1) & 0x11111111u));
}

template <bool GU>
__global__ void __launch_bounds__(B2Cfg<GU>::kThreads, B2Cfg<GU>::kCtas)
    bank2_mxf4_kernel(const __grid_constant__ CUtensorMap map_b, const B2Params p) {
  using C = B2Cfg<GU>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;                                  // [kRing][B terms | B atom | 2-bit tiles]
  uint8_t* dec = smem + C::kRing * C::kStage;            // [2][mats][128 rows][64 B] e2m1, 64-byte swizzle
  uint8_t* sfa_atom = dec + 2 * C::kDec;                 // 512 bytes of 127
  float* xs = reinterpret_cast<float*>(sfa_atom + kAtom);  // [16 token rows][64 groups] row sums
  uint64_t* bars = reinterpret_cast<uint64_t*>(xs + C::kXsFloats);
  // bars: full[R], empty[R], dfull[2], dempty[2], afull[2], aempty[2], drain, xs_full, xs_empty
  constexpr int NB = 2 * C::kRing + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NB);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_trigger();
  pdl_wait();
  const int first = *p.begin;
  const int n_items = (*p.count - first) * p.MT;
  if ((int)blockIdx.x >= n_items) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) {
      const int k = i - 2 * C::kRing;
      // empty: the MMA commit and the epilogue threads (done with the
      // stage's scales and biases); dfull: the expand threads; aempty,
      // xs_full, xs_empty: the epilogue threads
      const uint32_t cnt = (i >= C::kRing && i < 2 * C::kRing) ? 1u + C::kEpiThreads
                           : (k == 0 || k == 1)                  ? (uint32_t)C::kExpThreads
                           : (k == 6 || k == 7 || k == 9 || k == 10) ? (uint32_t)C::kEpiThreads
                                                                     : 1u;
      mbar_init(smem_u32(bars + i), cnt);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < kAtom / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sfa_atom)[i] = 0x7F7F7F7Fu;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Guard g{abort_flag, p.status, p.limit_ns};
  auto full = [&](int r) { return smem_u32(bars + r); };
  auto empty = [&](int r) { return smem_u32(bars + C::kRing + r); };
  auto dfull = [&](int d) { return smem_u32(bars + 2 * C::kRing + d); };
  auto dempty = [&](int d) { return smem_u32(bars + 2 * C::kRing + 2 + d); };
  auto afull = [&](int b) { return smem_u32(bars + 2 * C::kRing + 4 + b); };
  auto aempty = [&](int b) { return smem_u32(bars + 2 * C::kRing + 6 + b); };
  const uint32_t drain = smem_u32(bars + 2 * C::kRing + 8);
  const uint32_t xs_full = smem_u32(bars + 2 * C::kRing + 9), xs_empty = smem_u32(bars + 2 * C::kRing + 10);
  auto stage = [&](int r) { return ring + (size_t)r * C::kStage; };
  const int G = p.KC * 2;  // groups along K

  if (warp == 0) {
    // ================= copies
    if (lane == 0) {
      int kg = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int ti = first + item / p.MT, mt = item % p.MT;
        const int4 tile = p.tiles[ti];
        const uint8_t* a_src =
            p.a_tiles + ((size_t)(tile.x - p.expert_base) * p.MT + mt) * (size_t)G * C::kNumMat * kB2Tile;
        for (int kc = 0; kc < p.KC; ++kc, ++kg) {
          const int r = kg % C::kRing, u = kg / C::kRing;
          if (u > 0 && !mbar_wait_sleep(empty(r), (u - 1) & 1, g, 1u)) {
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(stage(r));
          mbar_expect_tx(full(r), (uint32_t)(C::kB + kAtom + C::kSrc));
          tma_load_4d(st, &map_b, full(r), 0, tile.y, 0, kc);
          bulk_load(st + C::kB, p.sfb + ((size_t)ti * p.KC + kc) * 2 * kAtom, kAtom, full(r));
          bulk_load(st + C::kB + kAtom, a_src + (size_t)kc * C::kSrc, C::kSrc, full(r));
        }
      }
      if (*abort_flag) {  // copies in flight land before the CTA exits
        for (int k = max(0, kg - C::kRing); k < kg; ++k) {
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(full(k % C::kRing), (k / C::kRing) & 1))
            if (global_ns() - t0 > p.limit_ns) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issue: per chunk, per group j (the 32-byte half
    // j of every 64-byte operand row), one MMA per matrix into buffer j
    if (lane == 0) {
      const uint32_t sfa_col = tmem + C::kSfa;
      tc_cp_scales(sfa_col, sf_desc(smem_u32(sfa_atom)));
      const uint64_t a_base = umma_desc_sw64(smem_u32(dec));
      const uint64_t b_base = umma_desc_sw64(smem_u32(ring));
      int kg = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        for (int kc = 0; kc < p.KC; ++kc, ++kg) {
          const int r = kg % C::kRing, d = kg & 1;
          if (!mbar_wait_sleep(full(r), (kg / C::kRing) & 1, g, 2u) || !mbar_wait_sleep(dfull(d), (kg >> 1) & 1, g, 4u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfb_col = tmem + C::kSfa + 4 + 4 * r;
          tc_cp_scales(sfb_col, sf_desc(smem_u32(stage(r) + C::kB)));
          const uint64_t so = (uint64_t)((uint32_t)(r * C::kStage) >> 4);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (kg > 0 && !mbar_wait_sleep(aempty(j), (kg - 1) & 1, g, 8u)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int m = 0; m < C::kNumMat; ++m)
              umma_fp4(tmem + (uint32_t)((m * 2 + j) * C::kN),
                       a_base + (uint64_t)((uint32_t)(d * C::kDec + m * kQM * 64 + j * 32) >> 4), b_base + so + (j * 32 >> 4),
                       fp4_idesc(2 * j, 2 * j, C::kN), sfa_col, sfb_col, 0u);
            umma_commit(afull(j));
          }
          if (!ok) break;
          umma_commit(empty(r));
          umma_commit(dempty(d));
        }
      }
      if (!ok) {  // MMAs already issued finish before TMEM is released
        umma_commit(drain);
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(drain, 0))
          if (global_ns() - t0 > p.limit_ns) break;
      }
    }
    __syncwarp();
  } else if (warp >= 2 + C::kEpiThreads / 32) {
    // ================= expand (thread = row, every matrix), both groups of
    // each chunk, into the two-deep ring of e2m1 tiles
    const int r = threadIdx.x - 64 - C::kEpiThreads;
    int kg = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      for (int kc = 0; kc < p.KC; ++kc, ++kg) {
        const int rr = kg % C::kRing, d = kg & 1;
        bool w_ok = mbar_wait_sleep(full(rr), (kg / C::kRing) & 1, g, 32u);
        if (w_ok && kg >= 2) w_ok = mbar_wait_sleep(dempty(d), ((kg >> 1) - 1) & 1, g, 64u);
        if (!__all_sync(0xFFFFFFFFu, w_ok)) {  // warp-uniform exits
          ok = false;
          break;
        }
        const uint8_t* src = stage(rr) + C::kB + kAtom;
        const int sw = (r >> 1) & 3;  // 64-byte swizzle: 16-byte chunk c of row r at c ^ ((r >> 1) & 3)
#pragma unroll
        for (int mat = 0; mat < C::kNumMat; ++mat) {
          uint8_t* drow = dec + (size_t)d * C::kDec + (size_t)(mat * kQM + r) * 64;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint4 q = *reinterpret_cast<const uint4*>(src + (size_t)(j * C::kNumMat + mat) * kB2Tile + r * 16);
            const uint2 e0 = codes_to_e2m1(q.x), e1 = codes_to_e2m1(q.y), e2 = codes_to_e2m1(q.z),
                        e3 = codes_to_e2m1(q.w);
            // row bytes [32 j, 32 j + 32): 16-byte chunks 2j, 2j + 1
            *reinterpret_cast<uint4*>(drow + (((2 * j) ^ sw) << 4)) = make_uint4(e0.x, e0.y, e1.x, e1.y);
            *reinterpret_cast<uint4*>(drow + (((2 * j + 1) ^ sw) << 4)) = make_uint4(e2.x, e2.y, e3.x, e3.y);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(dfull(d));
      }
    }
  } else {
    // ================= epilogue (warps 2..5: row r = TMEM lane, both
    // matrices): per group, acc += s * (sum of the six terms' columns) +
    // b * (the group's row sum); at the end of an item SiTU-GLU and h's
    // terms (gate/up) or o (down)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int et = threadIdx.x - 64;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    int kg = 0, it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
      const int ti = first + item / p.MT, mt = item % p.MT;
      const int4 tile = p.tiles[ti];
      // the item's per-group sums of its token rows (latent rows by token,
      // h rows by slot; rows past the tile 0) into shared memory, once
      if (it > 0 && !__all_sync(0xFFFFFFFFu, mbar_wait_sleep(xs_empty, (it - 1) & 1, g, 256u))) break;
      for (int i = et; i < kBsDecodeRows * G; i += C::kEpiThreads) {
        const int n = i / G, gg = i - n * G;
        float v = 0.f;
        if (n < tile.z) {
          const int sl = tile.y + n;
          v = GU ? p.xsum[(size_t)(p.perm[sl] / p.K) * G + gg]
                 : p.hsum_in[(size_t)sl * (2 * G) + 2 * gg] + p.hsum_in[(size_t)sl * (2 * G) + 2 * gg + 1];
        }
        xs[n * 64 + gg] = v;
      }
      mbar_arrive(xs_full);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_sleep(xs_full, it & 1, g, 512u))) break;
      float acc[C::kNumMat][kBsDecodeRows];
#pragma unroll
      for (int m = 0; m < C::kNumMat; ++m)
#pragma unroll
        for (int n = 0; n < kBsDecodeRows; ++n) acc[m][n] = 0.f;
      for (int kc = 0; kc < p.KC && ok; ++kc, ++kg) {
        const int rr = kg % C::kRing;
        // the stage's scales and biases (the wait makes its copies visible here)
        bool w_ok = mbar_wait_sleep(full(rr), (kg / C::kRing) & 1, g, 16u);
        if (!__all_sync(0xFFFFFFFFu, w_ok)) {
          ok = false;
          break;
        }
        const uint8_t* src = stage(rr) + C::kB + kAtom;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float sc[C::kNumMat], bi[C::kNumMat];
#pragma unroll
          for (int m = 0; m < C::kNumMat; ++m) {
            const uint8_t* tl = src + (size_t)(j * C::kNumMat + m) * kB2Tile;
            sc[m] = bf16_to_f32(*reinterpret_cast<const uint16_t*>(tl + 2048 + 2 * r));
            bi[m] = bf16_to_f32(*reinterpret_cast<const uint16_t*>(tl + 2304 + 2 * r));
          }
          w_ok = mbar_wait_sleep(afull(j), kg & 1, g, 16u);
          if (!__all_sync(0xFFFFFFFFu, w_ok)) {  // warp-uniform before the TMEM loads
            ok = false;
            break;
          }
          tc_fence_after();
          const int gg = 2 * kc + j;
          // eight tokens per pass: the six terms' columns 16 t + n of every
          // matrix, loaded together (one wait)
#pragma unroll
          for (int ps = 0; ps < kBsDecodeRows / 8; ++ps) {
            if (8 * ps < tile.z) {  // warp-uniform
              float v[48 * C::kNumMat];
              const uint32_t col0 = lane_base + (uint32_t)(j * C::kN + 8 * ps);
              if constexpr (C::kNumMat == 2)
                tmem_ld2x6x8_stride16(col0, col0 + 2 * C::kN, v);
              else
                tmem_ld6x8_stride16(col0, v);
#pragma unroll
              for (int m = 0; m < C::kNumMat; ++m) {
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                  if (8 * ps + n < tile.z) {
                    const float* vm = v + 48 * m;
                    const float dsum = ((vm[n] + vm[n + 8]) + (vm[n + 16] + vm[n + 24])) + (vm[n + 32] + vm[n + 40]);
                    float& a = acc[m][8 * ps + n];
                    a = fmaf(sc[m], dsum, a);
                    a = fmaf(bi[m], xs[(8 * ps + n) * 64 + gg], a);
                  }
                }
              }
            }
          }
          tc_fence_before();
          mbar_arrive(aempty(j));
        }
        if (!ok) break;
        mbar_arrive(empty(rr));  // done with the stage's scales and biases
      }
      mbar_arrive(xs_empty);  // the item's row sums are no longer read
      if (!ok || *abort_flag) break;
      // ---- outputs of the item
      const int m_out = mt * kQM + r;
      if constexpr (GU) {
        // h = SiTU-GLU(gate, up) as bf16, its six e2m1 terms over the warp's
        // 32 rows (one scale group of the down GEMM's K) and the per-32-row
        // sums of h
        const int KCo = p.ld_out / kQK;
        uint8_t* atoms = p.hsf + (((size_t)ti * KCo + (m_out >> 7)) * 2) * kAtom + ((m_out >> 5) & 3);
        unsigned long long my_sc = 0;
#pragma unroll
        for (int n = 0; n < kBsDecodeRows; ++n) {
          if (n < tile.z) {  // warp-uniform
            const size_t row = (size_t)(tile.y + n);
            const uint16_t hb = f32_to_bf16(situ_fast(acc[0][n], acc[1][n], p.beta, p.beta_lin));
            p.h[row * p.ld_out + m_out] = hb;
            float rr = bf16_to_f32(hb);
            float hsum = rr;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) hsum += __shfl_xor_sync(0xFFFFFFFFu, hsum, o);
            if (lane == 0) p.hsum[row * (p.ld_out / 32) + (m_out >> 5)] = hsum;
            uint32_t qn = 0;
            unsigned long long scw = 0;
#pragma unroll
            for (int t = 0; t < kFp4Terms; ++t) {
              const uint32_t sb = e2m1_scale_byte(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(rr))));
              uint32_t qb = 0;
              if (sb != 255u) {
                qb = to_e2m1x2(0.f, rr * exp2_any(127 - (int)sb)) & 0xFu;
                rr = fmaf(-from_e2m1x2(qb).x, exp2_any((int)sb - 127), rr);
              } else {
                rr = 0.f;
              }
              qn |= qb << (4 * t);
              scw |= (unsigned long long)sb << (8 * t);
            }
            const uint32_t qo = __shfl_down_sync(0xFFFFFFFFu, qn, 1);
            if (!(lane & 1)) {
#pragma unroll
              for (int t = 0; t < kFp4Terms; ++t)
                p.hq[(((size_t)(m_out >> 7) * kFp4Terms + t) * p.rows_max + row) * 64 + ((m_out & 127) >> 1)] =
                    (uint8_t)(((qn >> (4 * t)) & 0xFu) | (((qo >> (4 * t)) & 0xFu) << 4));
            }
            if (lane == n) my_sc = scw;
          }
        }
        if (lane < tile.z && lane < kBsDecodeRows) {
#pragma unroll
          for (int t = 0; t < kFp4Terms; ++t)
            atoms[act_scale_byte(t, lane, kBsDecodeRows)] = (uint8_t)(my_sc >> (8 * t));
        }
      } else {
#pragma unroll
        for (int n = 0; n < kBsDecodeRows; ++n)
          if (n < tile.z) p.o[(size_t)(tile.y + n) * p.ld_out + m_out] = acc[0][n];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

// Per-64-column sums of bf16 rows (fp32, a fixed tree over the warp): one
// warp per (row, group).
__global__ void group_sums_kernel(const uint16_t* __restrict__ x, int rows, int cols, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int G = cols / 64;
  const long long n = (long long)rows * G;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (long long wi = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; wi < n; wi += nw) {
    const int rw = (int)(wi / G), gg = (int)(wi - (long long)rw * G);
    const uint32_t v = *reinterpret_cast<const uint32_t*>(x + (size_t)rw * cols + gg * 64 + 2 * lane);
    float s = __uint_as_float(v << 16) + __uint_as_float(v & 0xFFFF0000u);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (lane == 0) out[wi] = s;
  }
}

// ------------------------------------------------------------------ host helpers
bool encode(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// e2m1 tiles [nbox][128 rows][64 bytes]; one copy = `depth` adjacent tiles,
// each landing as 128 rows of 128 bytes (16-byte slots) with a 128-byte swizzle.
bool map_e2m1(CUtensorMap* map, const void* base, long long nbox, int depth) {
  const cuuint64_t dims[3] = {(cuuint64_t)kQK, (cuuint64_t)kQM, (cuuint64_t)nbox};
  const cuuint64_t strides[2] = {(cuuint64_t)kQK / 2, (cuuint64_t)kQM * kQK / 2};
  const cuuint32_t box[3] = {(cuuint32_t)kQK, (cuuint32_t)kQM, (cuuint32_t)depth};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// The same tiles as bytes: each lands dense, 128 rows of 64 bytes with the
// 64-byte swizzle (the layout kind::mxf4 reads).
bool map_e2m1_dense(CUtensorMap* map, const void* base, long long nbox, int depth) {
  const cuuint64_t dims[3] = {(cuuint64_t)kQK / 2, (cuuint64_t)kQM, (cuuint64_t)nbox};
  const cuuint64_t strides[2] = {(cuuint64_t)kQK / 2, (cuuint64_t)kQM * kQK / 2};
  const cuuint32_t box[3] = {(cuuint32_t)kQK / 2, (cuuint32_t)kQM, (cuuint32_t)depth};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}
// e2m1 activation terms q[KC][kFp4Terms][rows_max][64]: box 64 x box_rows x
// all terms x nk chunks, 64-byte swizzle; in shared memory
// [chunk][term][row][64].
bool map_terms_fp4(CUtensorMap* map, const void* base, int KC, int rows_max, int box_rows, int nk) {
  const cuuint64_t dims[4] = {64, (cuuint64_t)rows_max, kFp4Terms, (cuuint64_t)KC};
  const cuuint64_t strides[3] = {64, (cuuint64_t)rows_max * 64, (cuuint64_t)kFp4Terms * rows_max * 64};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, kFp4Terms, (cuuint32_t)nk};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}
// Activation terms q[KC][2][rows_max][128]: box 128 x box_rows x 2 terms x
// nk chunks, 128-byte swizzle; in shared memory [chunk][term][row][128].
bool map_terms(CUtensorMap* map, const void* base, int KC, int rows_max, int box_rows, int nk) {
  const cuuint64_t dims[4] = {(cuuint64_t)kQK, (cuuint64_t)rows_max, 2, (cuuint64_t)KC};
  const cuuint64_t strides[3] = {(cuuint64_t)kQK, (cuuint64_t)rows_max * kQK, (cuuint64_t)2 * rows_max * kQK};
  const cuuint32_t box[4] = {(cuuint32_t)kQK, (cuuint32_t)box_rows, 2, (cuuint32_t)nk};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

struct BsWs {
  int rows_max;       // slots: max_tokens * K
  int rows_fp4;       // slots of the decode-size layout: min(max_tokens, kBsDecodeMaxT) * K
  int max_tiles;      // bound on the tile list length
  // latent rows: terms [L/128][2][rows_max][128] e4m3 (prefill tiles) or
  // [L/128][kFp4Terms][rows_fp4][64] e2m1 (decode tiles); atoms
  // [max_tiles][L/128][2][512]
  uint8_t *lq, *lsf;
  uint8_t *hq, *hsf;  // h rows: the same over I
  int* slot_tile;     // [rows_max]: tile << 8 | row within the tile
  float* part;        // K-split partial sums (T = 1): kBsMaxSplit planes of K rows of I (gate), I (up), L (down)
  float *xsum, *hsum; // second bank at decode sizes: per-64-column latent sums by token, per-32-row h sums by slot
  int* sched;         // the expert kernels' item counters (gate/up, down), zeroed by the quantiser
  size_t total;
};
BsWs bs_ws_view(void* base, const Dims& d, int max_tokens) {
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  const size_t R = (size_t)max_tokens * d.K;
  const size_t Rf = (size_t)std::min(max_tokens, kBsDecodeMaxT) * d.K;
  // tiles hold at least one slot and at most one expert: <= E + R / 16 whatever the tile height
  const size_t MT = (size_t)d.E + R / 16 + 1;
  auto terms = [&](size_t C) { return std::max(2 * R * C, (size_t)kFp4Terms * Rf * C / 2); };
  const size_t sizes[9] = {terms(d.L),
                           MT * (d.L / kQK) * 2 * kAtom,
                           terms(d.I),
                           MT * (d.I / kQK) * 2 * kAtom,
                           R * sizeof(int),
                           (size_t)kBsMaxSplit * d.K * (2 * d.I + d.L) * sizeof(float),
                           (size_t)std::min(max_tokens, kBsDecodeMaxT) * (d.L / 64) * sizeof(float),
                           Rf * (d.I / 32) * sizeof(float),
                           2 * sizeof(int)};
  uint8_t* b = static_cast<uint8_t*>(base);
  uint8_t* ptr[9];
  size_t off = 0;
  for (int i = 0; i < 9; ++i) {
    ptr[i] = b ? b + off : nullptr;
    off += up(sizes[i]);
  }
  return BsWs{(int)R,  (int)Rf, (int)MT, ptr[0], ptr[1], ptr[2], ptr[3], reinterpret_cast<int*>(ptr[4]),
              reinterpret_cast<float*>(ptr[5]), reinterpret_cast<float*>(ptr[6]), reinterpret_cast<float*>(ptr[7]),
              reinterpret_cast<int*>(ptr[8]), off};
}

template <int MODE, int NQ>
cudaError_t launch_bs(const BsPlan& p, const uint8_t* wq, const uint8_t* sfa, int n_exp, int rows, int cols,
                      const uint8_t* q, const uint8_t* sfb, int rows_max, const int4* tiles, const int* count,
                      BsParams prm, cudaStream_t s) {
  using C = BsCfg<MODE, NQ>;
  CUtensorMap ma, mb;
  const int KC = cols / kQK, MT = rows / kQM;
  if (MT % C::kRB) return cudaErrorInvalidValue;
  const long long nbox = (long long)n_exp * MT * KC * C::kMats;
  const bool mapped = C::kFp4 ? map_e2m1_dense(&ma, wq, nbox, C::kABox) && map_terms_fp4(&mb, q, KC, rows_max, NQ, C::kNK)
                              : map_e2m1(&ma, wq, nbox, C::kABox) && map_terms(&mb, q, KC, rows_max, NQ, C::kNK);
  if (!mapped) return cudaErrorInvalidValue;
  prm.sfa = sfa;
  prm.sfb = sfb;
  prm.MT = MT / C::kRB;  // work items per tile
  prm.KC = KC;
  prm.KS = (KC + C::kNK - 1) / C::kNK;
  prm.tiles = tiles;
  prm.count = count;
  prm.rows_max = rows_max;
  prm.status = p.status;
  prm.limit_ns = p.limit_ns;
  prm.withhold_item = MODE == BS_GATEUP ? p.withhold_item : -1;
  return launch_pdl(bs_stream_kernel<MODE, NQ>, C::kCtas * p.num_sms, C::kThreads, C::kSmem, s, ma, mb, prm);
}

}  // namespace

size_t bs_weight_bytes(const Dims& d) {
  const size_t E = d.E, I = d.I, L = d.L;
  return E * 2 * I * L / 2 + E * 2 * I * L / 32 + E * L * I / 2 + E * L * I / 32;
}

cudaError_t bs_e2m1_boxes(const uint8_t* packed, int ne, int rows, int cols, int n_mat, int mat, uint8_t* out,
                          cudaStream_t s) {
  e2m1_boxes_kernel<<<1024, 256, 0, s>>>(packed, ne, rows, cols, n_mat, mat, out);
  return cudaGetLastError();
}

cudaError_t bs_scale_atoms(const uint8_t* scale, int ne, int rows, int cols, int n_mat, int mat, uint8_t* out,
                           cudaStream_t s) {
  scale_atoms_kernel<<<1024, 256, 0, s>>>(scale, ne, rows, cols, n_mat, mat, out);
  return cudaGetLastError();
}

size_t bs_ws_bytes(const Dims& d, int max_tokens) { return bs_ws_view(nullptr, d, max_tokens).total; }

int* bs_slot_tile(const BsPlan& p) { return bs_ws_view(p.ws, p.dims, p.max_tokens).slot_tile; }

cudaError_t prepare_bs_kernels() {
  cudaError_t e = cudaSuccess;
  auto set = [&](const void* f, int bytes) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  };
  set((const void*)bs_stream_kernel<BS_GATEUP, kBsSmallRows>, BsCfg<BS_GATEUP, kBsSmallRows>::kSmem);
  set((const void*)bs_stream_kernel<BS_DOWN, kBsSmallRows>, BsCfg<BS_DOWN, kBsSmallRows>::kSmem);
  set((const void*)bs_stream_kernel<BS_GATEUP, kBsDecodeRows>, BsCfg<BS_GATEUP, kBsDecodeRows>::kSmem);
  set((const void*)bs_stream_kernel<BS_DOWN, kBsDecodeRows>, BsCfg<BS_DOWN, kBsDecodeRows>::kSmem);
  set((const void*)bs_stream_kernel<BS_GATEUP, kBsPrefillRows>, BsCfg<BS_GATEUP, kBsPrefillRows>::kSmem);
  set((const void*)bs_stream_kernel<BS_DOWN, kBsPrefillRows>, BsCfg<BS_DOWN, kBsPrefillRows>::kSmem);
  set((const void*)bank2_mxf4_kernel<true>, B2Cfg<true>::kSmem);
  set((const void*)bank2_mxf4_kernel<false>, B2Cfg<false>::kSmem);
  return e;
}

cudaError_t bs_quantize_latent(const BsPlan& p, const Work& w, int T, const Dims& d, int tile_rows,
                               const int* n_local, cudaStream_t s) {
  const int TK = T * d.K;
  if (TK <= 0) return cudaSuccess;
  if (T > p.max_tokens || (tile_rows != kBsSmallRows && tile_rows != kBsDecodeRows && tile_rows != kBsPrefillRows) ||
      (tile_rows == kBsSmallRows && T > kBsSmallMaxT))
    return cudaErrorInvalidValue;
  const int stack = tile_rows;
  const BsWs ws = bs_ws_view(p.ws, d, p.max_tokens);
  const bool fp4 = tile_rows != kBsPrefillRows;
  if (!fp4) {
    // prefill tiles: each token's row split once, its terms written to the
    // token's K slots (the split is ALU work, the copies a memory stream)
    const long long th = (long long)T * ((d.L / kQK + kQuantChunks - 1) / kQuantChunks);
    const int tb = (int)std::min<long long>((th * 16 + 255) / 256, 8LL * p.num_sms);
    return launch_pdl(quant_rows_kernel, tb, 256, 0, s, w.lat, (const int*)nullptr, d.K, T, n_local, d.L,
                      ws.rows_max, (const int*)ws.slot_tile, stack, ws.lq, ws.lsf, (const int*)w.slot, ws.sched);
  }
  // decode tiles: each token's row split once, its six terms written to
  // the token's K slots (K <= 32)
  if (d.K > 32 || d.L % kQK) return cudaErrorInvalidValue;
  const dim3 grid(T, (d.L / kQK + kTokChunks - 1) / kTokChunks);
  return launch_pdl(quant_tok_fp4_kernel, grid, kTokThreads, 0, s, (const uint16_t*)w.lat, d.K, d.L, n_local,
                    ws.rows_fp4,
                    (const int*)ws.slot_tile, stack, ws.lq, ws.lsf, (const int*)w.slot, ws.sched);
}

// Best K split for `items` decode work items of `ks` K steps over `ctas`
// persistent CTAs: the one with the fewest item-times on the busiest CTA
// (every part keeps at least one K step).
int bs_best_split(int items, int ks, int ctas) {
  int best = 1;
  double best_t = 1e30;
  for (int sp = 1; sp <= std::min(kBsMaxSplit, ks); ++sp) {
    const double t = (double)((items * sp + ctas - 1) / ctas) / sp;
    if (t < best_t - 1e-9) {
      best_t = t;
      best = sp;
    }
  }
  return best;
}

int bs_split_gateup(const BsPlan& p, const Dims& d, int T) {
  using C = BsCfg<BS_GATEUP, kBsDecodeRows>;
  const int ks = (d.L / kQK + C::kNK - 1) / C::kNK;
  return T == 1 ? bs_best_split(d.K * (d.I / kQM), ks, C::kCtas * p.num_sms) : 1;
}
int bs_split_down(const BsPlan& p, const Dims& d, int T) {
  using C = BsCfg<BS_DOWN, kBsDecodeRows>;
  const int ks = (d.I / kQK + C::kNK - 1) / C::kNK;
  return T == 1 ? bs_best_split(d.K * (d.L / kQM), ks, C::kCtas * p.num_sms) : 1;
}
float* bs_down_parts(const BsPlan& p, const Dims& d) {
  return bs_ws_view(p.ws, d, p.max_tokens).part + (size_t)kBsMaxSplit * d.K * 2 * d.I;
}

// The gate/up K parts of a T = 1 forward added in part order, then SiTU-GLU
// and the h outputs of the gate/up epilogue (bf16 h, its e2m1 terms and
// scale atoms for the down kernel): one warp per (slot, 32 rows of I), a
// row per lane, the 32 rows one scale group of the down GEMM's K.  With an
// expert shard only the shard's own slots [0, *rows_dev) are finished: the
// other slots have no partial sums and no tile this forward.
template <int kHStack>
__global__ void __launch_bounds__(256) bs_gateup_finish_kernel(const BsParams p, const int* __restrict__ slot_tile,
                                                               int TK, const int* __restrict__ rows_dev) {
  pdl_trigger();
  pdl_wait();
  if (rows_dev) TK = min(TK, *rows_dev);
  constexpr int kHTerms = BsCfg<BS_DOWN, kHStack>::kTerms;
  const int lane = threadIdx.x & 31;
  const int G = p.ld_out / 32, KCo = p.ld_out / kQK;
  const int nw = (int)((gridDim.x * blockDim.x) >> 5);
  for (int wi = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); wi < TK * G; wi += nw) {
    const int sl = wi / G, m = (wi - sl * G) * 32 + lane;
    float gs = 0.f, us = 0.f;
    for (int part = 0; part < p.n_split; ++part) {
      const size_t at = ((size_t)part * p.part_rows + sl) * p.ld_out + m;
      gs += p.part_a[at];
      us += p.part_b[at];
    }
    const uint16_t hb = f32_to_bf16(situ_fast(gs, us, p.beta, p.beta_lin));
    p.h[(size_t)sl * p.ld_out + m] = hb;
    float rr = bf16_to_f32(hb);
    uint32_t qn = 0;
    unsigned long long sc = 0;
#pragma unroll
    for (int t = 0; t < kHTerms; ++t) {
      const uint32_t sb = e2m1_scale_byte(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(rr))));
      uint32_t qb = 0;
      if (sb != 255u) {
        qb = to_e2m1x2(0.f, rr * exp2_any(127 - (int)sb)) & 0xFu;
        rr = fmaf(-from_e2m1x2(qb).x, exp2_any((int)sb - 127), rr);
      } else {
        rr = 0.f;
      }
      qn |= qb << (4 * t);
      sc |= (unsigned long long)sb << (8 * t);
    }
    const uint32_t qo = __shfl_down_sync(0xFFFFFFFFu, qn, 1);
    if (!(lane & 1)) {
#pragma unroll
      for (int t = 0; t < kHTerms; ++t)
        p.hq[(((size_t)(m >> 7) * kHTerms + t) * p.rows_max + sl) * 64 + ((m & 127) >> 1)] =
            (uint8_t)(((qn >> (4 * t)) & 0xFu) | (((qo >> (4 * t)) & 0xFu) << 4));
    }
    if (lane == 0) {  // the group's scales are the same on every lane
      const int st = slot_tile[sl];
      uint8_t* atoms = p.hsf + (((size_t)(st >> 8) * KCo + (m >> 7)) * 2) * kAtom + ((m >> 5) & 3);
#pragma unroll
      for (int t = 0; t < kHTerms; ++t) atoms[act_scale_byte(t, st & 0xFF, kHStack)] = (uint8_t)(sc >> (8 * t));
    }
  }
}

cudaError_t bs_stream_gateup(const BsPlan& p, const BsWeights& bw, const int4* tiles, const int* tile_count,
                             const Work& w, int T, const Dims& d, int tile_rows, cudaStream_t s, int n_split,
                             const int* n_local) {
  const int TK = T * d.K;
  if (TK <= 0) return cudaSuccess;
  if (T > p.max_tokens || n_split < 1 || n_split > kBsMaxSplit ||
      (n_split > 1 && (T != 1 || tile_rows > kBsDecodeRows)))
    return cudaErrorInvalidValue;
  const BsWs ws = bs_ws_view(p.ws, d, p.max_tokens);
  BsParams prm{};
  prm.ld_out = d.I;
  prm.h = w.h;
  prm.hq = ws.hq;
  prm.hsf = ws.hsf;
  prm.beta = d.beta;
  prm.beta_lin = d.beta_lin;
  prm.n_split = n_split;
  prm.part_rows = TK;
  prm.part_a = ws.part;
  prm.part_b = ws.part + (size_t)kBsMaxSplit * d.K * d.I;
  prm.next_item = ws.sched;
  if (n_split > 1) {
    const bool small = tile_rows == kBsSmallRows;
    cudaError_t e = small ? launch_bs<BS_GATEUP, kBsSmallRows>(p, bw.gu_q, bw.gu_sf, bw.n_exp, d.I, d.L, ws.lq, ws.lsf,
                                                                ws.rows_fp4, tiles, tile_count, prm, s)
                          : launch_bs<BS_GATEUP, kBsDecodeRows>(p, bw.gu_q, bw.gu_sf, bw.n_exp, d.I, d.L, ws.lq,
                                                                 ws.lsf, ws.rows_fp4, tiles, tile_count, prm, s);
    if (e != cudaSuccess) return e;
    prm.rows_max = ws.rows_fp4;
    const int warps = TK * (d.I / 32);
    return launch_pdl(small ? bs_gateup_finish_kernel<kBsSmallRows> : bs_gateup_finish_kernel<kBsDecodeRows>,
                      (warps + 7) / 8, 256, 0, s, prm, (const int*)ws.slot_tile, TK, n_local);
  }
  if (tile_rows == kBsSmallRows)
    return launch_bs<BS_GATEUP, kBsSmallRows>(p, bw.gu_q, bw.gu_sf, bw.n_exp, d.I, d.L, ws.lq, ws.lsf, ws.rows_fp4,
                                              tiles, tile_count, prm, s);
  if (tile_rows == kBsDecodeRows)
    return launch_bs<BS_GATEUP, kBsDecodeRows>(p, bw.gu_q, bw.gu_sf, bw.n_exp, d.I, d.L, ws.lq, ws.lsf, ws.rows_fp4,
                                               tiles, tile_count, prm, s);
  if (tile_rows == kBsPrefillRows)
    return launch_bs<BS_GATEUP, kBsPrefillRows>(p, bw.gu_q, bw.gu_sf, bw.n_exp, d.I, d.L, ws.lq, ws.lsf, ws.rows_max,
                                                tiles, tile_count, prm, s);
  return cudaErrorInvalidValue;
}

cudaError_t bs_stream_down(const BsPlan& p, const BsWeights& bw, const int4* tiles, const int* tile_count,
                           const Work& w, int T, const Dims& d, int tile_rows, cudaStream_t s, int n_split) {
  const int TK = T * d.K;
  if (TK <= 0) return cudaSuccess;
  if (T > p.max_tokens || n_split < 1 || n_split > kBsMaxSplit ||
      (n_split > 1 && (T != 1 || tile_rows > kBsDecodeRows)))
    return cudaErrorInvalidValue;
  const BsWs ws = bs_ws_view(p.ws, d, p.max_tokens);
  BsParams prm{};
  prm.ld_out = d.L;
  prm.o = w.o;
  prm.n_split = n_split;
  prm.part_rows = TK;
  prm.part_a = ws.part + (size_t)kBsMaxSplit * d.K * 2 * d.I;  // the combine adds the parts
  prm.next_item = ws.sched + 1;
  if (tile_rows == kBsSmallRows)
    return launch_bs<BS_DOWN, kBsSmallRows>(p, bw.d_q, bw.d_sf, bw.n_exp, d.L, d.I, ws.hq, ws.hsf, ws.rows_fp4, tiles,
                                            tile_count, prm, s);
  if (tile_rows == kBsDecodeRows)
    return launch_bs<BS_DOWN, kBsDecodeRows>(p, bw.d_q, bw.d_sf, bw.n_exp, d.L, d.I, ws.hq, ws.hsf, ws.rows_fp4, tiles,
                                             tile_count, prm, s);
  if (tile_rows == kBsPrefillRows)
    return launch_bs<BS_DOWN, kBsPrefillRows>(p, bw.d_q, bw.d_sf, bw.n_exp, d.L, d.I, ws.hq, ws.hsf, ws.rows_max, tiles,
                                              tile_count, prm, s);
  return cudaErrorInvalidValue;
}

cudaError_t bs_bank2_experts(const BsPlan& p, const uint8_t* gu2_tiles, const uint8_t* d2_tiles, int bank2_begin,
                             const int4* tiles, const int* tile_count, const Work& w, int T, const Dims& d,
                             cudaStream_t s) {
  const int TK = T * d.K;
  if (TK <= 0) return cudaSuccess;
  // (the kernel stages the per-group row sums of a tile: at most 64 groups of 64 along K)
  if (T > p.max_tokens || T > kBsDecodeMaxT || d.L % kQK || d.I % kQK || d.L > 4096 || d.I > 4096)
    return cudaErrorInvalidValue;
  const BsWs ws = bs_ws_view(p.ws, d, p.max_tokens);
  const int G = d.L / 64;
  const long long warps = (long long)T * G;
  cudaError_t e = launch_pdl(group_sums_kernel, (int)std::min<long long>((warps + 7) / 8, 8LL * p.num_sms), 256, 0,
                             s, (const uint16_t*)w.lat, T, d.L, ws.xsum);
  if (e != cudaSuccess) return e;
  CUtensorMap m1, m2;
  if (!map_terms_fp4(&m1, ws.lq, d.L / kQK, ws.rows_fp4, kBsDecodeRows, 1) ||
      !map_terms_fp4(&m2, ws.hq, d.I / kQK, ws.rows_fp4, kBsDecodeRows, 1))
    return cudaErrorInvalidValue;
  B2Params q{};
  q.a_tiles = gu2_tiles;
  q.expert_base = bank2_begin;
  q.MT = d.I / kQM;
  q.KC = d.L / kQK;
  q.tiles = tiles;
  q.count = tile_count;
  q.begin = tile_count + 1;
  q.sfb = ws.lsf;
  q.xsum = ws.xsum;
  q.perm = w.perm;
  q.K = d.K;
  q.h = w.h;
  q.hq = ws.hq;
  q.hsf = ws.hsf;
  q.hsum = ws.hsum;
  q.ld_out = d.I;
  q.rows_max = ws.rows_fp4;
  q.beta = d.beta;
  q.beta_lin = d.beta_lin;
  q.status = p.status;
  q.limit_ns = p.limit_ns;
  e = launch_pdl(bank2_mxf4_kernel<true>, B2Cfg<true>::kCtas * p.num_sms, B2Cfg<true>::kThreads,
                 B2Cfg<true>::kSmem, s, m1, q);
  if (e != cudaSuccess) return e;
  B2Params q2 = q;
  q2.a_tiles = d2_tiles;
  q2.MT = d.L / kQM;
  q2.KC = d.I / kQK;
  q2.sfb = ws.hsf;
  q2.xsum = nullptr;
  q2.hsum_in = ws.hsum;
  q2.h = nullptr;
  q2.hq = nullptr;
  q2.hsf = nullptr;
  q2.hsum = nullptr;
  q2.o = w.o;
  q2.ld_out = d.L;
  return launch_pdl(bank2_mxf4_kernel<false>, B2Cfg<false>::kCtas * p.num_sms, B2Cfg<false>::kThreads,
                    B2Cfg<false>::kSmem, s, m2, q2);
}

}  // namespace k3
