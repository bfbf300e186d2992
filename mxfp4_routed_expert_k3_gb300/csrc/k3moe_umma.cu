// k3moe_umma.cu -- tcgen05 kernels with bf16 operands: MMA with fp32
// accumulators in tensor memory, operands staged in shared memory by TMA.
//
//   umma_gemm_kernel         the dense projections at T > 64 (router +
//                            down_proj fused, up_proj, the shared experts):
//                            D[m, n] = sum_k W[m, k] X[n, k], a 128-row
//                            weight block (M side) x up to 256 token rows (N
//                            side), both K-major; epilogue by a DenseOut rule
//                            (fp32 logits / bf16 latent, SiTU-GLU pairs, an
//                            added term).
//   umma_dense_stream_kernel the same projections at T <= 64: split-K over
//   + dense_reduce_kernel    all SMs, fp32 partials, ordered reduction.
//   bank2_gemm_kernel        the second bank's 2-bit experts above decode
//                            sizes (decoded exactly to bf16 hi + lo).
// plus the tile-list builders the grouped expert kernels read.
//
// Warp roles: warp 0 issues the TMA copies, one lane of warp 1 issues the
// MMAs, a warpgroup (warp w reads TMEM lanes 32*(w%4)..+31) runs the
// epilogue.  Every wait on an mbarrier is bounded: past the limit the kernel
// records a status bit, raises a shared abort flag that releases the other
// roles, waits (bounded) for its own copies in flight, frees TMEM and
// returns.
#include <cuda.h>

#include <algorithm>
#include <cstdio>

#include "k3moe_device.cuh"
#include "k3moe_tc.cuh"
#include "k3moe_umma.h"

namespace k3 {

constexpr int kBM = 128;        // weight rows per tile (MMA M)
constexpr int kBK = 64;         // input columns per stage (one 128-byte swizzle row of bf16)
constexpr int kThreads = 192;

// Second-bank (2-bit affine) tile: 128 weight rows x 64 input columns of
// one matrix -- row r's 64 codes (four per byte, low bits first) at
// [16 r, 16 r + 16), then the rows' bf16 scales at 2048 + 2 r and bf16
// biases at 2304 + 2 r (one group of 64 per row per tile: the tile is one
// quantisation group wide).
constexpr int kTile2Bytes = 2560;
constexpr int kTile2MaxRows = 96;  // token rows of a second-bank tile's box at most

// The tensor cores' fp32 accumulation drifts by about 2^-24 (relative) per
// accumulation step, so a long K loop into one accumulator loses more than
// an fp32 FMA chain.  kAcc accumulators take the K steps in turn (each sees
// K/(16*kAcc) steps) and the epilogue adds them with round-to-nearest fp32.
// Tiles of 256 token rows (an MMA instruction costs about the pipe time of
// an N = 256 one whatever its N).
struct GCfg {
  static constexpr int kBN = 256;                  // token rows per tile (MMA N)
  static constexpr int kABytes = kBM * kBK * 2;    // 16 KB
  static constexpr int kBBytes = kBN * kBK * 2;    // 32 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = 4;
  static constexpr int kAcc = 2;
  static constexpr int kAccStride = 256;           // TMEM columns between accumulators
  static constexpr int kTmemCols = 512;
  static constexpr int kSmem = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
  static_assert(kAcc * kAccStride <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

// One output element of a dense projection (DenseOut, glu == 0).
__device__ __forceinline__ void dense_store1(const DenseOut& o, int M, int t, int m, float v) {
  if (m < o.split) {
    o.out_f32[(size_t)t * o.split + m] = v;
  } else {
    const size_t i = (size_t)t * (M - o.split) + (m - o.split);
    uint16_t b = f32_to_bf16(v);
    if (o.add_bf16) b = f32_to_bf16(bf16_to_f32(b) + bf16_to_f32(o.add_bf16[i]));
    o.out_bf16[i] = b;
  }
}
// Rows m..m+3 (m % 4 == 0) of token t.
__device__ __forceinline__ void dense_store4(const DenseOut& o, int M, int t, int m, float4 a) {
  if (o.glu) {
    const uint32_t h = pack_bf16x2(situ_fast(a.x, a.y, o.beta, o.beta_lin), situ_fast(a.z, a.w, o.beta, o.beta_lin));
    *reinterpret_cast<uint32_t*>(o.out_bf16 + (size_t)t * (M >> 1) + (m >> 1)) = h;
    return;
  }
  if (o.add_bf16 && m >= o.split && !(o.split & 3) && !((M - o.split) & 3)) {
    // bf16 rows with an added term: its four values in one load, before
    // the store (four loads behind four stores would run one by one)
    const size_t i = (size_t)t * (M - o.split) + (m - o.split);
    const uint2 ad = *reinterpret_cast<const uint2*>(o.add_bf16 + i);
    const float2 a01 = unpack_bf16x2(ad.x), a23 = unpack_bf16x2(ad.y);
    auto r = [](float v, float add) { return bf16_to_f32(f32_to_bf16(bf16_to_f32(f32_to_bf16(v)) + add)); };
    *reinterpret_cast<uint2*>(o.out_bf16 + i) =
        make_uint2(pack_bf16x2(r(a.x, a01.x), r(a.y, a01.y)), pack_bf16x2(r(a.z, a23.x), r(a.w, a23.y)));
    return;
  }
  dense_store1(o, M, t, m, a.x);
  dense_store1(o, M, t, m + 1, a.y);
  dense_store1(o, M, t, m + 2, a.z);
  dense_store1(o, M, t, m + 3, a.w);
}

// Per-tile description for grouped GEMMs: x = expert, y = first row (slot),
// z = valid rows, w = MMA N (rows rounded up to 16).  The kernel takes
// tiles [*begin, *count) (begin NULL: from 0), both read on the device.
struct TileList {
  const int4* tiles;
  const int* count;
  const int* begin = nullptr;
};

struct Params {
  // operand sources
  const uint8_t* a_tiles;  // second bank: 2-bit tiles
  int expert_base;         // weight index of a tile = its expert id - expert_base
  int MT;                  // weight row tiles per matrix
  int KS;                  // K / 64
  int M;                   // weight rows (DENSE edge masking)
  // token tiling
  TileList list;           // second bank
  int T, tn;               // DENSE: tokens and rows per tile; second bank: token box rows
  // epilogue
  DenseOut dout;           // DENSE
  float* out_f32;          // second bank down: o per slot
  uint16_t* out_bf16;      // second bank gate/up: h per slot
  int ld_out;              // I or L (row length of h / o)
  float beta, beta_lin;
  unsigned* status;
  uint64_t limit_ns;
};

// Dense projection of a token tile: D = W[mt block] . X[tile]^T over K,
// one CTA per (128-row block, token tile).  Warp 0 issues the 2-D TMA copies
// of both operands, one lane of warp 1 the MMAs (K steps alternating over
// kAcc accumulators), warps 2..5 the epilogue (DenseOut rule).
__global__ void __launch_bounds__(kThreads, 1) umma_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                                                                const __grid_constant__ CUtensorMap map_b,
                                                                const Params p) {
  using C = GCfg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  // bars: [0, S) full, [S, 2S) empty, [2S] tmem_full
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x;
  const int row0 = blockIdx.y * p.tn;
  const int rows = min(p.tn, p.T - row0);
  const int n_mma = (rows + 15) & ~15;
  if (rows <= 0) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2 * C::kStages + 1; ++s) mbar_init(smem_u32(bars + s), 1u);
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
  auto empty = [&](int s) { return smem_u32(bars + C::kStages + s); };
  const uint32_t tmem_full = smem_u32(bars + 2 * C::kStages);
  auto stage_a = [&](int s) { return smem + (size_t)s * C::kStageBytes; };
  auto stage_b = [&](int s) { return smem + (size_t)s * C::kStageBytes + C::kABytes; };

  if (warp == 0) {
    // ================= TMA producer
    int issued = 0;
    if (lane == 0) {
      for (int ks = 0; ks < p.KS; ++ks) {
        const int s = ks % C::kStages, u = ks / C::kStages;
        if (u > 0 && !mbar_wait(empty(s), (u - 1) & 1, g, 1u)) break;
        mbar_expect_tx(full(s), C::kABytes + C::kBBytes);
        tma_load_2d(smem_u32(stage_b(s)), &map_b, full(s), ks * kBK, row0);
        tma_load_2d(smem_u32(stage_a(s)), &map_a, full(s), ks * kBK, mt * kBM);
        ++issued;
      }
      if (*abort_flag) {
        // let our own copies land before the CTA's shared memory goes away
        for (int ks = max(0, issued - C::kStages); ks < issued; ++ks) {
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(full(ks % C::kStages), (ks / C::kStages) & 1))
            if (global_ns() - t0 > p.limit_ns) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kBM, n_mma);
      bool ok = true;
      for (int ks = 0; ks < p.KS && ok; ++ks) {
        const int s = ks % C::kStages;
        if (!(ok = mbar_wait(full(s), (ks / C::kStages) & 1, g, 2u))) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(stage_a(s)), b0 = smem_u32(stage_b(s));
        const uint32_t acc_col = (uint32_t)((ks % C::kAcc) * C::kAccStride);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma_bf16(tmem + acc_col, umma_desc_sw128(a0 + kk * 32), umma_desc_sw128(b0 + kk * 32), idesc,
                    (ks >= C::kAcc || kk) ? 1u : 0u);
        umma_commit(empty(s));
      }
      umma_commit(tmem_full);
      if (!ok) {
        // the MMAs already issued must finish before TMEM is released
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(tmem_full, 0))
          if (global_ns() - t0 > p.limit_ns) break;
      }
    }
    __syncwarp();
  } else {
    // ================= epilogue (warps 2..5: TMEM lane quarter warp % 4)
    if (mbar_wait(tmem_full, 0, g, 16u) && !*abort_flag) {
      tc_fence_after();
      const int quarter = warp & 3;
      const int m = mt * kBM + quarter * 32 + lane;
      const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
      // accumulators that hold a part of the sum: every K accumulator that
      // received at least one k step
      const int n_acc = min(C::kAcc, p.KS);
      for (int j0 = 0; j0 < n_mma; j0 += 32) {
        float acc[32];
        tmem_ld32(lane_addr + j0, acc);
        for (int a = 1; a < n_acc; ++a) {
          float part[32];
          tmem_ld32(lane_addr + a * C::kAccStride + j0, part);
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[j] += part[j];
        }
        if (p.dout.glu) {
          // gate/up row pairs sit in neighbouring lanes of this warp
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float partner = __shfl_xor_sync(0xFFFFFFFFu, acc[j], 1);
            if (!(m & 1) && m < p.M && j0 + j < rows)
              p.dout.out_bf16[(size_t)(row0 + j0 + j) * (p.M >> 1) + (m >> 1)] =
                  f32_to_bf16(situ_fast(acc[j], partner, p.dout.beta, p.dout.beta_lin));
          }
        } else if (m < p.M && p.dout.add_bf16 && m >= p.dout.split) {
          // the added term's 32 values loaded before any store (the output
          // and the added tensor are both bf16 arrays, so loads placed
          // after stores would wait for them one by one)
          const int Mb = p.M - p.dout.split;
          float addv[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            addv[j] = (j0 + j < rows)
                          ? bf16_to_f32(p.dout.add_bf16[(size_t)(row0 + j0 + j) * Mb + (m - p.dout.split)])
                          : 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j0 + j < rows)
              p.dout.out_bf16[(size_t)(row0 + j0 + j) * Mb + (m - p.dout.split)] =
                  f32_to_bf16(bf16_to_f32(f32_to_bf16(acc[j])) + addv[j]);
        } else if (m < p.M) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j0 + j < rows) dense_store1(p.dout, p.M, row0 + j0 + j, m, acc[j]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

// =====================================================================
// Second bank (2-bit affine experts): a persistent kernel over the work
// items (tile of the tile list's second-bank slice, 128-row weight block),
// the blocks of one tile consecutive so that CTAs running at the same time
// share its token rows in L2.  The compressed 2-bit tiles and the token
// rows stream through a deep ring; eight decode warps expand each k step's
// weights into bf16 hi and lo tiles (w = scale * q + bias is exact in fp32;
// hi = bf16(w), lo = bf16(w - hi)) in a two-deep ring; one thread issues
// the MMAs (hi and lo of each matrix into accumulators of their own); the
// epilogue adds them and applies SiTU-GLU (gate/up) or stores o (down).
// Decoded tiles are 8x the size of the compressed ones, so keeping them out
// of the copy ring lets a CTA keep many compressed stages in flight.
// =====================================================================
template <bool GU>
struct B2Cfg {
  static constexpr int kNumMat = GU ? 2 : 1;
  static constexpr int kBN = kTile2MaxRows;                    // token rows per box at most
  static constexpr int kABytes = kBM * kBK * 2;                // one bf16 tile: 16 KB
  static constexpr int kBBytes = kBN * kBK * 2;                // room for the largest token box: 10 KB
  static constexpr int kSrc = kNumMat * kTile2Bytes;           // compressed weights of a k step
  static constexpr int kRingStage = kBBytes + (kSrc + 1023) / 1024 * 1024;
  static constexpr int kDecBytes = kNumMat * 2 * kABytes;      // hi and lo of each matrix
  static constexpr int kRing = GU ? 5 : 10;
  static constexpr int kAcc = GU ? 1 : 2;                      // K split over accumulators
  static constexpr int kAccStride = 128, kMatStride = 256;
  static constexpr int kThreads = 320;                         // TMA, MMA, 8 decode warps (4 of them epilogue)
  static constexpr int kNB = 2 * kRing + 7;                    // barriers
  static constexpr int kSmem = 2 * kDecBytes + kRing * kRingStage + 1024 + 512;
  static_assert(kNumMat * 2 * kAcc * kAccStride <= 512, "TMEM budget");
  static_assert(kAccStride >= kBN && (kNumMat == 1 || 2 * kAcc * kAccStride <= kMatStride), "accumulator layout");
  static_assert(8 * kNB + 8 <= 512, "barrier area");
  static_assert(kSmem <= 232448, "shared memory budget");
};

template <bool GU>
__global__ void __launch_bounds__(B2Cfg<GU>::kThreads, 1)
    bank2_gemm_kernel(const __grid_constant__ CUtensorMap map_b, const Params p) {
  using C = B2Cfg<GU>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* dec = smem;                           // [2][kNumMat][hi, lo][128 x 64 bf16]
  uint8_t* ring = smem + 2 * C::kDecBytes;       // [kRing][B | compressed weights]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + C::kRing * C::kRingStage);
  // bars: full[R], empty[R], dfull[2], dempty[2], tmem_full, tmem_empty, drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNB);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int first = p.list.begin ? *p.list.begin : 0;
  const int n_items = (*p.list.count - first) * p.MT;
  if ((int)blockIdx.x >= n_items) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNB; ++i) {
      const bool dfull_bar = i >= 2 * C::kRing && i < 2 * C::kRing + 2;
      const bool tmem_empty_bar = i == 2 * C::kRing + 5;
      mbar_init(smem_u32(bars + i), dfull_bar ? 256u : tmem_empty_bar ? 128u : 1u);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Guard g{abort_flag, p.status, p.limit_ns};
  auto full = [&](int r) { return smem_u32(bars + r); };
  auto empty = [&](int r) { return smem_u32(bars + C::kRing + r); };
  auto dfull = [&](int d) { return smem_u32(bars + 2 * C::kRing + d); };
  auto dempty = [&](int d) { return smem_u32(bars + 2 * C::kRing + 2 + d); };
  const uint32_t tmem_full = smem_u32(bars + 2 * C::kRing + 4);
  const uint32_t tmem_empty = smem_u32(bars + 2 * C::kRing + 5);
  const uint32_t drain = smem_u32(bars + 2 * C::kRing + 6);
  auto stage_b = [&](int r) { return ring + (size_t)r * C::kRingStage; };
  auto stage_w = [&](int r) { return ring + (size_t)r * C::kRingStage + C::kBBytes; };
  auto dec_tile = [&](int d, int m, int part) { return dec + (size_t)d * C::kDecBytes + (m * 2 + part) * C::kABytes; };
  const uint32_t b_tx = (uint32_t)(p.tn * kBK * 2);  // one token box

  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0) {
      int kg = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int4 tile = p.list.tiles[first + item / p.MT];
        const int mt = item % p.MT, e = tile.x - p.expert_base;
        const uint8_t* a_src = p.a_tiles + ((size_t)(e * p.MT + mt) * p.KS) * C::kSrc;
        for (int ks = 0; ks < p.KS; ++ks, ++kg) {
          const int r = kg % C::kRing, u = kg / C::kRing;
          if (u > 0 && !mbar_wait(empty(r), (u - 1) & 1, g, 1u)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full(r), b_tx + C::kSrc);
          tma_load_2d(smem_u32(stage_b(r)), &map_b, full(r), ks * kBK, tile.y);
          bulk_load(smem_u32(stage_w(r)), a_src + (size_t)ks * C::kSrc, C::kSrc, full(r));
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
    // ================= MMA issuer
    if (lane == 0) {
      int kg = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
        const int n_mma = p.list.tiles[first + item / p.MT].w;
        const uint32_t idesc = umma_idesc_bf16(kBM, n_mma);
        if (it > 0 && !mbar_wait(tmem_empty, (it - 1) & 1, g, 2u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < p.KS; ++ks, ++kg) {
          const int r = kg % C::kRing, d = kg & 1;
          if (!mbar_wait(full(r), (kg / C::kRing) & 1, g, 2u) || !mbar_wait(dfull(d), (kg >> 1) & 1, g, 4u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b0 = smem_u32(stage_b(r));
          const int acc_k = ks % C::kAcc;
#pragma unroll
          for (int m = 0; m < C::kNumMat; ++m)
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              const uint32_t a0 = smem_u32(dec_tile(d, m, part));
              const uint32_t acc = (uint32_t)(m * C::kMatStride + (acc_k * 2 + part) * C::kAccStride);
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk)
                umma_bf16(tmem + acc, umma_desc_sw128(a0 + kk * 32), umma_desc_sw128(b0 + kk * 32), idesc,
                          (ks >= C::kAcc || kk) ? 1u : 0u);
            }
          umma_commit(empty(r));
          umma_commit(dempty(d));
        }
        if (ok) umma_commit(tmem_full);
      }
      if (!ok) {  // MMAs already issued finish before TMEM is released
        umma_commit(drain);
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(drain, 0))
          if (global_ns() - t0 > p.limit_ns) break;
      }
    }
    __syncwarp();
  } else {
    // ================= decode (warps 2..9: row dt % 128, columns 32 * (dt / 128) ..),
    // then the epilogue of each item on warps 2..5 (TMEM lane quarter warp % 4)
    const int dt = threadIdx.x - 64;
    const int r = dt & 127, half = dt >> 7;
    int kg = 0, it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
      for (int ks = 0; ks < p.KS; ++ks, ++kg) {
        const int rr = kg % C::kRing, d = kg & 1;
        if (!mbar_wait(full(rr), (kg / C::kRing) & 1, g, 8u) ||
            (kg >= 2 && !mbar_wait(dempty(d), ((kg >> 1) - 1) & 1, g, 32u))) {
          ok = false;
          break;
        }
        const uint8_t* stg = stage_w(rr);
#pragma unroll
        for (int m = 0; m < C::kNumMat; ++m) {
          const uint8_t* tl = stg + m * kTile2Bytes;
          const uint2 q = *reinterpret_cast<const uint2*>(tl + (size_t)r * 16 + half * 8);  // 32 codes
          const float sc = bf16_to_f32(*reinterpret_cast<const uint16_t*>(tl + 2048 + 2 * r));
          const float bi = bf16_to_f32(*reinterpret_cast<const uint16_t*>(tl + 2304 + 2 * r));
          // the row's four levels w_q = scale * q + bias (q = 0..3), as bf16
          // hi = bf16(w_q) and lo = bf16(w_q - hi), packed two per word: level
          // q occupies bytes 2q, 2q + 1 of the pair {H23:H01} (and {L23:L01})
          const float w0 = fmaf(sc, 0.f, bi), w1 = fmaf(sc, 1.f, bi);
          const float w2 = fmaf(sc, 2.f, bi), w3 = fmaf(sc, 3.f, bi);
          const uint32_t H01 = pack_bf16x2(w0, w1), H23 = pack_bf16x2(w2, w3);
          const float2 h01 = unpack_bf16x2(H01), h23 = unpack_bf16x2(H23);
          const uint32_t L01 = pack_bf16x2(w0 - h01.x, w1 - h01.y), L23 = pack_bf16x2(w2 - h23.x, w3 - h23.y);
          uint8_t* row_hi = dec_tile(d, m, 0) + (size_t)r * 128;
          uint8_t* row_lo = dec_tile(d, m, 1) + (size_t)r * 128;
          const uint32_t words[2] = {q.x, q.y};
#pragma unroll
          for (int c = 0; c < 4; ++c) {  // columns 8 c8 .. 8 c8 + 7, c8 = 4 half + c
            const int c8 = 4 * half + c;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              // four codes c0..c3 (two bits each, low first) -> byte i of sp
              // holds c_i -> the byte_perm selectors of the pairs (c0, c1)
              // and (c2, c3): nibbles 2 c_i, 2 c_i + 1 (the bytes of level c_i)
              const uint32_t x = (words[c >> 1] >> (16 * (c & 1) + 8 * b)) & 0xFFu;
              const uint32_t ev = x & 0x33u, od = x & 0xCCu;
              const uint32_t sp = ((ev * 0x1001u) & 0x30003u) | ((od * 0x40040u) & 0x3000300u);
              const uint32_t z = sp * 0x22u + 0x10101010u;
              hi[2 * b] = __byte_perm(H01, H23, z & 0xFFFFu);
              hi[2 * b + 1] = __byte_perm(H01, H23, z >> 16);
              lo[2 * b] = __byte_perm(L01, L23, z & 0xFFFFu);
              lo[2 * b + 1] = __byte_perm(L01, L23, z >> 16);
            }
            const int sw = (c8 ^ (r & 7)) << 4;
            *reinterpret_cast<uint4*>(row_hi + sw) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(row_lo + sw) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(dfull(d));
      }
      if (!ok || warp >= 6) continue;
      // ---- epilogue of this item
      if (!mbar_wait(tmem_full, it & 1, g, 16u) || *abort_flag) {
        ok = false;
        continue;
      }
      tc_fence_after();
      const int4 tile = p.list.tiles[first + item / p.MT];
      const int mt = item % p.MT, row0 = tile.y, rows = tile.z, n_mma = tile.w;
      const int quarter = warp & 3;
      const int m = mt * kBM + quarter * 32 + lane;
      const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
      const int n_acc = min(C::kAcc, p.KS) * 2;
      for (int j0 = 0; j0 < n_mma; j0 += 16) {
        float acc[16];
        tmem_ld16(lane_addr + j0, acc);
        for (int a = 1; a < n_acc; ++a) {
          float part[16];
          tmem_ld16(lane_addr + a * C::kAccStride + j0, part);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] += part[j];
        }
        if (GU) {
          float up[16];
          tmem_ld16(lane_addr + C::kMatStride + j0, up);
          for (int a = 1; a < n_acc; ++a) {
            float part[16];
            tmem_ld16(lane_addr + C::kMatStride + a * C::kAccStride + j0, part);
#pragma unroll
            for (int j = 0; j < 16; ++j) up[j] += part[j];
          }
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j0 + j < rows)
              p.out_bf16[(size_t)(row0 + j0 + j) * p.ld_out + m] =
                  f32_to_bf16(situ_fast(acc[j], up[j], p.beta, p.beta_lin));
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j0 + j < rows) p.out_f32[(size_t)(row0 + j0 + j) * p.ld_out + m] = acc[j];
        }
      }
      tc_fence_before();
      mbar_arrive(tmem_empty);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

constexpr int kMinTileRows = 16;  // the shortest tile height of a list with more than one tile per expert
constexpr int kDThreads = 192;

// =====================================================================
// Streaming dense GEMM for small T (decode): D = W . X^T with W bf16
// [M, K] (the weights, M side) and X bf16 [T <= 64, K] (N side).  Work items
// are (128-row tile, K chunk) so that every SM streams weights even though
// M / 128 is small (35 tiles for router + down_proj); each item writes its
// fp32 partial sums to part[chunk][t][m], and dense_reduce_kernel (launched
// right after, programmatic dependent launch) adds the chunks in order over
// all SMs.  A and B come by 2-D TMA (128-byte swizzle); D is double buffered
// in TMEM so the epilogue of one item overlaps the next item's MMAs.
// =====================================================================
constexpr int kDNB = 64;  // max tokens
struct DCfg {
  static constexpr int kABytes = kBM * kBK * 2;   // 16 KB
  static constexpr int kBBytes = kDNB * kBK * 2;  // 8 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = 4;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 512;
};

struct DenseStreamParams {
  int MT, KS, nkc, ks_per_chunk, M, T;
  uint32_t b_bytes;  // bytes of one token-row box: 128 x (T rounded up to 16)
  float* part;       // [nkc][T][M] fp32 partial sums
  unsigned* status;
  uint64_t limit_ns;
};

__global__ void __launch_bounds__(kDThreads, 1) umma_dense_stream_kernel(const __grid_constant__ CUtensorMap map_a,
                                                                         const __grid_constant__ CUtensorMap map_b,
                                                                         const DenseStreamParams p) {
  using C = DCfg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  // bars: full[S], free[S], tmem_full[2], tmem_empty[2]
  const int NB = 2 * C::kStages + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NB);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.MT * p.nkc;
  pdl_trigger();
  if ((int)blockIdx.x >= n_items) {
    pdl_wait();
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) mbar_init(smem_u32(bars + i), i >= 2 * C::kStages + 2 ? 128u : 1u);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto sfree = [&](int s) { return smem_u32(bars + C::kStages + s); };
  auto tfull = [&](int b) { return smem_u32(bars + 2 * C::kStages + b); };
  auto tempty = [&](int b) { return smem_u32(bars + 2 * C::kStages + 2 + b); };
  auto stage_a = [&](int s) { return smem + (size_t)s * C::kStageBytes; };
  auto stage_b = [&](int s) { return smem + (size_t)s * C::kStageBytes + C::kABytes; };
  // The weights are static: the first ring of weight tiles is requested
  // before the preceding kernel has finished (only the token rows, which
  // that kernel may write, wait for it).  Each stage's barrier expects the
  // weight and the token bytes at once; the token copy completes it later.
  int n_pre = 0;
  if (warp == 0 && lane == 0) {
    for (int item = blockIdx.x; item < n_items && n_pre < C::kStages; item += gridDim.x) {
      const int mt = item % p.MT, kc = item / p.MT;
      const int k0 = kc * p.ks_per_chunk, k1 = min(p.KS, k0 + p.ks_per_chunk);
      for (int ks = k0; ks < k1 && n_pre < C::kStages; ++ks, ++n_pre) {
        mbar_expect_tx(full(n_pre), C::kABytes + p.b_bytes);
        tma_load_2d(smem_u32(stage_a(n_pre)), &map_a, full(n_pre), ks * kBK, mt * kBM);
      }
    }
  }
  pdl_wait();
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Guard g{abort_flag, p.status, p.limit_ns};
  const int n_mma = (p.T + 15) & ~15;

  if (warp == 0) {
    if (lane == 0) {
      int kg = 0, issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int mt = item % p.MT, kc = item / p.MT;
        const int k0 = kc * p.ks_per_chunk, k1 = min(p.KS, k0 + p.ks_per_chunk);
        for (int ks = k0; ks < k1; ++ks, ++kg) {
          const int s = kg % C::kStages, u = kg / C::kStages;
          if (kg < n_pre) {  // weights already requested: the token rows only
            tma_load_2d(smem_u32(stage_b(s)), &map_b, full(s), ks * kBK, 0);
            ++issued;
            continue;
          }
          if (u > 0 && !mbar_wait(sfree(s), (u - 1) & 1, g, 1u)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full(s), C::kABytes + p.b_bytes);
          tma_load_2d(smem_u32(stage_a(s)), &map_a, full(s), ks * kBK, mt * kBM);
          tma_load_2d(smem_u32(stage_b(s)), &map_b, full(s), ks * kBK, 0);
          ++issued;
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
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kBM, n_mma);
      int kg = 0, it = 0, done = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
        const int kc = item / p.MT, buf = it & 1;
        const int k0 = kc * p.ks_per_chunk, k1 = min(p.KS, k0 + p.ks_per_chunk);
        // the epilogue must have drained this accumulator buffer (used two items ago)
        if (it >= 2 && !mbar_wait(tempty(buf), ((it >> 1) - 1) & 1, g, 64u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = k0; ks < k1; ++ks, ++kg) {
          const int s = kg % C::kStages;
          if (!(ok = mbar_wait(full(s), (kg / C::kStages) & 1, g, 2u))) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(stage_a(s)), b0 = smem_u32(stage_b(s));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(tmem + buf * kDNB, umma_desc_sw128(a0 + kk * 32), umma_desc_sw128(b0 + kk * 32), idesc,
                      (ks > k0 || kk) ? 1u : 0u);
          umma_commit(sfree(s));
        }
        if (ok) {
          umma_commit(tfull(buf));
          ++done;
        }
      }
      if (!ok) {
        umma_commit(tfull(0));
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(tfull(0), ((done + 1) >> 1) & 1))
          if (global_ns() - t0 > p.limit_ns) break;
      }
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
      const int mt = item % p.MT, kc = item / p.MT, buf = it & 1;
      if (!mbar_wait(tfull(buf), (it >> 1) & 1, g, 16u) || *abort_flag) break;
      tc_fence_after();
      const int m = mt * kBM + r;
      float* dst = p.part + (size_t)kc * p.T * p.M + m;
      for (int j0 = 0; j0 < n_mma; j0 += 32) {
        float acc[32];
        tmem_ld32(lane_base + buf * kDNB + j0, acc);
        if (m < p.M) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j0 + j < p.T) dst[(size_t)(j0 + j) * p.M] = acc[j];
        }
      }
      tc_fence_before();
      mbar_arrive(tempty(buf));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// Ordered split-K reduction: D[t, m] = sum over chunks c = 0, 1, ... of
// part[c][t][m] (fp32, chunk order fixed, so results do not depend on
// scheduling), then the dense output rule (DenseOut).  One thread per four
// consecutive rows of one token; all chunk loads of a thread are issued
// before the sum.
constexpr int kReduceMaxChunks = 16;
__global__ void __launch_bounds__(256) dense_reduce_kernel(const float* __restrict__ part, int nkc, int T, int M,
                                                           DenseOut o) {
  pdl_trigger();
  pdl_wait();
  const int M4 = M >> 2;
  const long long total = (long long)T * M4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / M4), m = (int)(i % M4) * 4;
    float4 v[kReduceMaxChunks];
#pragma unroll
    for (int c = 0; c < kReduceMaxChunks; ++c)
      if (c < nkc) v[c] = __ldcg(reinterpret_cast<const float4*>(part + ((size_t)c * T + t) * M + m));
    float4 a = v[0];
#pragma unroll
    for (int c = 1; c < kReduceMaxChunks; ++c)
      if (c < nkc) {
        a.x += v[c].x;
        a.y += v[c].y;
        a.z += v[c].z;
        a.w += v[c].w;
      }
    dense_store4(o, M, t, m, a);
  }
}

// ------------------------------------------------------------------ helpers
// Gather the latent rows into slot order: lat_perm[s] = lat[perm[s] / K].
__global__ void gather_rows_kernel(const uint16_t* __restrict__ lat, const int* __restrict__ perm, int TK, int K,
                                   int L, uint16_t* __restrict__ out) {
  const int vec = L / 8;
  const long long total = (long long)TK * vec;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int s = (int)(i / vec), v = (int)(i - (long long)s * vec);
    const int t = perm[s] / K;
    reinterpret_cast<uint4*>(out)[(size_t)s * vec + v] = reinterpret_cast<const uint4*>(lat)[(size_t)t * vec + v];
  }
}

// Tiles of at most bn_max rows per active expert, rows split evenly and
// rounded up to 16: tiles[i] = {expert, first slot, rows, MMA N}.
__global__ void __launch_bounds__(1024) build_tiles_kernel(const int* __restrict__ active,
                                                           const int* __restrict__ offsets, int bn_max,
                                                           int4* __restrict__ tiles, int* __restrict__ count,
                                                           int* __restrict__ slot_tile, int split_expert) {
  __shared__ int warp_tot[32];
  __shared__ int carry, n_first;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_act = active[0];
  if (threadIdx.x == 0) {
    carry = 0;
    n_first = 0;
  }
  __syncthreads();
  for (int a0 = 0; a0 < n_act; a0 += 1024) {
    const int a = a0 + threadIdx.x;
    int e = 0, c = 0, nsub = 0;
    if (a < n_act) {
      e = active[1 + a];
      c = offsets[e + 1] - offsets[e];
      nsub = (c + bn_max - 1) / bn_max;
    }
    // exclusive scan of nsub over the block
    int incl = nsub;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int wv = warp_tot[lane];
      int wi = wv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, wi, o);
        if (lane >= o) wi += v;
      }
      warp_tot[lane] = wi - wv;
    }
    __syncthreads();
    const int base = carry + warp_tot[warp] + incl - nsub;
    // tiles of experts below split_expert come first (experts ascend): their
    // number is where the second bank's tiles begin
    if (a < n_act && nsub > 0 && e < split_expert) atomicAdd(&n_first, nsub);
    if (a < n_act && nsub > 0) {
      const int per = (c + nsub - 1) / nsub;
      const int tn = min((per + 15) & ~15, bn_max);  // tiles never exceed bn_max rows
      for (int j = 0; j < nsub; ++j) {
        const int r0 = j * tn;
        const int rows = min(tn, c - r0);
        tiles[base + j] = make_int4(e, offsets[e] + r0, rows, (rows + 15) & ~15);
        if (slot_tile)
          for (int n = 0; n < rows; ++n) slot_tile[offsets[e] + r0 + n] = ((base + j) << 8) | n;
      }
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry = base + nsub;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    count[0] = carry;
    count[1] = n_first;
  }
}

// Second-bank weights into 2-bit tiles: n_mat matrices [rows, cols] per
// expert (codes [rows, cols/4] u8, scale and bias [rows, cols/64] bf16);
// tile (m, mt, ks) of expert e at out + ((e * n_mat_stride + (mt * KS + ks)
// * step + offset) * kTile2Bytes, one thread per 16-byte row of codes or
// per row's scale / bias pair.
__global__ void bank2_tiles_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ sc,
                                   const uint16_t* __restrict__ bi, int ne, int rows, int cols,
                                   uint8_t* __restrict__ out, size_t mat_stride_tiles, int step, int offset) {
  const int KS = cols / 64, MT = rows / kBM;
  const long long per_tile = 2 * kBM;  // 128 code rows + 128 scale/bias rows
  const long long total = (long long)ne * MT * KS * per_tile;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const int w = (int)(g % per_tile);
    const long long tl = g / per_tile;
    const int ks = (int)(tl % KS), mt = (int)((tl / KS) % MT);
    const int e = (int)(tl / ((long long)KS * MT));
    uint8_t* tile = out + ((size_t)e * mat_stride_tiles + ((size_t)mt * KS + ks) * step + offset) * kTile2Bytes;
    const int r = w % kBM;
    const size_t row = (size_t)e * rows + (size_t)mt * kBM + r;
    if (w < kBM) {
      *reinterpret_cast<uint4*>(tile + (size_t)r * 16) =
          *reinterpret_cast<const uint4*>(q + row * (cols / 4) + (size_t)ks * 16);
    } else {
      reinterpret_cast<uint16_t*>(tile + 2048)[r] = sc[row * (cols / 64) + ks];
      reinterpret_cast<uint16_t*>(tile + 2304)[r] = bi[row * (cols / 64) + ks];
    }
  }
}

// ------------------------------------------------------------------ host side
namespace {

// 2-D bf16 map of a row-major [rows, cols] matrix, box [box_rows, 64], 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int rows, int cols, int box_rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct UmmaWs {
  int4* tiles;
  int* count;
  uint16_t* lat_perm;
  float* part;
};

constexpr int kMaxChunks = kReduceMaxChunks;  // split-K chunks of the small-T dense GEMM

// Workspace carve-up; sizes are bounds for any T <= max_tokens:
//   tiles: at most T*K/kMinTileRows + (experts with work) entries (kMinTileRows is the
//          smallest tile height used), lat_perm: T*K rows of L,
//   part : kMaxChunks * kDNB * max(E + L, H) fp32 partial sums.
struct WsLayout {
  size_t tiles_off, count_off, lat_off, part_off, total;
};
WsLayout ws_layout(const Dims& d, int max_tokens) {
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  // every tile list holds tiles of at least kMinTileRows rows (one expert
  // each), or shorter ones only where no expert has more slots than a tile
  // holds (one tile per expert): at most E + T*K / kMinTileRows of them
  const size_t max_tiles = (size_t)max_tokens * d.K / kMinTileRows + d.E + 1;
  WsLayout l;
  l.tiles_off = 0;
  l.count_off = up(max_tiles * sizeof(int4));
  l.lat_off = l.count_off + 256;
  l.part_off = l.lat_off + up((size_t)max_tokens * d.K * d.L * 2);
  l.total = l.part_off + up(dense_small_part_floats(std::max(d.E + d.L, d.H)) * sizeof(float));
  return l;
}

UmmaWs ws_view(const UmmaPlan& p, const Dims& d, int max_tokens) {
  const WsLayout l = ws_layout(d, max_tokens);
  uint8_t* b = static_cast<uint8_t*>(p.ws);
  UmmaWs w;
  w.tiles = reinterpret_cast<int4*>(b + l.tiles_off);
  w.count = reinterpret_cast<int*>(b + l.count_off);
  w.lat_perm = reinterpret_cast<uint16_t*>(b + l.lat_off);
  w.part = reinterpret_cast<float*>(b + l.part_off);
  return w;
}

}  // namespace

cudaError_t prepare_umma_kernels() {
  cudaError_t e = cudaFuncSetAttribute(umma_dense_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DCfg::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(umma_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GCfg::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bank2_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             B2Cfg<true>::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bank2_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             B2Cfg<false>::kSmem);
  return e;
}

UmmaPlan umma_plan(const Dims& d, int max_tokens) {
  UmmaPlan p;
  p.max_tokens = max_tokens;
  p.dims = d;
  p.ws_bytes = ws_layout(d, max_tokens).total;
  return p;
}


int umma_dense_launches() { return 1; }

cudaError_t umma_dense(const UmmaPlan& p, const uint16_t* W, int M, int K, const uint16_t* X, int T,
                       const DenseOut& o, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (o.glu && (M % 2 || !o.out_bf16)) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  constexpr int BN = GCfg::kBN;
  if (!make_map(&ma, W, M, K, kBM) || !make_map(&mb, X, T, K, BN)) return cudaErrorInvalidValue;
  const int ntile = (T + BN - 1) / BN;
  const int per = (T + ntile - 1) / ntile;
  Params prm{};
  prm.MT = (M + kBM - 1) / kBM;
  prm.KS = K / kBK;
  prm.M = M;
  prm.T = T;
  prm.tn = (per + 15) & ~15;
  prm.dout = o;
  prm.status = p.status;
  prm.limit_ns = p.limit_ns;
  const int ny = (T + prm.tn - 1) / prm.tn;
  umma_gemm_kernel<<<dim3(prm.MT, ny), kThreads, GCfg::kSmem, s>>>(ma, mb, prm);
  return cudaGetLastError();
}

// slot -> (tile << 8 | row) for every row of every tile: one warp per tile,
// its rows' entries written together (consecutive slots).
__global__ void __launch_bounds__(256) slot_tile_kernel(const int4* __restrict__ tiles, const int* __restrict__ count,
                                                        int* __restrict__ slot_tile) {
  pdl_trigger();
  pdl_wait();
  const int n_tiles = *count;
  const int lane = threadIdx.x & 31;
  const int nw = (int)((gridDim.x * blockDim.x) >> 5);
  for (int ti = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); ti < n_tiles; ti += nw) {
    const int4 t = tiles[ti];
    for (int n = lane; n < t.z; n += 32) slot_tile[t.y + n] = (ti << 8) | n;
  }
}

cudaError_t umma_stream_tiles(const UmmaPlan& p, const Work& w, int T, const Dims& d, int bn_max, int* slot_tile,
                              int split_expert, cudaStream_t s) {
  if (T * d.K <= 0) return cudaSuccess;
  if (bn_max < kMinTileRows || bn_max > 255) return cudaErrorInvalidValue;  // list capacity, slot map row field
  UmmaWs ws = ws_view(p, p.dims, p.max_tokens);
  // the list in one CTA (a scan over the active experts); the slot map,
  // T*K scattered entries, by all SMs afterwards
  build_tiles_kernel<<<1, 1024, 0, s>>>(w.active, w.offsets, bn_max, ws.tiles, ws.count, nullptr, split_expert);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !slot_tile) return e;
  const int max_tiles = std::min(p.dims.E, T * d.K) + T * d.K / kMinTileRows + 1;
  return launch_pdl(slot_tile_kernel, std::min((max_tiles + 7) / 8, 8 * p.num_sms), 256, 0, s, (const int4*)ws.tiles,
                    (const int*)ws.count, slot_tile);
}

cudaError_t bank2_tiles(const uint8_t* q, const uint16_t* sc, const uint16_t* bi, int ne, int rows, int cols,
                        uint8_t* out, size_t mat_stride_tiles, int step, int offset, cudaStream_t s) {
  if (rows % kBM || cols % 64) return cudaErrorInvalidValue;
  bank2_tiles_kernel<<<152 * 8, 256, 0, s>>>(q, sc, bi, ne, rows, cols, out, mat_stride_tiles, step, offset);
  return cudaGetLastError();
}

size_t bank2_tile_bytes(int rows, int cols) { return (size_t)(rows / kBM) * (cols / 64) * kTile2Bytes; }

// The second bank's experts: tiles [count[1], count[0]) of the tile list
// (experts >= bank2_begin, whose weights sit at index expert - bank2_begin),
// slot-ordered bf16 latent rows, gate/up with SiTU-GLU -> h, down -> o.
cudaError_t umma_bank2_experts(const UmmaPlan& p, const uint8_t* gu2_tiles, const uint8_t* d2_tiles, int bank2_begin,
                               int n_bank2, int tile_rows, const Work& w, int T, const Dims& d, cudaStream_t s) {
  const int TK = T * d.K;
  if (TK <= 0) return cudaSuccess;
  // token boxes as high as the largest MMA N of the tiles (their rows
  // rounded up to 16): 16 at decode sizes, 96 for 88-row prefill tiles
  const int box_rows = (tile_rows + 15) & ~15;
  if (tile_rows <= 0 || box_rows > kTile2MaxRows) return cudaErrorInvalidValue;  // box room and TMEM layout
  UmmaWs ws = ws_view(p, p.dims, p.max_tokens);
  gather_rows_kernel<<<152 * 8, 256, 0, s>>>(w.lat, w.perm, TK, d.K, d.L, ws.lat_perm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mb1, mb2;
  if (!make_map(&mb1, ws.lat_perm, TK, d.L, box_rows) || !make_map(&mb2, w.h, TK, d.I, box_rows))
    return cudaErrorInvalidValue;
  // at most one tile per second-bank expert with work plus one per 16 slots
  const int max_tiles = std::min(n_bank2, TK) + TK / kMinTileRows + 1;
  Params g{};
  g.a_tiles = gu2_tiles;
  g.expert_base = bank2_begin;
  g.MT = d.I / kBM;
  g.KS = d.L / kBK;
  g.M = d.I;
  g.list = TileList{ws.tiles, ws.count, ws.count + 1};
  g.out_bf16 = w.h;
  g.ld_out = d.I;
  g.beta = d.beta;
  g.beta_lin = d.beta_lin;
  g.status = p.status;
  g.limit_ns = p.limit_ns;
  g.tn = box_rows;
  // persistent: one CTA per SM at most (the items are counted on the device)
  bank2_gemm_kernel<true><<<std::min(p.num_sms, g.MT * max_tiles), B2Cfg<true>::kThreads, B2Cfg<true>::kSmem, s>>>(
      mb1, g);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  Params dn = g;
  dn.a_tiles = d2_tiles;
  dn.MT = d.L / kBM;
  dn.KS = d.I / kBK;
  dn.M = d.L;
  dn.out_bf16 = nullptr;
  dn.out_f32 = w.o;
  dn.ld_out = d.L;
  bank2_gemm_kernel<false><<<std::min(p.num_sms, dn.MT * max_tiles), B2Cfg<false>::kThreads, B2Cfg<false>::kSmem,
                             s>>>(mb2, dn);
  return cudaGetLastError();
}

void umma_tile_list(const UmmaPlan& p, int4** tiles, int** count, int* bn_max) {
  UmmaWs ws = ws_view(p, p.dims, p.max_tokens);
  *tiles = ws.tiles;
  *count = ws.count;
  *bn_max = kMinTileRows;
}

size_t dense_small_part_floats(int M) { return (size_t)kMaxChunks * kDNB * (size_t)M; }
int umma_dense_small_launches() { return 2; }

cudaError_t umma_dense_small(const UmmaPlan& p, const uint16_t* W, int M, int K, const uint16_t* X, int T,
                             const DenseOut& o, float* part, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (T > kDNB || M % 4 || (o.glu && !o.out_bf16)) return cudaErrorInvalidValue;
  if (!part) {
    if ((size_t)M > (size_t)std::max(p.dims.E + p.dims.L, p.dims.H)) return cudaErrorInvalidValue;
    part = ws_view(p, p.dims, p.max_tokens).part;
  }
  CUtensorMap ma, mb;
  const int n_mma = (T + 15) & ~15;  // token rows per box (the MMA's N)
  if (!make_map(&ma, W, M, K, kBM) || !make_map(&mb, X, T, K, n_mma)) return cudaErrorInvalidValue;
  DenseStreamParams q{};
  q.MT = (M + kBM - 1) / kBM;
  q.KS = K / kBK;
  q.b_bytes = (uint32_t)(n_mma * kBK * 2);
  // K chunks per row tile: as many as keep every (row tile, chunk) item in
  // one wave of the grid (a second wave for a few items doubles the time)
  const int fit = (2 * p.num_sms) / q.MT;
  const int nkc0 = std::max(1, std::min({fit, q.KS, kMaxChunks}));
  q.ks_per_chunk = (q.KS + nkc0 - 1) / nkc0;
  q.nkc = (q.KS + q.ks_per_chunk - 1) / q.ks_per_chunk;
  q.M = M;
  q.T = T;
  q.part = part;
  q.status = p.status;
  q.limit_ns = p.limit_ns;
  const int items = q.MT * q.nkc;
  cudaError_t e =
      launch_pdl(umma_dense_stream_kernel, std::min(items, 2 * p.num_sms), kDThreads, DCfg::kSmem, s, ma, mb, q);
  if (e != cudaSuccess) return e;
  const long long threads = (long long)T * (M / 4);
  const int blocks = (int)std::min<long long>((threads + 255) / 256, 8LL * p.num_sms);
  return launch_pdl(dense_reduce_kernel, blocks, 256, 0, s, (const float*)part, q.nkc, T, M, o);
}

}  // namespace k3
