// k3moe_bs.cu -- MXFP4 expert GEMMs on the block-scaled tensor cores.
//
// tcgen05.mma kind::mxf8f6f4 multiplies e2m1 (A) by e4m3 (B) with one
// UE8M0 scale per 32 elements of K on each side and accumulates in fp32:
//   D[m, n] += sum_k (a[m, k] 2^(SA[m, k/32]-127)) (b[n, k] 2^(SB[n, k/32]-127)).
// A is an expert weight exactly as the checkpoint stores it (e2m1 nibbles,
// low nibble first; e8m0 scale per 32 along the input dimension: kimi-k3-mlx
// README, "Tiers"; K3_ARTIFACT_AUDIT section 4.3), so no CUDA-core work
// touches the weights: TMA moves the packed nibbles into shared memory in
// the 16-byte-slot layout the tensor core reads (16U4_ALIGN16B), and the
// scales go to tensor memory with tcgen05.cp.
//
// B carries the bf16 activations (latent rows, then h) as two e4m3 terms
// per element with per-32 scales:  x = q0 2^(S0-127) + q1 2^(S1-127),
//   S0 = max(E - 7, 0) for the block's largest biased bf16 exponent E, so
//        |x| 2^(127-S0) < 2^8 (inside e4m3's range), q0 = RN_e4m3 of that;
//   S1 = max(S0 - 4, 0), q1 = RN_e4m3((x 2^(127-S0) - q0) 2^(S0-S1)).
// The first term keeps the top 4 significant bits, the remainder has at
// most 4 more, so the split is exact for every element within 2^13 of its
// block's largest magnitude; smaller elements keep an absolute error below
// 2^(S0-127-13).  Two MMAs (one per term) accumulate into the same D.
//
// Tile scheme (decode sizes): M = 128 weight rows, N = 32 token rows (one
// tile of the expert's slots), K = 128 input columns per stage (four MMAs of
// K = 32 per term and matrix).  Warp 0 issues the copies, warp 1 the MMAs,
// warps 2..5 run the epilogue from a double-buffered accumulator.  Every
// wait is bounded (status bit + shared abort flag, as in the bf16 kernels).
#include <cuda.h>

#include <algorithm>

#include "k3moe_bs.h"
#include "k3moe_device.cuh"
#include "k3moe_tc.cuh"

namespace k3 {

namespace {

constexpr int kQM = 128;   // weight rows per tile (MMA M)
constexpr int kQN = 32;    // token rows per tile (MMA N)
constexpr int kQK = 128;   // input columns per stage
constexpr int kAtom = 512; // scale bytes per 128 rows x 128 columns
constexpr int kBsThreads = 192;
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

// Slot-ordered rows: dst row s = src row (perm ? perm[s] / K : s).  A half
// warp covers 128 columns (8 per lane, 4 lanes per scale block); the loop
// runs per warp so that both halves always meet at the shuffles.
__global__ void quant_rows_kernel(const uint16_t* __restrict__ src, const int* __restrict__ perm, int K, int rows,
                                  int C, uint8_t* __restrict__ q0, uint8_t* __restrict__ q1, uint8_t* __restrict__ sf0,
                                  uint8_t* __restrict__ sf1) {
  const int hl = threadIdx.x & 15, half = (threadIdx.x >> 4) & 1;
  const int KC = C / kQK;
  const long long nwork = (long long)rows * KC;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long wi = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; 2 * wi < nwork; wi += nwarps) {
    const long long i = 2 * wi + half;
    const bool valid = i < nwork;
    const int s = valid ? (int)(i / KC) : 0, kc = valid ? (int)(i - (long long)s * KC) : 0;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (valid) {
      const int t = perm ? perm[s] / K : s;
      v = *reinterpret_cast<const uint4*>(src + (size_t)t * C + kc * kQK + hl * 8);
    }
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
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
    if (!valid) continue;
    const size_t off = (size_t)s * C + kc * kQK + hl * 8;
    *reinterpret_cast<uint2*>(q0 + off) = make_uint2(a0, b0);
    *reinterpret_cast<uint2*>(q1 + off) = make_uint2(a1, b1);
    if ((hl & 3) == 0) {
      const size_t so = ((size_t)s * KC + kc) * 16 + (hl >> 2);
      sf0[so] = (uint8_t)s0;
      sf1[so] = (uint8_t)s1;
    }
  }
}

// ------------------------------------------------------------------ tcgen05 block-scaled pieces
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
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
// UE8M0 scales, M = 128, N = 32, scale-factor ids (byte of the scale column).
__device__ __forceinline__ uint32_t bs_idesc(uint32_t sfa_id, uint32_t sfb_id) {
  return (sfb_id << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(kQN >> 3) << 17) | (1u << 23) |
         ((uint32_t)(kQM >> 4) << 24) | (sfa_id << 29);
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

template <int MODE>
struct BsCfg {
  static constexpr int kNumA = (MODE == BS_GATEUP) ? 2 : 1;
  static constexpr int kA = kQM * kQK;  // e2m1 tile in 16-byte slots (8 data + 8 padding bytes per 16 codes)
  static constexpr int kB = kQN * kQK;  // one e4m3 term
  static constexpr int kOffB = kNumA * kA;
  static constexpr int kOffSfa = kOffB + 2 * kB;
  static constexpr int kOffSfb = kOffSfa + kNumA * kAtom;
  static constexpr int kStageBytes = (kOffSfb + 2 * kAtom + 1023) / 1024 * 1024;
  static constexpr int kStages = (MODE == BS_GATEUP) ? 5 : 8;
  static constexpr uint32_t kTx = kNumA * kA + 2 * kB + kNumA * kAtom + 2 * kAtom;
  static constexpr int kDCols = kNumA * kQN;      // one accumulator buffer (gate, up)
  static constexpr int kSfCols = 4 * (kNumA + 2); // scale columns per stage: SFA per matrix, SFB per term
  static constexpr int kSfBase = 2 * kDCols;
  static constexpr int kTmemCols = 256;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
  static_assert(kSfBase + kStages * kSfCols <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct BsParams {
  const uint8_t* sfa;  // weight scale atoms
  int MT, KC;          // weight row tiles, input-column chunks
  const int4* tiles;   // {expert, first slot, rows, -}
  const int* count;
  int ld_out;          // GATEUP: I, DOWN: L
  uint16_t* h;         // GATEUP outputs
  uint8_t *hq0, *hq1, *hsf0, *hsf1;
  float* o;            // DOWN output
  float beta, beta_lin;
  unsigned* status;
  uint64_t limit_ns;
};

template <int MODE>
__global__ void __launch_bounds__(kBsThreads, 1)
    bs_stream_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_q0,
                     const __grid_constant__ CUtensorMap map_q1, const __grid_constant__ CUtensorMap map_s0,
                     const __grid_constant__ CUtensorMap map_s1, const BsParams p) {
  using C = BsCfg<MODE>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  // bars: full[S], free[S], dfull[2], dempty[2], drain
  constexpr int NB = 2 * C::kStages + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NB);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_items = *p.count * p.MT;
  if ((int)blockIdx.x >= n_items) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) {
      const bool is_empty = i >= 2 * C::kStages + 2 && i < 2 * C::kStages + 4;
      mbar_init(smem_u32(bars + i), is_empty ? 128u : 1u);
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
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int4 tile = p.tiles[item / p.MT];
        const int mt = item - (item / p.MT) * p.MT;
        const int z = (MODE == BS_GATEUP) ? 2 * tile.x : tile.x;
        const uint8_t* sfa = p.sfa + (((size_t)tile.x * p.MT + mt) * p.KC) * C::kNumA * kAtom;
        for (int kc = 0; kc < p.KC; ++kc, ++kg) {
          const int s = kg % C::kStages, u = kg / C::kStages;
          if (u > 0 && !mbar_wait(sfree(s), (u - 1) & 1, g, 1u)) {
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(stage(s));
          mbar_expect_tx(full(s), C::kTx);
          tma_load_3d(st, &map_a, full(s), kc * kQK, mt * kQM, z);
          if (MODE == BS_GATEUP) tma_load_3d(st + C::kA, &map_a, full(s), kc * kQK, mt * kQM, z + 1);
          tma_load_2d(st + C::kOffB, &map_q0, full(s), kc * kQK, tile.y);
          tma_load_2d(st + C::kOffB + C::kB, &map_q1, full(s), kc * kQK, tile.y);
          bulk_load(st + C::kOffSfa, sfa + (size_t)kc * C::kNumA * kAtom, C::kNumA * kAtom, full(s));
          tma_load_2d(st + C::kOffSfb, &map_s0, full(s), kc * 16, tile.y);
          tma_load_2d(st + C::kOffSfb + kAtom, &map_s1, full(s), kc * 16, tile.y);
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
    // ================= MMA issue
    if (lane == 0) {
      int kg = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
        const int buf = it & 1;
        if (it >= 2 && !mbar_wait(dempty(buf), ((it >> 1) - 1) & 1, g, 2u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + buf * C::kDCols;
        for (int kc = 0; kc < p.KC; ++kc, ++kg) {
          const int s = kg % C::kStages;
          if (!mbar_wait(full(s), (kg / C::kStages) & 1, g, 4u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(stage(s));
          const uint32_t sfc = tmem + C::kSfBase + s * C::kSfCols;
#pragma unroll
          for (int a = 0; a < C::kNumA; ++a) tc_cp_scales(sfc + 4 * a, sf_desc(st + C::kOffSfa + a * kAtom));
          tc_cp_scales(sfc + 4 * C::kNumA, sf_desc(st + C::kOffSfb));
          tc_cp_scales(sfc + 4 * C::kNumA + 4, sf_desc(st + C::kOffSfb + kAtom));
#pragma unroll
          for (int kb = 0; kb < kQK / 32; ++kb) {
            const uint32_t idesc = bs_idesc(kb, kb);
#pragma unroll
            for (int a = 0; a < C::kNumA; ++a)
#pragma unroll
              for (int t = 0; t < 2; ++t)
                umma_bs(d0 + a * kQN, umma_desc_sw128(st + a * C::kA + kb * 32),
                        umma_desc_sw128(st + C::kOffB + t * C::kB + kb * 32), idesc, sfc + 4 * a,
                        sfc + 4 * C::kNumA + 4 * t, (kc | kb | t) ? 1u : 0u);
          }
          umma_commit(sfree(s));
        }
        if (!ok) break;
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
    // ================= epilogue (warps 2..5: lane quarter warp % 4)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
      const int buf = it & 1;
      if (!mbar_wait(dfull(buf), (it >> 1) & 1, g, 8u)) break;
      tc_fence_after();
      const int4 tile = p.tiles[item / p.MT];
      const int mt = item - (item / p.MT) * p.MT;
      const int m = mt * kQM + r;
      float acc[32];
      tmem_ld32(lane_base + buf * C::kDCols, acc);
      if (MODE == BS_GATEUP) {
        float up[32];
        tmem_ld32(lane_base + buf * C::kDCols + kQN, up);
        tc_fence_before();
        mbar_arrive(dempty(buf));
        const int KCo = p.ld_out / kQK;
        const int b = m >> 5;
#pragma unroll
        for (int j = 0; j < kQN; ++j) {
          if (j < tile.z) {
            const size_t row = (size_t)(tile.y + j);
            const uint16_t hb = f32_to_bf16(situ_fast(acc[j], up[j], p.beta, p.beta_lin));
            p.h[row * p.ld_out + m] = hb;
            const uint32_t emax = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(hb >> 7) & 0xFFu);
            const uint32_t s0 = term0_scale(emax), s1 = term1_scale(s0);
            const uint32_t q = split_e4m3(bf16_to_f32(hb), s0, s1);
            p.hq0[row * p.ld_out + m] = (uint8_t)q;
            p.hq1[row * p.ld_out + m] = (uint8_t)(q >> 8);
            if (lane == 0) {
              const size_t so = (row * KCo + (b >> 2)) * 16 + (b & 3);
              p.hsf0[so] = (uint8_t)s0;
              p.hsf1[so] = (uint8_t)s1;
            }
          }
        }
      } else {
        tc_fence_before();
        mbar_arrive(dempty(buf));
#pragma unroll
        for (int j = 0; j < kQN; ++j)
          if (j < tile.z) p.o[(size_t)(tile.y + j) * p.ld_out + m] = acc[j];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

// ------------------------------------------------------------------ host helpers
// e2m1 weights [nmat][rows][cols/2] as a 3-D map, box 128 codes x 128 rows,
// landing in 16-byte slots with a 128-byte swizzle.
bool map_e2m1(CUtensorMap* map, const void* base, int nmat, int rows, int cols) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)nmat};
  const cuuint64_t strides[2] = {(cuuint64_t)cols / 2, (cuuint64_t)rows * cols / 2};
  const cuuint32_t box[3] = {(cuuint32_t)kQK, (cuuint32_t)kQM, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// bytes [rows][cols], box box_cols x box_rows
bool map_u8(CUtensorMap* map, const void* base, int rows, int cols, int box_rows, int box_cols,
            CUtensorMapSwizzle sw) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct BsWs {
  uint8_t *lq0, *lq1, *lsf0, *lsf1;  // latent rows, slot order [TKmax][L], [TKmax][L/128][16]
  uint8_t *hq0, *hq1, *hsf0, *hsf1;  // h rows [TKmax][I], [TKmax][I/128][16]
  size_t total;
};
BsWs bs_ws_view(void* base, const Dims& d, int max_tokens) {
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  const size_t TK = (size_t)std::min(max_tokens, kBsMaxTokens) * d.K;
  const size_t sizes[8] = {TK * d.L, TK * d.L, TK * d.L / 8, TK * d.L / 8, TK * d.I, TK * d.I, TK * d.I / 8,
                           TK * d.I / 8};
  uint8_t* b = static_cast<uint8_t*>(base);
  uint8_t* ptr[8];
  size_t off = 0;
  for (int i = 0; i < 8; ++i) {
    ptr[i] = b ? b + off : nullptr;
    off += up(sizes[i]);
  }
  return BsWs{ptr[0], ptr[1], ptr[2], ptr[3], ptr[4], ptr[5], ptr[6], ptr[7], off};
}

template <int MODE>
cudaError_t launch_bs(const BsPlan& p, const uint8_t* wq, const uint8_t* sfa, int nmat, int rows, int cols,
                      const uint8_t* q0, const uint8_t* q1, const uint8_t* sf0, const uint8_t* sf1, int TK,
                      const int4* tiles, const int* count, BsParams prm, cudaStream_t s) {
  CUtensorMap ma, m0, m1, s0, s1;
  const int KC = cols / kQK;
  if (!map_e2m1(&ma, wq, nmat, rows, cols) || !map_u8(&m0, q0, TK, cols, kQN, kQK, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !map_u8(&m1, q1, TK, cols, kQN, kQK, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !map_u8(&s0, sf0, TK, KC * 16, kQN, 16, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !map_u8(&s1, sf1, TK, KC * 16, kQN, 16, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  prm.sfa = sfa;
  prm.MT = rows / kQM;
  prm.KC = KC;
  prm.tiles = tiles;
  prm.count = count;
  prm.status = p.status;
  prm.limit_ns = p.limit_ns;
  bs_stream_kernel<MODE><<<p.num_sms, kBsThreads, BsCfg<MODE>::kSmem, s>>>(ma, m0, m1, s0, s1, prm);
  return cudaGetLastError();
}

}  // namespace

size_t bs_weight_bytes(const Dims& d) {
  const size_t E = d.E, I = d.I, L = d.L;
  return E * 2 * I * L / 2 + E * 2 * I * L / 32 + E * L * I / 2 + E * L * I / 32;
}

cudaError_t bs_scale_atoms(const uint8_t* scale, int ne, int rows, int cols, int n_mat, int mat, uint8_t* out,
                           cudaStream_t s) {
  scale_atoms_kernel<<<1024, 256, 0, s>>>(scale, ne, rows, cols, n_mat, mat, out);
  return cudaGetLastError();
}

size_t bs_ws_bytes(const Dims& d, int max_tokens) { return bs_ws_view(nullptr, d, max_tokens).total; }

cudaError_t prepare_bs_kernels() {
  cudaError_t e = cudaFuncSetAttribute(bs_stream_kernel<BS_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BsCfg<BS_GATEUP>::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bs_stream_kernel<BS_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BsCfg<BS_DOWN>::kSmem);
  return e;
}

cudaError_t bs_quantize_latent(const BsPlan& p, const Work& w, int T, const Dims& d, cudaStream_t s) {
  const int TK = T * d.K;
  if (TK <= 0) return cudaSuccess;
  if (T > std::min(p.max_tokens, kBsMaxTokens)) return cudaErrorInvalidValue;
  const BsWs ws = bs_ws_view(p.ws, d, p.max_tokens);
  const long long halves = (long long)TK * (d.L / kQK);
  const int blocks = (int)std::min<long long>((halves * 16 + 255) / 256, 4LL * p.num_sms);
  quant_rows_kernel<<<blocks, 256, 0, s>>>(w.lat, w.perm, d.K, TK, d.L, ws.lq0, ws.lq1, ws.lsf0, ws.lsf1);
  return cudaGetLastError();
}

cudaError_t bs_stream_gateup(const BsPlan& p, const BsWeights& bw, const int4* tiles, const int* tile_count,
                             const Work& w, int T, const Dims& d, cudaStream_t s) {
  const int TK = T * d.K;
  if (TK <= 0) return cudaSuccess;
  if (T > std::min(p.max_tokens, kBsMaxTokens)) return cudaErrorInvalidValue;
  const BsWs ws = bs_ws_view(p.ws, d, p.max_tokens);
  BsParams prm{};
  prm.ld_out = d.I;
  prm.h = w.h;
  prm.hq0 = ws.hq0;
  prm.hq1 = ws.hq1;
  prm.hsf0 = ws.hsf0;
  prm.hsf1 = ws.hsf1;
  prm.beta = d.beta;
  prm.beta_lin = d.beta_lin;
  return launch_bs<BS_GATEUP>(p, bw.gu_q, bw.gu_sf, 2 * d.E, d.I, d.L, ws.lq0, ws.lq1, ws.lsf0, ws.lsf1, TK, tiles,
                              tile_count, prm, s);
}

cudaError_t bs_stream_down(const BsPlan& p, const BsWeights& bw, const int4* tiles, const int* tile_count,
                           const Work& w, int T, const Dims& d, cudaStream_t s) {
  const int TK = T * d.K;
  if (TK <= 0) return cudaSuccess;
  if (T > std::min(p.max_tokens, kBsMaxTokens)) return cudaErrorInvalidValue;
  const BsWs ws = bs_ws_view(p.ws, d, p.max_tokens);
  BsParams prm{};
  prm.ld_out = d.L;
  prm.o = w.o;
  return launch_bs<BS_DOWN>(p, bw.d_q, bw.d_sf, d.E, d.L, d.I, ws.hq0, ws.hq1, ws.hsf0, ws.hsf1, TK, tiles,
                            tile_count, prm, s);
}

}  // namespace k3
