// k3moe_decode.cu -- the layer's CUDA-core kernels: dense GEMV for small
// token counts, router top-K, the token->expert permutation, the grouped
// MXFP4 expert GEMVs (gate/up with the SiTU-GLU epilogue, and down), the
// weighted combine + RMSNorm, and the MXFP4 re-layout / dequant kernels.
//
// At decode sizes every one of these is bound by HBM bandwidth (the expert
// kernels stream MXFP4 tiles once; per weight they issue about two
// instructions), so they are written as streaming kernels: coalesced
// 16-byte loads, work items sized so the grid covers the 152 SMs several
// times, activations staged once per CTA in shared memory.
#include <algorithm>
#include <cfloat>
#include <climits>

#include "k3moe_device.cuh"
#include "k3moe_internal.h"

namespace k3 {

// =====================================================================
// Dense GEMV:  Y[t, m] = sum_k W[m, k] * X[t, k]
//   W bf16 [M, K] row-major, X bf16 [T, K]; fp32 accumulation.
//   rows m <  split -> out_f32 [t * split + m]            (router logits)
//   rows m >= split -> out_bf16[t * (M - split) + m - split] (bf16, RNE)
// One warp owns two rows; lanes stride over K in 16-byte vectors; tokens
// are processed TG at a time (each pass re-reads the rows).
// =====================================================================
template <int TG>
__global__ void __launch_bounds__(256) dense_gemv_kernel(const uint16_t* __restrict__ W, int M, int K,
                                                         const uint16_t* __restrict__ X, int T, int split,
                                                         float* __restrict__ out_f32,
                                                         uint16_t* __restrict__ out_bf16) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = (blockIdx.x * 8 + warp) * 2;
  if (m0 >= M) return;
  const bool has1 = (m0 + 1) < M;
  const uint4* w0 = reinterpret_cast<const uint4*>(W + (size_t)m0 * K);
  const uint4* w1 = reinterpret_cast<const uint4*>(W + (size_t)(has1 ? m0 + 1 : m0) * K);
  const int nvec = K >> 3;
  for (int t0 = 0; t0 < T; t0 += TG) {
    const int tn = min(TG, T - t0);
    float acc0[TG], acc1[TG];
#pragma unroll
    for (int t = 0; t < TG; ++t) acc0[t] = acc1[t] = 0.f;
    for (int v0 = lane; v0 < nvec; v0 += 32 * 4) {
      uint4 a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + 32 * u;
        if (v < nvec) {
          a[u] = __ldg(w0 + v);
          b[u] = __ldg(w1 + v);
        } else {
          a[u] = b[u] = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + 32 * u;
        if (v >= nvec) break;
        const uint32_t wa[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
        const uint32_t wb[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
#pragma unroll
        for (int t = 0; t < TG; ++t) {
          if (t < tn) {
            const uint4 xv = __ldg(reinterpret_cast<const uint4*>(X + (size_t)(t0 + t) * K) + v);
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 xf = unpack_bf16x2(xw[i]);
              const float2 fa = unpack_bf16x2(wa[i]);
              const float2 fb = unpack_bf16x2(wb[i]);
              acc0[t] = fmaf(fa.x, xf.x, acc0[t]);
              acc0[t] = fmaf(fa.y, xf.y, acc0[t]);
              acc1[t] = fmaf(fb.x, xf.x, acc1[t]);
              acc1[t] = fmaf(fb.y, xf.y, acc1[t]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TG; ++t) {
      if (t >= tn) break;
      const float s0 = warp_sum(acc0[t]);
      const float s1 = warp_sum(acc1[t]);
      if (lane == 0) {
        const int tt = t0 + t;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int m = m0 + rr;
          if (rr == 1 && !has1) break;
          const float v = rr ? s1 : s0;
          if (m < split)
            out_f32[(size_t)tt * split + m] = v;
          else
            out_bf16[(size_t)tt * (M - split) + (m - split)] = f32_to_bf16(v);
        }
      }
    }
  }
}

cudaError_t launch_dense_gemv(const uint16_t* W, int M, int K, const uint16_t* X, int T, int split,
                              float* out_f32, uint16_t* out_bf16, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int blocks = (M + 15) / 16;
  if (T <= 1)
    dense_gemv_kernel<1><<<blocks, 256, 0, s>>>(W, M, K, X, T, split, out_f32, out_bf16);
  else if (T <= 2)
    dense_gemv_kernel<2><<<blocks, 256, 0, s>>>(W, M, K, X, T, split, out_f32, out_bf16);
  else if (T <= 4)
    dense_gemv_kernel<4><<<blocks, 256, 0, s>>>(W, M, K, X, T, split, out_f32, out_bf16);
  else
    dense_gemv_kernel<8><<<blocks, 256, 0, s>>>(W, M, K, X, T, split, out_f32, out_bf16);
  return cudaGetLastError();
}

// =====================================================================
// Router top-K (kimi-k3-mlx README, "Architecture" table: sigmoid router,
// e_score_correction_bias added for selection only).  One CTA per token:
//   s[e] = 1 / (1 + exp(-logit[e])),  key[e] = s[e] + bias[e] (fp32);
//   the K largest keys (ties -> lower expert id), in descending key order;
//   w[k] = s[idx[k]] / sum_k s[idx[k]] * rsf (sum in k order, fp32), or
//   s * rsf without renormalisation.
// The K-th largest key is found exactly by a most-significant-digit-first
// radix select (four 8-bit digits) over an order-preserving integer image of
// the fp32 keys; keys above it are taken, keys equal to it by ascending id.
// The K winners are then ordered by (key desc, id asc) with a warp bitonic
// sort.  256 threads, ceil(E / 256) keys per thread.
// =====================================================================
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <int EPT>
__global__ void __launch_bounds__(256) topk_cta_kernel(const float* __restrict__ logits, int E, int ld,
                                                       const float* __restrict__ bias, int K, int norm_topk,
                                                       float rsf, int32_t* __restrict__ idx,
                                                       float* __restrict__ w) {
  __shared__ int hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need, n_cand, n_eq;
  __shared__ unsigned long long cand[32];
  __shared__ float cand_s[32];
  __shared__ int eq_e[2048];
  __shared__ float eq_s[2048];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* row = logits + (size_t)t * ld;
  uint32_t u[EPT];
  float sc[EPT];
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int e = tid + 256 * j;
    u[j] = 0u;  // below every key's image (the image of -inf is 0x007FFFFF)
    sc[j] = 0.f;
    if (e < E) {
      const float sg = 1.0f / (1.0f + expf(-row[e]));
      sc[j] = sg;
      u[j] = ordered_bits(sg + bias[e]);
    }
  }
  // ---- radix select of the K-th largest image
  uint32_t prefix = 0u;
  int need = K;
#pragma unroll 1
  for (int pass = 3; pass >= 0; --pass) {
    const int shift = 8 * pass;
    const uint32_t hmask = pass == 3 ? 0u : (0xFFFFFFFFu << (shift + 8));
    hist[tid] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < EPT; ++j)
      if (u[j] != 0u && (u[j] & hmask) == prefix) atomicAdd(&hist[(u[j] >> shift) & 255u], 1);
    __syncthreads();
    if (warp == 0) {
      // lane l holds digits 255-8l .. 248-8l (descending)
      int c[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[255 - 8 * lane - i];
        tot += c[i];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
      }
      const int excl = incl - tot;
      const unsigned owner = __ballot_sync(0xFFFFFFFFu, excl < need && need <= incl);
      if (lane == __ffs(owner) - 1) {
        int acc = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc + c[i] >= need) {
            s_prefix = prefix | ((uint32_t)(255 - 8 * lane - i) << shift);
            s_need = need - acc;
            break;
          }
          acc += c[i];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
  }
  // ---- the K winners: images above the K-th, then `need` of the equal ones by ascending id
  if (tid == 0) {
    n_cand = 0;
    n_eq = 0;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int e = tid + 256 * j;
    if (u[j] > prefix) {
      const int k = atomicAdd(&n_cand, 1);
      cand[k] = ((unsigned long long)u[j] << 32) | (0xFFFFFFFFu - (uint32_t)e);
      cand_s[k] = sc[j];
    } else if (u[j] == prefix && u[j] != 0u) {
      const int k = atomicAdd(&n_eq, 1);
      eq_e[k] = e;
      eq_s[k] = sc[j];
    }
  }
  __syncthreads();
  if (tid == 0) {
    int k = n_cand;
    // the `need` lowest ids among the equal keys (all of them in the usual case need == n_eq)
    for (int r = 0; r < need; ++r) {
      int best = -1;
      for (int i = 0; i < n_eq; ++i)
        if (eq_e[i] >= 0 && (best < 0 || eq_e[i] < eq_e[best])) best = i;
      cand[k] = ((unsigned long long)prefix << 32) | (0xFFFFFFFFu - (uint32_t)eq_e[best]);
      cand_s[k] = eq_s[best];
      eq_e[best] = -1;
      ++k;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // bitonic sort of the K (<= 32) winners, descending; lanes >= K hold 0
    unsigned long long v = lane < K ? cand[lane] : 0ull;
    float sv = lane < K ? cand_s[lane] : 0.f;
#pragma unroll
    for (int k2 = 2; k2 <= 32; k2 <<= 1) {
#pragma unroll
      for (int j2 = k2 >> 1; j2 > 0; j2 >>= 1) {
        const unsigned long long ov = __shfl_xor_sync(0xFFFFFFFFu, v, j2);
        const float os = __shfl_xor_sync(0xFFFFFFFFu, sv, j2);
        const bool up = (lane & k2) == 0;      // this block sorts descending when up
        const bool lower = (lane & j2) == 0;   // this lane keeps the larger value when lower == up
        const bool take = (lower == up) ? (ov > v) : (ov < v);
        if (take) {
          v = ov;
          sv = os;
        }
      }
    }
    float sum = 0.f;
    for (int k = 0; k < K; ++k) sum += __shfl_sync(0xFFFFFFFFu, sv, k);
    if (lane < K) {
      idx[(size_t)t * K + lane] = (int32_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
      w[(size_t)t * K + lane] = (norm_topk ? sv / sum : sv) * rsf;
    }
  }
}

cudaError_t launch_topk(const float* logits, int T, int E, int ld, const float* bias, int K, int norm_topk,
                        float rsf, int32_t* idx, float* w, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (K > 32 || E > 2048 || K > E) return cudaErrorInvalidValue;
  auto kernel = E <= 256 ? topk_cta_kernel<1> : E <= 1024 ? topk_cta_kernel<4> : topk_cta_kernel<8>;
  return launch_pdl(kernel, T, 256, 0, s, logits, E, ld, bias, K, norm_topk, rsf, idx, w);
}

// =====================================================================
// Token -> expert permutation ("sort the (token, expert) pairs by expert",
// kimi-k3-mlx README, REAP section): counts, offsets, a stable order of the
// T*K assignments grouped by expert (slot -> t*K + k), its inverse, and the
// list of experts that received work.  Three kernels; deterministic.
// =====================================================================
__global__ void __launch_bounds__(kPermChunk) perm_hist_kernel(const int32_t* __restrict__ idx, int TK, int E,
                                                               ExpertShard sh, int* __restrict__ blk_hist) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int a = blockIdx.x * kPermChunk + threadIdx.x;
  if (a < TK) atomicAdd(&hist[sh.bucket(idx[a])], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blk_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int wv = warp_tot[lane];
    int wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += n;
    }
    warp_tot[lane] = wi - wv;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + incl - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) perm_scan_kernel(int* __restrict__ blk_hist, int nblk, int E, int TK,
                                                         ExpertShard sh, int* __restrict__ counts,
                                                         int* __restrict__ offsets, int* __restrict__ active) {
  __shared__ int warp_tot[32];
  __shared__ int total_s, carry_off, carry_act;
  if (threadIdx.x == 0) {
    carry_off = 0;
    carry_act = 0;
  }
  __syncthreads();
  for (int e0 = 0; e0 < E; e0 += 1024) {
    const int e = e0 + threadIdx.x;
    int tot = 0;
    if (e < E) {
      // per-block prefix of this expert's count, in block order
      for (int b = 0; b < nblk; ++b) {
        const int c = blk_hist[(size_t)b * E + e];
        blk_hist[(size_t)b * E + e] = tot;
        tot += c;
      }
      counts[e] = tot;
    }
    const int ex = block_exclusive_scan(tot, warp_tot, &total_s);
    const int add_off = carry_off;
    if (e < E) offsets[e] = add_off + ex;
    const int flag = (e < sh.n_listed && tot > 0) ? 1 : 0;
    const int add_tot = total_s;
    const int ax = block_exclusive_scan(flag, warp_tot, &total_s);
    if (flag) active[1 + carry_act + ax] = e;
    __syncthreads();
    if (threadIdx.x == 0) {
      carry_off += add_tot;
      carry_act += total_s;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    offsets[E] = TK;
    active[0] = carry_act;
  }
}

__global__ void __launch_bounds__(kPermChunk) perm_scatter_kernel(const int32_t* __restrict__ idx, int TK, int E,
                                                                  ExpertShard sh, const int* __restrict__ blk_prefix,
                                                                  const int* __restrict__ offsets,
                                                                  int* __restrict__ perm, int* __restrict__ slot) {
  extern __shared__ int run[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) run[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int a = blockIdx.x * kPermChunk + threadIdx.x;
  const bool valid = a < TK;
  const int e = valid ? sh.bucket(idx[a]) : -1;
  const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  const bool leader = (__ffs(peers) - 1) == lane;
  int base = 0;
  for (int w = 0; w < kPermChunk / 32; ++w) {
    if (warp == w && valid) {
      base = run[e];
      __syncwarp(peers);
      if (leader) run[e] = base + __popc(peers);
    }
    __syncthreads();
  }
  if (valid) {
    const int s = offsets[e] + blk_prefix[(size_t)blockIdx.x * E + e] + base + rank;
    perm[s] = a;
    slot[a] = s;
  }
}

cudaError_t launch_permute(const int32_t* idx, int T, int K, const ExpertShard& sh, int* blk_hist, int* counts,
                           int* offsets, int* active, int* perm, int* slot, cudaStream_t s) {
  const int TK = T * K;
  if (TK <= 0) return cudaSuccess;
  const int E = sh.n_buckets;
  const int nblk = (TK + kPermChunk - 1) / kPermChunk;
  const size_t sm = sizeof(int) * (size_t)E;
  perm_hist_kernel<<<nblk, kPermChunk, sm, s>>>(idx, TK, E, sh, blk_hist);
  perm_scan_kernel<<<1, 1024, 0, s>>>(blk_hist, nblk, E, TK, sh, counts, offsets, active);
  perm_scatter_kernel<<<nblk, kPermChunk, sm, s>>>(idx, TK, E, sh, blk_hist, offsets, perm, slot);
  return cudaGetLastError();
}

// =====================================================================
// Permutation for small batches (T*K <= 1024) in ONE CTA, from the top-K
// of the top-K kernel: the per-expert histogram, offsets, active list, the
// stable slot order and its inverse (same results as the three
// permutation kernels), and the tile list of the streaming expert kernels
// (tiles of at most bn_max slots per expert: {expert, first slot, rows,
// rows rounded up to 16}).
// =====================================================================
__global__ void __launch_bounds__(1024) perm_small_kernel(const int32_t* __restrict__ idx, int T, int E, int K,
                                                          ExpertShard sh, int* __restrict__ counts,
                                                          int* __restrict__ offsets,
                                                          int* __restrict__ active, int* __restrict__ perm,
                                                          int* __restrict__ slot, int bn_max,
                                                          int4* __restrict__ tiles, int* __restrict__ tile_count,
                                                          int* __restrict__ slot_tile, int split_expert) {
  __shared__ int hist[2048];   // assignments per bucket, then placement cursors, then tile heights
  __shared__ int base[2048];   // first slot of each bucket, then (for active experts) first tile
  __shared__ int placed[1024]; // assignment ids, grouped by bucket in arbitrary order within a bucket
  __shared__ int act_s[1024];  // the active experts
  __shared__ int warp_tot[32];
  __shared__ int total_s, n_first;
  pdl_trigger();
  pdl_wait();
  const int TK = T * K;
  for (int e = threadIdx.x; e < E; e += 1024) hist[e] = 0;
  __syncthreads();
  const int a = threadIdx.x;
  const int e_a = a < TK ? sh.bucket(idx[a]) : -1;
  if (a < TK) atomicAdd(&hist[e_a], 1);
  __syncthreads();
  // offsets and active list (experts in chunks of 1024)
  int carry_off = 0, carry_act = 0;
  for (int e0 = 0; e0 < E; e0 += 1024) {
    const int e = e0 + threadIdx.x;
    const int c = e < E ? hist[e] : 0;
    const int ex = block_exclusive_scan(c, warp_tot, &total_s);
    if (e < E) {
      base[e] = carry_off + ex;
      counts[e] = c;
      offsets[e] = carry_off + ex;
    }
    carry_off += total_s;
    const int flag = (c > 0 && e < sh.n_listed) ? 1 : 0;
    const int ax = block_exclusive_scan(flag, warp_tot, &total_s);
    if (flag) {
      active[1 + carry_act + ax] = e;
      act_s[carry_act + ax] = e;
    }
    carry_act += total_s;
  }
  if (threadIdx.x == 0) {
    offsets[E] = TK;
    active[0] = carry_act;
    n_first = 0;
  }
  // The stable slot order: an assignment's rank in its bucket is the number
  // of smaller assignment ids there.  Expert buckets hold at most T entries
  // (an expert is chosen at most once per token), so the rank is counted
  // over the bucket's placed ids; the shard's bucket of other experts (up to
  // T*K entries) takes an exclusive scan of its membership instead.
  const bool other = a < TK && e_a == sh.n_listed && sh.n_buckets > sh.n_listed;
  const int orank = block_exclusive_scan(other ? 1 : 0, warp_tot, &total_s);  // (synchronises)
  for (int e = threadIdx.x; e < E; e += 1024) hist[e] = 0;  // placement cursors
  __syncthreads();
  if (a < TK && !other) placed[base[e_a] + atomicAdd(&hist[e_a], 1)] = a;
  __syncthreads();
  int rank = 0, sl = 0;
  if (a < TK) {
    rank = orank;
    if (!other) {
      rank = 0;
      const int b0 = base[e_a], n = hist[e_a];
      for (int j = 0; j < n; ++j) rank += placed[b0 + j] < a ? 1 : 0;
    }
    sl = base[e_a] + rank;
    perm[sl] = a;
    slot[a] = sl;
  }
  // tile list over the active experts (at most TK of them)
  const int n_act = carry_act;
  int nsub = 0, e_t = 0, c_t = 0, tn = 0;
  if (threadIdx.x < n_act) {
    e_t = act_s[threadIdx.x];
    c_t = hist[e_t];
    nsub = (c_t + bn_max - 1) / bn_max;
    const int per = (c_t + nsub - 1) / nsub;
    tn = min((per + 15) & ~15, bn_max);  // tiles never exceed bn_max rows
  }
  const int tb = block_exclusive_scan(nsub, warp_tot, &total_s);  // (synchronises)
  // tiles of experts below split_expert come first (experts ascend)
  if (nsub > 0 && e_t < split_expert) atomicAdd(&n_first, nsub);
  for (int j = 0; j < nsub; ++j) {
    const int r0 = j * tn;
    const int rows = min(tn, c_t - r0);
    tiles[tb + j] = make_int4(e_t, base[e_t] + r0, rows, (rows + 15) & ~15);
  }
  __syncthreads();
  if (slot_tile) {
    // slot -> (tile, row): rank r of an expert's slots is row r % tn of its
    // tile r / tn (tn = the expert's tile height)
    if (nsub > 0) {
      hist[e_t] = tn;
      base[e_t] = tb;
    }
    __syncthreads();
    if (a < TK && !other) slot_tile[sl] = ((base[e_a] + rank / hist[e_a]) << 8) | (rank % hist[e_a]);
  }
  if (threadIdx.x == 0) {
    tile_count[0] = total_s;
    tile_count[1] = n_first;
  }
}

cudaError_t launch_route_small(const float* logits, int T, int E, const float* bias, int K, int norm_topk, float rsf,
                               const ExpertShard& sh, int32_t* idx, float* w, int* counts, int* offsets, int* active,
                               int* perm, int* slot, int bn_max, int4* tiles, int* tile_count, int* slot_tile,
                               int split_expert, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  // tiles of at least 16 rows (the tile list's capacity), or shorter ones
  // when no expert can have more slots than a tile (T <= bn_max: one tile
  // per expert); row field of 8 bits
  if (T * K > 1024 || E > 2048 || sh.n_buckets > 2048 || bn_max < 1 || bn_max > 255 || (bn_max < 16 && T > bn_max))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_topk(logits, T, E, E, bias, K, norm_topk, rsf, idx, w, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(perm_small_kernel, 1, 1024, 0, s, idx, T, sh.n_buckets, K, sh, counts, offsets, active, perm, slot,
                    bn_max, tiles, tile_count, slot_tile, split_expert);
}

// =====================================================================
// SiTU-GLU in fp32 (kimi-k3-mlx README, "Architecture" table and
// "Porting notes" item 1): beta*tanh(g/beta)*sigmoid(g) * beta_lin*tanh(u/beta_lin).
// =====================================================================
__device__ __forceinline__ float situ_glu(float g, float u, float beta, float beta_lin) {
  const float sig = 1.0f / (1.0f + expf(-g));
  return beta * tanhf(g / beta) * sig * beta_lin * tanhf(u / beta_lin);
}

// Accumulate sum_i w_i * x_i over one 32-column scale group held in the
// 16-byte chunk q (decoded exactly to bf16 with the group's scale, then
// widened to fp32), for NT staged token rows (xs rows of `ld` floats,
// starting at column x0).
template <int NT>
__device__ __forceinline__ void group_dot(const uint4& q, const ScaleMul& sm, const float* __restrict__ xs, int ld,
                                          int x0, int nt, float part[NT]) {
  const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t o[4];
    tile_word_to_bf16(wd[j], sm, o);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
        const float4 xa = *reinterpret_cast<const float4*>(xs + (size_t)t * ld + x0 + 8 * j);
        const float4 xb = *reinterpret_cast<const float4*>(xs + (size_t)t * ld + x0 + 8 * j + 4);
        unsigned long long acc = pack_f32x2(part[t], 0.f);
        acc = ffma2(((unsigned long long)(o[0] & 0xFFFF0000u) << 32) | (o[0] << 16), pack_f32x2(xa.x, xa.y), acc);
        acc = ffma2(((unsigned long long)(o[1] & 0xFFFF0000u) << 32) | (o[1] << 16), pack_f32x2(xa.z, xa.w), acc);
        acc = ffma2(((unsigned long long)(o[2] & 0xFFFF0000u) << 32) | (o[2] << 16), pack_f32x2(xb.x, xb.y), acc);
        acc = ffma2(((unsigned long long)(o[3] & 0xFFFF0000u) << 32) | (o[3] << 16), pack_f32x2(xb.z, xb.w), acc);
        const float2 r = unpack_f32x2(acc);
        part[t] = r.x + r.y;
      }
    }
  }
}

// Stage nb token rows (bf16, length len, row index from `rows_of`) as fp32.
template <typename RowOf>
__device__ __forceinline__ void stage_rows(float* xs, const uint16_t* __restrict__ src, int len, int nb,
                                           RowOf rows_of) {
  for (int i = threadIdx.x; i < nb * len; i += blockDim.x) {
    const int j = i / len, c = i - j * len;
    xs[(size_t)j * len + c] = bf16_to_f32(src[rows_of(j) * len + c]);
  }
}

// =====================================================================
// Grouped MXFP4 gate/up GEMV + SiTU-GLU.  Work item (a, mt): active expert
// a, output rows [128 mt, 128 mt + 128) of both w1 (gate) and w3 (up).
// Threads 0..127 stream gate rows, 128..255 the matching up rows; each
// thread's row tile is read once per pass of up to TB tokens.
//   h[slot, j] = bf16(SiTU(W1_e[j] . lat[t], W3_e[j] . lat[t]))
// =====================================================================
template <int TB>
__global__ void __launch_bounds__(256) gateup_gemv_kernel(const uint8_t* __restrict__ gu_tiles,
                                                          const uint16_t* __restrict__ lat,
                                                          const int* __restrict__ active,
                                                          const int* __restrict__ offsets,
                                                          const int* __restrict__ perm, int Ktop, int L, int I,
                                                          float beta, float beta_lin, uint16_t* __restrict__ h) {
  extern __shared__ float xs[];  // [TB, L] staged activations
  __shared__ float ubuf[TB][128];
  const int n_mt = I / kTileRows;
  const int a = blockIdx.x / n_mt, mt = blockIdx.x - (blockIdx.x / n_mt) * n_mt;
  if (a >= active[0]) return;
  const int e = active[1 + a];
  const int s0 = offsets[e], n = offsets[e + 1] - s0;
  const int tid = threadIdx.x, r = tid & 127;
  const bool is_up = tid >= 128;
  const int KS = L / kTileCols;
  const uint8_t* base =
      gu_tiles + ((size_t)(e * n_mt + mt) * KS) * 2 * kTileBytes + (is_up ? kTileBytes : 0);
  for (int p0 = 0; p0 < n; p0 += TB) {
    const int nb = min(TB, n - p0);
    __syncthreads();
    stage_rows(xs, lat, L, nb, [&](int j) { return (size_t)(perm[s0 + p0 + j] / Ktop); });
    __syncthreads();
    float acc[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[t] = 0.f;
    const uint8_t* tile = base;
    uint4 c0 = __ldg(reinterpret_cast<const uint4*>(tile) + r);
    uint4 c1 = __ldg(reinterpret_cast<const uint4*>(tile) + 128 + r);
    uint32_t sc = __ldg(reinterpret_cast<const uint16_t*>(tile + kTilePackedBytes) + r);
    for (int ks = 0; ks < KS; ++ks) {
      uint4 n0 = c0, n1 = c1;
      uint32_t nsc = sc;
      if (ks + 1 < KS) {
        const uint8_t* nt = tile + 2 * kTileBytes;
        n0 = __ldg(reinterpret_cast<const uint4*>(nt) + r);
        n1 = __ldg(reinterpret_cast<const uint4*>(nt) + 128 + r);
        nsc = __ldg(reinterpret_cast<const uint16_t*>(nt + kTilePackedBytes) + r);
      }
      group_dot<TB>(c0, scale_multipliers(sc & 0xFFu), xs, L, ks * kTileCols, nb, acc);
      group_dot<TB>(c1, scale_multipliers(sc >> 8), xs, L, ks * kTileCols + 32, nb, acc);
      c0 = n0;
      c1 = n1;
      sc = nsc;
      tile += 2 * kTileBytes;
    }
    if (is_up) {
#pragma unroll
      for (int t = 0; t < TB; ++t) ubuf[t][r] = acc[t];
    }
    __syncthreads();
    if (!is_up) {
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        if (t < nb)
          h[(size_t)(s0 + p0 + t) * I + mt * kTileRows + r] = f32_to_bf16(situ_glu(acc[t], ubuf[t][r], beta, beta_lin));
      }
    }
  }
}

cudaError_t launch_gateup_gemv(const uint8_t* gu_tiles, const uint16_t* lat, const int* active,
                               const int* offsets, const int* perm, int max_active, const Dims& d,
                               uint16_t* h, cudaStream_t s) {
  constexpr int TB = 4;
  const int grid = max_active * (d.I / kTileRows);
  if (grid <= 0) return cudaSuccess;
  const size_t sm = sizeof(float) * (size_t)TB * d.L;
  gateup_gemv_kernel<TB><<<grid, 256, sm, s>>>(gu_tiles, lat, active, offsets, perm, d.K, d.L, d.I, d.beta,
                                               d.beta_lin, h);
  return cudaGetLastError();
}

// =====================================================================
// Grouped MXFP4 down GEMV.  Work item (a, mt): active expert a, output rows
// [128 mt, 128 mt + 128) of w2.  Threads t and t+128 take the two halves of
// the input columns of row t; the halves are added in a fixed order.
//   o[slot, l] = W2_e[l] . h[slot]   (fp32)
// =====================================================================
template <int TB>
__global__ void __launch_bounds__(256) down_gemv_kernel(const uint8_t* __restrict__ d_tiles,
                                                        const uint16_t* __restrict__ h,
                                                        const int* __restrict__ active,
                                                        const int* __restrict__ offsets, int L, int I,
                                                        float* __restrict__ o) {
  extern __shared__ float xs[];  // [TB, I]
  __shared__ float half1[TB][128];
  const int n_mt = L / kTileRows;
  const int a = blockIdx.x / n_mt, mt = blockIdx.x - (blockIdx.x / n_mt) * n_mt;
  if (a >= active[0]) return;
  const int e = active[1 + a];
  const int s0 = offsets[e], n = offsets[e + 1] - s0;
  const int tid = threadIdx.x, r = tid & 127, hf = tid >> 7;
  const int KS = I / kTileCols, ks_begin = hf * (KS / 2), ks_end = hf ? KS : KS / 2;
  const uint8_t* base = d_tiles + ((size_t)(e * n_mt + mt) * KS) * kTileBytes;
  for (int p0 = 0; p0 < n; p0 += TB) {
    const int nb = min(TB, n - p0);
    __syncthreads();
    stage_rows(xs, h, I, nb, [&](int j) { return (size_t)(s0 + p0 + j); });
    __syncthreads();
    float acc[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[t] = 0.f;
    const uint8_t* tile = base + (size_t)ks_begin * kTileBytes;
    uint4 c0 = __ldg(reinterpret_cast<const uint4*>(tile) + r);
    uint4 c1 = __ldg(reinterpret_cast<const uint4*>(tile) + 128 + r);
    uint32_t sc = __ldg(reinterpret_cast<const uint16_t*>(tile + kTilePackedBytes) + r);
    for (int ks = ks_begin; ks < ks_end; ++ks) {
      uint4 n0 = c0, n1 = c1;
      uint32_t nsc = sc;
      if (ks + 1 < ks_end) {
        const uint8_t* nt = tile + kTileBytes;
        n0 = __ldg(reinterpret_cast<const uint4*>(nt) + r);
        n1 = __ldg(reinterpret_cast<const uint4*>(nt) + 128 + r);
        nsc = __ldg(reinterpret_cast<const uint16_t*>(nt + kTilePackedBytes) + r);
      }
      group_dot<TB>(c0, scale_multipliers(sc & 0xFFu), xs, I, ks * kTileCols, nb, acc);
      group_dot<TB>(c1, scale_multipliers(sc >> 8), xs, I, ks * kTileCols + 32, nb, acc);
      c0 = n0;
      c1 = n1;
      sc = nsc;
      tile += kTileBytes;
    }
    if (hf) {
#pragma unroll
      for (int t = 0; t < TB; ++t) half1[t][r] = acc[t];
    }
    __syncthreads();
    if (!hf) {
#pragma unroll
      for (int t = 0; t < TB; ++t)
        if (t < nb) o[(size_t)(s0 + p0 + t) * L + mt * kTileRows + r] = acc[t] + half1[t][r];
    }
  }
}

cudaError_t launch_down_gemv(const uint8_t* d_tiles, const uint16_t* h, const int* active, const int* offsets,
                             int max_active, const Dims& d, float* o, cudaStream_t s) {
  constexpr int TB = 4;
  const int grid = max_active * (d.L / kTileRows);
  if (grid <= 0) return cudaSuccess;
  const size_t sm = sizeof(float) * (size_t)TB * d.I;
  down_gemv_kernel<TB><<<grid, 256, sm, s>>>(d_tiles, h, active, offsets, d.L, d.I, o);
  return cudaGetLastError();
}

// =====================================================================
// Weighted combine (k order, fp32) + RMSNorm over the latent (kimi-k3-mlx
// README, REAP section caveat: RMSNorm on the combined expert output,
// before up_proj).  One CTA per token.
//   SAL: also the REAP saliency term of each (token, k): w_k ||o_k||_2
//        (kimi-k3-mlx README, "REAP expert pruning": S_j = 1/|C| sum_x
//        g_j(x) ||e_j(x)||_2), from the o rows the combine reads anyway.
//   PARTIAL: an expert shard's partial combine: only slots below *n_local
//        (the shard's own experts) are added, and c itself (fp32) goes to
//        c_out instead of through RMSNorm.
// The sum of squares for RMSNorm is taken on c scaled by a power of two
// whenever the plain sum overflows fp32 (|c| above ~1e17), which gives the
// same bits as the plain formula wherever that one is finite.
// =====================================================================
template <bool SAL, bool PARTIAL>
__global__ void __launch_bounds__(1024) combine_rmsnorm_kernel(const float* __restrict__ o,
                                                               const int* __restrict__ slot,
                                                               const float* __restrict__ topk_w,
                                                               const uint16_t* __restrict__ gamma, int K, int L,
                                                               float eps, uint16_t* __restrict__ n,
                                                               float* __restrict__ sal_tk,
                                                               const int* __restrict__ n_local,
                                                               float* __restrict__ c_out, int o_parts,
                                                               size_t o_part_stride) {
  // One CTA per token; thread i owns latent columns 4i..4i+3 (plus further
  // groups of 4*blockDim.x when L is larger); the K slot rows of a column
  // group are loaded together so their latencies overlap.
  extern __shared__ float cs[];  // [L]
  __shared__ int sl[32];
  __shared__ float wk[32];
  __shared__ float red[32];
  __shared__ float red_k[SAL ? 32 : 1][33];
  __shared__ int kloc[32];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < K) {
    const int sv = slot[(size_t)t * K + threadIdx.x];
    sl[threadIdx.x] = sv;
    wk[threadIdx.x] = topk_w[(size_t)t * K + threadIdx.x];
    kloc[threadIdx.x] = PARTIAL ? (sv < *n_local) : 1;  // other shards' slots hold no output
  }
  __syncthreads();
  float ss = 0.f;
  float sq[SAL ? 32 : 1];
#pragma unroll
  for (int k = 0; k < (SAL ? 32 : 1); ++k) sq[k] = 0.f;
  for (int c4 = threadIdx.x; c4 < L / 4; c4 += blockDim.x) {
    float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k0 = 0; k0 < 32; k0 += 8) {  // eight slot rows in flight at a time, added in k order
      if (k0 >= K) break;
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k0 + k < K && (!PARTIAL || kloc[k0 + k]))
          v[k] = __ldg(reinterpret_cast<const float4*>(o + (size_t)sl[k0 + k] * L) + c4);
      // o split in K parts (T = 1): the parts are added in part order
      for (int pp = 1; pp < o_parts; ++pp) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k0 + k < K && (!PARTIAL || kloc[k0 + k])) {
            const float4 q = __ldg(reinterpret_cast<const float4*>(o + pp * o_part_stride + (size_t)sl[k0 + k] * L) + c4);
            v[k].x += q.x;
            v[k].y += q.y;
            v[k].z += q.z;
            v[k].w += q.w;
          }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k0 + k < K && (!PARTIAL || kloc[k0 + k])) {
          const float wv = wk[k0 + k];
          c.x = fmaf(wv, v[k].x, c.x);
          c.y = fmaf(wv, v[k].y, c.y);
          c.z = fmaf(wv, v[k].z, c.z);
          c.w = fmaf(wv, v[k].w, c.w);
          if (SAL) {
            float& q = sq[SAL ? k0 + k : 0];
            q = fmaf(v[k].x, v[k].x, q);
            q = fmaf(v[k].y, v[k].y, q);
            q = fmaf(v[k].z, v[k].z, q);
            q = fmaf(v[k].w, v[k].w, q);
          }
        }
      }
    }
    if (PARTIAL) {
      reinterpret_cast<float4*>(c_out + (size_t)t * L)[c4] = c;
      continue;
    }
    reinterpret_cast<float4*>(cs)[c4] = c;
    ss = fmaf(c.x, c.x, ss);
    ss = fmaf(c.y, c.y, ss);
    ss = fmaf(c.z, c.z, ss);
    ss = fmaf(c.w, c.w, ss);
  }
  if (SAL) {
    // ||o_k||^2: per warp in a fixed tree, then over warps in order
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      if (k >= K) break;
      const float v = warp_sum(sq[SAL ? k : 0]);
      if (lane == 0) red_k[SAL ? warp : 0][k] = v;
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  const int nw = (int)(blockDim.x >> 5);
  float tot = 0.f;
  for (int i = 0; i < nw; ++i) tot += red[i];
  if (SAL && threadIdx.x < K) {
    float q = 0.f;
    for (int i = 0; i < nw; ++i) q += red_k[SAL ? i : 0][threadIdx.x];
    sal_tk[(size_t)t * K + threadIdx.x] = kloc[threadIdx.x] ? wk[threadIdx.x] * sqrtf(q) : 0.f;
  }
  if (PARTIAL) return;
  float scale = 1.f;  // power of two applied to c before squaring
  if (!(tot <= 3.0e38f)) {
    // the plain sum of squares overflowed: take it again on c * 2^-e, e
    // the exponent of max|c| (exact scaling, same rounding)
    float mx = 0.f;
    for (int c4 = threadIdx.x; c4 < L / 4; c4 += blockDim.x) {
      const float4 c = reinterpret_cast<const float4*>(cs)[c4];
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(c.x), fabsf(c.y)), fmaxf(fabsf(c.z), fabsf(c.w))));
    }
    mx = warp_max(mx);
    __syncthreads();
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = 0.f;
    for (int i = 0; i < nw; ++i) mx = fmaxf(mx, red[i]);
    if (mx <= 3.0e38f) {  // finite c: rescale; an inf or NaN in c stays as it is
      int ex;
      frexpf(mx, &ex);
      scale = ldexpf(1.f, -ex);
      float s2 = 0.f;
      for (int c4 = threadIdx.x; c4 < L / 4; c4 += blockDim.x) {
        const float4 c = reinterpret_cast<const float4*>(cs)[c4];
        s2 = fmaf(c.x * scale, c.x * scale, s2);
        s2 = fmaf(c.y * scale, c.y * scale, s2);
        s2 = fmaf(c.z * scale, c.z * scale, s2);
        s2 = fmaf(c.w * scale, c.w * scale, s2);
      }
      s2 = warp_sum(s2);
      __syncthreads();
      if (lane == 0) red[warp] = s2;
      __syncthreads();
      tot = 0.f;
      for (int i = 0; i < nw; ++i) tot += red[i];
    }
  }
  // scale = 2^-e: c / sqrt(mean(c^2) + eps) = (c 2^-e) / sqrt(mean((c 2^-e)^2) + eps 2^-2e)
  const float inv = 1.0f / sqrtf(tot / (float)L + eps * scale * scale);
  for (int c4 = threadIdx.x; c4 < L / 4; c4 += blockDim.x) {
    float4 c = reinterpret_cast<const float4*>(cs)[c4];
    c.x *= scale;
    c.y *= scale;
    c.z *= scale;
    c.w *= scale;
    const uint2 g = __ldg(reinterpret_cast<const uint2*>(gamma) + c4);
    const float2 g01 = unpack_bf16x2(g.x), g23 = unpack_bf16x2(g.y);
    uint2 out;
    out.x = pack_bf16x2(c.x * inv * g01.x, c.y * inv * g01.y);
    out.y = pack_bf16x2(c.z * inv * g23.x, c.w * inv * g23.y);
    reinterpret_cast<uint2*>(n + (size_t)t * L)[c4] = out;
  }
}

// REAP saliency accumulation: for every expert with work, the terms of its
// slots (in slot order: tokens ascending) are added in a fixed order and
// the sum is added to the expert's fp64 running total; the token count of
// the calibration set grows by T.  One warp per active expert; the launch
// is ordered on the stream, so no two updates of a total overlap.
__global__ void __launch_bounds__(256) saliency_accumulate_kernel(const float* __restrict__ sal_tk,
                                                                  const int* __restrict__ perm,
                                                                  const int* __restrict__ offsets,
                                                                  const int* __restrict__ active, int T,
                                                                  double* __restrict__ sal_sum,
                                                                  unsigned long long* __restrict__ sal_tokens) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int n_act = active[0];
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int nw = (int)((gridDim.x * blockDim.x) >> 5);
  for (int i = gw; i < n_act; i += nw) {
    const int e = active[1 + i];
    double acc = 0.0;
    for (int sidx = offsets[e] + lane; sidx < offsets[e + 1]; sidx += 32) acc += (double)sal_tk[perm[sidx]];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (lane == 0) sal_sum[e] += acc;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *sal_tokens += (unsigned long long)T;
}

// One-time kernel attributes (dynamic shared memory above 48 KB), set when a
// context is created so that forward calls stay capturable.
cudaError_t prepare_decode_kernels(const Dims& d) {
  cudaError_t e = cudaFuncSetAttribute(gateup_gemv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(sizeof(float) * 4 * d.L));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(down_gemv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(sizeof(float) * 4 * d.I));
  const int sm = (int)(sizeof(float) * d.L);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(combine_rmsnorm_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(combine_rmsnorm_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(combine_rmsnorm_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(combine_rmsnorm_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
  return e;
}

cudaError_t launch_combine_rmsnorm(const float* o, const int* slot, const float* topk_w, const uint16_t* gamma,
                                   int T, int K, const Dims& d, uint16_t* n, float* sal_tk, const int* n_local,
                                   float* c_out, cudaStream_t s, int o_parts, size_t o_part_stride) {
  if (T <= 0) return cudaSuccess;
  if (K < 1 || K > 32 || (c_out && !n_local)) return cudaErrorInvalidValue;
  const int threads = std::min(1024, ((d.L / 4 + 31) / 32) * 32);
  const size_t sm = sizeof(float) * d.L;
  auto kernel = c_out ? (sal_tk ? combine_rmsnorm_kernel<true, true> : combine_rmsnorm_kernel<false, true>)
                      : (sal_tk ? combine_rmsnorm_kernel<true, false> : combine_rmsnorm_kernel<false, false>);
  return launch_pdl(kernel, T, threads, sm, s, o, slot, topk_w, gamma, K, d.L, d.rms_eps, n, sal_tk, n_local, c_out,
                    o_parts, o_part_stride);
}

cudaError_t launch_saliency_accumulate(const float* sal_tk, const int* perm, const int* offsets, const int* active,
                                       int T, int E, double* sal_sum, unsigned long long* sal_tokens,
                                       cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int blocks = std::max(1, std::min((E * 32 + 255) / 256, 152));
  return launch_pdl(saliency_accumulate_kernel, blocks, 256, 0, s, sal_tk, perm, offsets, active, T, sal_sum,
                    sal_tokens);
}

// =====================================================================
// Checkpoint MXFP4 -> tile format.  n_mat matrices [rows, cols] (packed
// [rows, cols/2], scale [rows, cols/32]); tile (m, mt, ks) goes to
// tiles + ((m * mat_stride_tiles) + (mt * KS + ks) * tile_step + tile_offset) * kTileBytes.
// One thread per 32-bit word of a tile (1024 packed words + 64 scale words).
// =====================================================================
__global__ void relayout_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scale, int n_mat,
                                int rows, int cols, uint8_t* __restrict__ tiles, size_t mat_stride_tiles,
                                int tile_step, int tile_offset) {
  const int KS = cols / kTileCols, MT = rows / kTileRows;
  const long long words_per_tile = kTileBytes / 4;  // 1088
  const long long total = (long long)n_mat * MT * KS * words_per_tile;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const int w = (int)(g % words_per_tile);
    const long long tile_lin = g / words_per_tile;
    const int ks = (int)(tile_lin % KS);
    const int mt = (int)((tile_lin / KS) % MT);
    const int m = (int)(tile_lin / ((long long)KS * MT));
    uint8_t* tile = tiles + ((size_t)m * mat_stride_tiles + ((size_t)mt * KS + ks) * tile_step + tile_offset) *
                                (size_t)kTileBytes;
    uint32_t word;
    if (w < 1024) {
      const int ch = w >> 2, j = w & 3;
      const int c = ch >> 7, r = ch & 127;
      const size_t row = (size_t)m * rows + (size_t)mt * kTileRows + r;
      const int col0 = ks * kTileCols + c * 32 + j * 8;
      const uint8_t* src = packed + row * (cols / 2) + col0 / 2;
      word = tile_word_from_checkpoint(src[0], src[1], src[2], src[3]);
    } else {
      const int sw = w - 1024;  // bytes 4sw..4sw+3: rows 2sw, 2sw+1, groups 0 and 1
      const size_t row0 = (size_t)m * rows + (size_t)mt * kTileRows + 2 * sw;
      const uint8_t* s0 = scale + row0 * (cols / 32) + ks * 2;
      const uint8_t* s1 = s0 + cols / 32;
      word = (uint32_t)s0[0] | ((uint32_t)s0[1] << 8) | ((uint32_t)s1[0] << 16) | ((uint32_t)s1[1] << 24);
    }
    reinterpret_cast<uint32_t*>(tile)[w] = word;
  }
}

cudaError_t launch_relayout(const uint8_t* packed, const uint8_t* scale, int n_mat, int rows, int cols,
                            uint8_t* tiles, size_t mat_stride_tiles, int tile_step, int tile_offset,
                            cudaStream_t s) {
  relayout_kernel<<<152 * 8, 256, 0, s>>>(packed, scale, n_mat, rows, cols, tiles, mat_stride_tiles, tile_step,
                                          tile_offset);
  return cudaGetLastError();
}

// =====================================================================
// Standalone dequant (checkpoint layout in, row-major out) through the same
// tile-word re-layout and decoders as the expert kernels.
//   kind 0: bf16 (the tensor-core tile producer's decoder)
//   kind 1: the same values widened to fp32 (as the CUDA-core GEMVs use them)
// One thread per 8 consecutive columns of a row.
// =====================================================================
__global__ void dequant_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scale, int rows,
                               int cols, void* __restrict__ out, int kind) {
  const long long total = (long long)rows * (cols / 8);
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(g / (cols / 8));
    const int col0 = (int)(g % (cols / 8)) * 8;
    const uint8_t* src = packed + (size_t)r * (cols / 2) + col0 / 2;
    const uint32_t q = tile_word_from_checkpoint(src[0], src[1], src[2], src[3]);
    const uint32_t S = scale[(size_t)r * (cols / 32) + col0 / 32];
    if (kind == 0) {
      uint32_t o4[4];
      tile_word_to_bf16(q, scale_multipliers(S), o4);
      *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(out) + (size_t)r * cols + col0) =
          make_uint4(o4[0], o4[1], o4[2], o4[3]);
    } else {
      uint32_t o4[4];
      tile_word_to_bf16(q, scale_multipliers(S), o4);
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (size_t)r * cols + col0);
      const float2 a = unpack_bf16x2(o4[0]), b = unpack_bf16x2(o4[1]), c = unpack_bf16x2(o4[2]),
                   d = unpack_bf16x2(o4[3]);
      dst[0] = make_float4(a.x, a.y, b.x, b.y);
      dst[1] = make_float4(c.x, c.y, d.x, d.y);
    }
  }
}

cudaError_t launch_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols, void* out,
                           int kind, cudaStream_t s) {
  const long long total = (long long)rows * (cols / 8);
  if (total <= 0) return cudaSuccess;
  const int blocks = (int)std::min<long long>((total + 255) / 256, 152LL * 16);
  dequant_kernel<<<blocks, 256, 0, s>>>(packed, scale, rows, cols, out, kind);
  return cudaGetLastError();
}

}  // namespace k3
