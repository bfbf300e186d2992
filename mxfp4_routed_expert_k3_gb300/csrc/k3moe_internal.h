// k3moe_internal.h -- launchers shared between the library's translation
// units (host side only; no torch types).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace k3 {

struct Dims {
  int H, L, E, K, I;
  float beta, beta_lin, rms_eps, rsf;
  int norm_topk;
};

// The experts a context computes: ids [begin, begin + n_listed) of the
// router's E, renumbered from 0.  The permutation sorts the T*K selections
// into n_buckets buckets: local experts in their own, every other expert in
// one last bucket (n_buckets = n_listed + 1) whose slots come after all
// local ones and get no work; without a shard n_buckets = n_listed = E.
struct ExpertShard {
  int begin = 0, n_listed = 0, n_buckets = 0;
  __host__ __device__ __forceinline__ int bucket(int e) const {
    const int l = e - begin;
    return (l >= 0 && l < n_listed) ? l : n_listed;
  }
};

// Workspace views for one forward call (all device memory).
struct Work {
  float* logits;      // [Tm, E]
  uint16_t* lat;      // [Tm, L]
  int* counts;        // [E]
  int* offsets;       // [E + 1]
  int* active;        // [E + 1]: n_active, then expert ids
  int* perm;          // [Tm * K] slot -> t*K + k
  int* slot;          // [Tm * K] t*K + k -> slot
  int* blk_hist;      // [nblk_max, E]
  uint16_t* h;        // [Tm * K, I]
  float* o;           // [Tm * K, L]
  uint16_t* n;        // [Tm, L]
  unsigned* status;   // device status word
};

// ---- k3moe_api.cu: the per-thread message returned by k3moe_last_error(NULL)
void set_thread_error(const char* msg);

// ---- k3moe_decode.cu
cudaError_t launch_dense_gemv(const uint16_t* W, int M, int K, const uint16_t* X, int T, int split,
                              float* out_f32, uint16_t* out_bf16, cudaStream_t s);
cudaError_t launch_topk(const float* logits, int T, int E, int ld, const float* bias, int K, int norm_topk,
                        float rsf, int32_t* idx, float* w, cudaStream_t s);
constexpr int kPermChunk = 1024;
cudaError_t launch_permute(const int32_t* idx, int T, int K, const ExpertShard& sh, int* blk_hist, int* counts,
                           int* offsets, int* active, int* perm, int* slot, cudaStream_t s);
cudaError_t launch_gateup_gemv(const uint8_t* gu_tiles, const uint16_t* lat, const int* active,
                               const int* offsets, const int* perm, int max_active, const Dims& d,
                               uint16_t* h, cudaStream_t s);
cudaError_t launch_down_gemv(const uint8_t* d_tiles, const uint16_t* h, const int* active, const int* offsets,
                             int max_active, const Dims& d, float* o, cudaStream_t s);
cudaError_t prepare_decode_kernels(const Dims& d);
// T*K <= 1024: top-K (one CTA per token) + permutation and streaming tile
// list in one CTA
cudaError_t launch_route_small(const float* logits, int T, int E, const float* bias, int K, int norm_topk, float rsf,
                               const ExpertShard& sh, int32_t* idx, float* w, int* counts, int* offsets, int* active,
                               int* perm, int* slot, int bn_max, int4* tiles, int* tile_count, int* slot_tile,
                               int split_expert, cudaStream_t s);
// n = RMSNorm(sum_k topk_w[t,k] o[slot[t,k]]) for K slots per token.
// sal_tk (optional, [T*K]): also w_k ||o_k||_2 per (token, k), the REAP
// saliency terms.  c_out (optional, [T, L] fp32): write the combine itself
// instead of n, adding only slots below *n_local (an expert shard's part).
// o_parts > 1: o is the sum of that many planes o_part_stride floats apart
// (a K-split down GEMM), added in plane order.
cudaError_t launch_combine_rmsnorm(const float* o, const int* slot, const float* topk_w, const uint16_t* gamma,
                                   int T, int K, const Dims& d, uint16_t* n, float* sal_tk, const int* n_local,
                                   float* c_out, cudaStream_t s, int o_parts = 1, size_t o_part_stride = 0);
// sal_sum[e] += the terms of expert e's slots (slot order), *sal_tokens += T
cudaError_t launch_saliency_accumulate(const float* sal_tk, const int* perm, const int* offsets, const int* active,
                                       int T, int E, double* sal_sum, unsigned long long* sal_tokens,
                                       cudaStream_t s);
cudaError_t launch_relayout(const uint8_t* packed, const uint8_t* scale, int n_mat, int rows, int cols,
                            uint8_t* tiles, size_t mat_stride_tiles, int tile_step, int tile_offset,
                            cudaStream_t s);
cudaError_t launch_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols, void* out,
                           int kind, cudaStream_t s);

}  // namespace k3
