// k3moe_umma.h -- tcgen05 kernels with bf16 operands: the dense projections
// (router + down_proj, up_proj, shared experts) at every T, the second
// bank's 2-bit experts above decode sizes, and the expert tile lists.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "k3moe_internal.h"

namespace k3 {

// Where a dense projection's fp32 sums D[t, m] (t < T tokens, m < M weight
// rows) go:
//   glu == 0: rows m < split -> out_f32[t * split + m] (fp32);
//             rows m >= split -> out_bf16[t * (M - split) + m - split] =
//             bf16(D), or, with add_bf16, bf16(bf16(D) + add_bf16[same index]);
//   glu == 1: the weight rows are gate/up pairs (row 2j gate, 2j + 1 up) and
//             out_bf16[t * (M / 2) + j] = bf16(SiTU-GLU(D[t, 2j], D[t, 2j + 1]))
//             with temperatures beta, beta_lin.
struct DenseOut {
  int split = 0;
  float* out_f32 = nullptr;
  uint16_t* out_bf16 = nullptr;
  const uint16_t* add_bf16 = nullptr;
  int glu = 0;
  float beta = 4.f, beta_lin = 25.f;
};

struct UmmaPlan {
  int max_tokens = 0;
  size_t ws_bytes = 256;  // workspace this path needs (tile list, slot-ordered latent rows)
  void* ws = nullptr;
  unsigned* status = nullptr;  // device status word (bounded waits report here)
  int num_sms = 152;
  Dims dims{};  // the context's layer dimensions (workspace layout)
  uint64_t limit_ns = 2000000000ull;
};

cudaError_t prepare_umma_kernels();
UmmaPlan umma_plan(const Dims& d, int max_tokens);
cudaError_t umma_dense(const UmmaPlan& p, const uint16_t* W, int M, int K, const uint16_t* X, int T,
                       const DenseOut& o, cudaStream_t s);
int umma_dense_launches();
// T <= 64: split-K streaming dense GEMM over all SMs writing fp32 partials
// to `part` (at least dense_small_part_floats(M) floats; a context's own
// buffer when null), then an ordered reduction of the chunks (two launches)
cudaError_t umma_dense_small(const UmmaPlan& p, const uint16_t* W, int M, int K, const uint16_t* X, int T,
                             const DenseOut& o, float* part, cudaStream_t s);
int umma_dense_small_launches();
size_t dense_small_part_floats(int M);
// Tile list over the experts with work (tiles of at most bn_max slots),
// slot -> tile map, and count[1] = the tiles of experts below split_expert
// (they come first).
cudaError_t umma_stream_tiles(const UmmaPlan& p, const Work& w, int T, const Dims& d, int bn_max, int* slot_tile,
                              int split_expert, cudaStream_t s);
// Second bank (2-bit affine experts): re-layout into 2-bit tiles at load,
// and the bank's gate/up + down over tiles [count[1], count[0]).
cudaError_t bank2_tiles(const uint8_t* q, const uint16_t* sc, const uint16_t* bi, int ne, int rows, int cols,
                        uint8_t* out, size_t mat_stride_tiles, int step, int offset, cudaStream_t s);
size_t bank2_tile_bytes(int rows, int cols);  // one matrix of one expert
cudaError_t umma_bank2_experts(const UmmaPlan& p, const uint8_t* gu2_tiles, const uint8_t* d2_tiles, int bank2_begin,
                               int n_bank2, int tile_rows, const Work& w, int T, const Dims& d, cudaStream_t s);
// where the grouped expert kernels read their tile list (and the shortest
// tile height any list uses)
void umma_tile_list(const UmmaPlan& p, int4** tiles, int** count, int* bn_max);

}  // namespace k3
