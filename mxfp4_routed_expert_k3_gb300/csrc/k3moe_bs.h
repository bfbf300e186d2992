// k3moe_bs.h -- block-scaled tensor-core path for the MXFP4 expert GEMMs:
// the e2m1 weights and their e8m0 scales go to the tensor cores as they are
// stored.  Two tile kinds: decode tiles (16 token rows, up to T = 128) use
// tcgen05.mma kind::mxf4 with the bf16 activations carried as six
// block-scaled e2m1 terms; prefill tiles (88 token rows) use
// kind::mxf8f6f4 with the activations written exactly as the sum of two
// block-scaled e4m3 terms.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "k3moe_internal.h"

namespace k3 {

// Expert weights in the block-scaled layout (device memory).
//   gu_q : [E][I/128][L/128][2][128][64] e2m1 nibbles in checkpoint order,
//          one contiguous 8 KB block per 128 x 128 tile, gate then up
//   gu_sf: [E][I/128][L/128][2][512] e8m0 scale atoms (gate, up)
//   d_q  : [E][L/128][I/128][128][64]
//   d_sf : [E][L/128][I/128][512]
struct BsWeights {
  int n_exp = 0;  // experts held (a shard's own count)
  uint8_t* gu_q = nullptr;
  uint8_t* gu_sf = nullptr;
  uint8_t* d_q = nullptr;
  uint8_t* d_sf = nullptr;
};
size_t bs_weight_bytes(const Dims& d);  // for d.E experts
// Packed nibbles [ne][rows][cols/2] into the box layout above (slot `mat`
// of n_mat matrices per expert).
cudaError_t bs_e2m1_boxes(const uint8_t* packed, int ne, int rows, int cols, int n_mat, int mat, uint8_t* out,
                          cudaStream_t s);
// Scale atoms of n_mat matrices [ne][rows][cols/32] into out (layout above;
// mat_stride atoms between experts, `mat` selects the slot in an atom pair).
cudaError_t bs_scale_atoms(const uint8_t* scale, int ne, int rows, int cols, int n_mat, int mat, uint8_t* out,
                           cudaStream_t s);

struct BsPlan {
  int max_tokens = 0;     // largest T (workspace bound)
  void* ws = nullptr;
  size_t ws_bytes = 0;
  unsigned* status = nullptr;
  uint64_t limit_ns = 2000000000ull;
  int num_sms = 152;
  Dims dims{};
  int withhold_item = -1;  // test hook (see k3moe_test_withhold_copies)
};
// Tile heights (token rows per tile, the MMA's N bound): decode-size batches
// use short tiles (every weight byte streamed once per forward; the six
// activation terms of the 16 rows form one 96-row MMA operand), larger
// batches taller ones (fewer weight re-reads and MMA instructions per
// token).  A block-scaled MMA instruction costs about the same pipe time
// for any N up to 192, so the prefill tile is as tall as the gate/up
// kernel's four-stage ring allows: 88 rows (N = 176), which keeps an
// expert of up to 176 slots -- nearly every expert of a uniform T = 8192
// batch, ~146 +- 12 slots -- at two tiles.
constexpr int kBsSmallRows = 8;
constexpr int kBsSmallMaxT = 8;     // largest T run on 8-row decode tiles (no expert has more slots)
constexpr int kBsDecodeRows = 16;
constexpr int kBsPrefillRows = 88;
constexpr int kBsDecodeMaxT = 128;  // largest T run on decode tiles
constexpr int kBsMaxSplit = 4;      // most K parts of a T = 1 work item
// The token-tile height of the expert kernels for T tokens; the second
// bank's decode kernel works on 16-row tiles only.
inline int bs_tile_rows(int T, bool bank2 = false) {
  return (T <= kBsSmallMaxT && !bank2) ? kBsSmallRows : T <= kBsDecodeMaxT ? kBsDecodeRows : kBsPrefillRows;
}
size_t bs_ws_bytes(const Dims& d, int max_tokens);
// slot -> (tile << 8 | row in tile), written by the tile-list builders
int* bs_slot_tile(const BsPlan& p);
cudaError_t prepare_bs_kernels();

// Slot-ordered latent rows (lat[perm[s] / K]) written as the block-scaled
// terms of the expert kernels' B operand (six e2m1 terms for decode tiles,
// two e4m3 terms for prefill tiles) and their scales as per-tile atoms
// (needs the tile list's slot map; tile_rows is the tile height the expert
// kernels will use).
// n_local (device, optional): an expert shard's slot count; slots from there
// on belong to other shards and are skipped.
cudaError_t bs_quantize_latent(const BsPlan& p, const Work& w, int T, const Dims& d, int tile_rows,
                               const int* n_local, cudaStream_t s);
// gate/up over the tile list (tiles of at most tile_rows rows): h (bf16,
// slot order) and its block-scaled terms for the down GEMM.
// At T = 1 the K experts give K x (rows / 128) work items, fewer than twice
// the persistent CTAs, so the busiest CTA would take two items: each item's
// K range is then split in n_split parts (the bs_split_* choice) whose fp32
// partial sums are added in part order -- for gate/up by a finish kernel
// (SiTU-GLU and h's terms), for down by the combine (bs_down_parts, planes
// of T*K rows of L).
int bs_split_gateup(const BsPlan& p, const Dims& d, int T);
int bs_split_down(const BsPlan& p, const Dims& d, int T);
float* bs_down_parts(const BsPlan& p, const Dims& d);
cudaError_t bs_stream_gateup(const BsPlan& p, const BsWeights& bw, const int4* tiles, const int* tile_count,
                             const Work& w, int T, const Dims& d, int tile_rows, cudaStream_t s, int n_split = 1,
                             const int* n_local = nullptr);
// down: o (fp32, slot order)
cudaError_t bs_stream_down(const BsPlan& p, const BsWeights& bw, const int4* tiles, const int* tile_count,
                           const Work& w, int T, const Dims& d, int tile_rows, cudaStream_t s, int n_split = 1);
// The second bank's experts at decode sizes (T <= kBsDecodeMaxT): tiles
// [tile_count[1], tile_count[0]) of the list (experts >= bank2_begin, 2-bit
// tiles at index expert - bank2_begin), on kind::mxf4 against the same
// e2m1 activation terms as the first bank: gate/up -> h (and its terms),
// down -> o.
cudaError_t bs_bank2_experts(const BsPlan& p, const uint8_t* gu2_tiles, const uint8_t* d2_tiles, int bank2_begin,
                             const int4* tiles, const int* tile_count, const Work& w, int T, const Dims& d,
                             cudaStream_t s);

}  // namespace k3
