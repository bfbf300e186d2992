/*
 * k3moe.h -- C ABI of the GB300 (sm_103a) Kimi-K3 Stable LatentMoE
 * routed-expert layer.
 *
 * The layer, for each token x (7168-d, bf16) independently:
 *   1. router    logit[e] = x . Wr[e] (fp32 accumulate); s = sigmoid(logit);
 *                key = s + e_score_correction_bias[e] (selection only);
 *                the top-K keys give topk_idx; topk_w = s / sum(s) * rsf.
 *   2. down_proj lat = bf16(Wd . x), 7168 -> 3584.
 *   3. experts   for each selected expert e: g = W1_e . lat, u = W3_e . lat,
 *                h = bf16(beta tanh(g/beta) sigmoid(g) beta_lin tanh(u/beta_lin)),
 *                o = W2_e . h; W1/W3/W2 are MXFP4 (e2m1 nibbles, low nibble
 *                first, one e8m0 scale per 32 along the input dimension).
 *   4. combine   c = sum_k topk_w[k] * o_k, in k order, fp32.
 *   5. RMSNorm   n = bf16(c / sqrt(mean(c^2) + eps) * gamma).
 *   6. up_proj   y = bf16(Wu . n), 3584 -> 7168.
 * Passages defining these steps (page title, section):
 *   kimi-k3-mlx README, "Architecture" table (896 routed experts, top-16,
 *     sigmoid router + aux-loss-free e_score_correction_bias, Stable
 *     LatentMoE down_proj -> experts -> RMSNorm -> up_proj in a 3584-d
 *     latent, SiTU-GLU with beta = 4 and beta_lin = 25, MXFP4 source format
 *     with group 32); "Porting notes" item 1 (SiTU-GLU in fp32); "Tiers"
 *     (low-bits-first e2m1 codes, e8m0 scales); "REAP expert pruning"
 *     closing caveat (RMSNorm on the combined expert output, before up_proj).
 *   K3_ARTIFACT_AUDIT, section 4.3 (expert tensor shapes and the group of 32)
 *     and section 6 (router weight [896,7168] bf16, fp32 correction bias).
 * The renormalisation of the selected scores and the routed scaling factor
 * are not fixed by the pages; they are configuration fields here.
 *
 * Conventions
 *   - Every function returns K3MOE_OK (0) or a negative K3MOE_E* code; no
 *     C++ exception crosses this boundary.  The message of the last failure
 *     of a context is available from k3moe_last_error(); failures that
 *     happen without a context (bad arguments to k3moe_create) are reported
 *     by k3moe_last_error(NULL) on the calling thread.
 *   - bf16 values are passed as uint16_t bit patterns (or void* to them).
 *   - "device" pointers are CUDA device (or managed) memory on the context's
 *     device; "host" pointers are ordinary CPU memory.  The library never
 *     takes ownership of caller memory.
 *   - Argument checks happen on the host before anything is launched.
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define K3MOE_OK 0
#define K3MOE_EINVAL (-1)    /* bad argument or unsupported dimension */
#define K3MOE_ENOMEM (-2)    /* device or host allocation failed */
#define K3MOE_ECUDA (-3)     /* a CUDA runtime/driver call failed */
#define K3MOE_ETIMEOUT (-4)  /* a bounded device-side wait gave up */
#define K3MOE_EBADSCALE (-5) /* an e8m0 scale byte was 0xFF (NaN) */
#define K3MOE_ESTATE (-6)    /* call out of order (e.g. forward before load_weights) */

typedef struct k3moe_ctx k3moe_ctx; /* opaque; owned by the library */

/* Layer configuration.  Dimensions must satisfy: hidden, latent and inter
 * are multiples of 128; top_k <= 32 and top_k <= n_experts <= 2048;
 * group == 32.  max_tokens bounds T in every forward call; the workspace
 * is sized for it at create time and forward never allocates. */
typedef struct {
  int hidden;      /* H: 7168 for K3 */
  int latent;      /* L: 3584 */
  int n_experts;   /* E: 896 */
  int top_k;       /* K: 16 */
  int inter;       /* I: moe_intermediate_size, 3072 */
  int group;       /* MXFP4 scale group along the input dimension: 32 */
  float beta;      /* SiTU-GLU gate temperature: 4 */
  float beta_lin;  /* SiTU-GLU linear-branch temperature: 25 */
  float rms_eps;   /* RMSNorm epsilon: 1e-6 */
  float routed_scaling; /* multiplies topk_w: 1.0 */
  int norm_topk;   /* 1: topk_w = s / sum of the selected s; 0: topk_w = s */
  int max_tokens;  /* largest T a forward call may pass */
  int spin_timeout_ms; /* limit of any device-side wait; 0 selects 2000 ms */
  int force_path;  /* 0: the library's choice (path 4 for every T);
                      1: CUDA-core kernels everywhere (an independent
                         implementation kept as a cross-check);
                      4: tensor-core dense projections (split-K for
                         T <= 64) and the expert GEMMs on the block-scaled
                         MXFP4 tensor cores (e2m1 weights and e8m0 scales
                         as stored; up to T = 128 tcgen05 kind::mxf4 on
                         tiles of 16 token rows (8 for T <= 8 without a
                         second bank) with the activations as six
                         block-scaled e2m1 terms, above that
                         kind::mxf8f6f4 on tiles of 88 rows with two exact
                         e4m3 terms; the terms of a tile form one MMA
                         operand).
                      Other values: EINVAL. */
  /* Shared experts (kimi-k3-mlx README, "Architecture" table: 2 shared
   * experts on every token; "Porting notes" item 3: they act on the 7168-d
   * residual, not the latent; "Parameter budget": 12.2 B parameters, i.e.
   * intermediate 3072 each).  0 = the routed layer alone.  With Is =
   * n_shared * shared_inter (a multiple of 128), the block output becomes
   *   y = bf16(y_routed + z),  z = bf16(W2s . bf16(SiTU(W1s . x, W3s . x)))
   * (the experts summed: one MLP over their concatenated intermediate).
   * Needs force_path 0 or 4. */
  int n_shared;
  int shared_inter;
  /* Expert shard (expert parallelism: Kimi-K3-Alis-MLX-Dynamic model card,
   * "Performance" and "Usage" -- dense weights replicated, the routed
   * experts split between two machines).  expert_count = 0: the context
   * holds all n_experts experts.  Otherwise it holds experts
   * [expert_begin, expert_begin + expert_count): load_weights takes the
   * expert tensors of those experts only, while the router, bias and dense
   * weights stay whole.  A shard has no whole forward; it runs
   * k3moe_forward_partial, the callers sum the shards' partial combines
   * (one all-reduce), and k3moe_finish completes the block.  Needs
   * force_path 0 or 4. */
  int expert_begin;
  int expert_count;
  /* Two-bank graded experts (kimi-k3-mlx README, "REAP expert pruning",
   * graded mode and the two-bank SwitchGLU: the most salient experts keep
   * MXFP4, the next ones a lower bit width, each bank owning a contiguous
   * range of expert ids).  0: one MXFP4 bank.  Otherwise experts
   * [0, bank2_begin) are MXFP4 (the w1/w3/w2 tensors hold those only) and
   * experts [bank2_begin, n_experts) are 2-bit affine (the b2_* tensors):
   * w = scale * q + bias, q in {0..3} packed four per byte low bits first,
   * one bf16 scale and bias per 64 inputs of a row (2.5 bits per weight,
   * the pages' 2-bit tier).  The permutation sorts the selections by expert,
   * so each bank's slots form one contiguous slice; the slice boundary is
   * found on the device and each bank's kernels read it there (no host
   * synchronisation).  Needs force_path 0 or 4 and no expert shard. */
  int bank2_begin;
} k3moe_config;

/* Host arrays in checkpoint layout, experts stacked along dim 0.  Row-major;
 * packed MXFP4 rows hold element 2i in the low nibble of byte i. */
typedef struct {
  const uint16_t* router_w;    /* [E, H] bf16   (gate.weight)                 */
  const float* router_bias;    /* [E]    f32    (e_score_correction_bias)     */
  const uint16_t* down_proj;   /* [L, H] bf16                                 */
  const uint8_t* w1_packed;    /* [E, I, L/2]   gate weight_packed            */
  const uint8_t* w1_scale;     /* [E, I, L/32]  gate weight_scale (e8m0)      */
  const uint8_t* w3_packed;    /* [E, I, L/2]   up                            */
  const uint8_t* w3_scale;     /* [E, I, L/32]                                */
  const uint8_t* w2_packed;    /* [E, L, I/2]   down                          */
  const uint8_t* w2_scale;     /* [E, L, I/32]                                */
  const uint16_t* norm_w;      /* [L]    bf16   RMSNorm weight (gamma)        */
  const uint16_t* up_proj;     /* [H, L] bf16                                 */
  /* shared experts (read only when cfg.n_shared > 0; Is = n_shared *
   * shared_inter, expert s owning intermediate rows [s*shared_inter, ...)) */
  const uint16_t* shared_w1;   /* [Is, H] bf16  gate                          */
  const uint16_t* shared_w3;   /* [Is, H] bf16  up                            */
  const uint16_t* shared_w2;   /* [H, Is] bf16  down                          */
  /* second bank (read only when cfg.bank2_begin > 0; E2 = n_experts -
   * bank2_begin experts, expert bank2_begin + i at index i) */
  const uint8_t* b2_w1q;       /* [E2, I, L/4]  gate codes                    */
  const uint16_t* b2_w1s;      /* [E2, I, L/64] bf16 scales                   */
  const uint16_t* b2_w1b;      /* [E2, I, L/64] bf16 biases                   */
  const uint8_t* b2_w3q;       /* up, as gate                                 */
  const uint16_t* b2_w3s;
  const uint16_t* b2_w3b;
  const uint8_t* b2_w2q;       /* [E2, L, I/4]  down codes                    */
  const uint16_t* b2_w2s;      /* [E2, L, I/64]                               */
  const uint16_t* b2_w2b;
} k3moe_weights;

/* Creates a context on `cuda_device` and allocates its device workspace for
 * cfg->max_tokens tokens.  On success *out owns the context; release it
 * with k3moe_destroy.  Errors: EINVAL (bad config or device), ECUDA,
 * ENOMEM. */
int k3moe_create(const k3moe_config* cfg, int cuda_device, k3moe_ctx** out);

/* Copies the weights (host memory, checkpoint layout) to the device.  The
 * MXFP4 tensors are regrouped (values unchanged) into 128 x 128 blocks of
 * nibbles and 512-byte scale atoms for the block-scaled expert kernels
 * (path 4); contexts created with force_path 1 also keep a copy in
 * 128-row x 64-column tiles for the CUDA-core kernels.  Any scale byte equal
 * to 0xFF is rejected with EBADSCALE before anything is copied.  May be
 * called again to replace the weights.  Synchronous. */
int k3moe_load_weights(k3moe_ctx* ctx, const k3moe_weights* w);

/* One layer forward for T tokens, enqueued on `cuda_stream` (a
 * cudaStream_t; NULL = the legacy default stream).  Asynchronous: returns
 * after launching.  Device pointers:
 *   x        [T, H] bf16 input
 *   y        [T, H] bf16 output
 *   topk_idx [T, K] int32 output: selected experts, descending key; ties
 *            go to the lower expert id
 *   topk_w   [T, K] fp32 output: routing weights in the same order
 * T == 0 is a no-op.  T > max_tokens or T < 0 returns EINVAL.  Performs no
 * allocation and no host synchronisation; a device-side timeout is
 * reported by the next k3moe_status. */
int k3moe_forward(k3moe_ctx* ctx, const void* x, int T, void* y, int32_t* topk_idx,
                  float* topk_w, void* cuda_stream);

/* The same forward with HOST buffers (x_host [T,H] bf16, y_host [T,H] bf16,
 * idx_host [T,K], w_host [T,K]; any of the three outputs may be NULL):
 * copies x to the device, runs the layer, copies the results back and
 * synchronises the stream.  Pinned host memory gives the fastest copies. */
int k3moe_forward_host(k3moe_ctx* ctx, const void* x_host, int T, void* y_host,
                       int32_t* idx_host, float* w_host, void* cuda_stream);

/* Synchronises the context's device, then reports and clears the device
 * status word: K3MOE_OK, or K3MOE_ETIMEOUT if a bounded wait gave up, or
 * ECUDA if a pending CUDA error was found. */
int k3moe_status(k3moe_ctx* ctx);

/* Message of the last failure on `ctx` (or, for NULL, of the last
 * k3moe_create failure on this thread).  Never NULL; owned by the library,
 * valid until the next call on the same context. */
const char* k3moe_last_error(const k3moe_ctx* ctx);

/* Frees the device memory of the context and the context itself.  NULL is
 * a no-op. */
void k3moe_destroy(k3moe_ctx* ctx);

/* ---- expert parallelism: the block split at the combine ---- */

/* The routed chain of one forward up to the score-weighted combine, for
 * this context's experts only: router and top-K over all experts (topk_idx
 * and topk_w as in k3moe_forward, global expert ids), then
 *   c_partial[t] = sum over k in k order, for the selected experts this
 *                  context holds, of topk_w[t,k] * o_k     (fp32, [T, L])
 * and no RMSNorm.  For a context without a shard c_partial is the whole
 * combine.  The shards' c_partial are summed by the caller (one fp32
 * all-reduce of [T, L]; for two shards, c_0 + c_1), because RMSNorm needs
 * the whole combine.  Device pointers, 16-byte aligned; asynchronous on
 * `cuda_stream`; no allocation.  The REAP saliency, when enabled, covers
 * this context's experts (sums indexed by local expert id). */
int k3moe_forward_partial(k3moe_ctx* ctx, const void* x, int T, float* c_partial, int32_t* topk_idx,
                          float* topk_w, void* cuda_stream);

/* The rest of the block for a given combine c_sum [T, L] fp32 (device):
 * n = bf16(c_sum / sqrt(mean(c_sum^2) + eps) * gamma), y = bf16(Wu . n),
 * plus the shared experts of x when configured (x [T, H] bf16 device; may
 * be NULL otherwise).  k3moe_finish(k3moe_forward_partial(x)) on a context
 * without a shard equals k3moe_forward(x).  Asynchronous; no allocation. */
int k3moe_finish(k3moe_ctx* ctx, const void* x, const float* c_sum, int T, void* y, void* cuda_stream);

/* ---- step entry points (the hot path's steps, callable on their own) ---- */

/* MXFP4 -> bf16 dequantisation of a [rows, cols] matrix in checkpoint
 * layout (device pointers: packed [rows, cols/2] u8, scale [rows, cols/32]
 * u8, out [rows, cols] bf16), using the same device decoding routines as
 * the expert kernels (checkpoint bytes -> tile word -> bf16).  kind 0: bf16
 * out (value = e2m1 * 2^(S-127), exact for scale bytes 0..252, IEEE
 * overflow above); kind 1: the same values widened to fp32 (out is then
 * [rows, cols] float), as the CUDA-core kernels use them.  Requires
 * cols % 64 == 0.
 * Asynchronous on `cuda_stream`.  The decoding definition is the "Tiers"
 * section of the kimi-k3-mlx README (same encoding, low bits first, e8m0
 * scales) and K3_ARTIFACT_AUDIT section 4.3 (group 32). */
int k3moe_mxfp4_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols,
                        void* out, int kind, void* cuda_stream);

/* Router step on its own: logits = x . Wr^T into the caller's scratch
 * `logits` [T, E] fp32 (device), then top-K selection and weights with the
 * forward's top-K kernel.  The logits come from a CUDA-core GEMV with fp32
 * FMA chains (k3moe_forward computes them on the tensor cores, fused with
 * down_proj), so the two can differ in the last bits of a logit.  Device pointers: x [T,H] bf16,
 * router_w [E,H] bf16, bias [E] f32, topk_idx [T,K], topk_w [T,K].
 * Requires H % 128 == 0, 1 <= K <= 32, K <= E <= 2048.  Asynchronous. */
int k3moe_route(const void* x, int T, const void* router_w, const float* bias, int E, int H, int K,
                int norm_topk, float routed_scaling, float* logits, int32_t* topk_idx, float* topk_w,
                void* cuda_stream);

/* Router step that allocates nothing, for callers that must not allocate
 * device memory when they route: code running while a CUDA graph is being
 * captured, code living inside another framework's memory pool or under a
 * fixed memory budget, services that forbid allocation after start-up.  (The
 * pages have no counterpart; this is a property of this library's API.)
 * Same inputs, outputs and results as k3moe_route, but the [T, E] fp32
 * logits scratch is a file-scope __device__ array of 131072 floats (512 KiB)
 * that every GPU loading the library holds until the process exits.
 * T * E > 131072 returns K3MOE_EINVAL.  The array's device address is
 * looked up with the calling thread's current device and CUDA context, and
 * cached per context: outside stream capture every call looks it up again
 * (so a context rebuilt after cudaDeviceReset gets a fresh address), while
 * a call made during stream capture uses the cached address of its
 * context.  So the first call on a device (and the first one after a
 * device reset) must come before any stream capture; a first call made
 * during capture returns K3MOE_ESTATE.  Calls never allocate.
 * All calls share the one array and it keeps the last call's contents
 * (nothing here needs it zeroed): calls that overlap on the GPU, from any
 * stream or thread, race on it.  Errors are reported by
 * k3moe_last_error(NULL) on the calling thread. */
int k3moe_route_noalloc(const void* x, int T, const void* router_w, const float* bias, int E, int H, int K,
                        int norm_topk, float routed_scaling, int32_t* topk_idx, float* topk_w,
                        void* cuda_stream);

/* ---- REAP saliency (calibration by-product of the forward) ---- */

/* REAP expert saliency (kimi-k3-mlx README, "REAP expert pruning"):
 *   S_j = (1/|C|) sum over calibration tokens x of g_j(x) ||e_j(x)||_2,
 * g_j(x) the routing weight of expert j for x (topk_w; zero when j is not
 * selected) and e_j(x) the expert's output o in the latent (fp32, before
 * the combine).  With k3moe_saliency(ctx, 1), every later forward (eager
 * or replayed from a captured graph) also adds, for each expert, the terms
 * of its selections to a running fp64 sum -- per expert in slot order (the
 * tokens ascending), so the totals do not depend on scheduling -- and adds
 * T to a token count; both live on the device and start at zero.
 * k3moe_saliency_read synchronises the device and copies the E sums
 * (`sums`, host, may be NULL) and the token count (`tokens`, host, may be
 * NULL); S_j = sums[j] / tokens.  k3moe_saliency_reset zeroes both
 * (synchronising first).  Enabling adds two launches' work to a forward
 * (the per-slot norms in the combine kernel, one accumulation kernel). */
int k3moe_saliency(k3moe_ctx* ctx, int enable);
int k3moe_saliency_read(k3moe_ctx* ctx, double* sums, int n_experts, unsigned long long* tokens);
int k3moe_saliency_reset(k3moe_ctx* ctx);

/* ---- inspection (tests and tools) ---- */

enum {
  K3MOE_BUF_LOGITS = 0, /* [T, E] f32   router logits of the last forward       */
  K3MOE_BUF_LAT = 1,    /* [T, L] bf16  latent after down_proj                   */
  K3MOE_BUF_COUNTS = 2, /* [E]    i32   assignments per expert                   */
  K3MOE_BUF_OFFSETS = 3,/* [E+1]  i32   exclusive prefix sum of COUNTS           */
  K3MOE_BUF_PERM = 4,   /* [T*K]  i32   slot -> t*K + k, grouped by expert, stable */
  K3MOE_BUF_SLOT = 5,   /* [T*K]  i32   t*K + k -> slot                          */
  K3MOE_BUF_H = 6,      /* [T*K, I] bf16 SiTU-GLU output per slot                */
  K3MOE_BUF_O = 7,      /* [T*K, L] f32 expert output per slot                   */
  K3MOE_BUF_N = 8,      /* [T, L] bf16  RMSNorm output                           */
  K3MOE_BUF_ACTIVE = 9, /* [E+1]  i32   number of experts with work, then their ids */
  K3MOE_BUF_SHARED_H = 10, /* [T, Is] bf16 shared experts' SiTU-GLU output      */
  K3MOE_BUF_SHARED_Z = 11  /* [T, H] bf16  shared experts' output z              */
};

/* Copies `bytes` bytes of an internal buffer (K3MOE_BUF_*) of the last
 * forward into host memory `dst` (synchronises the device).  EINVAL if
 * `bytes` exceeds the buffer. */
int k3moe_fetch(k3moe_ctx* ctx, int which, void* dst, size_t bytes);

enum {
  K3MOE_Q_WORKSPACE_BYTES = 0, /* device workspace bytes                       */
  K3MOE_Q_WEIGHT_BYTES = 1,    /* device weight bytes                          */
  K3MOE_Q_LAUNCHES_LAST = 2,   /* kernels launched by the last forward          */
  K3MOE_Q_PATH_LAST = 3,       /* path of the last forward (1 or 4) */
  K3MOE_Q_DEVICE = 4           /* CUDA device ordinal                          */
};

/* Failure detection.  k3moe_check_guards synchronises the device and checks
 * the 256-byte guard bands the library keeps after every workspace buffer
 * (filled with 0xA5 at create): K3MOE_OK, or K3MOE_ESTATE naming the first
 * band a kernel wrote into.  k3moe_test_withhold_copies is a test hook: the
 * next forward's block-scaled gate/up kernel issues no copies for the first
 * pipeline stage of one work item, so that the CTA's bounded waits run out
 * (after spin_timeout_ms), it records K3MOE_ETIMEOUT in the status word,
 * frees its tensor memory and returns; k3moe_status reports it and clears
 * it, and later forwards are unaffected (the hook acts once).  Only that
 * forward's outputs are invalid. */
int k3moe_check_guards(k3moe_ctx* ctx);
int k3moe_test_withhold_copies(k3moe_ctx* ctx);

/* Reads a counter or size of the context into *value. */
int k3moe_query(const k3moe_ctx* ctx, int what, long long* value);

/* Per-step timing.  With profiling enabled, every later forward records a
 * CUDA event on its stream before its first launch and after each launch
 * group (router+down_proj, top-k + permute, tile list, latent terms,
 * gate/up, down, second bank, combine+RMSNorm, up_proj; the groups a
 * forward runs depend on T and the configuration).  k3moe_profile_read waits for the events of the last
 * forward and writes the elapsed milliseconds of each group to ms[0..max)
 * and the number of groups to *count; k3moe_profile_name gives the group's
 * name (a static string, "" out of range).  The events are also recorded
 * inside a captured CUDA graph, so replays can be read the same way. */
int k3moe_profile(k3moe_ctx* ctx, int enable);
int k3moe_profile_read(k3moe_ctx* ctx, float* ms, int max_entries, int* count);
const char* k3moe_profile_name(const k3moe_ctx* ctx, int i);

#ifdef __cplusplus
}
#endif

#endif /* K3MOE_H */
