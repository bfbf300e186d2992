// k3moe_api.cu -- host implementation of the C ABI declared in
// include/k3moe.h: context lifetime, weight loading (with the MXFP4 tile
// re-layout), argument checks and the per-forward launch sequence.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/k3moe.h"
#include "k3moe_device.cuh"
#include "k3moe_internal.h"
#include "k3moe_bs.h"
#include "k3moe_umma.h"

namespace {

thread_local std::string g_create_error = "no error";

constexpr size_t kGuardBytes = 256;
constexpr int kGuardByte = 0xA5;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

namespace k3 {
void set_thread_error(const char* msg) { g_create_error = msg; }
}  // namespace k3

struct k3moe_ctx {
  k3moe_config cfg{};
  int device = 0;
  k3::Dims d{};
  // device weights
  uint16_t* wcat = nullptr;     // [E + L, H]: router rows, then down_proj rows
  float* bias = nullptr;        // [E]
  uint16_t* gamma = nullptr;    // [L]
  uint16_t* wu = nullptr;       // [H, L]
  uint8_t* gu_tiles = nullptr;  // [E][I/128][L/64][2][tile]
  uint8_t* d_tiles = nullptr;   // [E][L/128][I/64][tile]
  // shared experts: gate/up rows interleaved (2j gate_j, 2j+1 up_j), so a
  // GEMM epilogue finds both halves of SiTU-GLU in neighbouring rows
  int Is = 0;                   // n_shared * shared_inter (0: none)
  uint16_t* wsh_gu = nullptr;   // [2 Is, H]
  uint16_t* wsh_d = nullptr;    // [H, Is]
  uint16_t* sh_h = nullptr;     // workspace [Tm, Is]
  uint16_t* sh_z = nullptr;     // workspace [Tm, H]
  float* sh_part = nullptr;     // workspace: split-K partials of the side stream
  cudaStream_t side = nullptr;  // the shared experts run here, beside the routed chain
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // expert shard: experts [shard.begin, shard.begin + E_local) of the router's E
  k3::ExpertShard shard{};
  int E_local = 0;
  bool sharded = false;
  // second bank (two-bank graded experts): experts >= bank2_begin in 2-bit tiles
  int bank2_begin = 0;           // 0: one bank
  uint8_t* gu2_tiles = nullptr;  // [E2][I/128][L/64][2][2560]
  uint8_t* d2_tiles = nullptr;   // [E2][L/128][I/64][2560]
  int* iota = nullptr;   // workspace [Tm]: 0, 1, 2, ... (RMSNorm of a given combine)
  bool test_withhold = false;  // test hook: the next forward's gate/up kernel withholds one stage's copies
  // guard bands: 256 bytes of kGuardByte after every workspace buffer, to
  // catch a kernel writing past the end of its buffer (k3moe_check_guards)
  std::vector<uint8_t*> guards;
  float* ones = nullptr; // workspace [Tm]: 1.0
  // REAP saliency accumulation (off unless enabled)
  bool sal_on = false;
  float* sal_tk = nullptr;          // workspace [Tm * K]: w_k ||o_k|| of the last forward
  double* sal_sum = nullptr;        // [E] running sums (zero at create and reset)
  unsigned long long* sal_tokens = nullptr;  // calibration tokens accumulated
  size_t weight_bytes = 0;
  bool loaded = false;
  // workspace
  void* ws = nullptr;
  size_t ws_bytes = 0;
  k3::Work w{};
  size_t sz_logits = 0, sz_lat = 0, sz_counts = 0, sz_offsets = 0, sz_active = 0, sz_perm = 0, sz_h = 0, sz_o = 0,
         sz_n = 0;
  uint16_t* x_stage = nullptr;
  uint16_t* y_stage = nullptr;
  int32_t* idx_stage = nullptr;
  float* w_stage = nullptr;
  k3::UmmaPlan umma{};
  k3::BsPlan bs{};
  k3::BsWeights bw{};
  long long launches_last = 0;
  int path_last = 0;
  int split_dn_last = 1;  // K parts of the last forward's down GEMM (o lives in part planes when > 1)
  int T_last = 0;
  // optional per-step timing: events around each launch group of a forward
  static constexpr int kMaxProf = 16;
  bool prof = false;
  int prof_n = 0;
  cudaEvent_t prof_ev[kMaxProf + 1] = {};
  const char* prof_name[kMaxProf] = {};
  std::string err = "no error";
};

namespace {

int fail(k3moe_ctx* c, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (c)
    c->err = buf;
  else
    g_create_error = buf;
  return code;
}

int cuda_fail(k3moe_ctx* c, cudaError_t e, const char* what) {
  return fail(c, e == cudaErrorMemoryAllocation ? K3MOE_ENOMEM : K3MOE_ECUDA, "%s: %s (%s)", what,
              cudaGetErrorName(e), cudaGetErrorString(e));
}

#define K3_CUDA(c, call, what)                 \
  do {                                         \
    cudaError_t e_ = (call);                   \
    if (e_ != cudaSuccess) return cuda_fail(c, e_, what); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_config(const k3moe_config* c) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "config is NULL");
  if (c->hidden <= 0 || c->latent <= 0 || c->inter <= 0 || c->n_experts <= 0 || c->top_k <= 0)
    return fail(nullptr, K3MOE_EINVAL, "dimensions must be positive");
  if (c->hidden % 128 || c->latent % 128 || c->inter % 128)
    return fail(nullptr, K3MOE_EINVAL, "hidden, latent and inter must be multiples of 128 (got %d, %d, %d)",
                c->hidden, c->latent, c->inter);
  if (c->group != 32) return fail(nullptr, K3MOE_EINVAL, "only MXFP4 group 32 is supported (got %d)", c->group);
  if (c->top_k > 32 || c->top_k > c->n_experts || c->n_experts > 2048)
    return fail(nullptr, K3MOE_EINVAL, "need top_k <= 32, top_k <= n_experts <= 2048");
  if (c->max_tokens < 1 || c->max_tokens > (1 << 20))
    return fail(nullptr, K3MOE_EINVAL, "max_tokens must be in [1, 2^20] (got %d)", c->max_tokens);
  if (!(c->rms_eps >= 0.f) || !(c->beta > 0.f) || !(c->beta_lin > 0.f))
    return fail(nullptr, K3MOE_EINVAL, "beta, beta_lin must be > 0 and rms_eps >= 0");
  if (c->spin_timeout_ms < 0) return fail(nullptr, K3MOE_EINVAL, "spin_timeout_ms must be >= 0");
  if (c->force_path != 0 && c->force_path != 1 && c->force_path != 4)
    return fail(nullptr, K3MOE_EINVAL, "force_path must be 0, 1 or 4 (got %d)", c->force_path);
  if (c->n_shared < 0 || c->shared_inter < 0 || (c->n_shared > 0) != (c->shared_inter > 0))
    return fail(nullptr, K3MOE_EINVAL, "n_shared and shared_inter must both be 0 or both positive");
  if (c->n_shared > 0) {
    const long long Is = (long long)c->n_shared * c->shared_inter;
    if (Is % 128 || Is > (1 << 16))
      return fail(nullptr, K3MOE_EINVAL, "n_shared * shared_inter must be a multiple of 128 and <= 65536");
    if (c->force_path == 1)
      return fail(nullptr, K3MOE_EINVAL, "shared experts need force_path 0 or 4 (tensor-core dense GEMMs)");
  }
  if (c->expert_begin < 0 || c->expert_count < 0 || c->expert_begin + c->expert_count > c->n_experts ||
      (c->expert_count == 0 && c->expert_begin != 0))
    return fail(nullptr, K3MOE_EINVAL, "expert shard [%d, %d + %d) outside [0, n_experts=%d)", c->expert_begin,
                c->expert_begin, c->expert_count, c->n_experts);
  if (c->expert_count > 0 && c->expert_count < c->n_experts && c->force_path == 1)
    return fail(nullptr, K3MOE_EINVAL, "an expert shard needs force_path 0 or 4");
  if (c->bank2_begin < 0 || c->bank2_begin >= c->n_experts)
    return fail(nullptr, K3MOE_EINVAL, "bank2_begin must be 0 (one bank) or in [1, n_experts) (got %d)",
                c->bank2_begin);
  if (c->bank2_begin > 0 && ((c->expert_count > 0 && c->expert_count < c->n_experts) ||
                             (c->force_path != 0 && c->force_path != 4)))
    return fail(nullptr, K3MOE_EINVAL, "a second bank needs force_path 0 or 4 and no expert shard");
  return K3MOE_OK;
}

}  // namespace

extern "C" {

int k3moe_create(const k3moe_config* cfg, int cuda_device, k3moe_ctx** out) {
  if (!out) return fail(nullptr, K3MOE_EINVAL, "out is NULL");
  *out = nullptr;
  int rc = check_config(cfg);
  if (rc) return rc;
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess || ndev == 0)
    return fail(nullptr, K3MOE_ECUDA, "no CUDA device available (%s)", cudaGetErrorString(e));
  if (cuda_device < 0 || cuda_device >= ndev)
    return fail(nullptr, K3MOE_EINVAL, "device %d out of range [0, %d)", cuda_device, ndev);
  cudaDeviceProp prop;
  if ((e = cudaGetDeviceProperties(&prop, cuda_device)) != cudaSuccess)
    return fail(nullptr, K3MOE_ECUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
  if (prop.major != 10 || prop.minor != 3)
    return fail(nullptr, K3MOE_EINVAL, "this library is built for sm_103a (GB300); device %d is sm_%d%d",
                cuda_device, prop.major, prop.minor);
  if ((e = cudaSetDevice(cuda_device)) != cudaSuccess)
    return fail(nullptr, K3MOE_ECUDA, "cudaSetDevice: %s", cudaGetErrorString(e));

  k3moe_ctx* c = new k3moe_ctx();
  c->cfg = *cfg;
  if (c->cfg.spin_timeout_ms == 0) c->cfg.spin_timeout_ms = 2000;
  c->device = cuda_device;
  c->d = k3::Dims{cfg->hidden, cfg->latent, cfg->n_experts, cfg->top_k, cfg->inter, cfg->beta, cfg->beta_lin,
                  cfg->rms_eps, cfg->routed_scaling, cfg->norm_topk};
  const size_t Tm = (size_t)cfg->max_tokens, H = cfg->hidden, L = cfg->latent, E = cfg->n_experts,
               K = cfg->top_k, I = cfg->inter;
  const size_t nblk = (Tm * K + k3::kPermChunk - 1) / k3::kPermChunk;
  c->sz_logits = Tm * E * 4;
  c->sz_lat = Tm * L * 2;
  c->E_local = cfg->expert_count > 0 ? cfg->expert_count : cfg->n_experts;
  c->sharded = c->E_local < cfg->n_experts;
  c->shard.begin = c->sharded ? cfg->expert_begin : 0;
  c->shard.n_listed = c->E_local;
  c->shard.n_buckets = c->sharded ? c->E_local + 1 : c->E_local;
  c->bank2_begin = cfg->bank2_begin;
  // bucket arrays: counts [buckets], offsets and active [buckets + 1]
  c->sz_counts = (E + 1) * 4;
  c->sz_offsets = (E + 2) * 4;
  c->sz_active = (E + 2) * 4;
  c->sz_perm = Tm * K * 4;
  c->sz_h = Tm * K * I * 2;
  c->sz_o = Tm * K * L * 4;
  c->sz_n = Tm * L * 2;
  c->umma = k3::umma_plan(c->d, (int)Tm);
  const size_t bs_bytes = k3::bs_ws_bytes(c->d, (int)Tm);
  c->Is = cfg->n_shared * cfg->shared_inter;
  const size_t Is = (size_t)c->Is;
  const size_t sh_part = Is ? k3::dense_small_part_floats((int)std::max(2 * Is, H)) * 4 : 0;
  const size_t parts[] = {c->sz_logits, c->sz_lat,   c->sz_counts, c->sz_offsets, c->sz_active, c->sz_perm,
                          c->sz_perm,   nblk * (E + 1) * 4, c->sz_h, c->sz_o,       c->sz_n,      256,
                          Tm * H * 2,   Tm * H * 2,   Tm * K * 4,  Tm * K * 4,    c->umma.ws_bytes, bs_bytes,
                          Tm * Is * 2,  Is ? Tm * H * 2 : 0, sh_part,   Tm * K * 4,  E * 8 + 8,  Tm * 4,  Tm * 4};
  size_t total = 0;
  for (size_t p : parts) total += align_up(p, 256) + kGuardBytes;
  e = cudaMalloc(&c->ws, total);
  if (e != cudaSuccess) {
    fail(nullptr, K3MOE_ENOMEM, "workspace of %zu bytes for max_tokens=%d: %s", total, cfg->max_tokens,
         cudaGetErrorString(e));
    delete c;
    return K3MOE_ENOMEM;
  }
  c->ws_bytes = total;
  char* p = static_cast<char*>(c->ws);
  auto take = [&](size_t n) {
    char* r = p;
    p += align_up(n, 256);
    c->guards.push_back(reinterpret_cast<uint8_t*>(p));
    p += kGuardBytes;
    return r;
  };
  c->w.logits = (float*)take(parts[0]);
  c->w.lat = (uint16_t*)take(parts[1]);
  c->w.counts = (int*)take(parts[2]);
  c->w.offsets = (int*)take(parts[3]);
  c->w.active = (int*)take(parts[4]);
  c->w.perm = (int*)take(parts[5]);
  c->w.slot = (int*)take(parts[6]);
  c->w.blk_hist = (int*)take(parts[7]);
  c->w.h = (uint16_t*)take(parts[8]);
  c->w.o = (float*)take(parts[9]);
  c->w.n = (uint16_t*)take(parts[10]);
  c->w.status = (unsigned*)take(parts[11]);
  c->x_stage = (uint16_t*)take(parts[12]);
  c->y_stage = (uint16_t*)take(parts[13]);
  c->idx_stage = (int32_t*)take(parts[14]);
  c->w_stage = (float*)take(parts[15]);
  c->umma.ws = take(parts[16]);
  c->umma.status = c->w.status;
  c->umma.num_sms = prop.multiProcessorCount;
  c->umma.limit_ns = (uint64_t)c->cfg.spin_timeout_ms * 1000000ull;
  c->bs.ws = take(parts[17]);
  c->sh_h = (uint16_t*)take(parts[18]);
  c->sh_z = (uint16_t*)take(parts[19]);
  c->sh_part = (float*)take(parts[20]);
  c->sal_tk = (float*)take(parts[21]);
  c->sal_sum = (double*)take(parts[22]);
  c->sal_tokens = (unsigned long long*)(c->sal_sum + E);
  c->iota = (int*)take(parts[23]);
  c->ones = (float*)take(parts[24]);
  c->bs.ws_bytes = bs_bytes;
  c->bs.max_tokens = (int)Tm;
  c->bs.status = c->w.status;
  c->bs.num_sms = prop.multiProcessorCount;
  c->bs.limit_ns = c->umma.limit_ns;
  c->bs.dims = c->d;
  e = cudaMemset(c->ws, 0, total);
  for (uint8_t* gp : c->guards)
    if (e == cudaSuccess) e = cudaMemset(gp, kGuardByte, kGuardBytes);
  if (e == cudaSuccess) {
    std::vector<int> iota(Tm);
    std::vector<float> ones(Tm, 1.0f);
    for (size_t i = 0; i < Tm; ++i) iota[i] = (int)i;
    e = cudaMemcpy(c->iota, iota.data(), Tm * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(c->ones, ones.data(), Tm * 4, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = k3::prepare_decode_kernels(c->d);
  if (e == cudaSuccess) e = k3::prepare_umma_kernels();
  if (e == cudaSuccess) e = k3::prepare_bs_kernels();
  if (e == cudaSuccess && c->Is) e = cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking);
  if (e == cudaSuccess && c->Is) e = cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess && c->Is) e = cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    fail(nullptr, K3MOE_ECUDA, "workspace / kernel setup: %s", cudaGetErrorString(e));
    cudaFree(c->ws);
    delete c;
    return K3MOE_ECUDA;
  }
  *out = c;
  return K3MOE_OK;
}

void k3moe_destroy(k3moe_ctx* c) {
  if (!c) return;
  cudaSetDevice(c->device);
  cudaDeviceSynchronize();
  cudaFree(c->ws);
  cudaFree(c->wcat);
  cudaFree(c->bias);
  cudaFree(c->gamma);
  cudaFree(c->wu);
  cudaFree(c->gu_tiles);
  cudaFree(c->d_tiles);
  cudaFree(c->bw.gu_q);
  cudaFree(c->wsh_gu);
  cudaFree(c->wsh_d);
  cudaFree(c->gu2_tiles);
  cudaFree(c->d2_tiles);
  if (c->side) cudaStreamDestroy(c->side);
  if (c->ev_fork) cudaEventDestroy(c->ev_fork);
  if (c->ev_join) cudaEventDestroy(c->ev_join);
  for (cudaEvent_t ev : c->prof_ev)
    if (ev) cudaEventDestroy(ev);
  delete c;
}

const char* k3moe_last_error(const k3moe_ctx* c) { return c ? c->err.c_str() : g_create_error.c_str(); }

int k3moe_load_weights(k3moe_ctx* c, const k3moe_weights* wt) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  if (!wt) return fail(c, K3MOE_EINVAL, "weights is NULL");
  const void* ptrs[] = {wt->router_w,  wt->router_bias, wt->down_proj, wt->w1_packed, wt->w1_scale, wt->w3_packed,
                        wt->w3_scale,  wt->w2_packed,   wt->w2_scale,  wt->norm_w,    wt->up_proj};
  for (const void* q : ptrs)
    if (!q) return fail(c, K3MOE_EINVAL, "a weight pointer is NULL");
  if (c->Is && (!wt->shared_w1 || !wt->shared_w3 || !wt->shared_w2))
    return fail(c, K3MOE_EINVAL, "the context has shared experts but a shared weight pointer is NULL");
  if (c->bank2_begin) {
    const void* b2[] = {wt->b2_w1q, wt->b2_w1s, wt->b2_w1b, wt->b2_w3q, wt->b2_w3s,
                        wt->b2_w3b, wt->b2_w2q, wt->b2_w2s, wt->b2_w2b};
    for (const void* q : b2)
      if (!q) return fail(c, K3MOE_EINVAL, "the context has a second bank but a b2_* pointer is NULL");
  }
  // the router, bias and dense weights cover all Er experts; the expert
  // tensors hold this context's E (its shard, or all of them)
  // (with a second bank the MXFP4 tensors hold its first bank2_begin experts)
  const size_t H = c->d.H, L = c->d.L, Er = c->d.E, I = c->d.I;
  const size_t E = c->bank2_begin ? (size_t)c->bank2_begin : (size_t)c->E_local;
  k3::Dims dx = c->d;
  dx.E = (int)E;
  const size_t n_gu_scale = E * I * (L / 32), n_d_scale = E * L * (I / 32);
  const uint8_t* scales[] = {wt->w1_scale, wt->w3_scale, wt->w2_scale};
  const size_t nscales[] = {n_gu_scale, n_gu_scale, n_d_scale};
  const char* names[] = {"w1_scale", "w3_scale", "w2_scale"};
  for (int i = 0; i < 3; ++i) {
    const void* hit = memchr(scales[i], 0xFF, nscales[i]);
    if (hit)
      return fail(c, K3MOE_EBADSCALE, "%s holds the e8m0 NaN byte 0xFF at offset %zu", names[i],
                  (size_t)((const uint8_t*)hit - scales[i]));
  }
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  const size_t gu_bytes = E * (I / 128) * (L / 64) * 2 * (size_t)k3::kTileBytes;
  const size_t d_bytes = E * (L / 128) * (I / 64) * (size_t)k3::kTileBytes;
  // The tile copy of the experts serves the CUDA-core path (1) only; the
  // default (path 4) reads the block-scaled copy alone.
  const bool want_tiles = c->cfg.force_path == 1;
  if (!c->wcat) {
    K3_CUDA(c, cudaMalloc(&c->wcat, (Er + L) * H * 2), "cudaMalloc(router+down_proj)");
    K3_CUDA(c, cudaMalloc(&c->bias, Er * 4), "cudaMalloc(bias)");
    K3_CUDA(c, cudaMalloc(&c->gamma, L * 2), "cudaMalloc(gamma)");
    K3_CUDA(c, cudaMalloc(&c->wu, H * L * 2), "cudaMalloc(up_proj)");
    if (want_tiles) {
      K3_CUDA(c, cudaMalloc(&c->gu_tiles, gu_bytes), "cudaMalloc(gate/up tiles)");
      K3_CUDA(c, cudaMalloc(&c->d_tiles, d_bytes), "cudaMalloc(down tiles)");
    }
    // block-scaled layout: one allocation, carved as gu_q | gu_sf | d_q | d_sf
    K3_CUDA(c, cudaMalloc(&c->bw.gu_q, k3::bs_weight_bytes(dx)), "cudaMalloc(block-scaled experts)");
    c->bw.n_exp = (int)E;
    c->bw.gu_sf = c->bw.gu_q + E * 2 * I * L / 2;
    c->bw.d_q = c->bw.gu_sf + E * 2 * I * L / 32;
    c->bw.d_sf = c->bw.d_q + E * L * I / 2;
    c->weight_bytes = (Er + L) * H * 2 + Er * 4 + L * 2 + H * L * 2 + (want_tiles ? gu_bytes + d_bytes : 0) +
                      k3::bs_weight_bytes(dx);
  }
  c->loaded = false;
  K3_CUDA(c, cudaMemcpy(c->wcat, wt->router_w, Er * H * 2, cudaMemcpyHostToDevice), "copy router_w");
  K3_CUDA(c, cudaMemcpy(c->wcat + Er * H, wt->down_proj, L * H * 2, cudaMemcpyHostToDevice), "copy down_proj");
  K3_CUDA(c, cudaMemcpy(c->bias, wt->router_bias, Er * 4, cudaMemcpyHostToDevice), "copy bias");
  K3_CUDA(c, cudaMemcpy(c->gamma, wt->norm_w, L * 2, cudaMemcpyHostToDevice), "copy norm_w");
  K3_CUDA(c, cudaMemcpy(c->wu, wt->up_proj, H * L * 2, cudaMemcpyHostToDevice), "copy up_proj");
  if (c->Is) {
    const size_t Is = (size_t)c->Is;
    if (!c->wsh_gu) {
      K3_CUDA(c, cudaMalloc(&c->wsh_gu, 2 * Is * H * 2), "cudaMalloc(shared gate/up)");
      K3_CUDA(c, cudaMalloc(&c->wsh_d, H * Is * 2), "cudaMalloc(shared down)");
      c->weight_bytes += 3 * Is * H * 2;
    }
    // gate row j -> row 2j, up row j -> row 2j + 1
    K3_CUDA(c, cudaMemcpy2D(c->wsh_gu, 2 * H * 2, wt->shared_w1, H * 2, H * 2, Is, cudaMemcpyHostToDevice),
            "copy shared_w1");
    K3_CUDA(c, cudaMemcpy2D(c->wsh_gu + H, 2 * H * 2, wt->shared_w3, H * 2, H * 2, Is, cudaMemcpyHostToDevice),
            "copy shared_w3");
    K3_CUDA(c, cudaMemcpy(c->wsh_d, wt->shared_w2, H * Is * 2, cudaMemcpyHostToDevice), "copy shared_w2");
  }

  // Experts: stage a chunk of experts of one tensor, re-lay into tiles.
  const size_t per_expert_packed = I * L / 2, per_expert_scale = I * L / 32;  // same for w1/w3/w2
  size_t chunk = std::max<size_t>(1, (size_t)(256u << 20) / per_expert_packed);
  chunk = std::min(chunk, E);
  uint8_t *st_p = nullptr, *st_s = nullptr;
  K3_CUDA(c, cudaMalloc(&st_p, chunk * per_expert_packed), "cudaMalloc(staging)");
  cudaError_t e = cudaMalloc(&st_s, chunk * per_expert_scale);
  if (e != cudaSuccess) {
    cudaFree(st_p);
    return cuda_fail(c, e, "cudaMalloc(staging)");
  }
  struct Job {
    const uint8_t *p, *s;
    int rows, cols;
    uint8_t* tiles;
    size_t mat_stride;
    int step, offset;
  } jobs[3] = {
      {wt->w1_packed, wt->w1_scale, (int)I, (int)L, c->gu_tiles, (I / 128) * (L / 64) * 2, 2, 0},
      {wt->w3_packed, wt->w3_scale, (int)I, (int)L, c->gu_tiles, (I / 128) * (L / 64) * 2, 2, 1},
      {wt->w2_packed, wt->w2_scale, (int)L, (int)I, c->d_tiles, (L / 128) * (I / 64), 1, 0},
  };
  int rc = K3MOE_OK;
  for (const Job& j : jobs) {
    if (!want_tiles) break;
    for (size_t e0 = 0; e0 < E && rc == K3MOE_OK; e0 += chunk) {
      const size_t ne = std::min(chunk, E - e0);
      if ((e = cudaMemcpy(st_p, j.p + e0 * per_expert_packed, ne * per_expert_packed, cudaMemcpyHostToDevice)) ||
          (e = cudaMemcpy(st_s, j.s + e0 * per_expert_scale, ne * per_expert_scale, cudaMemcpyHostToDevice)) ||
          (e = k3::launch_relayout(st_p, st_s, (int)ne, j.rows, j.cols,
                                   j.tiles + e0 * j.mat_stride * (size_t)k3::kTileBytes, j.mat_stride, j.step,
                                   j.offset, 0)) ||
          (e = cudaDeviceSynchronize()))
        rc = cuda_fail(c, e, "expert re-layout");
    }
  }
  // block-scaled layout: nibbles unchanged, regrouped into contiguous
  // 128 x 128 boxes (gate and up of an expert adjacent); scales into
  // 512-byte atoms
  struct QJob {
    const uint8_t* p;
    int rows, cols, n_mat, mat;
    uint8_t* out;
  } qjobs[3] = {{wt->w1_packed, (int)I, (int)L, 2, 0, c->bw.gu_q},
                {wt->w3_packed, (int)I, (int)L, 2, 1, c->bw.gu_q},
                {wt->w2_packed, (int)L, (int)I, 1, 0, c->bw.d_q}};
  for (const QJob& j : qjobs) {
    for (size_t e0 = 0; e0 < E && rc == K3MOE_OK; e0 += chunk) {
      const size_t ne = std::min(chunk, E - e0);
      if ((e = cudaMemcpy(st_p, j.p + e0 * per_expert_packed, ne * per_expert_packed, cudaMemcpyHostToDevice)) ||
          (e = k3::bs_e2m1_boxes(st_p, (int)ne, j.rows, j.cols, j.n_mat, j.mat,
                                 j.out + e0 * j.n_mat * per_expert_packed, 0)) ||
          (e = cudaDeviceSynchronize()))
        rc = cuda_fail(c, e, "block-scaled expert boxes");
    }
  }
  struct SJob {
    const uint8_t* s;
    int rows, cols, n_mat, mat;
    uint8_t* out;
  } sjobs[3] = {{wt->w1_scale, (int)I, (int)L, 2, 0, c->bw.gu_sf},
                {wt->w3_scale, (int)I, (int)L, 2, 1, c->bw.gu_sf},
                {wt->w2_scale, (int)L, (int)I, 1, 0, c->bw.d_sf}};
  for (const SJob& j : sjobs) {
    for (size_t e0 = 0; e0 < E && rc == K3MOE_OK; e0 += chunk) {
      const size_t ne = std::min(chunk, E - e0);
      const size_t atoms_per_expert = (size_t)(j.rows / 128) * (j.cols / 128) * j.n_mat;
      if ((e = cudaMemcpy(st_s, j.s + e0 * per_expert_scale, ne * per_expert_scale, cudaMemcpyHostToDevice)) ||
          (e = k3::bs_scale_atoms(st_s, (int)ne, j.rows, j.cols, j.n_mat, j.mat,
                                  j.out + e0 * atoms_per_expert * 512, 0)) ||
          (e = cudaDeviceSynchronize()))
        rc = cuda_fail(c, e, "block-scaled scale atoms");
    }
  }
  cudaFree(st_p);
  cudaFree(st_s);
  if (rc) return rc;
  if (c->bank2_begin) {
    // second bank: 2-bit codes + bf16 scale/bias into 2-bit tiles (gate and
    // up of one (expert, row tile, k step) adjacent); staged per expert
    const size_t E2 = (size_t)(c->d.E - c->bank2_begin);
    const size_t gu_t = k3::bank2_tile_bytes((int)I, (int)L), d_t = k3::bank2_tile_bytes((int)L, (int)I);
    if (!c->gu2_tiles) {
      K3_CUDA(c, cudaMalloc(&c->gu2_tiles, E2 * 2 * gu_t), "cudaMalloc(second-bank gate/up)");
      K3_CUDA(c, cudaMalloc(&c->d2_tiles, E2 * d_t), "cudaMalloc(second-bank down)");
      c->weight_bytes += E2 * (2 * gu_t + d_t);
    }
    struct B2Job {
      const uint8_t* q;
      const uint16_t *sc, *bi;
      int rows, cols, step, offset;
      uint8_t* out;
      size_t stride_tiles;
    } b2jobs[3] = {{wt->b2_w1q, wt->b2_w1s, wt->b2_w1b, (int)I, (int)L, 2, 0, c->gu2_tiles, 2 * gu_t / 2560},
                   {wt->b2_w3q, wt->b2_w3s, wt->b2_w3b, (int)I, (int)L, 2, 1, c->gu2_tiles, 2 * gu_t / 2560},
                   {wt->b2_w2q, wt->b2_w2s, wt->b2_w2b, (int)L, (int)I, 1, 0, c->d2_tiles, d_t / 2560}};
    const size_t nq = I * L / 4, ns = I * (L / 64);  // per expert and matrix (same for w2)
    uint8_t* stage = nullptr;
    K3_CUDA(c, cudaMalloc(&stage, nq + 2 * ns * 2), "cudaMalloc(staging)");
    for (const B2Job& j : b2jobs) {
      for (size_t e2 = 0; e2 < E2 && rc == K3MOE_OK; ++e2) {
        uint16_t* st_sc = reinterpret_cast<uint16_t*>(stage + nq);
        uint16_t* st_bi = st_sc + ns;
        if ((e = cudaMemcpy(stage, j.q + e2 * nq, nq, cudaMemcpyHostToDevice)) ||
            (e = cudaMemcpy(st_sc, j.sc + e2 * ns, ns * 2, cudaMemcpyHostToDevice)) ||
            (e = cudaMemcpy(st_bi, j.bi + e2 * ns, ns * 2, cudaMemcpyHostToDevice)) ||
            (e = k3::bank2_tiles(stage, st_sc, st_bi, 1, j.rows, j.cols, j.out + e2 * j.stride_tiles * 2560,
                                 j.stride_tiles, j.step, j.offset, 0)) ||
            (e = cudaDeviceSynchronize()))
          rc = cuda_fail(c, e, "second-bank tiles");
      }
    }
    cudaFree(stage);
    if (rc) return rc;
  }
  c->loaded = true;
  return K3MOE_OK;
}

// The block for T tokens, in one of three modes:
//   c_out == c_in == NULL: the whole block, x -> y;
//   c_out != NULL: the routed chain up to the combine: c_out = the partial
//                  combine of this context's experts (an expert shard's
//                  part; all experts without a shard), no RMSNorm;
//   c_in != NULL:  the rest of the block for a given combine c_in: shared
//                  experts of x, RMSNorm(c_in), up_proj -> y.
static int forward_impl(k3moe_ctx* c, const void* x, int T, void* y, int32_t* idx, float* wts,
                        cudaStream_t s, float* c_out = nullptr, const float* c_in = nullptr) {
  const k3::Dims& d = c->d;
  const bool routed = c_in == nullptr;  // router, permutation, experts, combine
  const bool tail = c_out == nullptr;   // shared experts, RMSNorm, up_proj
  k3::Work& w = c->w;
  // path: 4 (default) tensor-core dense projections and the experts on the
  // block-scaled MXFP4 tensor cores; 1 CUDA-core kernels everywhere (an
  // independent implementation kept as a cross-check)
  int path = c->cfg.force_path;
  if (path == 0) path = 4;
  c->bs.withhold_item = c->test_withhold ? 0 : -1;
  c->test_withhold = false;  // one forward only
  c->path_last = path;
  long long n = 0;
  cudaError_t e;
  c->prof_n = 0;
  // While a graph is being captured, event records must be "external" to be
  // updated by every replay and readable outside the graph; outside capture
  // that flag is not allowed.
  unsigned ev_flags = cudaEventRecordDefault;
  if (c->prof) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(s, &cs)) != cudaSuccess) return cuda_fail(c, e, "cudaStreamIsCapturing");
    if (cs == cudaStreamCaptureStatusActive) ev_flags = cudaEventRecordExternal;
    if ((e = cudaEventRecordWithFlags(c->prof_ev[0], s, ev_flags)) != cudaSuccess)
      return cuda_fail(c, e, "profile event");
  }
#define K3_LAUNCH(expr, count, what)                                                    \
  do {                                                                                  \
    if ((e = (expr)) != cudaSuccess) return cuda_fail(c, e, what);                      \
    n += (count);                                                                       \
    if (c->prof && c->prof_n < k3moe_ctx::kMaxProf) {                                   \
      c->prof_name[c->prof_n] = what;                                                   \
      if ((e = cudaEventRecordWithFlags(c->prof_ev[++c->prof_n], s, ev_flags)) != cudaSuccess) \
        return cuda_fail(c, e, "profile event");                                        \
    }                                                                                   \
  } while (0)
  // Shared experts (on the residual x, independent of the routed chain):
  // gate/up with the SiTU-GLU epilogue -> sh_h, down -> sh_z; up_proj adds
  // sh_z.  They run on the context's side stream, forked here and joined
  // before up_proj, so their weight stream overlaps the routing and
  // expert-permutation latency of the routed chain.  With per-group
  // profiling they run on `s` instead, as groups of their own.
  auto shared_launch = [&](cudaStream_t q, float* part) -> cudaError_t {
    k3::DenseOut o_gu;
    o_gu.glu = 1;
    o_gu.out_bf16 = c->sh_h;
    o_gu.beta = d.beta;
    o_gu.beta_lin = d.beta_lin;
    k3::DenseOut o_dn;
    o_dn.out_bf16 = c->sh_z;
    cudaError_t r;
    if (T <= 64) {
      r = k3::umma_dense_small(c->umma, c->wsh_gu, 2 * c->Is, d.H, (const uint16_t*)x, T, o_gu, part, q);
      if (r == cudaSuccess) r = k3::umma_dense_small(c->umma, c->wsh_d, d.H, c->Is, c->sh_h, T, o_dn, part, q);
    } else {
      r = k3::umma_dense(c->umma, c->wsh_gu, 2 * c->Is, d.H, (const uint16_t*)x, T, o_gu, q);
      if (r == cudaSuccess) r = k3::umma_dense(c->umma, c->wsh_d, d.H, c->Is, c->sh_h, T, o_dn, q);
    }
    return r;
  };
  const int shared_launches = c->Is ? 2 * (T <= 64 ? k3::umma_dense_small_launches() : k3::umma_dense_launches()) : 0;
  const bool shared_side = tail && c->Is && !c->prof;
  if (shared_side) {
    if ((e = cudaEventRecord(c->ev_fork, s)) != cudaSuccess) return cuda_fail(c, e, "fork event");
    if ((e = cudaStreamWaitEvent(c->side, c->ev_fork, 0)) != cudaSuccess) return cuda_fail(c, e, "fork wait");
    if ((e = shared_launch(c->side, c->sh_part)) != cudaSuccess) return cuda_fail(c, e, "shared experts");
    if ((e = cudaEventRecord(c->ev_join, c->side)) != cudaSuccess) return cuda_fail(c, e, "join event");
    n += shared_launches;
  }
  // the slots of this context's experts: all of them without a shard
  const int* n_local = w.offsets + c->shard.n_listed;
  if (routed) {
  // router logits (fp32) and the latent (bf16) from one pass over [Wr; Wd]
  k3::DenseOut o_route;
  o_route.split = d.E;
  o_route.out_f32 = w.logits;
  o_route.out_bf16 = w.lat;
  if (path == 4 && T <= 64) {
    K3_LAUNCH(k3::umma_dense_small(c->umma, c->wcat, d.E + d.L, d.H, (const uint16_t*)x, T, o_route, nullptr, s),
              k3::umma_dense_small_launches(), "router + down_proj");
  } else if (path == 4) {
    K3_LAUNCH(k3::umma_dense(c->umma, c->wcat, d.E + d.L, d.H, (const uint16_t*)x, T, o_route, s),
              k3::umma_dense_launches(), "router + down_proj");
  } else {
    K3_LAUNCH(k3::launch_dense_gemv(c->wcat, d.E + d.L, d.H, (const uint16_t*)x, T, d.E, w.logits, w.lat, s), 1,
              "router + down_proj");
  }
  const bool fused_route = path == 4 && T * d.K <= 1024;
  const int split_expert = c->bank2_begin ? c->bank2_begin : (1 << 30);
  if (fused_route) {
    int4* tiles;
    int* tile_count;
    int bn;
    k3::umma_tile_list(c->umma, &tiles, &tile_count, &bn);
    // with the slot -> tile map (the tiles have bs_tile_rows(T) <= bn rows)
    int* slot_tile = k3::bs_slot_tile(c->bs);
    bn = k3::bs_tile_rows(T, c->bank2_begin != 0);
    K3_LAUNCH(k3::launch_route_small(w.logits, T, d.E, c->bias, d.K, d.norm_topk, d.rsf, c->shard, idx, wts,
                                     w.counts, w.offsets, w.active, w.perm, w.slot, bn, tiles, tile_count, slot_tile,
                                     split_expert, s),
              2, "top-k + permute");
  } else {
    K3_LAUNCH(k3::launch_topk(w.logits, T, d.E, d.E, c->bias, d.K, d.norm_topk, d.rsf, idx, wts, s), 1, "top-k");
    K3_LAUNCH(k3::launch_permute(idx, T, d.K, c->shard, w.blk_hist, w.counts, w.offsets, w.active, w.perm, w.slot,
                                 s),
              3, "permute");
  }
  const int max_active = std::min(d.E, T * d.K);
  int split_gu = 1, split_dn = 1;  // K parts of the T = 1 expert kernels
  if (path == 4) {
    int4* tiles;
    int* tile_count;
    int bn;
    k3::umma_tile_list(c->umma, &tiles, &tile_count, &bn);
    bn = k3::bs_tile_rows(T, c->bank2_begin != 0);
    if (!fused_route)
      K3_LAUNCH(k3::umma_stream_tiles(c->umma, w, T, d, bn, k3::bs_slot_tile(c->bs), split_expert, s), 2,
                "tile list");
    K3_LAUNCH(k3::bs_quantize_latent(c->bs, w, T, d, bn, c->sharded ? n_local : nullptr, s), bn <= 16 ? 1 : 2,
              bn <= 16 ? "latent rows -> e2m1 terms" : "latent rows -> e4m3 terms");
    // with a second bank the block-scaled kernels take the first bank's
    // tiles [0, count[1]) and the second bank's kernels the rest: the split
    // is read on the device, no host synchronisation
    const int* count_a = c->bank2_begin ? tile_count + 1 : tile_count;
    // T = 1: the K experts' work items are split along K (both kernels)
    split_gu = c->bank2_begin ? 1 : k3::bs_split_gateup(c->bs, d, T);
    split_dn = c->bank2_begin ? 1 : k3::bs_split_down(c->bs, d, T);
    K3_LAUNCH(k3::bs_stream_gateup(c->bs, c->bw, tiles, count_a, w, T, d, bn, s, split_gu,
                                                c->sharded ? n_local : nullptr), split_gu > 1 ? 2 : 1,
              "gate/up");
    K3_LAUNCH(k3::bs_stream_down(c->bs, c->bw, tiles, count_a, w, T, d, bn, s, split_dn), 1, "down");
    if (c->bank2_begin && bn == k3::kBsDecodeRows)
      K3_LAUNCH(k3::bs_bank2_experts(c->bs, c->gu2_tiles, c->d2_tiles, c->bank2_begin, tiles, tile_count, w, T, d, s),
                3, "second bank (2-bit)");
    else if (c->bank2_begin)
      K3_LAUNCH(k3::umma_bank2_experts(c->umma, c->gu2_tiles, c->d2_tiles, c->bank2_begin, d.E - c->bank2_begin, bn,
                                       w, T, d, s),
                3, "second bank (2-bit)");
  } else {
    K3_LAUNCH(k3::launch_gateup_gemv(c->gu_tiles, w.lat, w.active, w.offsets, w.perm, max_active, d, w.h, s), 1,
              "gate/up");
    K3_LAUNCH(k3::launch_down_gemv(c->d_tiles, w.h, w.active, w.offsets, max_active, d, w.o, s), 1, "down");
  }
  // with a K-split down GEMM the combine reads o as the sum of its parts
  const float* o_src = split_dn > 1 ? k3::bs_down_parts(c->bs, d) : w.o;
  c->split_dn_last = split_dn;
  c->T_last = T;
  K3_LAUNCH(k3::launch_combine_rmsnorm(o_src, w.slot, wts, c->gamma, T, d.K, d, w.n, c->sal_on ? c->sal_tk : nullptr,
                                       n_local, c_out, s, split_dn, (size_t)T * d.K * d.L),
            1, c_out ? "partial combine" : "combine + RMSNorm");
  if (c->sal_on)
    K3_LAUNCH(k3::launch_saliency_accumulate(c->sal_tk, w.perm, w.offsets, w.active, T, d.E, c->sal_sum,
                                             c->sal_tokens, s),
              1, "REAP saliency");
  } else {
    // RMSNorm of the given combine: one "slot" per token (slot t = row t of
    // c_in) with weight 1, so c = c_in exactly
    K3_LAUNCH(k3::launch_combine_rmsnorm(c_in, c->iota, c->ones, c->gamma, T, 1, d, w.n, nullptr, nullptr, nullptr, s),
              1, "RMSNorm");
  }
  if (!tail) {
    c->launches_last = n;
    return K3MOE_OK;
  }
  if (c->Is && !shared_side)
    K3_LAUNCH(shared_launch(s, c->sh_part), shared_launches, "shared experts");
  if (shared_side && (e = cudaStreamWaitEvent(s, c->ev_join, 0)) != cudaSuccess) return cuda_fail(c, e, "join wait");
  k3::DenseOut o_up;
  o_up.out_bf16 = (uint16_t*)y;
  o_up.add_bf16 = c->Is ? c->sh_z : nullptr;
  if (path == 4 && T <= 64) {
    K3_LAUNCH(k3::umma_dense_small(c->umma, c->wu, d.H, d.L, w.n, T, o_up, nullptr, s),
              k3::umma_dense_small_launches(), "up_proj");
  } else if (path == 4) {
    K3_LAUNCH(k3::umma_dense(c->umma, c->wu, d.H, d.L, w.n, T, o_up, s), k3::umma_dense_launches(), "up_proj");
  } else {
    K3_LAUNCH(k3::launch_dense_gemv(c->wu, d.H, d.L, w.n, T, 0, nullptr, (uint16_t*)y, s), 1, "up_proj");
  }
#undef K3_LAUNCH
  c->launches_last = n;
  return K3MOE_OK;
}

int k3moe_forward(k3moe_ctx* c, const void* x, int T, void* y, int32_t* topk_idx, float* topk_w,
                  void* cuda_stream) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  if (!c->loaded) return fail(c, K3MOE_ESTATE, "forward before load_weights");
  if (T < 0 || T > c->cfg.max_tokens)
    return fail(c, K3MOE_EINVAL, "T=%d outside [0, max_tokens=%d]", T, c->cfg.max_tokens);
  if (T == 0) {
    c->launches_last = 0;
    return K3MOE_OK;
  }
  if (!x || !y || !topk_idx || !topk_w) return fail(c, K3MOE_EINVAL, "a device pointer is NULL");
  if (!aligned16(x) || !aligned16(y) || !aligned16(topk_idx) || !aligned16(topk_w))
    return fail(c, K3MOE_EINVAL, "x, y, topk_idx and topk_w must be 16-byte aligned");
  if (c->sharded)
    return fail(c, K3MOE_ESTATE, "an expert shard has no whole forward: use k3moe_forward_partial and k3moe_finish");
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  return forward_impl(c, x, T, y, topk_idx, topk_w, (cudaStream_t)cuda_stream);
}

int k3moe_forward_partial(k3moe_ctx* c, const void* x, int T, float* c_partial, int32_t* topk_idx, float* topk_w,
                          void* cuda_stream) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  if (!c->loaded) return fail(c, K3MOE_ESTATE, "forward before load_weights");
  if (T < 0 || T > c->cfg.max_tokens)
    return fail(c, K3MOE_EINVAL, "T=%d outside [0, max_tokens=%d]", T, c->cfg.max_tokens);
  if (T == 0) {
    c->launches_last = 0;
    return K3MOE_OK;
  }
  if (!x || !c_partial || !topk_idx || !topk_w) return fail(c, K3MOE_EINVAL, "a device pointer is NULL");
  if (!aligned16(x) || !aligned16(c_partial) || !aligned16(topk_idx) || !aligned16(topk_w))
    return fail(c, K3MOE_EINVAL, "x, c_partial, topk_idx and topk_w must be 16-byte aligned");
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  return forward_impl(c, x, T, nullptr, topk_idx, topk_w, (cudaStream_t)cuda_stream, c_partial, nullptr);
}

int k3moe_finish(k3moe_ctx* c, const void* x, const float* c_sum, int T, void* y, void* cuda_stream) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  if (!c->loaded) return fail(c, K3MOE_ESTATE, "finish before load_weights");
  if (T < 0 || T > c->cfg.max_tokens)
    return fail(c, K3MOE_EINVAL, "T=%d outside [0, max_tokens=%d]", T, c->cfg.max_tokens);
  if (T == 0) {
    c->launches_last = 0;
    return K3MOE_OK;
  }
  if (!c_sum || !y || (c->Is && !x)) return fail(c, K3MOE_EINVAL, "a device pointer is NULL");
  if (!aligned16(c_sum) || !aligned16(y) || (x && !aligned16(x)))
    return fail(c, K3MOE_EINVAL, "x, c_sum and y must be 16-byte aligned");
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  return forward_impl(c, x, T, y, nullptr, nullptr, (cudaStream_t)cuda_stream, nullptr, c_sum);
}

int k3moe_forward_host(k3moe_ctx* c, const void* x_host, int T, void* y_host, int32_t* idx_host, float* w_host,
                       void* cuda_stream) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  if (!c->loaded) return fail(c, K3MOE_ESTATE, "forward before load_weights");
  if (T < 0 || T > c->cfg.max_tokens)
    return fail(c, K3MOE_EINVAL, "T=%d outside [0, max_tokens=%d]", T, c->cfg.max_tokens);
  if (T == 0) return K3MOE_OK;
  if (!x_host) return fail(c, K3MOE_EINVAL, "x_host is NULL");
  if (c->sharded)
    return fail(c, K3MOE_ESTATE, "an expert shard has no whole forward: use k3moe_forward_partial and k3moe_finish");
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  cudaStream_t s = (cudaStream_t)cuda_stream;
  const size_t H = c->d.H, K = c->d.K;
  K3_CUDA(c, cudaMemcpyAsync(c->x_stage, x_host, (size_t)T * H * 2, cudaMemcpyHostToDevice, s), "copy x");
  int rc = forward_impl(c, c->x_stage, T, c->y_stage, c->idx_stage, c->w_stage, s);
  if (rc) return rc;
  if (y_host)
    K3_CUDA(c, cudaMemcpyAsync(y_host, c->y_stage, (size_t)T * H * 2, cudaMemcpyDeviceToHost, s), "copy y");
  if (idx_host)
    K3_CUDA(c, cudaMemcpyAsync(idx_host, c->idx_stage, (size_t)T * K * 4, cudaMemcpyDeviceToHost, s), "copy idx");
  if (w_host)
    K3_CUDA(c, cudaMemcpyAsync(w_host, c->w_stage, (size_t)T * K * 4, cudaMemcpyDeviceToHost, s), "copy w");
  K3_CUDA(c, cudaStreamSynchronize(s), "cudaStreamSynchronize");
  return K3MOE_OK;
}

int k3moe_status(k3moe_ctx* c) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  K3_CUDA(c, cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  unsigned st = 0;
  K3_CUDA(c, cudaMemcpy(&st, c->w.status, 4, cudaMemcpyDeviceToHost), "read status");
  if (st) {
    unsigned zero = 0;
    K3_CUDA(c, cudaMemcpy(c->w.status, &zero, 4, cudaMemcpyHostToDevice), "clear status");
    return fail(c, K3MOE_ETIMEOUT, "a device-side wait gave up (status word 0x%08x)", st);
  }
  return K3MOE_OK;
}

int k3moe_fetch(k3moe_ctx* c, int which, void* dst, size_t bytes) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  if (!dst && bytes) return fail(c, K3MOE_EINVAL, "dst is NULL");
  const void* src = nullptr;
  size_t cap = 0;
  switch (which) {
    case K3MOE_BUF_LOGITS: src = c->w.logits; cap = c->sz_logits; break;
    case K3MOE_BUF_LAT: src = c->w.lat; cap = c->sz_lat; break;
    case K3MOE_BUF_COUNTS: src = c->w.counts; cap = c->sz_counts; break;
    case K3MOE_BUF_OFFSETS: src = c->w.offsets; cap = c->sz_offsets; break;
    case K3MOE_BUF_PERM: src = c->w.perm; cap = c->sz_perm; break;
    case K3MOE_BUF_SLOT: src = c->w.slot; cap = c->sz_perm; break;
    case K3MOE_BUF_H: src = c->w.h; cap = c->sz_h; break;
    case K3MOE_BUF_O: src = c->w.o; cap = c->sz_o; break;
    case K3MOE_BUF_N: src = c->w.n; cap = c->sz_n; break;
    case K3MOE_BUF_ACTIVE: src = c->w.active; cap = c->sz_active; break;
    case K3MOE_BUF_SHARED_H: src = c->sh_h; cap = (size_t)c->cfg.max_tokens * c->Is * 2; break;
    case K3MOE_BUF_SHARED_Z: src = c->sh_z; cap = c->Is ? (size_t)c->cfg.max_tokens * c->d.H * 2 : 0; break;
    default: return fail(c, K3MOE_EINVAL, "unknown buffer %d", which);
  }
  if (bytes > cap) return fail(c, K3MOE_EINVAL, "buffer %d holds %zu bytes, %zu requested", which, cap, bytes);
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  K3_CUDA(c, cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  if (which == K3MOE_BUF_O && c->split_dn_last > 1) {
    // the down GEMM ran in K parts: o is their sum, in part order, as the
    // combine formed it
    const size_t plane = (size_t)c->T_last * c->d.K * c->d.L;
    std::vector<float> parts(plane * c->split_dn_last);
    K3_CUDA(c, cudaMemcpy(parts.data(), k3::bs_down_parts(c->bs, c->d), parts.size() * 4, cudaMemcpyDeviceToHost),
            "fetch");
    std::vector<float> o(plane);
    for (size_t i = 0; i < plane; ++i) {
      float v = parts[i];
      for (int pp = 1; pp < c->split_dn_last; ++pp) v += parts[pp * plane + i];
      o[i] = v;
    }
    memcpy(dst, o.data(), std::min(bytes, plane * 4));
    return K3MOE_OK;
  }
  K3_CUDA(c, cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost), "fetch");
  return K3MOE_OK;
}

int k3moe_query(const k3moe_ctx* c, int what, long long* value) {
  if (!c || !value) return fail(nullptr, K3MOE_EINVAL, "ctx or value is NULL");
  switch (what) {
    case K3MOE_Q_WORKSPACE_BYTES: *value = (long long)c->ws_bytes; return K3MOE_OK;
    case K3MOE_Q_WEIGHT_BYTES: *value = (long long)c->weight_bytes; return K3MOE_OK;
    case K3MOE_Q_LAUNCHES_LAST: *value = c->launches_last; return K3MOE_OK;
    case K3MOE_Q_PATH_LAST: *value = c->path_last; return K3MOE_OK;
    case K3MOE_Q_DEVICE: *value = c->device; return K3MOE_OK;
    default: return fail(nullptr, K3MOE_EINVAL, "unknown query %d", what);
  }
}

int k3moe_test_withhold_copies(k3moe_ctx* c) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  c->test_withhold = true;
  return K3MOE_OK;
}

int k3moe_check_guards(k3moe_ctx* c) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  K3_CUDA(c, cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  std::vector<uint8_t> band(kGuardBytes);
  for (size_t i = 0; i < c->guards.size(); ++i) {
    K3_CUDA(c, cudaMemcpy(band.data(), c->guards[i], kGuardBytes, cudaMemcpyDeviceToHost), "read guard band");
    for (size_t j = 0; j < kGuardBytes; ++j)
      if (band[j] != (uint8_t)kGuardByte)
        return fail(c, K3MOE_ESTATE, "guard band after workspace buffer %zu overwritten at byte %zu", i, j);
  }
  return K3MOE_OK;
}

int k3moe_saliency(k3moe_ctx* c, int enable) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  c->sal_on = enable != 0;
  return K3MOE_OK;
}

int k3moe_saliency_read(k3moe_ctx* c, double* sums, int n_experts, unsigned long long* tokens) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  if (n_experts != c->d.E) return fail(c, K3MOE_EINVAL, "n_experts %d != the context's %d", n_experts, c->d.E);
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  K3_CUDA(c, cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  if (sums) K3_CUDA(c, cudaMemcpy(sums, c->sal_sum, (size_t)c->d.E * 8, cudaMemcpyDeviceToHost), "read sums");
  if (tokens) K3_CUDA(c, cudaMemcpy(tokens, c->sal_tokens, 8, cudaMemcpyDeviceToHost), "read token count");
  return K3MOE_OK;
}

int k3moe_saliency_reset(k3moe_ctx* c) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  K3_CUDA(c, cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  K3_CUDA(c, cudaMemset(c->sal_sum, 0, (size_t)c->d.E * 8 + 8), "clear saliency");
  return K3MOE_OK;
}

int k3moe_profile(k3moe_ctx* c, int enable) {
  if (!c) return fail(nullptr, K3MOE_EINVAL, "ctx is NULL");
  K3_CUDA(c, cudaSetDevice(c->device), "cudaSetDevice");
  if (enable && !c->prof_ev[0])
    for (cudaEvent_t& ev : c->prof_ev) K3_CUDA(c, cudaEventCreate(&ev), "cudaEventCreate");
  c->prof = enable != 0;
  c->prof_n = 0;
  return K3MOE_OK;
}

int k3moe_profile_read(k3moe_ctx* c, float* ms, int max_entries, int* count) {
  if (!c || !count) return fail(c, K3MOE_EINVAL, "ctx or count is NULL");
  *count = c->prof_n;
  for (int i = 0; i < c->prof_n && i < max_entries && ms; ++i) {
    K3_CUDA(c, cudaEventSynchronize(c->prof_ev[i + 1]), "cudaEventSynchronize");
    K3_CUDA(c, cudaEventElapsedTime(&ms[i], c->prof_ev[i], c->prof_ev[i + 1]), "cudaEventElapsedTime");
  }
  return K3MOE_OK;
}

const char* k3moe_profile_name(const k3moe_ctx* c, int i) {
  if (!c || i < 0 || i >= c->prof_n) return "";
  return c->prof_name[i];
}

int k3moe_mxfp4_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols, void* out, int kind,
                        void* cuda_stream) {
  if (!packed || !scale || !out) return fail(nullptr, K3MOE_EINVAL, "a pointer is NULL");
  if (rows < 0 || cols < 0 || cols % 64) return fail(nullptr, K3MOE_EINVAL, "need rows >= 0 and cols %% 64 == 0");
  if (kind != 0 && kind != 1) return fail(nullptr, K3MOE_EINVAL, "kind must be 0 (bf16) or 1 (fp32)");
  if (!aligned16(out)) return fail(nullptr, K3MOE_EINVAL, "out must be 16-byte aligned");
  cudaError_t e = k3::launch_dequant(packed, scale, rows, cols, out, kind, (cudaStream_t)cuda_stream);
  if (e != cudaSuccess) return fail(nullptr, K3MOE_ECUDA, "dequant launch: %s", cudaGetErrorString(e));
  return K3MOE_OK;
}

int k3moe_route(const void* x, int T, const void* router_w, const float* bias, int E, int H, int K, int norm_topk,
                float routed_scaling, float* logits, int32_t* topk_idx, float* topk_w, void* cuda_stream) {
  if (T < 0) return fail(nullptr, K3MOE_EINVAL, "T < 0");
  if (T == 0) return K3MOE_OK;
  if (!x || !router_w || !bias || !logits || !topk_idx || !topk_w)
    return fail(nullptr, K3MOE_EINVAL, "a pointer is NULL");
  if (H <= 0 || H % 128 || K < 1 || K > 32 || K > E || E > 2048)
    return fail(nullptr, K3MOE_EINVAL, "need H %% 128 == 0, 1 <= K <= 32, K <= E <= 2048");
  if (!aligned16(x) || !aligned16(router_w)) return fail(nullptr, K3MOE_EINVAL, "x and router_w must be 16-byte aligned");
  cudaStream_t s = (cudaStream_t)cuda_stream;
  cudaError_t e = k3::launch_dense_gemv((const uint16_t*)router_w, E, H, (const uint16_t*)x, T, E, logits, nullptr, s);
  if (e == cudaSuccess) e = k3::launch_topk(logits, T, E, E, bias, K, norm_topk, routed_scaling, topk_idx, topk_w, s);
  if (e != cudaSuccess) return fail(nullptr, K3MOE_ECUDA, "route launch: %s", cudaGetErrorString(e));
  return K3MOE_OK;
}

}  // extern "C"
