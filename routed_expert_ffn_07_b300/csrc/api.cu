// Host side of the C ABI declared in include/moe.h: argument validation, the workspace, the
// order of launches per layer, and the whole-stack CUDA graph.
//
// The stack of 48 MoE layers runs as one recorded CUDA graph, so no synchronous driver call
// sits between layers ('Strata はなぜ少ない VRAM でも速いのか' (modeldock.net), section
// '1 トークン、三者の分担').
#include <cstdio>
#include <cstring>
#include <map>
#include <vector>

#include "../../include/moe.h"
#include "common.cuh"

namespace moe {
cudaError_t launch_route(const RouteArgs& a, int nblocks_dispatch, cudaStream_t st);
cudaError_t route_kernels_init();
cudaError_t gemv_kernels_init(int num_sms);
cudaError_t launch_experts_gemv(const ExpertArgs& a, int wfmt, cudaStream_t st, cudaEvent_t mid, cudaEvent_t mid2);
size_t gemv_smem_gu(int wfmt, int T, int d, int E, int K);
size_t gemv_smem_dn(int T, int K, int E);
cudaError_t gemm_kernels_init(int num_sms);
cudaError_t fused_kernels_init(int num_sms);
cudaError_t launch_bounded_wait_selftest(unsigned long long* counter, long long budget, unsigned* result,
                                         cudaStream_t st);
bool fused_shape_ok(int T, int d, int f, int E, int K);
cudaError_t launch_decode_fused(const RouteArgs& r, const ExpertArgs& x, const FusedExtra& fx, cudaStream_t st);
size_t fused_layout_bytes(int n_exp, int d, int f);
cudaError_t fused_repack(const void* gu_q, const void* gu_s, const void* dn_q, const void* dn_s, int n_exp, int d,
                         int f, void* out, cudaStream_t st);
size_t gemm_workspace_bytes(int max_tokens, int d, int f, int E, int K);
bool gemm_shape_ok(int d, int f);
void* gemm_maps_new();
void gemm_maps_free(void* p);
cudaError_t gemm_build_maps(void* maps, int E, int d, int f, int has_shared, const void* gu_q, const void* gu_s,
                            const void* dn_q, const void* dn_s, const void* sh_gu_q, const void* sh_gu_s,
                            const void* sh_dn_q, const void* sh_dn_s);
cudaError_t launch_experts_gemm(const ExpertArgs& a, const void* maps, const void* act_maps, void* gemm_ws,
                                cudaStream_t st, cudaEvent_t mid, cudaEvent_t mid2);
cudaError_t gemm_build_act_maps(void* ws, int T, int d, int f, int E, int K, void* out);
size_t gemm_act_maps_bytes();
constexpr int kDispatchBlockHost = 256;
constexpr int kTimingEvents = 5;  // before route, after route, after stage A, after stage B, end
constexpr int kFusedMaxTokensHost = 8;    // the one-launch decode layer's limit
constexpr int kFusedDefaultTokens = 4;    // decode and 1 + 3 verify
}  // namespace moe

using namespace moe;

struct LayerW {
  moe_layer_weights w;
  bool set = false;
  void* maps = nullptr;  // TMA descriptors of the layer's planes (tensor-core path only)
  void* dnb = nullptr;   // decode-layout copy of the experts (one-launch decode path only)
};

struct moe_ctx {
  moe_config cfg;
  int device = 0;
  int num_sms = 148;
  std::vector<LayerW> layers;
  char* slab = nullptr;
  size_t slab_bytes = 0;
  // workspace views
  float* logits;
  int32_t* idx;
  float* w;
  int32_t* counts;
  int32_t* offs;
  int32_t* perm;
  int32_t* active;
  int32_t* n_active;
  int32_t* stats;
  int4* slots;
  unsigned* ticket;
  unsigned* status;
  int32_t* blockhist;
  float* h;
  void* gemm_ws;
  void* xnorm;
  void* stack_x;
  void* host_x;
  void* host_y;
  int nblocks_max;
  cudaStream_t cap_stream = nullptr;
  std::map<int, cudaGraphExec_t> graphs;
  bool gemm_ok = false;          // tensor-core path available for this config
  void* act_maps = nullptr;      // TMA descriptors of the workspace activation buffers
  int gemv_max_tokens = 4;       // T <= this runs the GEMV experts (when the grouped GEMM is available)
  int fused_max_tokens = 0;      // T <= this runs the one-launch decode layer (0: off)
  unsigned long long* grid_bar = nullptr;  // grid-barrier counter of the one-launch decode layer
  bool fused_capable = false;    // the one-launch decode layer serves this config (T = 1 at least)
  float* part = nullptr;         // its per-CTA partial outputs [#SM][min(max_tokens, 8)][d]
  // stage timing
  std::vector<cudaEvent_t> tev;
  int t_next = 0;
  int t_used = 0;
};

static size_t act_size(int act) { return act == MOE_ACT_BF16 ? 2 : 4; }

// Largest T <= want (and <= max_tokens) that the one-launch decode layer serves for this config.
static int fused_limit(const moe_config& c, int want) {
  int best = 0;
  if (c.wfmt == MOE_W_INT4_G32)
    for (int t = 1; t <= want && t <= c.max_tokens; ++t)
      if (fused_shape_ok(t, c.d, c.f, c.n_experts, c.top_k)) best = t;
  return best;
}
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static size_t up256(size_t n) { return (n + 255) & ~size_t(255); }

static thread_local int g_last_cuda_error = 0;

#define CUDA_TRY(expr)                               \
  do {                                               \
    cudaError_t e_ = (expr);                         \
    if (e_ != cudaSuccess) {                         \
      g_last_cuda_error = (int)e_;                   \
      return MOE_ERR_CUDA;                           \
    }                                                \
  } while (0)

extern "C" {

int moe_version(void) { return 1; }

int moe_last_cuda_error(void) { return g_last_cuda_error; }

int moe_peek_cuda_error(void) { return (int)cudaPeekAtLastError(); }

const char* moe_cuda_error_string(int code) { return cudaGetErrorString(static_cast<cudaError_t>(code)); }

const char* moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or format";
    case MOE_ERR_OOM: return "workspace allocation failed";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_NOT_SET: return "layer weights not set";
    case MOE_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

moe_status moe_create(const moe_config* cfg, moe_handle* out) {
  if (!cfg || !out) return MOE_ERR_INVALID_ARG;
  const moe_config c = *cfg;
  if (c.d <= 0 || c.f <= 0 || c.n_experts <= 0 || c.n_layers <= 0 || c.max_tokens <= 0) return MOE_ERR_INVALID_ARG;
  if (c.top_k < 1 || c.top_k > c.n_experts || c.top_k > kMaxK) return MOE_ERR_INVALID_ARG;
  if (c.n_experts > kMaxE) return MOE_ERR_UNSUPPORTED;
  if (c.act != MOE_ACT_BF16 && c.act != MOE_ACT_F32) return MOE_ERR_INVALID_ARG;
  if (c.wfmt != MOE_W_INT4_G32 && c.wfmt != MOE_W_F32) return MOE_ERR_INVALID_ARG;
  if (c.has_shared != 0 && c.has_shared != 1) return MOE_ERR_INVALID_ARG;
  if (c.prenorm != 0 && c.prenorm != 1) return MOE_ERR_INVALID_ARG;
  if (c.prenorm && !(c.norm_eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (c.d % 4 || c.f % 4) return MOE_ERR_UNSUPPORTED;
  if (c.wfmt == MOE_W_INT4_G32) {
    if (c.d % 128 || c.f % 128) return MOE_ERR_UNSUPPORTED;
    if (c.d > 4096 || c.f > 1024) return MOE_ERR_UNSUPPORTED;  // GEMV lane mapping limits
    if (c.max_tokens > kSmallT && !gemm_shape_ok(c.d, c.f)) return MOE_ERR_UNSUPPORTED;  // tensor-core path needed
  } else {
    if (c.max_tokens > kSmallT) return MOE_ERR_UNSUPPORTED;   // fp32 experts: GEMV path only
  }
  if (c.max_tokens > 65536) return MOE_ERR_UNSUPPORTED;

  moe_ctx* h = new (std::nothrow) moe_ctx();
  if (!h) return MOE_ERR_OOM;
  h->cfg = c;
  h->layers.resize(c.n_layers);
  if (cudaGetDevice(&h->device) != cudaSuccess) {
    delete h;
    return MOE_ERR_CUDA;
  }
  cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  h->gemm_ok = c.wfmt == MOE_W_INT4_G32 && gemm_shape_ok(c.d, c.f);
  if (!h->gemm_ok) h->gemv_max_tokens = kSmallT;
  if (route_kernels_init() != cudaSuccess || gemv_kernels_init(h->num_sms) != cudaSuccess ||
      (h->gemm_ok && gemm_kernels_init(h->num_sms) != cudaSuccess) ||
      (c.wfmt == MOE_W_INT4_G32 && fused_kernels_init(h->num_sms) != cudaSuccess)) {
    delete h;
    return MOE_ERR_CUDA;
  }
  h->fused_max_tokens = fused_limit(c, kFusedDefaultTokens);
  h->fused_capable = fused_limit(c, 1) == 1;

  const int T = c.max_tokens, E = c.n_experts, K = c.top_k, d = c.d, f = c.f;
  const size_t as = act_size(c.act);
  h->nblocks_max = (T * K + kDispatchBlockHost - 1) / kDispatchBlockHost;
  size_t sz[24];
  int n = 0;
  sz[n++] = up256((size_t)T * E * 4);                 // logits
  sz[n++] = up256((size_t)T * K * 4);                 // idx
  sz[n++] = up256((size_t)T * K * 4);                 // w
  sz[n++] = up256((size_t)E * 4);                     // counts
  sz[n++] = up256((size_t)(E + 1) * 4);               // offs
  sz[n++] = up256((size_t)T * K * 4);                 // perm
  sz[n++] = up256((size_t)E * 4);                     // active
  sz[n++] = up256(4);                                 // n_active
  sz[n++] = up256((size_t)c.n_layers * 4);            // stats
  sz[n++] = up256((size_t)E * 16);                    // slot table
  sz[n++] = up256(4);                                 // ticket
  sz[n++] = up256(4);                                 // status
  sz[n++] = up256(8);                                 // grid barrier
  sz[n++] = up256((size_t)h->nblocks_max * E * 4);    // blockhist
  const int TS = T < kSmallT ? T : kSmallT;
  sz[n++] = up256((size_t)(TS * K + TS) * f * 4);     // h (GEMV path)
  sz[n++] = h->gemm_ok ? up256(gemm_workspace_bytes(T, d, f, E, K)) : 0;
  sz[n++] = up256((size_t)T * d * as);                // xnorm
  sz[n++] = up256((size_t)T * d * as);                // stack x
  sz[n++] = up256((size_t)T * d * as);                // host x
  sz[n++] = up256((size_t)T * d * as);                // host y
  const int TF = T < kFusedMaxTokensHost ? T : kFusedMaxTokensHost;
  sz[n++] = h->fused_capable ? up256((size_t)h->num_sms * TF * d * 4) : 0;  // one-launch partials
  size_t total = 0;
  for (int i = 0; i < n; ++i) total += sz[i];
  if (cudaMalloc(&h->slab, total) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_OOM;
  }
  h->slab_bytes = total;
  char* p = h->slab;
  int i = 0;
  h->logits = reinterpret_cast<float*>(p); p += sz[i++];
  h->idx = reinterpret_cast<int32_t*>(p); p += sz[i++];
  h->w = reinterpret_cast<float*>(p); p += sz[i++];
  h->counts = reinterpret_cast<int32_t*>(p); p += sz[i++];
  h->offs = reinterpret_cast<int32_t*>(p); p += sz[i++];
  h->perm = reinterpret_cast<int32_t*>(p); p += sz[i++];
  h->active = reinterpret_cast<int32_t*>(p); p += sz[i++];
  h->n_active = reinterpret_cast<int32_t*>(p); p += sz[i++];
  h->stats = reinterpret_cast<int32_t*>(p); p += sz[i++];
  h->slots = reinterpret_cast<int4*>(p); p += sz[i++];
  h->ticket = reinterpret_cast<unsigned*>(p); p += sz[i++];
  h->status = reinterpret_cast<unsigned*>(p); p += sz[i++];
  h->grid_bar = reinterpret_cast<unsigned long long*>(p); p += sz[i++];
  h->blockhist = reinterpret_cast<int32_t*>(p); p += sz[i++];
  h->h = reinterpret_cast<float*>(p); p += sz[i++];
  h->gemm_ws = sz[i] ? p : nullptr; p += sz[i++];
  h->xnorm = p; p += sz[i++];
  h->stack_x = p; p += sz[i++];
  h->host_x = p; p += sz[i++];
  h->host_y = p; p += sz[i++];
  h->part = sz[i] ? reinterpret_cast<float*>(p) : nullptr; p += sz[i++];
  if (cudaMemset(h->slab, 0, total) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(h->slab);
    delete h;
    return MOE_ERR_CUDA;
  }
  if (h->gemm_ok) {
    h->act_maps = gemm_maps_new();
    if (!h->act_maps || gemm_build_act_maps(h->gemm_ws, T, d, f, E, K, h->act_maps) != cudaSuccess) {
      if (h->act_maps) gemm_maps_free(h->act_maps);
      cudaFree(h->slab);
      delete h;
      return MOE_ERR_CUDA;
    }
  }
  *out = h;
  return MOE_OK;
}

moe_status moe_set_layer(moe_handle h, int layer, const moe_layer_weights* w) {
  if (!h || !w || layer < 0 || layer >= h->cfg.n_layers) return MOE_ERR_INVALID_ARG;
  const bool q4 = h->cfg.wfmt == MOE_W_INT4_G32;
  const void* need[] = {w->router_w, w->gu_q, w->dn_q};
  for (const void* p : need)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (q4 && (!w->gu_s || !w->dn_s || !aligned16(w->gu_s) || !aligned16(w->dn_s))) return MOE_ERR_INVALID_ARG;
  if (w->router_b && !aligned16(w->router_b)) return MOE_ERR_INVALID_ARG;
  if (h->cfg.has_shared) {
    if (!w->sh_gu_q || !w->sh_dn_q || !aligned16(w->sh_gu_q) || !aligned16(w->sh_dn_q)) return MOE_ERR_INVALID_ARG;
    if (q4 && (!w->sh_gu_s || !w->sh_dn_s || !aligned16(w->sh_gu_s) || !aligned16(w->sh_dn_s)))
      return MOE_ERR_INVALID_ARG;
  }
  LayerW& L = h->layers[layer];
  if (h->gemm_ok) {
    if (!L.maps) L.maps = gemm_maps_new();
    if (!L.maps) return MOE_ERR_OOM;
    if (gemm_build_maps(L.maps, h->cfg.n_experts, h->cfg.d, h->cfg.f, h->cfg.has_shared, w->gu_q, w->gu_s, w->dn_q,
                        w->dn_s, w->sh_gu_q, w->sh_gu_s, w->sh_dn_q, w->sh_dn_s) != cudaSuccess) {
      L.set = false;
      return MOE_ERR_INVALID_ARG;
    }
  }
  if (h->fused_capable) {
    // the one-launch decode layer reads the experts in its own fragment order: copy them once, here
    const moe_config& c = h->cfg;
    const size_t rb = (fused_layout_bytes(c.n_experts, c.d, c.f) + 255) & ~size_t(255);
    const size_t sb = c.has_shared ? fused_layout_bytes(1, c.d, c.f) : 0;
    if (!L.dnb && cudaMalloc(&L.dnb, rb + sb) != cudaSuccess) {
      cudaGetLastError();
      L.dnb = nullptr;
      L.set = false;
      return MOE_ERR_OOM;
    }
    char* base = static_cast<char*>(L.dnb);
    // the weights may have been written on any stream: wait for the device before reading them
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = fused_repack(w->gu_q, w->gu_s, w->dn_q, w->dn_s, c.n_experts, c.d, c.f, base, nullptr);
    if (e == cudaSuccess && c.has_shared)
      e = fused_repack(w->sh_gu_q, w->sh_gu_s, w->sh_dn_q, w->sh_dn_s, 1, c.d, c.f, base + rb, nullptr);
    if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
    if (e != cudaSuccess) {
      g_last_cuda_error = (int)e;
      L.set = false;
      return MOE_ERR_CUDA;
    }
  }
  L.w = *w;
  L.set = true;
  return MOE_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ internal launch sequences
static RouteArgs make_route_args(moe_ctx* h, int layer, const void* x, int T, bool prenorm, int32_t* stat) {
  const moe_config& c = h->cfg;
  const moe_layer_weights& w = h->layers[layer].w;
  RouteArgs a;
  a.x = x;
  a.act = c.act;
  a.T = T;
  a.d = c.d;
  a.E = c.n_experts;
  a.K = c.top_k;
  a.Wr = w.router_w;
  a.bias = w.router_b;
  a.prenorm = prenorm ? 1 : 0;
  a.eps = c.norm_eps;
  a.xnorm = h->xnorm;
  a.logits = h->logits;
  a.idx = h->idx;
  a.w = h->w;
  a.counts = h->counts;
  a.offs = h->offs;
  a.perm = h->perm;
  a.active = h->active;
  a.n_active = h->n_active;
  a.stat = stat;
  a.slots = h->slots;
  a.blockhist = h->blockhist;
  a.ticket = h->ticket;
  a.status = h->status;
  return a;
}

static ExpertArgs make_expert_args(moe_ctx* h, int layer, const void* x, int T, void* y, const void* resid) {
  const moe_config& c = h->cfg;
  const moe_layer_weights& w = h->layers[layer].w;
  ExpertArgs a;
  a.T = T;
  a.d = c.d;
  a.f = c.f;
  a.E = c.n_experts;
  a.K = c.top_k;
  a.act = c.act;
  a.has_shared = c.has_shared;
  a.max_tokens = c.max_tokens;
  a.x = x;
  a.gu_q = w.gu_q;
  a.gu_s = static_cast<const __half*>(w.gu_s);
  a.dn_q = w.dn_q;
  a.dn_s = static_cast<const __half*>(w.dn_s);
  a.sh_gu_q = w.sh_gu_q;
  a.sh_gu_s = static_cast<const __half*>(w.sh_gu_s);
  a.sh_dn_q = w.sh_dn_q;
  a.sh_dn_s = static_cast<const __half*>(w.sh_dn_s);
  a.offs = h->offs;
  a.perm = h->perm;
  a.active = h->active;
  a.n_active = h->n_active;
  a.slots = h->slots;
  a.topk_w = h->w;
  a.h = h->h;
  a.y = y;
  a.resid = resid;
  a.status = h->status;
  return a;
}

// One layer: route (optionally on RMSNorm(x)), experts, combine (+ residual).
static cudaError_t enqueue_layer(moe_ctx* h, int layer, const void* x, int T, void* y, const void* resid,
                                 bool prenorm, cudaStream_t st) {
  cudaEvent_t* ev = nullptr;
  if (!h->tev.empty() && h->t_next + kTimingEvents <= (int)h->tev.size()) {
    ev = &h->tev[h->t_next];
    h->t_next += kTimingEvents;
    if (h->t_next / kTimingEvents > h->t_used) h->t_used = h->t_next / kTimingEvents;
  }
  cudaError_t e;
  if (ev && (e = record_timing_event(ev[0], st)) != cudaSuccess) return e;
  RouteArgs ra = make_route_args(h, layer, x, T, prenorm, h->stats + layer);
  if (T <= h->fused_max_tokens && h->layers[layer].dnb) {
    // one launch for the whole layer; its stages are not separated (all of it counts as "route")
    ExpertArgs ea = make_expert_args(h, layer, x, T, y, resid);
    const moe_config& c = h->cfg;
    char* base = static_cast<char*>(h->layers[layer].dnb);
    const size_t rb = (fused_layout_bytes(c.n_experts, c.d, c.f) + 255) & ~size_t(255);
    FusedExtra fx;
    fx.dl = base;
    fx.sh_dl = c.has_shared ? base + rb : nullptr;
    fx.part = h->part;
    fx.grid_bar = h->grid_bar;
    e = launch_decode_fused(ra, ea, fx, st);
    if (e != cudaSuccess) return e;
    for (int k = 1; ev && k < kTimingEvents; ++k)
      if ((e = record_timing_event(ev[k], st)) != cudaSuccess) return e;
    return cudaSuccess;
  }
  const int nb = (T * h->cfg.top_k + kDispatchBlockHost - 1) / kDispatchBlockHost;
  e = launch_route(ra, nb, st);
  if (e != cudaSuccess) return e;
  if (ev && (e = record_timing_event(ev[1], st)) != cudaSuccess) return e;
  const void* xin = prenorm ? h->xnorm : x;
  ExpertArgs ea = make_expert_args(h, layer, xin, T, y, resid);
  if (T <= h->gemv_max_tokens || !h->gemm_ok)
    e = launch_experts_gemv(ea, h->cfg.wfmt, st, ev ? ev[2] : nullptr, ev ? ev[3] : nullptr);
  else
    e = launch_experts_gemm(ea, h->layers[layer].maps, h->act_maps, h->gemm_ws, st, ev ? ev[2] : nullptr,
                            ev ? ev[3] : nullptr);
  if (e != cudaSuccess) return e;
  if (ev && (e = record_timing_event(ev[4], st)) != cudaSuccess) return e;
  return cudaSuccess;
}

static moe_status check_common(moe_handle h, int layer, const void* x, int T) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->cfg.n_layers) return MOE_ERR_INVALID_ARG;
  if (!x || !aligned16(x)) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!h->layers[layer].set) return MOE_ERR_NOT_SET;
  return MOE_OK;
}

extern "C" {

moe_status moe_route(moe_handle h, int layer, const void* x, int T, int32_t* topk_idx, float* topk_w,
                     int32_t* expert_offs, int32_t* perm, void* stream) {
  moe_status s = check_common(h, layer, x, T);
  if (s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaGetLastError());
  RouteArgs ra = make_route_args(h, layer, x, T, false, h->stats + layer);
  const int K = h->cfg.top_k, E = h->cfg.n_experts;
  const int nb = (T * K + kDispatchBlockHost - 1) / kDispatchBlockHost;
  CUDA_TRY(launch_route(ra, nb, st));
  if (topk_idx) CUDA_TRY(cudaMemcpyAsync(topk_idx, h->idx, (size_t)T * K * 4, cudaMemcpyDeviceToDevice, st));
  if (topk_w) CUDA_TRY(cudaMemcpyAsync(topk_w, h->w, (size_t)T * K * 4, cudaMemcpyDeviceToDevice, st));
  if (expert_offs) CUDA_TRY(cudaMemcpyAsync(expert_offs, h->offs, (size_t)(E + 1) * 4, cudaMemcpyDeviceToDevice, st));
  if (perm) CUDA_TRY(cudaMemcpyAsync(perm, h->perm, (size_t)T * K * 4, cudaMemcpyDeviceToDevice, st));
  return MOE_OK;
}

moe_status moe_layer_forward(moe_handle h, int layer, const void* x, int T, void* y, void* stream) {
  moe_status s = check_common(h, layer, x, T);
  if (s != MOE_OK) return s;
  if (!y || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  const size_t bytes = (size_t)T * h->cfg.d * act_size(h->cfg.act);
  const char* xb = static_cast<const char*>(x);
  const char* yb = static_cast<const char*>(y);
  if (xb < yb + bytes && yb < xb + bytes) return MOE_ERR_INVALID_ARG;  // y must not overlap x
  CUDA_TRY(cudaGetLastError());
  CUDA_TRY(enqueue_layer(h, layer, x, T, y, nullptr, false, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_layer_forward_host(moe_handle h, int layer, const void* x_host, int T, void* y_host, void* stream) {
  if (!h || !x_host || !y_host) return MOE_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->cfg.n_layers || T < 1 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!h->layers[layer].set) return MOE_ERR_NOT_SET;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)T * h->cfg.d * act_size(h->cfg.act);
  CUDA_TRY(cudaGetLastError());
  CUDA_TRY(cudaMemcpyAsync(h->host_x, x_host, bytes, cudaMemcpyHostToDevice, st));
  CUDA_TRY(enqueue_layer(h, layer, h->host_x, T, h->host_y, nullptr, false, st));
  CUDA_TRY(cudaMemcpyAsync(y_host, h->host_y, bytes, cudaMemcpyDeviceToHost, st));
  CUDA_TRY(cudaStreamSynchronize(st));
  return MOE_OK;
}

}  // extern "C"

static cudaError_t enqueue_stack(moe_ctx* h, int T, void* trace, cudaStream_t st) {
  const moe_config& c = h->cfg;
  const size_t bytes = (size_t)T * c.d * act_size(c.act);
  for (int l = 0; l < c.n_layers; ++l) {
    if (trace) {
      char* tl = static_cast<char*>(trace) + (size_t)l * 2 * bytes;
      cudaError_t e = cudaMemcpyAsync(tl, h->stack_x, bytes, cudaMemcpyDeviceToDevice, st);
      if (e != cudaSuccess) return e;
    }
    cudaError_t e = enqueue_layer(h, l, h->stack_x, T, h->stack_x, h->stack_x, c.prenorm != 0, st);
    if (e != cudaSuccess) return e;
    (void)0;
    if (trace) {
      // the normalised input of layer l (its expert input) was produced by the route step
      char* tl = static_cast<char*>(trace) + (size_t)l * 2 * bytes + bytes;
      const void* src = c.prenorm ? h->xnorm : nullptr;
      if (src) {
        e = cudaMemcpyAsync(tl, src, bytes, cudaMemcpyDeviceToDevice, st);
      } else {
        e = cudaMemcpyAsync(tl, static_cast<char*>(trace) + (size_t)l * 2 * bytes, bytes, cudaMemcpyDeviceToDevice, st);
      }
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

extern "C" {

moe_status moe_stack_forward(moe_handle h, void* x_inout, int T, void* trace, void* stream) {
  if (!h || !x_inout || !aligned16(x_inout)) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (trace && !aligned16(trace)) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < h->cfg.n_layers; ++l)
    if (!h->layers[l].set) return MOE_ERR_NOT_SET;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)T * h->cfg.d * act_size(h->cfg.act);
  CUDA_TRY(cudaGetLastError());
  CUDA_TRY(cudaMemcpyAsync(h->stack_x, x_inout, bytes, cudaMemcpyDeviceToDevice, st));
  if (trace) {
    CUDA_TRY(enqueue_stack(h, T, trace, st));
  } else {
    auto it = h->graphs.find(T);
    if (it == h->graphs.end()) {
      if (!h->cap_stream) CUDA_TRY(cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking));
      cudaGraph_t g = nullptr;
      CUDA_TRY(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
      cudaError_t e = enqueue_stack(h, T, nullptr, h->cap_stream);
      cudaError_t e2 = cudaStreamEndCapture(h->cap_stream, &g);
      if (e != cudaSuccess || e2 != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return MOE_ERR_CUDA;
      }
      cudaGraphExec_t ex = nullptr;
      e = cudaGraphInstantiate(&ex, g, 0);
      cudaGraphDestroy(g);
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      it = h->graphs.emplace(T, ex).first;
    }
    CUDA_TRY(cudaGraphLaunch(it->second, st));
  }
  CUDA_TRY(cudaMemcpyAsync(x_inout, h->stack_x, bytes, cudaMemcpyDeviceToDevice, st));
  return MOE_OK;
}

moe_status moe_get_active_counts(moe_handle h, int32_t* counts_host, void* stream) {
  if (!h || !counts_host) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaMemcpyAsync(counts_host, h->stats, (size_t)h->cfg.n_layers * 4, cudaMemcpyDeviceToHost, st));
  CUDA_TRY(cudaStreamSynchronize(st));
  return MOE_OK;
}

moe_status moe_get_device_status(moe_handle h, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  unsigned v = 0;
  CUDA_TRY(cudaMemcpy(&v, h->status, 4, cudaMemcpyDeviceToHost));
  if (v) CUDA_TRY(cudaMemset(h->status, 0, 4));
  if (v & kStatusTimeout) {
    // a grid barrier that gave up may hold a partial count: start the next launch from zero
    CUDA_TRY(cudaMemset(h->grid_bar, 0, 8));
    return MOE_ERR_TIMEOUT;
  }
  if (v) return MOE_ERR_DEVICE;
  return MOE_OK;
}

moe_status moe_selftest_bounded_waits(long long budget_cycles, void* stream) {
  if (budget_cycles < 1000 || budget_cycles > 2000000000ll) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned long long* counter = nullptr;
  unsigned* res = nullptr;
  CUDA_TRY(cudaMalloc(&counter, 8));
  cudaError_t e = cudaMalloc(&res, 8);
  if (e != cudaSuccess) {
    cudaFree(counter);
    g_last_cuda_error = (int)e;
    return MOE_ERR_CUDA;
  }
  unsigned hres[2] = {0, 0};
  e = cudaMemsetAsync(counter, 0, 8, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(res, 0, 8, st);
  if (e == cudaSuccess) e = launch_bounded_wait_selftest(counter, budget_cycles, res, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(hres, res, 8, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(counter);
  cudaFree(res);
  if (e != cudaSuccess) {
    g_last_cuda_error = (int)e;
    return MOE_ERR_CUDA;
  }
  if (hres[0] & 4u) return MOE_ERR_DEVICE;            // a wait that cannot succeed returned success
  if ((hres[0] & 3u) == 3u && (hres[1] & kStatusTimeout)) return MOE_ERR_TIMEOUT;
  return MOE_ERR_DEVICE;
}

int moe_set_option(moe_handle h, int option, int value) {
  if (!h) return -(int)MOE_ERR_INVALID_ARG;
  if (option == MOE_OPT_GEMV_MAX_TOKENS) {
    if (value < 0 || value > kSmallT) return -(int)MOE_ERR_INVALID_ARG;
    h->gemv_max_tokens = h->gemm_ok ? value : kSmallT;
    for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);  // captured graphs used the old path
    h->graphs.clear();
    return h->gemv_max_tokens;
  }
  if (option == MOE_OPT_FUSED_MAX_TOKENS) {
    if (value < 0 || value > kFusedMaxTokensHost) return -(int)MOE_ERR_INVALID_ARG;
    h->fused_max_tokens = fused_limit(h->cfg, value);
    for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
    h->graphs.clear();
    return h->fused_max_tokens;
  }
  return -(int)MOE_ERR_INVALID_ARG;
}

moe_status moe_timing_enable(moe_handle h, int n_records) {
  if (!h || n_records < 0 || n_records > (1 << 20)) return MOE_ERR_INVALID_ARG;
  for (cudaEvent_t e : h->tev) cudaEventDestroy(e);
  h->tev.clear();
  h->t_next = h->t_used = 0;
  cudaGetLastError();  // destroying an event that a live graph still records is reported here, not later
  for (int i = 0; i < kTimingEvents * n_records; ++i) {
    cudaEvent_t e;
    CUDA_TRY(cudaEventCreate(&e));
    h->tev.push_back(e);
  }
  return MOE_OK;
}

moe_status moe_timing_rewind(moe_handle h) {
  if (!h) return MOE_ERR_INVALID_ARG;
  h->t_next = 0;
  return MOE_OK;
}

moe_status moe_timing_read(moe_handle h, float* ms, int max_records, int* n_records, void* stream) {
  if (!h || !n_records || (max_records > 0 && !ms)) return MOE_ERR_INVALID_ARG;
  CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  const int n = h->t_used < max_records ? h->t_used : max_records;
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < kTimingEvents - 1; ++j)
      CUDA_TRY(cudaEventElapsedTime(&ms[(kTimingEvents - 1) * i + j], h->tev[kTimingEvents * i + j],
                                    h->tev[kTimingEvents * i + j + 1]));
  *n_records = n;
  return MOE_OK;
}

moe_status moe_destroy(moe_handle h) {
  if (!h) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  for (cudaEvent_t ev : h->tev) cudaEventDestroy(ev);
  for (LayerW& L : h->layers) {
    if (L.maps) gemm_maps_free(L.maps);
    if (L.dnb) cudaFree(L.dnb);
  }
  if (h->act_maps) gemm_maps_free(h->act_maps);
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->slab) cudaFree(h->slab);
  delete h;
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
