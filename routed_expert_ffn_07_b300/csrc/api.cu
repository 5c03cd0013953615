// Host side of the C ABI declared in include/moe.h: argument validation, the workspace, the
// order of launches per layer, and the whole-stack CUDA graph.
//
// The stack of 48 MoE layers runs as one recorded CUDA graph, so no synchronous driver call
// sits between layers ('Strata はなぜ少ない VRAM でも速いのか' (modeldock.net), section
// '1 トークン、三者の分担').
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <map>
#include <vector>

#include "../../include/moe.h"
#include "common.cuh"

namespace moe {
cudaError_t launch_route(const RouteArgs& a, int nblocks_dispatch, cudaStream_t st);
cudaError_t route_kernels_init();
cudaError_t gemv_kernels_init();
cudaError_t launch_experts_gemv(const ExpertArgs& a, int wfmt, cudaStream_t st, cudaEvent_t mid, cudaEvent_t mid2);
size_t gemv_smem_gu(int wfmt, int T, int d, int E, int K);
size_t gemv_smem_dn(int T, int K, int E);
cudaError_t gemm_kernels_init();
cudaError_t decode_kernels_init();
cudaError_t launch_bounded_wait_selftest(long long budget, unsigned* result_host, cudaStream_t st);
bool decode_shape_ok(int T, int d, int f, int E, int K, int nsm);
size_t decode_maps_bytes();
cudaError_t decode_build_maps(void* maps, int E, int d, int f, int nsm, int has_shared, const void* gu_q,
                              const void* gu_s, const void* dn_q, const void* dn_s, const void* sh_gu_q,
                              const void* sh_gu_s, const void* sh_dn_q, const void* sh_dn_s);
cudaError_t launch_decode_layer(const RouteArgs& r, const ExpertArgs& x, const void* maps, unsigned long long* hw,
                                unsigned long long* lgt, unsigned long long* launches, int nsm,
                                unsigned long long* timeline, cudaStream_t st);
int decode_timeline_events();
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
constexpr int kFusedMaxTokensHost = 16;   // the one-launch decode layer's limit
constexpr int kFusedDefaultTokens = 16;   // decode, 1 + 3 verify and small concurrent batches
}  // namespace moe

using namespace moe;

// ------------------------------------------------------------------ host-link copies
// Page-locked host memory mapped into the device's address space is read and written by a kernel
// directly; for the few KB of a decode step's activations this avoids two copy-engine transfers.
constexpr size_t kHostLinkMaxBytes = 256 * 1024;

__global__ void __launch_bounds__(256) host_link_copy_kernel(uint8_t* dst, const uint8_t* src, size_t n, int vec) {
  const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x, nt = (size_t)gridDim.x * blockDim.x;
  size_t done = 0;
  if (vec) {  // both ends 16-byte aligned
    const size_t nw = n / 16;
    for (size_t i = t; i < nw; i += nt) reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
    done = nw * 16;
  }
  for (size_t i = done + t; i < n; i += nt) dst[i] = src[i];
}

static cudaError_t launch_host_link_copy(void* dst, const void* src, size_t n, cudaStream_t st) {
  const int vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
  const size_t units = vec ? (n + 15) / 16 : n;
  const unsigned grid = (unsigned)std::max<size_t>(1, std::min<size_t>(64, (units + 255) / 256));
  host_link_copy_kernel<<<grid, 256, 0, st>>>(static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src), n, vec);
  return cudaGetLastError();
}

// The device address of page-locked, device-mapped host memory p, or null when p is anything else
// (pageable memory, device memory, another device's allocation).
static void* host_device_view(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  int mapped = 0;
  if (cudaDeviceGetAttribute(&mapped, cudaDevAttrCanMapHostMemory, dev) != cudaSuccess || !mapped) {
    cudaGetLastError();
    return nullptr;
  }
  return at.devicePointer;
}

struct LayerW {
  moe_layer_weights w;
  bool set = false;
  void* maps = nullptr;   // TMA descriptors of the layer's planes (grouped tensor-core path)
  void* dmaps = nullptr;  // TMA descriptors of the same planes for the one-launch decode layer
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
  unsigned long long* lgt = nullptr;  // the one-launch decode layer's published logits [16][E] (epoch-tagged)
  unsigned long long* launches = nullptr;  // and its launch counter (one per CTA per launch)
  bool fused_capable = false;    // the one-launch decode layer serves this config (T = 1 at least)
  unsigned long long* hw = nullptr;  // its gate/up results [T + T*K][f/2], epoch-tagged fp16 pairs (T <= 16)
  size_t hw_bytes = 0;
  unsigned long long* timeline = nullptr;  // its in-kernel timeline [#SM][events] (ns)
  bool timeline_on = false;
  unsigned long long* usage = nullptr;  // per-layer expert usage histogram [n_layers][E]
  bool usage_on = false;         // forward passes add their per-expert counts to `usage`
  int last_T = 0;                // T of the most recent routing enqueued on the handle
  // stage timing
  std::vector<cudaEvent_t> tev;
  int t_next = 0;
  int t_used = 0;
};

static size_t act_size(int act) { return act == MOE_ACT_BF16 ? 2 : 4; }

// Largest T <= want (and <= max_tokens) that the one-launch decode layer serves for this config.
static int fused_limit(const moe_config& c, int nsm, int want) {
  int best = 0;
  if (c.wfmt == MOE_W_INT4_G32 && c.act == MOE_ACT_BF16)
    for (int t = 1; t <= want && t <= c.max_tokens; ++t)
      if (decode_shape_ok(t, c.d, c.f, c.n_experts, c.top_k, nsm)) best = t;
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

namespace moe {
// Lets the entry points defined in other files report the CUDA error behind their MOE_ERR_CUDA.
void set_last_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }
}  // namespace moe

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
  if (route_kernels_init() != cudaSuccess || gemv_kernels_init() != cudaSuccess ||
      (h->gemm_ok && gemm_kernels_init() != cudaSuccess) ||
      (c.wfmt == MOE_W_INT4_G32 && decode_kernels_init() != cudaSuccess)) {
    delete h;
    return MOE_ERR_CUDA;
  }
  h->fused_max_tokens = fused_limit(c, h->num_sms, kFusedDefaultTokens);
  h->fused_capable = fused_limit(c, h->num_sms, 1) == 1;

  const int T = c.max_tokens, E = c.n_experts, K = c.top_k, d = c.d, f = c.f;
  const size_t as = act_size(c.act);
  h->nblocks_max = (T * K + kDispatchBlockHost - 1) / kDispatchBlockHost;
  std::vector<size_t> sz;
  sz.push_back(up256((size_t)T * E * 4));                 // logits
  sz.push_back(up256((size_t)T * K * 4));                 // idx
  sz.push_back(up256((size_t)T * K * 4));                 // w
  sz.push_back(up256((size_t)E * 4));                     // counts
  sz.push_back(up256((size_t)(E + 1) * 4));               // offs
  sz.push_back(up256((size_t)T * K * 4));                 // perm
  sz.push_back(up256((size_t)E * 4));                     // active
  sz.push_back(up256(4));                                 // n_active
  sz.push_back(up256((size_t)c.n_layers * 4));            // stats
  sz.push_back(up256((size_t)E * 16));                    // slot table
  sz.push_back(up256(4));                                 // ticket
  sz.push_back(up256(4));                                 // status
  sz.push_back(up256(8));                                 // one-launch layer: launch counter
  sz.push_back(up256((size_t)h->nblocks_max * E * 4));    // blockhist
  const int TS = T < kSmallT ? T : kSmallT;
  sz.push_back(up256((size_t)(TS * K + TS) * f * 4));     // h (GEMV path)
  sz.push_back(h->gemm_ok ? up256(gemm_workspace_bytes(T, d, f, E, K)) : 0);
  sz.push_back(up256((size_t)T * d * as));                // xnorm
  sz.push_back(up256((size_t)T * d * as));                // stack x
  sz.push_back(up256((size_t)T * d * as));                // host x
  sz.push_back(up256((size_t)T * d * as));                // host y
  const int TF = T < kFusedMaxTokensHost ? T : kFusedMaxTokensHost;
  sz.push_back(h->fused_capable ? up256((size_t)(TF + TF * K) * f * 4) : 0);   // one-launch gate/up results
  sz.push_back(h->fused_capable ? up256((size_t)kFusedMaxTokensHost * E * 8) : 0);  // its published logits
  sz.push_back(h->fused_capable ? up256((size_t)h->num_sms * decode_timeline_events() * 8) : 0);  // its timeline
  sz.push_back(up256((size_t)c.n_layers * E * 8));        // usage histogram
  size_t total = 0;
  for (size_t v : sz) total += v;
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
  h->launches = reinterpret_cast<unsigned long long*>(p); p += sz[i++];
  h->blockhist = reinterpret_cast<int32_t*>(p); p += sz[i++];
  h->h = reinterpret_cast<float*>(p); p += sz[i++];
  h->gemm_ws = sz[i] ? p : nullptr; p += sz[i++];
  h->xnorm = p; p += sz[i++];
  h->stack_x = p; p += sz[i++];
  h->host_x = p; p += sz[i++];
  h->host_y = p; p += sz[i++];
  h->hw = sz[i] ? reinterpret_cast<unsigned long long*>(p) : nullptr;
  h->hw_bytes = sz[i];
  p += sz[i++];
  h->lgt = sz[i] ? reinterpret_cast<unsigned long long*>(p) : nullptr; p += sz[i++];
  h->timeline = sz[i] ? reinterpret_cast<unsigned long long*>(p) : nullptr; p += sz[i++];
  h->usage = reinterpret_cast<unsigned long long*>(p); p += sz[i++];
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
    // the one-launch decode layer reads the same planes through its own TMA descriptors (host memory)
    if (!L.dmaps) L.dmaps = aligned_alloc(64, (decode_maps_bytes() + 63) & ~size_t(63));
    if (!L.dmaps) return MOE_ERR_OOM;
    const moe_config& c = h->cfg;
    if (decode_build_maps(L.dmaps, c.n_experts, c.d, c.f, h->num_sms, c.has_shared, w->gu_q, w->gu_s, w->dn_q, w->dn_s,
                          w->sh_gu_q, w->sh_gu_s, w->sh_dn_q, w->sh_dn_s) != cudaSuccess) {
      L.set = false;
      return MOE_ERR_INVALID_ARG;
    }
  }
  L.w = *w;
  L.set = true;
  return MOE_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ internal launch sequences
static RouteArgs make_route_args(moe_ctx* h, int layer, const void* x, int T, bool prenorm, int32_t* stat,
                                 bool count_usage) {
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
  a.usage = (count_usage && h->usage_on) ? h->usage + (size_t)layer * c.n_experts : nullptr;
  h->last_T = T;
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
  a.num_sms = h->num_sms;
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
  RouteArgs ra = make_route_args(h, layer, x, T, prenorm, h->stats + layer, true);
  if (T <= h->fused_max_tokens && h->layers[layer].dmaps) {
    // one launch for the whole layer; its stages are not separated (all of it counts as "route")
    ExpertArgs ea = make_expert_args(h, layer, x, T, y, resid);
    e = launch_decode_layer(ra, ea, h->layers[layer].dmaps, h->hw, h->lgt, h->launches, h->num_sms,
                            h->timeline_on ? h->timeline : nullptr, st);
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
  RouteArgs ra = make_route_args(h, layer, x, T, false, h->stats + layer, false);
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
  // A decode step's few KB cross the host link faster as loads and stores of a small kernel than as
  // two copy-engine transfers, when both buffers are page-locked and mapped into the device's space
  void* xd = bytes <= kHostLinkMaxBytes ? host_device_view(x_host) : nullptr;
  void* yd = xd ? host_device_view(y_host) : nullptr;
  if (xd && yd) {
    CUDA_TRY(launch_host_link_copy(h->host_x, xd, bytes, st));
    CUDA_TRY(enqueue_layer(h, layer, h->host_x, T, h->host_y, nullptr, false, st));
    CUDA_TRY(launch_host_link_copy(yd, h->host_y, bytes, st));
  } else {
    CUDA_TRY(cudaMemcpyAsync(h->host_x, x_host, bytes, cudaMemcpyHostToDevice, st));
    CUDA_TRY(enqueue_layer(h, layer, h->host_x, T, h->host_y, nullptr, false, st));
    CUDA_TRY(cudaMemcpyAsync(y_host, h->host_y, bytes, cudaMemcpyDeviceToHost, st));
  }
  CUDA_TRY(cudaStreamSynchronize(st));
  return MOE_OK;
}

}  // extern "C"

// Per-layer copies of the routing a traced stack used (each pointer may be null).
struct RouteRecord {
  int32_t* idx;   // [L][T*K]
  float* w;       // [L][T*K]
  int32_t* offs;  // [L][E+1]
  int32_t* perm;  // [L][T*K]
};

static cudaError_t copy_routing(moe_ctx* h, int T, int32_t* idx, float* w, int32_t* offs, int32_t* perm,
                                cudaStream_t st) {
  const size_t nk = (size_t)T * h->cfg.top_k * 4, ne = (size_t)(h->cfg.n_experts + 1) * 4;
  cudaError_t e = cudaSuccess;
  if (idx && e == cudaSuccess) e = cudaMemcpyAsync(idx, h->idx, nk, cudaMemcpyDeviceToDevice, st);
  if (w && e == cudaSuccess) e = cudaMemcpyAsync(w, h->w, nk, cudaMemcpyDeviceToDevice, st);
  if (offs && e == cudaSuccess) e = cudaMemcpyAsync(offs, h->offs, ne, cudaMemcpyDeviceToDevice, st);
  if (perm && e == cudaSuccess) e = cudaMemcpyAsync(perm, h->perm, nk, cudaMemcpyDeviceToDevice, st);
  return e;
}

static cudaError_t enqueue_stack(moe_ctx* h, int T, void* trace, const RouteRecord* rr, cudaStream_t st) {
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
    if (rr) {
      const size_t nk = (size_t)l * T * c.top_k, ne = (size_t)l * (c.n_experts + 1);
      e = copy_routing(h, T, rr->idx ? rr->idx + nk : nullptr, rr->w ? rr->w + nk : nullptr,
                       rr->offs ? rr->offs + ne : nullptr, rr->perm ? rr->perm + nk : nullptr, st);
      if (e != cudaSuccess) return e;
    }
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

static moe_status stack_forward(moe_handle h, void* x_inout, int T, void* trace, const RouteRecord* rr,
                                void* stream) {
  if (!h || !x_inout || !aligned16(x_inout)) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (trace && !aligned16(trace)) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < h->cfg.n_layers; ++l)
    if (!h->layers[l].set) return MOE_ERR_NOT_SET;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)T * h->cfg.d * act_size(h->cfg.act);
  CUDA_TRY(cudaGetLastError());
  CUDA_TRY(cudaMemcpyAsync(h->stack_x, x_inout, bytes, cudaMemcpyDeviceToDevice, st));
  if (trace || rr) {
    CUDA_TRY(enqueue_stack(h, T, trace, rr, st));
  } else {
    auto it = h->graphs.find(T);
    if (it == h->graphs.end()) {
      if (!h->cap_stream) CUDA_TRY(cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking));
      cudaGraph_t g = nullptr;
      CUDA_TRY(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
      cudaError_t e = enqueue_stack(h, T, nullptr, nullptr, h->cap_stream);
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

extern "C" {

moe_status moe_stack_forward(moe_handle h, void* x_inout, int T, void* trace, void* stream) {
  return stack_forward(h, x_inout, T, trace, nullptr, stream);
}

moe_status moe_stack_forward_traced(moe_handle h, void* x_inout, int T, void* trace, int32_t* route_idx,
                                    float* route_w, int32_t* route_offs, int32_t* route_perm, void* stream) {
  RouteRecord rr{route_idx, route_w, route_offs, route_perm};
  const bool any = route_idx || route_w || route_offs || route_perm;
  return stack_forward(h, x_inout, T, trace, any ? &rr : nullptr, stream);
}

moe_status moe_get_last_routing(moe_handle h, int T, int32_t* topk_idx, float* topk_w, int32_t* expert_offs,
                                int32_t* perm, void* stream) {
  if (!h || T < 1 || T != h->last_T) return MOE_ERR_INVALID_ARG;
  CUDA_TRY(copy_routing(h, T, topk_idx, topk_w, expert_offs, perm, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_usage_enable(moe_handle h, int on) {
  if (!h || (on != 0 && on != 1)) return MOE_ERR_INVALID_ARG;
  if (h->usage_on != (on != 0)) {
    h->usage_on = on != 0;
    for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);  // the graphs hold the old kernel arguments
    h->graphs.clear();
  }
  return MOE_OK;
}

moe_status moe_usage_read(moe_handle h, unsigned long long* counts_host, int reset, void* stream) {
  if (!h || !counts_host || (reset != 0 && reset != 1)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)h->cfg.n_layers * h->cfg.n_experts * 8;
  CUDA_TRY(cudaMemcpyAsync(counts_host, h->usage, bytes, cudaMemcpyDeviceToHost, st));
  if (reset) CUDA_TRY(cudaMemsetAsync(h->usage, 0, bytes, st));
  CUDA_TRY(cudaStreamSynchronize(st));
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
    // the one-launch layer restarts its epochs from 1: clear the epoch-tagged logits and h words,
    // whose old tags could otherwise match a new epoch
    CUDA_TRY(cudaMemset(h->launches, 0, 8));
    if (h->lgt) CUDA_TRY(cudaMemset(h->lgt, 0, (size_t)kFusedMaxTokensHost * h->cfg.n_experts * 8));
    if (h->hw) CUDA_TRY(cudaMemset(h->hw, 0, h->hw_bytes));
    return MOE_ERR_TIMEOUT;
  }
  if (v) return MOE_ERR_DEVICE;
  return MOE_OK;
}

moe_status moe_inject_device_status(moe_handle h, unsigned bits, void* stream) {
  if (!h || bits == 0 || (bits & ~(kStatusBadIndex | kStatusTimeout))) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  CUDA_TRY(cudaMemcpyAsync(&v, h->status, 4, cudaMemcpyDeviceToHost, st));
  CUDA_TRY(cudaStreamSynchronize(st));
  v |= bits;
  CUDA_TRY(cudaMemcpyAsync(h->status, &v, 4, cudaMemcpyHostToDevice, st));
  CUDA_TRY(cudaStreamSynchronize(st));
  return MOE_OK;
}

moe_status moe_selftest_bounded_waits(long long budget_cycles, void* stream) {
  if (budget_cycles < 1000 || budget_cycles > 2000000000ll) return MOE_ERR_INVALID_ARG;
  unsigned hres[2] = {0, 0};
  const cudaError_t e = launch_bounded_wait_selftest(budget_cycles, hres, static_cast<cudaStream_t>(stream));
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
  if (value == -1) {  // query
    if (option == MOE_OPT_GEMV_MAX_TOKENS) return h->gemv_max_tokens;
    if (option == MOE_OPT_FUSED_MAX_TOKENS) return h->fused_max_tokens;
    if (option == MOE_OPT_KERNEL_TIMELINE) return h->timeline_on ? 1 : 0;
    return -(int)MOE_ERR_INVALID_ARG;
  }
  if (option == MOE_OPT_GEMV_MAX_TOKENS) {
    if (value < 0 || value > kSmallT) return -(int)MOE_ERR_INVALID_ARG;
    h->gemv_max_tokens = h->gemm_ok ? value : kSmallT;
    for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);  // captured graphs used the old path
    h->graphs.clear();
    return h->gemv_max_tokens;
  }
  if (option == MOE_OPT_KERNEL_TIMELINE) {
    if (value != 0 && value != 1) return -(int)MOE_ERR_INVALID_ARG;
    if (!h->timeline) return value ? -(int)MOE_ERR_UNSUPPORTED : 0;
    h->timeline_on = value != 0;
    for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
    h->graphs.clear();
    return value;
  }
  if (option == MOE_OPT_FUSED_MAX_TOKENS) {
    if (value < 0 || value > kFusedMaxTokensHost) return -(int)MOE_ERR_INVALID_ARG;
    h->fused_max_tokens = fused_limit(h->cfg, h->num_sms, value);
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

moe_status moe_timeline_read(moe_handle h, unsigned long long* stamps_host, int capacity, int* n_ctas, int* n_events,
                             void* stream) {
  if (!h || !n_ctas || !n_events || (capacity > 0 && !stamps_host)) return MOE_ERR_INVALID_ARG;
  if (!h->timeline) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int ev = decode_timeline_events();
  const size_t n = std::min((size_t)capacity, (size_t)h->num_sms * ev);
  if (n) CUDA_TRY(cudaMemcpyAsync(stamps_host, h->timeline, n * 8, cudaMemcpyDeviceToHost, st));
  CUDA_TRY(cudaStreamSynchronize(st));
  *n_ctas = h->num_sms;
  *n_events = ev;
  return MOE_OK;
}

moe_status moe_destroy(moe_handle h) {
  if (!h) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  for (cudaEvent_t ev : h->tev) cudaEventDestroy(ev);
  for (LayerW& L : h->layers) {
    if (L.maps) gemm_maps_free(L.maps);
    if (L.dmaps) free(L.dmaps);
  }
  if (h->act_maps) gemm_maps_free(h->act_maps);
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->slab) cudaFree(h->slab);
  delete h;
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
