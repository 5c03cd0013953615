/*
 * Routed mixture-of-experts FFN layer for one B300 (sm_103a): C ABI.
 *
 * The layer is the one the Strata engine pages describe for Qwen3.8-Flash-Next:
 *   - 48 layers, each with 512 experts and a router that picks 10 of them per token, plus a
 *     shared expert that every token uses -- 'Strata はなぜ少ない VRAM でも速いのか'
 *     (modeldock.net), section '問題：1,250 億パラメータと 12 GB';
 *   - per layer the router runs, the chosen experts compute, the results are summed and the next
 *     layer starts, the 48-layer step replayed as one CUDA graph -- same page, section
 *     '1 トークン、三者の分担';
 *   - a verify pass runs 1 new + up to 3 drafted tokens through all 48 layers at once -- same
 *     page, section '予測してから検証する';
 *   - prefill runs chunks of thousands of tokens that reach almost every expert -- same page,
 *     section '長いプロンプトを読む：大きなまとまりで流す'.
 * The pages fix no formula, activation or number format.  This library computes:
 *   logits[t,e] = sum_j x[t,j] * router_w[e,j] (+ router_b[e])              (fp32)
 *   p = softmax over all E logits; keep the K largest logits (ties: lower expert index first);
 *   w[t,k] = p[idx[t,k]] / sum_k' p[idx[t,k']]                                (renormalised)
 *   FFN_e(x) = W_down,e ( silu(W_gate,e x) * (W_up,e x) ),  silu(z) = z / (1 + exp(-z))
 *   y[t] = sum_{k=0..K-1} w[t,k] FFN_{idx[t,k]}(x[t])  (+ FFN_shared(x[t]) with weight 1),
 *   summed in fp32 in a fixed order and rounded once to the output type (the GEMV and prefill
 *   paths: ascending k, the shared expert last; the one-launch decode layer: the routing weight
 *   is folded into h, each output row is owned by one CTA which sums the slots in slot order,
 *   the shared expert first, then the distinct experts ascending, and its warps' partial sums in
 *   warp order).
 *
 * Conventions (all entry points):
 *   - Pointers are DEVICE pointers owned by the caller unless a parameter says "host".
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default stream.  Every
 *     call is asynchronous on that stream unless stated otherwise; none synchronises it except
 *     moe_get_device_status and the *_host entry points.
 *   - Arguments are validated before anything is launched; on error nothing is launched and an
 *     error status is returned.  Status codes are returned, never printed.
 *   - The library allocates device memory only in moe_create (one workspace sized for
 *     max_tokens) and frees it in moe_destroy.  Every kernel reads the caller's weight planes
 *     where they are; there is no second copy of any weight.
 *   - A handle is not thread-safe, and calls made with one handle on different streams that
 *     overlap in time race on its workspace.
 *
 * Weight storage (our definition; the pages give none):
 *   MOE_W_INT4_G32: a matrix [rows x K] is stored row-major, two 4-bit two's-complement values per
 *     byte, the even column in the low nibble; 32 consecutive columns (16 bytes) form a group
 *     with one fp16 scale; value = q * scale, q in [-8, 7].  Scales: fp16 [rows x K/32].
 *   MOE_W_F32: the same matrices as plain fp32 [rows x K], no scales.
 *   Routed experts of a layer are stacked by expert index:
 *     gu_q  [E][2f][d/2] bytes   (rows 0..f-1 = gate, rows f..2f-1 = up), gu_s [E][2f][d/32] fp16
 *     dn_q  [E][d][f/2] bytes,                                             dn_s [E][d][f/32] fp16
 *   (fp32: gu [E][2f][d], dn [E][d][f]).  The shared expert uses the same per-expert layout.
 *   Router: router_w fp32 [E][d], router_b fp32 [E] or NULL.
 *   Every base pointer must be 16-byte aligned.  INT4 needs d % 128 == 0 and f % 128 == 0.
 * Activations: [T][d] row-major, bf16 (MOE_ACT_BF16) or fp32 (MOE_ACT_F32).
 */
#ifndef ROUTED_MOE_B300_MOE_H
#define ROUTED_MOE_B300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx* moe_handle;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size, T > max_tokens, ...        */
  MOE_ERR_UNSUPPORTED = 2, /* a shape or format this build does not implement                 */
  MOE_ERR_OOM = 3,         /* workspace allocation failed in moe_create                        */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call failed (including earlier asynchronous errors) */
  MOE_ERR_TIMEOUT = 5,     /* a device-side bounded wait gave up (reported by get_device_status) */
  MOE_ERR_NOT_SET = 6,     /* the layer's weights were never registered with moe_set_layer      */
  MOE_ERR_DEVICE = 7       /* a device-side check failed (reported by get_device_status)        */
} moe_status;

enum { MOE_ACT_F32 = 0, MOE_ACT_BF16 = 1 };
enum { MOE_W_F32 = 0, MOE_W_INT4_G32 = 1 };

typedef struct {
  int d;          /* hidden size                                                    */
  int f;          /* expert FFN width                                               */
  int n_experts;  /* E, routed experts per layer (<= 1024)                          */
  int top_k;      /* K, experts kept per token (1 <= K <= min(E, 32))               */
  int n_layers;   /* L                                                              */
  int max_tokens; /* largest T any call will pass (sizes the workspace)             */
  int has_shared; /* 1: every layer has a shared expert with weight 1               */
  int prenorm;    /* stack only: x <- x + MoE(RMSNorm(x)), RMSNorm without weight   */
  float norm_eps; /* RMSNorm epsilon                                                */
  int wfmt;       /* MOE_W_INT4_G32 or MOE_W_F32                                    */
  int act;        /* MOE_ACT_BF16 or MOE_ACT_F32                                    */
} moe_config;

typedef struct {
  const float* router_w; /* fp32 [E][d]                          */
  const float* router_b; /* fp32 [E] or NULL                     */
  const void* gu_q;      /* routed experts, gate/up (see above)  */
  const void* gu_s;
  const void* dn_q;      /* routed experts, down                 */
  const void* dn_s;
  const void* sh_gu_q;   /* shared expert (NULL if !has_shared)  */
  const void* sh_gu_s;
  const void* sh_dn_q;
  const void* sh_dn_s;
} moe_layer_weights;

/* Create a handle on the current CUDA device and allocate its workspace for cfg->max_tokens.
 * Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for bad configs, MOE_ERR_OOM if the
 * workspace cannot be allocated.  *out is set only on success. */
moe_status moe_create(const moe_config* cfg, moe_handle* out);

/* Register the weights of layer `layer` (0 <= layer < n_layers).  Stores the pointers (the memory
 * must stay valid while the handle uses it) and encodes, in host memory, the TMA descriptors of
 * the layer's planes for the tensor-core paths.  It neither allocates device memory, launches,
 * copies nor synchronises, so the weights may be written before or after this call (before the
 * first forward that uses them); a layer whose planes MOVE must be registered again.  Pointers
 * are checked for NULL (scales only for INT4, shared planes only with has_shared) and 16-byte
 * alignment; MOE_ERR_INVALID_ARG if a descriptor cannot be encoded, MOE_ERR_OOM if the host
 * memory for the descriptors cannot be had. */
moe_status moe_set_layer(moe_handle h, int layer, const moe_layer_weights* w);

/* Router + top-K + dispatch of one layer for T tokens (1 <= T <= max_tokens):
 *   topk_idx [T*K] int32, slot order = selection order (largest logit first, ties lower index);
 *   topk_w [T*K] fp32 renormalised weights;
 *   expert_offs [E+1] int32: assignments of expert e are perm[offs[e] .. offs[e+1]);
 *   perm [T*K] int32: assignment ids a = t*K + k stably sorted by expert (ascending t per expert).
 * Any of the four outputs may be NULL (not written).  x is [T][d] of the configured act type. */
moe_status moe_route(moe_handle h, int layer, const void* x, int T, int32_t* topk_idx, float* topk_w,
                     int32_t* expert_offs, int32_t* perm, void* stream);

/* y = MoE_layer(x) for T tokens.  x, y: [T][d] of the configured act type; y must not overlap x.
 * Which kernels run depends on T (see MOE_OPT_FUSED_MAX_TOKENS and MOE_OPT_GEMV_MAX_TOKENS): small T
 * runs the one-launch decode layer, larger T the grouped tensor-core GEMM. */
moe_status moe_layer_forward(moe_handle h, int layer, const void* x, int T, void* y, void* stream);

/* All n_layers layers in order, in place: x <- x + MoE_l(N(x)) with N = RMSNorm (no weight,
 * norm_eps) if cfg.prenorm, else the identity; the residual is added in fp32 and rounded once.
 * Replays one CUDA graph per T (captured at the first call with that T; capture happens on an
 * internal stream, so the first call for a T must not be made while `stream` is being captured).
 * trace: NULL, or a device buffer of n_layers*2*T*d activations receiving, per layer l, the
 * layer input x_l and the normalised input N(x_l) (both in the act type); with a trace the
 * layers are launched directly instead of through the graph. */
moe_status moe_stack_forward(moe_handle h, void* x_inout, int T, void* trace, void* stream);

/* moe_stack_forward with launches made one by one (no graph) and, per layer l, a device copy of the
 * routing the layer used: route_idx [L][T*K] int32, route_w [L][T*K] fp32, route_offs [L][E+1] int32,
 * route_perm [L][T*K] int32 (each may be NULL), with the meaning of moe_route's outputs.  trace as in
 * moe_stack_forward (may be NULL).  For checking a stack against a reference layer by layer. */
moe_status moe_stack_forward_traced(moe_handle h, void* x_inout, int T, void* trace, int32_t* route_idx,
                                    float* route_w, int32_t* route_offs, int32_t* route_perm, void* stream);

/* Device copy (asynchronous on `stream`) of the routing that the most recent layer enqueued on the
 * handle used -- by moe_layer_forward, moe_layer_forward_host, moe_route, or the last layer of
 * moe_stack_forward -- as computed by whichever kernels served it: topk_idx [T*K], topk_w [T*K],
 * expert_offs [E+1], perm [T*K], meanings as in moe_route (each may be NULL).  T must be the T of that
 * call (MOE_ERR_INVALID_ARG otherwise).  Must be enqueued before the next call that routes. */
moe_status moe_get_last_routing(moe_handle h, int T, int32_t* topk_idx, float* topk_w, int32_t* expert_offs,
                                int32_t* perm, void* stream);

/* Per-expert usage histogram ('Strata はなぜ少ない VRAM でも速いのか', section '粗から細へ：モデルを分ける
 * 四つの方法': the engine ranks experts by how often they are used).  With on = 1, every forward pass
 * (moe_layer_forward, moe_layer_forward_host, moe_stack_forward) adds, per layer l and expert e, the
 * number of (token, slot) assignments routed to e; moe_route does not count.  The counters are
 * uint64 [n_layers][E] inside the handle's workspace (zero at moe_create), added in the dispatch step
 * of every path, so they are exact.  Toggling drops the handle's captured stack graphs.
 * moe_usage_read copies them to counts_host (n_layers*E values), optionally zeroes them, and
 * synchronises `stream`. */
moe_status moe_usage_enable(moe_handle h, int on);
moe_status moe_usage_read(moe_handle h, unsigned long long* counts_host, int reset, void* stream);

/* End-to-end form of moe_layer_forward for HOST buffers: copies x_host to the device, runs the
 * layer, copies the result to y_host and synchronises `stream`.  When both buffers are page-locked
 * and mapped into the device's address space (cudaHostAlloc / cudaHostRegister under unified
 * addressing) and hold at most 256 KiB, a small kernel moves the bytes over the host link with loads
 * and stores; otherwise two cudaMemcpyAsync transfers do (pageable buffers work, synchronously).
 * Either way x_host is read and y_host written exactly once per call.  Blocks the calling thread
 * until done. */
moe_status moe_layer_forward_host(moe_handle h, int layer, const void* x_host, int T, void* y_host,
                                  void* stream);

/* Host copy of the per-layer count of distinct routed experts selected by the most recent
 * route of each layer (n_layers int32 values).  Synchronises `stream`. */
moe_status moe_get_active_counts(moe_handle h, int32_t* counts_host, void* stream);

/* Synchronises `stream` and reports pending errors: MOE_ERR_CUDA for a CUDA error,
 * MOE_ERR_DEVICE / MOE_ERR_TIMEOUT if a kernel recorded a failed check or an exhausted wait in
 * the handle's status word (which is then cleared). */
moe_status moe_get_device_status(moe_handle h, void* stream);

/* Free the workspace and any captured graphs.  Synchronises the device first. */
moe_status moe_destroy(moe_handle h);

/* Test hook (host-side fault injection): ORs `bits` (1 = a failed device-side check, 2 = a wait that
 * gave up) into the handle's device status word, exactly as a kernel that hit the condition would.
 * Synchronises `stream`.  A one-launch decode layer that finds the timeout bit set gives up at once
 * and writes NaN to y, until moe_get_device_status has reported the status and reset the layer's
 * launch state; nothing on the device faults or hangs. */
moe_status moe_inject_device_status(moe_handle h, unsigned bits, void* stream);

/* Self-test of the device-side bounded waits that every layer kernel uses (no model data, no
 * handle).  One small kernel waits on an mbarrier nobody arrives at and polls a word for an epoch
 * tag nobody writes, each with a budget of `budget_cycles` SM clocks (1000 .. 2e9).  Returns MOE_ERR_TIMEOUT
 * when both waits gave up and recorded "timeout" (the expected outcome), MOE_ERR_DEVICE if a wait
 * reported success, MOE_ERR_CUDA on a CUDA error.  Synchronises `stream`; the GPU context stays
 * usable afterwards.  Allocates nothing: the word and the result live in file-scope device memory
 * (concurrent self-tests on one device race on them). */
moe_status moe_selftest_bounded_waits(long long budget_cycles, void* stream);

/* Options (each returns the value in effect, or a negative moe_status on error; changing one
 * drops the handle's captured stack graphs; value -1 only queries the value in effect).
 * MOE_OPT_FUSED_MAX_TOKENS: calls with T <= value run the whole layer (router, selection,
 *   dispatch, experts on tensor cores, combine) as one kernel of one CTA per SM with grid-wide
 *   barriers (value 0..8, 0 = off; default 4; INT4 weights with d % 512 == 0, d <= 2048,
 *   f % 32 == 0, f <= 1024; the value in effect is clamped to what the shared-memory plan of the
 *   shape allows).  Its operands are fp16 (exact int4 codes and bf16 activations, w * h rounded
 *   once), accumulated in fp32.
 * MOE_OPT_GEMV_MAX_TOKENS: other calls with T <= value run the split-K GEMV experts, larger T the
 *   tensor-core grouped GEMM (value 0..16; default 4; the grouped GEMM needs INT4 weights with
 *   d % 256 == 0 and f % 256 == 0, otherwise the value is clamped to 16). */
enum { MOE_OPT_GEMV_MAX_TOKENS = 1, MOE_OPT_FUSED_MAX_TOKENS = 2, MOE_OPT_KERNEL_TIMELINE = 3 };
int moe_set_option(moe_handle h, int option, int value);

/* In-kernel timeline of the one-launch decode layer (tracing).  With MOE_OPT_KERNEL_TIMELINE = 1 every
 * launch of that layer writes, per CTA and event, the GPU global timer (ns) at its phase boundaries
 * (kernel entry, dependency wait passed, logits stored, grid barrier passed, routing done, first
 * gate/up unit landed, gate/up done, first down item landed, down done, y written, and the producer's
 * last gate/up issue, first and last down issue); each launch overwrites the previous one's stamps.
 * moe_timeline_read copies the most recent stamps ([n_ctas][n_events] uint64, at most `capacity`
 * values) to the host and synchronises `stream`; MOE_ERR_UNSUPPORTED when the config has no one-launch
 * layer. */
moe_status moe_timeline_read(moe_handle h, unsigned long long* stamps_host, int capacity, int* n_ctas, int* n_events,
                             void* stream);

/* Stage timing (tracing).  moe_timing_enable(h, n) creates 5*n CUDA events; afterwards every
 * layer enqueued by moe_layer_forward / moe_stack_forward (also inside a graph captured after
 * this call) records events before routing, after routing, after expert stage A, after expert
 * stage B and at the end, until n layer records are used.  Stages: decode (T <= 16) A = gate/up,
 * B = down + combine, C = 0; prefill A = fp16 staging + tile plan + gate/up GEMM, B = down GEMM,
 * C = combine.  moe_timing_read synchronises `stream` and writes, for each of the *n_records
 * recorded layers, 4 durations in milliseconds (route, A, B, C) into ms[4*i .. 4*i+3]
 * (capacity: max_records records); moe_timing_rewind restarts recording at record 0 (events of a
 * captured graph keep their record indices).  moe_timing_enable(h, 0) frees the events. */
moe_status moe_timing_enable(moe_handle h, int n_records);
moe_status moe_timing_rewind(moe_handle h);
moe_status moe_timing_read(moe_handle h, float* ms, int max_records, int* n_records, void* stream);

/* Routing without any allocation, for callers that cannot call cudaMalloc: code that runs while a
 * stream is being captured into a CUDA graph owned by another framework (allocating there is not
 * allowed), code that must stay inside a memory pool it was given, or latency-critical host
 * threads that cannot afford the device synchronisation cudaMalloc may cause.  The pages describe
 * no counterpart of this call: it exists only for such callers.
 * It computes exactly what moe_route computes (router + softmax + top-K + dispatch, no RMSNorm)
 * from plain pointers, without a handle: router_w fp32 [E][d], router_b fp32 [E] or NULL, x [T][d]
 * of type `act`; outputs as in moe_route (each may be NULL).  Its scratch (logits, counts, slot
 * table, ticket; 121,600 bytes) is one fixed device array inside this library, so it supports at
 * most T = 16 tokens, E = 1024 experts, K = 32 and T*d*4 <= 163,840 bytes; larger sizes return
 * MOE_ERR_UNSUPPORTED and launch nothing.  Every GPU that loads the library holds that array until
 * the process exits.  All calls on a device share it, so calls that overlap on the GPU (different
 * streams, or threads without ordering) race and give wrong results; the array keeps the last
 * call's contents.  The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture, and do not reset the device
 * (cudaDeviceReset) between calls: the address is kept for the life of the process.  No cudaMalloc,
 * cudaFree or allocating library call is made.  Its kernels make no device-side checks and never
 * wait, so there is no device status to read back; MOE_ERR_CUDA sets moe_last_cuda_error. */
moe_status moe_route_noalloc(const float* router_w, const float* router_b, const void* x, int act, int T, int d,
                             int E, int K, int32_t* topk_idx, float* topk_w, int32_t* expert_offs, int32_t* perm,
                             void* stream);

const char* moe_status_str(moe_status s);
int moe_version(void);

/* The CUDA error code behind the most recent MOE_ERR_CUDA returned on this host thread (0 if none),
 * and its text. */
int moe_last_cuda_error(void);
/* The CUDA runtime's pending error of this host thread (not cleared), for diagnostics. */
int moe_peek_cuda_error(void);
const char* moe_cuda_error_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* ROUTED_MOE_B300_MOE_H */
