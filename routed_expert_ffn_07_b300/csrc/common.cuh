// Shared device helpers and launch-argument structs of the routed MoE library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

constexpr int kActF32 = 0;
constexpr int kActBf16 = 1;
constexpr int kWF32 = 0;
constexpr int kWInt4 = 1;

constexpr int kSmallT = 16;   // T <= kSmallT: fused router + split-K GEMV experts
constexpr int kMaxK = 32;
constexpr int kMaxE = 1024;
constexpr int kRouterWarps = 8;
constexpr int kRouterExpertsPerBlock = 4;  // small-T router: 2 warps per expert row

// bits of the device status word
constexpr unsigned kStatusBadIndex = 1u;
constexpr unsigned kStatusTimeout = 2u;
constexpr unsigned kStatusRange = 4u;  // an fp16 tensor-core operand was out of the fp16 range

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sums N values (N = 2, 4 or 8) over the warp in five dependent shuffle steps in all: the first
// log2(N) steps exchange halves of the value list (each lane keeps the half its lane bit selects),
// the rest are a plain butterfly.  On return every lane holds the total of value index
// (lane >> 2) & (N - 1) when N == 8, (lane >> 3) & 3 when N == 4, (lane >> 4) & 1 when N == 2,
// i.e. value i's total sits in the lanes whose bits [5 - log2(N), 5) spell i.
template <int N>
__device__ __forceinline__ float warp_sum_multi(float (&v)[N]) {
  const int lane = threadIdx.x & 31;
  float w[N];
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = v[i];
  int n = N;
  int off = 16;
#pragma unroll
  for (; n > 1; n >>= 1, off >>= 1) {
    const bool up = (lane & off) != 0;  // keep the upper half of the list
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? w[i] : w[i + n / 2];
      const float keep = up ? w[i + n / 2] : w[i];
      w[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
#pragma unroll
  for (; off > 0; off >>= 1) w[0] += __shfl_xor_sync(0xffffffffu, w[0], off);
  return w[0];
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float load_act(const void* p, int act, size_t i) {
  if (act == kActBf16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  return static_cast<const float*>(p)[i];
}

__device__ __forceinline__ void store_act(void* p, int act, size_t i, float v) {
  if (act == kActBf16)
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(p)[i] = v;
}

// 8 consecutive activations starting at element i (i % 8 == 0, 16-byte aligned base): one 16-byte
// load for bf16, two for fp32.
__device__ __forceinline__ void load8_act(const void* p, int act, size_t i, float (&v)[8]) {
  if (act == kActBf16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p) + i));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  } else {
    const float4 a = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p) + i));
    const float4 b = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p) + i) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// Value of v after rounding to the activation type.
__device__ __forceinline__ float round_act(int act, float v) {
  return act == kActBf16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// int4 code byte b (0..3) of `lo` (offset-binary nibbles o = q + 8, one per byte) as the fp32
// value 0.5 + o/256: the byte lands in bits 16..23 under the exponent of 0.5, and o < 16 only
// touches mantissa bits 16..19.
__device__ __forceinline__ float v_lo(uint32_t lo, int b) {
  return __int_as_float(__byte_perm(lo, 0x3F000000u, 0x7054u | (b << 8)));
}

// Record a stage-timing event: inside stream capture it must become an external event node,
// outside capture it is a plain record.
inline cudaError_t record_timing_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, st);
}

// ------------------------------------------------------------------ launch arguments
struct RouteArgs {
  const void* x;     // [T][d] activations (layer input)
  int act, T, d, E, K;
  const float* Wr;   // [E][d]
  const float* bias; // [E] or null
  int prenorm;       // 1: route / compute on RMSNorm(x) rounded to the act type
  float eps;
  void* xnorm;       // [T][d] receives RMSNorm(x) when prenorm (written by block 0)
  float* logits;     // [T][E]
  int32_t* idx;      // [T][K]
  float* w;          // [T][K]
  int32_t* counts;   // [E]
  int32_t* offs;     // [E+1]
  int32_t* perm;     // [T*K]
  int32_t* active;   // [E] distinct experts, ascending
  int32_t* n_active; // [1]
  int32_t* stat;     // [1] or null: receives n_active (per-layer statistics)
  int4* slots;       // [E] per distinct expert s: {expert, first perm position, count, 0}
  int32_t* blockhist;// [nblocks][E] (large-T dispatch)
  unsigned* ticket;  // last-block-done counter (zero between launches)
  unsigned* status;  // device status word
  unsigned long long* usage;  // [E] or null: count[e] of this routing is added (usage histogram)
};

struct ExpertArgs {
  int T, d, f, E, K, act, has_shared;
  int max_tokens;         // the handle's max_tokens (fixes the workspace layout)
  int num_sms;            // the handle's device: SMs (persistent grids)
  const void* x;          // [T][d] expert input (normalised input in the stack)
  const void* gu_q;       // [E][2f][..] routed gate/up
  const __half* gu_s;
  const void* dn_q;       // [E][d][..] routed down
  const __half* dn_s;
  const void* sh_gu_q;
  const __half* sh_gu_s;
  const void* sh_dn_q;
  const __half* sh_dn_s;
  const int32_t* offs;
  const int32_t* perm;
  const int32_t* active;
  const int32_t* n_active;
  const int4* slots;      // [E] {expert, first perm position, count, 0}
  const float* topk_w;    // [T][K]
  float* h;               // [(T*K + T)][f] fp32 (GEMV path)
  void* y;                // [T][d]
  const void* resid;      // [T][d] or null: y = resid + moe
  unsigned* status;
};

}  // namespace moe
