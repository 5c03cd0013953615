// Decode / verify experts: split-K GEMV over the distinct experts the batch routed to (sm_103a).
//
// A decode step touches only the experts its tokens routed to, so its cost is the bytes of
// those experts ('Strata はなぜ少ない VRAM でも速いのか' (modeldock.net), section
// '1 トークン、三者の分担': the step is bound by how fast expert bytes stream; section
// '予測してから検証する': verifying several tokens costs only the extra experts they route to).
// Every distinct expert is read from HBM exactly once per layer, whatever the number of tokens
// routed to it, and all its tokens are served from that one read.
//
// Kernels (one launch each):
//   gu_*  : work item = (slot, 16 consecutive f indices); slot = a distinct routed expert or the
//           shared expert.  Each warp owns 2 f indices (gate row + up row each), each lane a fixed
//           set of 32-column groups, so one warp load instruction covers 512 contiguous bytes.
//           h = silu(gate . x) * (up . x) in fp32 -> workspace h[assignment][f].
//   dn_*  : block = 16 output rows; its warps split the slots; each lane owns one 32-column
//           group of h and reuses it for the 16 rows.  Per-assignment results land in shared
//           memory and are combined in fixed order (ascending k, shared expert last), plus the
//           optional residual, and rounded once to the activation type.
//
// int4 dot product without per-element integer->float conversion: a code o = q + 8 (offset
// binary, 0..15) placed in mantissa bits 16..19 under exponent 2^-1 is the fp32 value
// v = 0.5 + o/256 (one byte permute per element).  With x' = 256 x,
//   sum_k q_k x_k = sum_k v_k x'_k - 136 sum_k x_k,
// the second term precomputed per (token, group).  v_k x'_k is exact in fp32 for bf16 x; the
// accumulation is fp32; the group scale multiplies the group sum once.
#include "common.cuh"

namespace moe {

constexpr int kGuWarps = 8;             // warps per block of the gate/up kernel
constexpr int kGuFPerWarp = 2;          // f indices per warp
constexpr int kGuFPerItem = kGuWarps * kGuFPerWarp;  // 16
constexpr int kDnRows = 16;             // output rows per block of the down kernel
constexpr int kDnWarps = 16;
constexpr int kTB = 2;                  // tokens per register batch

// ------------------------------------------------------------------ slot -> (expert, tokens)
struct SlotInfo {
  int n;           // tokens routed to the slot
  bool shared;
  int e;
};

// Token list of slot s: tok[i] = token index, asg[i] = assignment row (t*K+k, or T*K+t for shared).
__device__ __forceinline__ SlotInfo slot_tokens(const ExpertArgs& a, int s, int n_act, int* tok, int* asg) {
  SlotInfo si;
  if (s < n_act) {
    const int e = a.active[s];
    const int b = a.offs[e], n = a.offs[e + 1] - b;
    for (int i = 0; i < n; ++i) {
      const int as = a.perm[b + i];
      tok[i] = as / a.K;
      asg[i] = as;
    }
    si.n = n;
    si.shared = false;
    si.e = e;
  } else {
    for (int i = 0; i < a.T; ++i) {
      tok[i] = i;
      asg[i] = a.T * a.K + i;
    }
    si.n = a.T;
    si.shared = true;
    si.e = -1;
  }
  return si;
}


// ------------------------------------------------------------------ gate/up, int4
// Persistent: one block per SM, 16 warps.  The (gate row, up row) pairs of all slots are numbered
// slot-major, p = slot * f + i, and split into one contiguous range per block; warp w of a block
// takes pairs w, w+16, ... of that range and keeps the next pair's loads in flight while it
// computes the current one.  All T tokens' activations are staged once per block in shared memory
// as x' = 256 x in a group-interleaved layout [t][m4=0..7][G][4], with 136 * (group sum) beside.
constexpr int kGuThreads = 512;
constexpr int kGuW = kGuThreads / 32;

template <int NG>
struct PairRegs {
  uint4 q[2][NG];
  __half2 s[NG];  // .x = gate scale, .y = up scale
};

template <int NG>
__device__ __forceinline__ void gu_load_pair(const ExpertArgs& a, const int4* slot_s, int n_act, int p, int lane,
                                             PairRegs<NG>& r) {
  const int d = a.d, f = a.f, G = d / 32;
  const int s = p / f, i = p - s * f;
  const uint8_t* gq;
  const __half* gs;
  if (s < n_act) {
    const int e = slot_s[s].x;
    gq = static_cast<const uint8_t*>(a.gu_q) + (size_t)e * 2 * f * (d / 2);
    gs = a.gu_s + (size_t)e * 2 * f * G;
  } else {
    gq = static_cast<const uint8_t*>(a.sh_gu_q);
    gs = a.sh_gu_s;
  }
#pragma unroll
  for (int j = 0; j < NG; ++j) {
    const int g = lane + 32 * j;
    if (g < G) {
      r.q[0][j] = ldg_nc_v4(gq + (size_t)i * (d / 2) + g * 16);
      r.q[1][j] = ldg_nc_v4(gq + (size_t)(f + i) * (d / 2) + g * 16);
      r.s[j] = __halves2half2(gs[(size_t)i * G + g], gs[(size_t)(f + i) * G + g]);
    } else {
      r.q[0][j] = r.q[1][j] = make_uint4(0, 0, 0, 0);
      r.s[j] = __float2half2_rn(0.f);
    }
  }
}

template <int NG>
__device__ __forceinline__ void gu_compute_pair(const ExpertArgs& a, const int4* slot_s, const int* perm_s,
                                                int n_act, int p, int lane, const float4* xq, const float* xs136,
                                                const PairRegs<NG>& r) {
  const int d = a.d, f = a.f, G = d / 32, K = a.K;
  const int s = p / f, i = p - s * f;
  int n, pbase;
  bool shared;
  if (s < n_act) {
    const int4 sl = slot_s[s];
    pbase = sl.y;
    n = sl.z;
    shared = false;
  } else {
    pbase = 0;
    n = a.T;
    shared = true;
  }
  for (int t0 = 0; t0 < n; t0 += kTB) {
    int tok[kTB];
#pragma unroll
    for (int tt = 0; tt < kTB; ++tt) {
      const int ti = t0 + tt < n ? t0 + tt : t0;
      tok[tt] = shared ? ti : perm_s[pbase + ti] / K;
    }
    float acc[2][kTB];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int tt = 0; tt < kTB; ++tt) acc[m][tt] = 0.f;
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      const int g = lane + 32 * j;
      if (g >= G) continue;
      float part[2][kTB];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int tt = 0; tt < kTB; ++tt) part[m][tt] = 0.f;
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        float4 xa[kTB], xb[kTB];
#pragma unroll
        for (int tt = 0; tt < kTB; ++tt) {
          const float4* xp = xq + (size_t)tok[tt] * 8 * G + g;
          xa[tt] = xp[(2 * wd) * G];
          xb[tt] = xp[(2 * wd + 1) * G];
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          uint32_t w32 = wd == 0 ? r.q[m][j].x : wd == 1 ? r.q[m][j].y : wd == 2 ? r.q[m][j].z : r.q[m][j].w;
          asm volatile("" : "+r"(w32));  // keep the dequantisation inside the token loop
          const uint32_t lo = (w32 & 0x0F0F0F0Fu) ^ 0x08080808u;
          const uint32_t hi = ((w32 >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
          const float v0 = v_lo(lo, 0), v1 = v_lo(hi, 0), v2 = v_lo(lo, 1), v3 = v_lo(hi, 1);
          const float v4 = v_lo(lo, 2), v5 = v_lo(hi, 2), v6 = v_lo(lo, 3), v7 = v_lo(hi, 3);
#pragma unroll
          for (int tt = 0; tt < kTB; ++tt) {
            float q = part[m][tt];
            q = fmaf(v0, xa[tt].x, q);
            q = fmaf(v1, xa[tt].y, q);
            q = fmaf(v2, xa[tt].z, q);
            q = fmaf(v3, xa[tt].w, q);
            q = fmaf(v4, xb[tt].x, q);
            q = fmaf(v5, xb[tt].y, q);
            q = fmaf(v6, xb[tt].z, q);
            q = fmaf(v7, xb[tt].w, q);
            part[m][tt] = q;
          }
        }
      }
      const float2 sc = __half22float2(r.s[j]);
#pragma unroll
      for (int tt = 0; tt < kTB; ++tt) {
        const float x136 = xs136[tok[tt] * G + g];
        acc[0][tt] = fmaf(sc.x, part[0][tt] - x136, acc[0][tt]);
        acc[1][tt] = fmaf(sc.y, part[1][tt] - x136, acc[1][tt]);
      }
    }
#pragma unroll
    for (int tt = 0; tt < kTB; ++tt) {
      if (t0 + tt >= n) continue;
      const float gsum = warp_sum(acc[0][tt]);
      const float usum = warp_sum(acc[1][tt]);
      if (lane == 0) {
        const int as = shared ? a.T * K + (t0 + tt) : perm_s[pbase + t0 + tt];
        a.h[(size_t)as * f + i] = silu(gsum) * usum;
      }
    }
  }
}

template <int NG>  // 32-column groups per lane per row (d = NG * 1024 at full width)
__global__ void __launch_bounds__(kGuThreads, 1) gu_int4_kernel(ExpertArgs a) {
  extern __shared__ float4 smem4[];
  const int d = a.d, f = a.f, G = d / 32, T = a.T, K = a.K;
  float4* xq = smem4;                                                     // [T][8][G] float4
  float* xs136 = reinterpret_cast<float*>(smem4 + (size_t)T * 8 * G);     // [T][G]
  int4* slot_s = reinterpret_cast<int4*>(xs136 + (size_t)T * G);          // [E]
  int* perm_s = reinterpret_cast<int*>(slot_s + a.E);                     // [T*K]
  __shared__ int n_act_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) n_act_s = *a.n_active;
  for (int i = threadIdx.x; i < T * K; i += blockDim.x) perm_s[i] = a.perm[i];
  __syncthreads();
  const int n_act = n_act_s;
  for (int i = threadIdx.x; i < n_act; i += blockDim.x) slot_s[i] = a.slots[i];
  __syncthreads();
  const int n_slots = n_act + a.has_shared;
  const int Np = n_slots * f;
  const int p0 = (int)((long long)Np * blockIdx.x / gridDim.x);
  const int p1 = (int)((long long)Np * (blockIdx.x + 1) / gridDim.x);
  PairRegs<NG> ra, rb;
  int p = p0 + warp;
  if (p < p1) gu_load_pair<NG>(a, slot_s, n_act, p, lane, ra);  // in flight while x is staged
  // stage x' = 256 x for all tokens, group-interleaved, and 136 * group sums
  const int nch = T * d / 8;
  for (int c0 = threadIdx.x; c0 < nch; c0 += 4 * blockDim.x) {
    float v[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * blockDim.x;
      if (c < nch) load8_act(a.x, a.act, (size_t)c * 8, v[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * blockDim.x;
      if (c < nch) {
        const int ti = (c * 8) / d, k = c * 8 - ti * d;
        const int g = k >> 5, m4 = (k & 31) >> 2;
        float4* dst = xq + ((size_t)ti * 8 + m4) * G + g;
        dst[0] = make_float4(v[u][0] * 256.f, v[u][1] * 256.f, v[u][2] * 256.f, v[u][3] * 256.f);
        dst[G] = make_float4(v[u][4] * 256.f, v[u][5] * 256.f, v[u][6] * 256.f, v[u][7] * 256.f);
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * G; i += blockDim.x) {
    const int ti = i / G, g = i - ti * G;
    const float* xb = reinterpret_cast<const float*>(xq) + (size_t)ti * 8 * G * 4;
    float sx = 0.f;
    for (int m = 0; m < 32; ++m) sx += xb[((m >> 2) * G + g) * 4 + (m & 3)];
    xs136[i] = sx * (136.0f / 256.0f);
  }
  __syncthreads();
  for (; p < p1; p += 2 * kGuW) {
    const int pn = p + kGuW;
    if (pn < p1) gu_load_pair<NG>(a, slot_s, n_act, pn, lane, rb);
    gu_compute_pair<NG>(a, slot_s, perm_s, n_act, p, lane, xq, xs136, ra);
    if (pn + kGuW < p1) gu_load_pair<NG>(a, slot_s, n_act, pn + kGuW, lane, ra);
    if (pn < p1) gu_compute_pair<NG>(a, slot_s, perm_s, n_act, pn, lane, xq, xs136, rb);
  }
}

// ------------------------------------------------------------------ down + combine, int4
// One lane per 32-column group of h (f/32 <= 32 lanes active); 16 rows per block.
// Shared memory: P [T*K + T][16] floats.
__global__ void __launch_bounds__(kDnWarps * 32, 1) dn_int4_kernel(ExpertArgs a) {
  extern __shared__ float P[];  // [T*K + T][kDnRows], then slot table [E] int4, perm [T*K]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, f = a.f, G = f / 32, T = a.T, K = a.K;
  int4* slot_s = reinterpret_cast<int4*>(P + (size_t)(T * K + T) * kDnRows);
  int* perm_s = reinterpret_cast<int*>(slot_s + a.E);
  __shared__ int n_act_s;
  const int j0 = blockIdx.x * kDnRows;
  if (threadIdx.x == 0) n_act_s = *a.n_active;
  for (int i = threadIdx.x; i < T * K; i += blockDim.x) perm_s[i] = a.perm[i];
  __syncthreads();
  const int n_act = n_act_s;
  for (int i = threadIdx.x; i < n_act; i += blockDim.x) slot_s[i] = a.slots[i];
  __syncthreads();
  const int n_slots = n_act + a.has_shared;
  const bool on = lane < G;
  for (int s = warp; s < n_slots; s += kDnWarps) {
    const bool shared = s >= n_act;
    const int4 sl = shared ? make_int4(-1, 0, T, 0) : slot_s[s];
    const uint8_t* q = shared ? static_cast<const uint8_t*>(a.sh_dn_q)
                              : static_cast<const uint8_t*>(a.dn_q) + (size_t)sl.x * d * (f / 2);
    const __half* sp = shared ? a.sh_dn_s : a.dn_s + (size_t)sl.x * d * G;
    uint4 wq[kDnRows];
    __half2 sch[kDnRows / 2];  // scales of rows (2r, 2r+1)
#pragma unroll
    for (int r = 0; r < kDnRows; ++r)
      wq[r] = on ? ldg_nc_v4(q + (size_t)(j0 + r) * (f / 2) + lane * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int r = 0; r < kDnRows; r += 2)
      sch[r / 2] = on ? __halves2half2(sp[(size_t)(j0 + r) * G + lane], sp[(size_t)(j0 + r + 1) * G + lane])
                      : __float2half2_rn(0.f);
    for (int i = 0; i < sl.z; ++i) {
      const int as = shared ? T * K + i : perm_s[sl.y + i];
      // the token's 32 h values of this lane's group, all loads issued together
      float4 hv[8];
      const float4* hp = reinterpret_cast<const float4*>(a.h + (size_t)as * f + (on ? lane : 0) * 32);
#pragma unroll
      for (int m = 0; m < 8; ++m) hv[m] = on ? __ldcg(hp + m) : make_float4(0.f, 0.f, 0.f, 0.f);
      float hsum = 0.f;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        hsum += (hv[m].x + hv[m].y) + (hv[m].z + hv[m].w);
        hv[m].x *= 256.f;
        hv[m].y *= 256.f;
        hv[m].z *= 256.f;
        hv[m].w *= 256.f;
      }
      const float h136 = hsum * 136.0f;
#pragma unroll
      for (int r = 0; r < kDnRows; ++r) {
        float pv = 0.f;
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          uint32_t w32 = wd == 0 ? wq[r].x : wd == 1 ? wq[r].y : wd == 2 ? wq[r].z : wq[r].w;
          asm volatile("" : "+r"(w32));  // keep the dequantisation inside the token loop
          const uint32_t lo = (w32 & 0x0F0F0F0Fu) ^ 0x08080808u;
          const uint32_t hi = ((w32 >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
          const float4 xa = hv[2 * wd], xb = hv[2 * wd + 1];
          pv = fmaf(v_lo(lo, 0), xa.x, pv);
          pv = fmaf(v_lo(hi, 0), xa.y, pv);
          pv = fmaf(v_lo(lo, 1), xa.z, pv);
          pv = fmaf(v_lo(hi, 1), xa.w, pv);
          pv = fmaf(v_lo(lo, 2), xb.x, pv);
          pv = fmaf(v_lo(hi, 2), xb.y, pv);
          pv = fmaf(v_lo(lo, 3), xb.z, pv);
          pv = fmaf(v_lo(hi, 3), xb.w, pv);
        }
        const float sr = (r & 1) ? __high2float(sch[r / 2]) : __low2float(sch[r / 2]);
        const float pr = on ? sr * (pv - h136) : 0.f;
        const float o = warp_sum(pr);
        if (lane == 0) P[(size_t)as * kDnRows + r] = o;
      }
    }
  }
  __syncthreads();
  // fixed-order combine: ascending k, shared expert last, optional residual, one rounding
  for (int i = threadIdx.x; i < T * kDnRows; i += blockDim.x) {
    const int t = i / kDnRows, r = i - t * kDnRows;
    float y = 0.f;
    for (int k = 0; k < K; ++k) y = fmaf(a.topk_w[t * K + k], P[(size_t)(t * K + k) * kDnRows + r], y);
    if (a.has_shared) y += P[(size_t)(T * K + t) * kDnRows + r];
    const size_t o = (size_t)t * d + j0 + r;
    if (a.resid) y = load_act(a.resid, a.act, o) + y;
    store_act(a.y, a.act, o, y);
  }
}

// ------------------------------------------------------------------ fp32 weights (tiny layer)
// Same decomposition; a lane owns float4 column chunks instead of int4 groups.
__global__ void __launch_bounds__(256) gu_f32_kernel(ExpertArgs a) {
  extern __shared__ float xs[];  // [T][d]
  __shared__ int tok_s[kSmallT], asg_s[kSmallT];
  __shared__ int n_s, shared_s, e_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, f = a.f;
  const int n_act = *a.n_active;
  const int n_slots = n_act + a.has_shared;
  const int items_per_slot = (f + kGuFPerItem - 1) / kGuFPerItem;
  const long long N = (long long)n_slots * items_per_slot;
  const long long beg = N * blockIdx.x / gridDim.x, end = N * (blockIdx.x + 1) / gridDim.x;
  int loaded = -1;
  for (long long it = beg; it < end; ++it) {
    const int s = (int)(it / items_per_slot), c = (int)(it % items_per_slot);
    if (s != loaded) {
      __syncthreads();
      if (threadIdx.x == 0) {
        const SlotInfo si = slot_tokens(a, s, n_act, tok_s, asg_s);
        n_s = si.n;
        shared_s = si.shared;
        e_s = si.e;
      }
      __syncthreads();
      for (int i = threadIdx.x; i < n_s * d; i += blockDim.x)
        xs[i] = load_act(a.x, a.act, (size_t)tok_s[i / d] * d + (i % d));
      __syncthreads();
      loaded = s;
    }
    const float* W = shared_s ? static_cast<const float*>(a.sh_gu_q)
                              : static_cast<const float*>(a.gu_q) + (size_t)e_s * 2 * f * d;
    for (int p = 0; p < kGuFPerWarp; ++p) {
      const int fi = c * kGuFPerItem + warp * kGuFPerWarp + p;
      if (fi >= f) continue;
      for (int i = 0; i < n_s; ++i) {
        float g = 0.f, u = 0.f;
        for (int k4 = lane; k4 < d / 4; k4 += 32) {
          const float4 xv = reinterpret_cast<const float4*>(xs + (size_t)i * d)[k4];
          const float4 wg = __ldg(reinterpret_cast<const float4*>(W + (size_t)fi * d) + k4);
          const float4 wu = __ldg(reinterpret_cast<const float4*>(W + (size_t)(f + fi) * d) + k4);
          g = fmaf(wg.x, xv.x, fmaf(wg.y, xv.y, fmaf(wg.z, xv.z, fmaf(wg.w, xv.w, g))));
          u = fmaf(wu.x, xv.x, fmaf(wu.y, xv.y, fmaf(wu.z, xv.z, fmaf(wu.w, xv.w, u))));
        }
        g = warp_sum(g);
        u = warp_sum(u);
        if (lane == 0) a.h[(size_t)asg_s[i] * f + fi] = silu(g) * u;
      }
    }
  }
}

__global__ void __launch_bounds__(kDnWarps * 32, 1) dn_f32_kernel(ExpertArgs a) {
  extern __shared__ float P[];
  __shared__ int tok_s[kDnWarps][kSmallT], asg_s[kDnWarps][kSmallT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, f = a.f, T = a.T, K = a.K;
  const int j0 = blockIdx.x * kDnRows;
  const int n_act = *a.n_active;
  const int n_slots = n_act + a.has_shared;
  for (int s = warp; s < n_slots; s += kDnWarps) {
    SlotInfo si;
    if (lane == 0) si = slot_tokens(a, s, n_act, tok_s[warp], asg_s[warp]);
    __syncwarp();
    si.n = __shfl_sync(0xffffffffu, si.n, 0);
    si.e = __shfl_sync(0xffffffffu, si.e, 0);
    si.shared = __shfl_sync(0xffffffffu, (int)si.shared, 0);
    const float* W = si.shared ? static_cast<const float*>(a.sh_dn_q)
                               : static_cast<const float*>(a.dn_q) + (size_t)si.e * d * f;
    for (int i = 0; i < si.n; ++i) {
      const int as = asg_s[warp][i];
      for (int r = 0; r < kDnRows; ++r) {
        const int j = j0 + r;
        float acc = 0.f;
        if (j < d) {
          for (int k4 = lane; k4 < f / 4; k4 += 32) {
            const float4 hv = __ldcg(reinterpret_cast<const float4*>(a.h + (size_t)as * f) + k4);
            const float4 wv = __ldg(reinterpret_cast<const float4*>(W + (size_t)j * f) + k4);
            acc = fmaf(wv.x, hv.x, fmaf(wv.y, hv.y, fmaf(wv.z, hv.z, fmaf(wv.w, hv.w, acc))));
          }
        }
        acc = warp_sum(acc);
        if (lane == 0) P[(size_t)as * kDnRows + r] = acc;
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * kDnRows; i += blockDim.x) {
    const int t = i / kDnRows, r = i - t * kDnRows;
    if (j0 + r >= d) continue;
    float y = 0.f;
    for (int k = 0; k < K; ++k) y = fmaf(a.topk_w[t * K + k], P[(size_t)(t * K + k) * kDnRows + r], y);
    if (a.has_shared) y += P[(size_t)(T * K + t) * kDnRows + r];
    const size_t o = (size_t)t * d + j0 + r;
    if (a.resid) y = load_act(a.resid, a.act, o) + y;
    store_act(a.y, a.act, o, y);
  }
}

// ------------------------------------------------------------------ launchers
cudaError_t gemv_kernels_init() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gu_int4_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024))) return e;
  if ((e = cudaFuncSetAttribute(gu_int4_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024))) return e;
  if ((e = cudaFuncSetAttribute(gu_int4_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024))) return e;
  if ((e = cudaFuncSetAttribute(gu_int4_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024))) return e;
  if ((e = cudaFuncSetAttribute(gu_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024))) return e;
  if ((e = cudaFuncSetAttribute(dn_int4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024))) return e;
  if ((e = cudaFuncSetAttribute(dn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024))) return e;
  return cudaSuccess;
}

size_t gemv_smem_gu(int wfmt, int T, int d, int E, int K) {
  if (wfmt == kWInt4)
    return (size_t)T * 8 * (d / 32) * sizeof(float4) + (size_t)T * (d / 32) * sizeof(float) + (size_t)E * sizeof(int4) +
           (size_t)T * K * sizeof(int);
  return (size_t)T * d * sizeof(float);
}

size_t gemv_smem_dn(int T, int K, int E) {
  return (size_t)(T * K + T) * kDnRows * sizeof(float) + (size_t)E * sizeof(int4) + (size_t)T * K * sizeof(int);
}

// Launches gate/up then down+combine for T <= kSmallT tokens.
cudaError_t launch_experts_gemv(const ExpertArgs& a, int wfmt, cudaStream_t st, cudaEvent_t mid, cudaEvent_t mid2) {
  const int dn_grid = (a.d + kDnRows - 1) / kDnRows;
  const size_t sm_gu = gemv_smem_gu(wfmt, a.T, a.d, a.E, a.K);
  const size_t sm_dn = gemv_smem_dn(a.T, a.K, a.E);
  if (wfmt == kWInt4) {
    const int G = a.d / 32;
    const int ng = (G + 31) / 32;
    const int grid = a.num_sms;
    switch (ng) {
      case 1: gu_int4_kernel<1><<<grid, kGuThreads, sm_gu, st>>>(a); break;
      case 2: gu_int4_kernel<2><<<grid, kGuThreads, sm_gu, st>>>(a); break;
      case 3: gu_int4_kernel<3><<<grid, kGuThreads, sm_gu, st>>>(a); break;
      case 4: gu_int4_kernel<4><<<grid, kGuThreads, sm_gu, st>>>(a); break;
      default: return cudaErrorInvalidValue;
    }
    if (mid) record_timing_event(mid, st);
    dn_int4_kernel<<<dn_grid, kDnWarps * 32, sm_dn, st>>>(a);
    if (mid2) record_timing_event(mid2, st);
  } else {
    gu_f32_kernel<<<a.num_sms, 256, sm_gu, st>>>(a);
    if (mid) record_timing_event(mid, st);
    dn_f32_kernel<<<dn_grid, kDnWarps * 32, sm_dn, st>>>(a);
    if (mid2) record_timing_event(mid2, st);
  }
  return cudaGetLastError();
}

}  // namespace moe
