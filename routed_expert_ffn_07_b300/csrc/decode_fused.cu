// Decode / verify layer in one launch (sm_103a): router logits, softmax + top-K, dispatch, the
// gate/up and down GEMVs of the selected and shared experts, and the fixed-order combine.
//
// A decode step streams the bytes of the experts its few tokens chose and little else
// ('Strata はなぜ少ない VRAM でも速いのか' (modeldock.net), section '1 トークン、三者の分担';
// verifying 1 + 3 drafted tokens adds only the experts the drafts pick, section
// '予測してから検証する').  With every expert in HBM the cost that remains besides those bytes is
// the chain router -> selection -> experts -> combine, so it runs in one kernel: one CTA per SM,
// all resident, two grid-wide barriers.
//
//   phase 1  every CTA scores its slice of the E experts for all T tokens (its router rows were
//            copied into shared memory before the previous kernel finished) and stores the
//            logits;                                                              [grid arrive]
//            meanwhile it runs its 8 columns of the shared expert (gate/up, SwiGLU and the
//            matching down columns): those weights do not depend on the routing;    [grid wait]
//   phase 2  every CTA reads all logits and repeats the selection (one warp per token) and the
//            dispatch in shared memory (identical, deterministic); CTA 0 publishes them;
//   phase 3  the routed work, (slot, f-column) in units of 8 columns numbered slot-major, is cut
//            into #CTA contiguous ranges.  A CTA streams, per window of at most 16 columns, the
//            gate and up rows of those columns and the down weights of the same columns (a
//            K-blocked copy of the down planes makes them one contiguous block) into a ring of
//            shared-memory stages, computes h = silu(g) * u for them and at once their share of
//            the down projection, w_k * W_down[:, cols] h[cols], for all d outputs.  No h leaves
//            the CTA; each CTA ends with a partial output [T][d];                 [grid barrier]
//   phase 4  each CTA sums the #CTA partials of its d / #CTA output rows in CTA order (a fixed
//            order: the run is bit-reproducible), adds the optional residual and writes y.
//
// The arithmetic per product is that of the split-K GEMV path: int4 codes become fp32 0.5 + o/256
// by one byte permute, x' = 256 x, sum q x = sum v x' - 136 sum x, one fp16 group scale per 32.
// Every wait is bounded; on timeout the CTA records MOE status "timeout", stops issuing and
// waits (bounded) for its copies in flight before exiting.
#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace moe {

constexpr int kFzWarps = 16;                     // consumer warps
constexpr int kFzThreads = (kFzWarps + 1) * 32;  // + one producer warp
constexpr int kFzMaxT = 8;
constexpr int kFzMaxStages = 8;
constexpr int kFzUnit = 8;                       // columns per down block and per work unit
constexpr int kFzWin = 16;                       // columns per stage window (one gate/up pair per warp)
constexpr int kFzSmemMax = 227 * 1024;
constexpr int kFzReduceLoads = 8;                // final sum: up to 32 * 8 CTAs
constexpr unsigned kFzSpinLimit = 1u << 24;      // grid-barrier polls, at least 32 ns apart
constexpr unsigned kFzProducerSleep = 200;        // ns between polls of the producer's waits
constexpr unsigned kFzConsumerSleep = 64;         // ns between polls of a waiting consumer warp

struct FusedArgs {
  const void* x;
  int act, T, d, E, K, f, has_shared, prenorm;
  float eps;
  void* xnorm;
  const float* Wr;
  const float* bias;
  float* logits;
  int32_t* idx;
  float* w;
  int32_t* counts;
  int32_t* offs;
  int32_t* perm;
  int32_t* active;
  int32_t* n_active;
  int32_t* stat;
  int4* slots;
  const uint8_t* gu_q;     // [E][2f][d/2] routed gate/up codes (rows 0..f-1 gate, f..2f-1 up)
  const __half* gu_s;      // [E][2f][d/32]
  const uint32_t* dnb_q;   // [E][f/8][d] routed down codes, K-blocked: word = 8 columns of one row
  const __half* dnb_s;     // [E][f/32][d] their scales
  const uint8_t* sh_gu_q;  // the shared expert, same layouts with E = 1
  const __half* sh_gu_s;
  const uint32_t* sh_dnb_q;
  const __half* sh_dnb_s;
  float* part;             // [gridDim.x][T][d] per-CTA partial outputs
  void* y;
  const void* resid;
  unsigned long long* grid_bar;  // grid-barrier arrival counter (only ever increases)
  unsigned* status;
  int ns;                  // ring stages
  int stage_bytes;
};

// ------------------------------------------------------------------ grid barrier
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Consumer-warp barrier (named barrier 1, the 512 consumer threads).
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kFzWarps * 32) : "memory"); }
// The same barrier, returning the AND of v over the consumer threads: every consumer gets the
// same verdict, so branches on it stay uniform across the named barriers that follow.
__device__ __forceinline__ bool consumers_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kFzWarps * 32)
      : "memory");
  return r != 0;
}

// Grid barrier on a 64-bit arrival counter that only ever increases.  At the start (after
// griddepcontrol.wait) one thread per CTA reads the counter and rounds it down to a multiple of
// gridDim.x: the previous launch's barriers are complete and fewer than gridDim.x arrivals of this
// launch's first barrier can precede the read, so every CTA gets the same base.  Barrier i of the launch is
// complete when the counter reaches base + (i + 1) * gridDim.x.  Arrival is a release reduction
// (no reply awaited); the wait polls with acquire loads.
__device__ __forceinline__ void grid_arrive(unsigned long long* bar) {
  __threadfence();
  asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(bar) : "memory");
}
__device__ __forceinline__ bool grid_wait(const unsigned long long* bar, unsigned long long target,
                                          volatile int* abort) {
  for (unsigned n = 0; ld_acquire_gpu(bar) < target; ++n) {
    if (n > kFzSpinLimit || *abort) return false;
    __nanosleep(32);
  }
  return true;
}

// ------------------------------------------------------------------ gate/up dot products
// 2*NP int4 rows against TB tokens of x' (group-interleaved [t][8][G] float4), all in shared memory:
// rows r < NP are gate rows p = r, rows r >= NP up rows p = r - NP, at gq/uq + min-clamped p*qrow
// (rows p >= np repeat row 0), scales at gs/us + p*G.  Lane-partial sums acc[r][tt]; each x' load
// is shared by all rows.  Lane = 32-column groups lane, lane+32, ...
template <int NG, int TB, int NP>
__device__ __forceinline__ void pairs_dot(const uint8_t* gq, const uint8_t* uq, const __half* gs, const __half* us,
                                          size_t qrow, int np, int G, const float4* xq, const float* xs136,
                                          const int (&tok)[TB], float (&acc)[2 * NP][TB], int lane) {
  constexpr int ROWS = 2 * NP;
#pragma unroll
  for (int r = 0; r < ROWS; ++r)
#pragma unroll
    for (int tt = 0; tt < TB; ++tt) acc[r][tt] = 0.f;
#pragma unroll 1
  for (int j = 0; j < NG; ++j) {
    const int g = lane + 32 * j;
    if (g >= G) continue;
    uint4 wq[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const int p = r < NP ? r : r - NP;
      const int pp = p < np ? p : 0;
      wq[r] = *reinterpret_cast<const uint4*>((r < NP ? gq : uq) + pp * qrow + g * 16);
    }
    float part[ROWS][TB];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
      for (int tt = 0; tt < TB; ++tt) part[r][tt] = 0.f;
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
      float4 xa[TB], xb[TB];
#pragma unroll
      for (int tt = 0; tt < TB; ++tt) {
        const float4* xp = xq + (size_t)tok[tt] * 8 * G + g;
        xa[tt] = xp[(2 * wd) * G];
        xb[tt] = xp[(2 * wd + 1) * G];
      }
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        const uint32_t w32 = wd == 0 ? wq[r].x : wd == 1 ? wq[r].y : wd == 2 ? wq[r].z : wq[r].w;
        const uint32_t lo = (w32 & 0x0F0F0F0Fu) ^ 0x08080808u;
        const uint32_t hi = ((w32 >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
        const float v0 = v_lo(lo, 0), v1 = v_lo(hi, 0), v2 = v_lo(lo, 1), v3 = v_lo(hi, 1);
        const float v4 = v_lo(lo, 2), v5 = v_lo(hi, 2), v6 = v_lo(lo, 3), v7 = v_lo(hi, 3);
#pragma unroll
        for (int tt = 0; tt < TB; ++tt) {
          float a2 = part[r][tt];
          a2 = fmaf(v0, xa[tt].x, a2);
          a2 = fmaf(v1, xa[tt].y, a2);
          a2 = fmaf(v2, xa[tt].z, a2);
          a2 = fmaf(v3, xa[tt].w, a2);
          a2 = fmaf(v4, xb[tt].x, a2);
          a2 = fmaf(v5, xb[tt].y, a2);
          a2 = fmaf(v6, xb[tt].z, a2);
          a2 = fmaf(v7, xb[tt].w, a2);
          part[r][tt] = a2;
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < TB; ++tt) {
      const float x136 = xs136[tok[tt] * G + g];
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        const int p = r < NP ? r : r - NP;
        const int pp = p < np ? p : 0;
        const float sc = __half2float((r < NP ? gs : us)[(size_t)pp * G + g]);
        acc[r][tt] = fmaf(sc, part[r][tt] - x136, acc[r][tt]);
      }
    }
  }
}

// ------------------------------------------------------------------ stages
// A stage holds at most kFzWin columns [col, col + n) of one expert, n a multiple of kFzUnit, all
// inside one kFzWin-aligned window (so inside one 32-column scale group of the down weights):
// the n gate rows and n up rows (d/2 code bytes, d/32 fp16 scales each), the n/8 down blocks
// ([d] words of 8 columns) and the [d] down scales of the group.  Byte offsets for d:
struct StageLayout {
  uint32_t uq, gs, us, dq, ds, bytes;
};
__host__ __device__ inline StageLayout stage_layout(int d) {
  const uint32_t qrow = (uint32_t)d / 2, srow = (uint32_t)d / 16;
  StageLayout L;
  L.uq = kFzWin * qrow;
  L.gs = 2u * kFzWin * qrow;
  L.us = L.gs + kFzWin * srow;
  L.dq = L.us + kFzWin * srow;
  L.ds = L.dq + (kFzWin / kFzUnit) * 4u * (uint32_t)d;
  L.bytes = L.ds + 2u * (uint32_t)d;
  return L;
}

// The bulk copies of one stage: expert e of the given planes, columns [col, col + n).
__device__ __forceinline__ void issue_stage(uint8_t* dst, const StageLayout& L, const uint8_t* gu_q,
                                            const __half* gu_s, const uint32_t* dnb_q, const __half* dnb_s, int e,
                                            int col, int n, int d, int f, uint64_t* bar) {
  const size_t qrow = (size_t)d / 2, G = (size_t)d / 32;
  const size_t rg = (size_t)e * 2 * f + col, ru = rg + f;
  const uint32_t nq = (uint32_t)(n * qrow), nsc = (uint32_t)(n * G * 2);
  const uint32_t nd = (uint32_t)(n / kFzUnit) * 4u * (uint32_t)d;
  tc::mbar_arrive_expect_tx(bar, 2 * nq + 2 * nsc + nd + 2u * (uint32_t)d);
  tc::bulk_g2s(dst, gu_q + rg * qrow, nq, bar);
  tc::bulk_g2s(dst + L.uq, gu_q + ru * qrow, nq, bar);
  tc::bulk_g2s(dst + L.gs, gu_s + rg * G, nsc, bar);
  tc::bulk_g2s(dst + L.us, gu_s + ru * G, nsc, bar);
  tc::bulk_g2s(dst + L.dq, dnb_q + ((size_t)e * (f / kFzUnit) + col / kFzUnit) * d, nd, bar);
  tc::bulk_g2s(dst + L.ds, dnb_s + ((size_t)e * (f / 32) + col / 32) * d, 2u * (uint32_t)d, bar);
}

// A CTA's routed work: units [pos, end) of kFzUnit columns, numbered slot-major (slot * f/8 + u).
// Stages are cut at slot boundaries and at kFzWin-column windows.
struct UnitRange {
  int pos, end;
};
__device__ __forceinline__ bool next_stage(UnitRange& r, int fu, int& s, int& col, int& n) {
  if (r.pos >= r.end) return false;
  s = r.pos / fu;
  const int u = r.pos - s * fu;
  constexpr int wu = kFzWin / kFzUnit;
  const int ue = min(min((u / wu + 1) * wu, fu), u + (r.end - r.pos));
  col = u * kFzUnit;
  n = (ue - u) * kFzUnit;
  r.pos += ue - u;
  return true;
}

// h of one column for TB tokens of a slot: the tokens of assignments perm_s[pb + t0 ..] (or, for
// the shared expert, pb < 0, tokens t0 ..); stores 256 * silu(g) * u at hcol[(t0 + tt) * kFzWin].
template <int NG, int TB>
__device__ __forceinline__ void col_h(const uint8_t* gq, const uint8_t* uq, const __half* gs, const __half* us,
                                      size_t qrow, int G, int t0, int pb, int K, const int* perm_s, const float4* xq,
                                      const float* xs136, float* hcol, int lane) {
  int tok[TB];
#pragma unroll
  for (int tt = 0; tt < TB; ++tt) tok[tt] = pb >= 0 ? perm_s[pb + t0 + tt] / K : t0 + tt;
  float acc[2][TB];
  pairs_dot<NG, TB, 1>(gq, uq, gs, us, qrow, 1, G, xq, xs136, tok, acc, lane);
  constexpr int NV = 2 * TB;             // gate values of the TB tokens, then up values
  constexpr int SH = NV == 4 ? 3 : 4;    // value i's total sits in the lanes with lane >> SH == i
  float vals[NV];
#pragma unroll
  for (int tt = 0; tt < TB; ++tt) {
    vals[tt] = acc[0][tt];
    vals[TB + tt] = acc[1][tt];
  }
  const float g = warp_sum_multi<NV>(vals);
  const float u = __shfl_down_sync(0xffffffffu, g, 16);  // the up value of the same token
  if (lane < 16 && (lane & ((1 << SH) - 1)) == 0) hcol[(t0 + (lane >> SH)) * kFzWin] = 256.f * (silu(g) * u);
}

// sum over the 8 columns of one down word (8 int4 codes of one row) of v * h', v = 0.5 + o/256.
__device__ __forceinline__ float dot8(uint32_t w, const float4& ha, const float4& hb, float acc) {
  const uint32_t lo = (w & 0x0F0F0F0Fu) ^ 0x08080808u, hi = ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
  acc = fmaf(v_lo(lo, 0), ha.x, acc);
  acc = fmaf(v_lo(hi, 0), ha.y, acc);
  acc = fmaf(v_lo(lo, 1), ha.z, acc);
  acc = fmaf(v_lo(hi, 1), ha.w, acc);
  acc = fmaf(v_lo(lo, 2), hb.x, acc);
  acc = fmaf(v_lo(hi, 2), hb.y, acc);
  acc = fmaf(v_lo(lo, 3), hb.z, acc);
  acc = fmaf(v_lo(hi, 3), hb.w, acc);
  return acc;
}

// One stage: h of its n columns for the nt tokens of its slot (assignments perm_s[pb ..], weights
// w_s; pb < 0: the shared expert, tokens 0 .. nt-1, weight 1), then the down share of those
// columns, y_s[t][r] += w * sum_{c in stage} W_down[r][c] h[t][c], every thread for its row quads.
// Uniform over the consumer threads (one consumers_sync inside).  hb: [kFzMaxT][kFzWin].
template <int NG>
__device__ __noinline__ void run_stage(const FusedArgs& a, const uint8_t* stg, const StageLayout& L, int n,
                                          int pb, int nt, const int* perm_s, const float* w_s, const float4* xq,
                                          const float* xs136, float* hb, float* y_s, int warp, int lane, int ctid) {
  const int d = a.d, G = d / 32, K = a.K;
  const size_t qrow = (size_t)d / 2;
  if (warp < n) {
    // gate/up: warp w computes column w, two tokens per pass where it can
    const uint8_t* gq = stg + (size_t)warp * qrow;
    const uint8_t* uq = stg + L.uq + (size_t)warp * qrow;
    const __half* gs = reinterpret_cast<const __half*>(stg + L.gs) + (size_t)warp * G;
    const __half* us = reinterpret_cast<const __half*>(stg + L.us) + (size_t)warp * G;
    int t0 = 0;
    for (; t0 + 2 <= nt; t0 += 2) col_h<NG, 2>(gq, uq, gs, us, qrow, G, t0, pb, K, perm_s, xq, xs136, hb + warp, lane);
    if (t0 < nt) col_h<NG, 1>(gq, uq, gs, us, qrow, G, t0, pb, K, perm_s, xq, xs136, hb + warp, lane);
  }
  consumers_sync();
  // down: 4 rows (one 16-byte group of words per block) per thread and pass
  const uint4* dq0 = reinterpret_cast<const uint4*>(stg + L.dq);
  const uint4* dq1 = reinterpret_cast<const uint4*>(stg + L.dq + 4u * (uint32_t)d);
  const uint2* dsq = reinterpret_cast<const uint2*>(stg + L.ds);
  const bool two = n > kFzUnit;
  #pragma unroll 1
  for (int qd = ctid; qd < d / 4; qd += kFzWarps * 32) {
    const uint4 w0 = dq0[qd];
    const uint4 w1 = two ? dq1[qd] : make_uint4(0u, 0u, 0u, 0u);
    const uint2 sv = dsq[qd];
    const float s0 = __half2float(__ushort_as_half((unsigned short)(sv.x & 0xFFFFu)));
    const float s1 = __half2float(__ushort_as_half((unsigned short)(sv.x >> 16)));
    const float s2 = __half2float(__ushort_as_half((unsigned short)(sv.y & 0xFFFFu)));
    const float s3 = __half2float(__ushort_as_half((unsigned short)(sv.y >> 16)));
    #pragma unroll 1
    for (int j = 0; j < nt; ++j) {
      const int as = pb >= 0 ? perm_s[pb + j] : 0;
      const int t = pb >= 0 ? as / K : j;
      const float wt = pb >= 0 ? w_s[as] : 1.f;
      const float4* hp = reinterpret_cast<const float4*>(hb + j * kFzWin);
      const float4 h0 = hp[0], h1 = hp[1];
      float hs = (h0.x + h0.y) + (h0.z + h0.w) + ((h1.x + h1.y) + (h1.z + h1.w));
      float a0 = dot8(w0.x, h0, h1, 0.f), a1 = dot8(w0.y, h0, h1, 0.f);
      float a2 = dot8(w0.z, h0, h1, 0.f), a3 = dot8(w0.w, h0, h1, 0.f);
      if (two) {
        const float4 h2 = hp[2], h3 = hp[3];
        hs += (h2.x + h2.y) + (h2.z + h2.w) + ((h3.x + h3.y) + (h3.z + h3.w));
        a0 = dot8(w1.x, h2, h3, a0);
        a1 = dot8(w1.y, h2, h3, a1);
        a2 = dot8(w1.z, h2, h3, a2);
        a3 = dot8(w1.w, h2, h3, a3);
      }
      // h' = 256 h and v = (q + 136) / 256: sum v h' - 136 sum h = sum q h
      hs *= 136.0f / 256.0f;
      const float ws = wt;
      float4* yp = reinterpret_cast<float4*>(y_s + (size_t)t * d) + qd;
      float4 yv = *yp;
      yv.x = fmaf(ws * s0, a0 - hs, yv.x);
      yv.y = fmaf(ws * s1, a1 - hs, yv.y);
      yv.z = fmaf(ws * s2, a2 - hs, yv.z);
      yv.w = fmaf(ws * s3, a3 - hs, yv.w);
      *yp = yv;
    }
  }
}

template <int NG>
__global__ void __launch_bounds__(kFzThreads, 1) decode_layer_kernel(const FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int T = a.T, d = a.d, E = a.E, K = a.K, f = a.f, G = d / 32;
  const int nc = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = a.ns, SB = a.stage_bytes;
  const StageLayout L = stage_layout(d);
  const int fu = f / kFzUnit, QD = d / 4;

  // this CTA's fixed shares
  const int e0 = (int)((long long)E * c / nc), ne = (int)((long long)E * (c + 1) / nc) - e0;  // router rows
  const int su0 = (int)((long long)fu * c / nc), su1 = (int)((long long)fu * (c + 1) / nc);  // shared units (<= 1)
  const int q0 = (int)((long long)QD * c / nc), q1 = (int)((long long)QD * (c + 1) / nc);    // output row quads
  const bool sh_on = a.has_shared && su1 > su0;

  // shared memory carve (all offsets 16-byte multiples); the router rows use ring stage 1 and the
  // shared-expert stage ring stage 0: both are done with before the routed stages are issued
  uint8_t* ring = smem_raw;
  float4* xq = reinterpret_cast<float4*>(ring + (size_t)NS * SB);  // x' = 256 x, [T][8][G] float4
  float* xs136 = reinterpret_cast<float*>(xq + (size_t)T * 8 * G);  // [T][G]: 136 * (sum of x per group)
  float* y_s = xs136 + (size_t)T * G;                               // [T][d] partial output
  int4* slot_s = reinterpret_cast<int4*>(y_s + (size_t)T * d);      // [T*K]
  int* perm_s = reinterpret_cast<int*>(slot_s + T * K);
  int* idx_s = perm_s + T * K;
  float* w_s = reinterpret_cast<float*>(idx_s + T * K);
  const float* wr_s = reinterpret_cast<const float*>(ring + SB);
  uint8_t* sh_stg = ring;

  __shared__ __align__(8) uint64_t full[kFzMaxStages], empty[kFzMaxStages], wr_full, sh_full, route_ready;
  __shared__ __align__(16) float hbuf[2][kFzMaxT * kFzWin];
  __shared__ float lpart[kFzWarps * kFzMaxT];
  __shared__ int s_srt[kFzMaxT * kMaxK];
  __shared__ float inv_s[kFzMaxT];
  __shared__ volatile int s_abort;
  __shared__ int s_nact, s_issued, s_ok;

  // This launch may start while the previous kernel in the stream is still finishing
  // (programmatic dependent launch): everything before griddepcontrol.wait touches only this CTA's
  // shared memory and read-only weights; activations, workspace and the barrier counter come after.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    #pragma unroll 1
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], kFzWarps);
    }
    tc::mbar_init(&wr_full, 1);
    tc::mbar_init(&sh_full, 1);
    tc::mbar_init(&route_ready, 1);
    s_abort = 0;
    s_issued = 0;
    s_ok = 1;
    tc::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kFzWarps) {
    // ================================================================ producer
    if (lane == 0) {
      if (ne > 0) {
        tc::mbar_arrive_expect_tx(&wr_full, (uint32_t)(ne * d * 4));
        tc::bulk_g2s(ring + SB, a.Wr + (size_t)e0 * d, (uint32_t)(ne * d * 4), &wr_full);
      }
      if (sh_on)
        issue_stage(sh_stg, L, a.sh_gu_q, a.sh_gu_s, a.sh_dnb_q, a.sh_dnb_s, 0, su0 * kFzUnit, kFzUnit, d, f, &sh_full);
      bool ok = tc::mbar_wait_sleepy(&route_ready, 0, &s_abort, kFzProducerSleep);
      int k = 0;
      if (ok) {
        const long long U = (long long)s_nact * fu;
        UnitRange ur{(int)(U * c / nc), (int)(U * (c + 1) / nc)};
        int s, col, n;
        while (next_stage(ur, fu, s, col, n)) {
          const int st = k % NS;
          if (!tc::mbar_wait_sleepy(&empty[st], ((k / NS) & 1) ^ 1u, &s_abort, kFzProducerSleep)) {
            ok = false;
            break;
          }
          issue_stage(ring + (size_t)st * SB, L, a.gu_q, a.gu_s, a.dnb_q, a.dnb_s, slot_s[s].x, col, n, d, f,
                      &full[st]);
          s_issued = ++k;
        }
      }
      if (!ok) {
        atomicOr(a.status, kStatusTimeout);
        s_abort = 1;
      }
    }
    __syncwarp();
  } else {
    // ================================================================ consumers
    const int ctid = threadIdx.x;
    bool ok = true;
    #pragma unroll 1
    for (int i = ctid; i < T * QD; i += kFzWarps * 32) reinterpret_cast<float4*>(y_s)[i] = make_float4(0.f, 0.f, 0.f, 0.f);

    asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous kernel's writes are visible
    // the barrier counter's base: the previous launch's barriers are complete and fewer than
    // gridDim.x arrivals of this launch's first barrier can precede this read
    unsigned long long bar_base = 0;
    if (ctid == 0) bar_base = ld_acquire_gpu(a.grid_bar) / nc * nc;

    // ---- phase 1: x (optionally RMS-normalised) as x' = 256 x, the router rows, the logits
    if (a.prenorm) {
      #pragma unroll 1
      for (int t = warp; t < T; t += kFzWarps) {
        float ss = 0.f;
        #pragma unroll 8
        for (int cc = lane; cc < d / 8; cc += 32) {
          float v[8];
          load8_act(a.x, a.act, (size_t)t * d + cc * 8, v);
#pragma unroll
          for (int q = 0; q < 8; ++q) ss = fmaf(v[q], v[q], ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) inv_s[t] = 1.0f / sqrtf(ss / (float)d + a.eps);
      }
      consumers_sync();
    }
    #pragma unroll 4
    for (int cc = ctid; cc < T * d / 8; cc += kFzWarps * 32) {
      float v[8];
      load8_act(a.x, a.act, (size_t)cc * 8, v);
      const int ti = (cc * 8) / d, kk = cc * 8 - ti * d;
      if (a.prenorm) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          v[q] = round_act(a.act, v[q] * inv_s[ti]);
          if (c == 0) store_act(a.xnorm, a.act, (size_t)cc * 8 + q, v[q]);
        }
      }
      const int g = kk >> 5, m4 = (kk & 31) >> 2;
      float4* dst = xq + ((size_t)ti * 8 + m4) * G + g;
      dst[0] = make_float4(v[0] * 256.f, v[1] * 256.f, v[2] * 256.f, v[3] * 256.f);
      dst[G] = make_float4(v[4] * 256.f, v[5] * 256.f, v[6] * 256.f, v[7] * 256.f);
    }
    consumers_sync();
    #pragma unroll 1
    for (int i = ctid; i < T * G; i += kFzWarps * 32) {
      const int ti = i / G, g = i - ti * G;
      const float* xb = reinterpret_cast<const float*>(xq) + (size_t)ti * 8 * G * 4;
      float sx = 0.f;
      #pragma unroll 1
      for (int m = 0; m < 32; ++m) sx += xb[((m >> 2) * G + g) * 4 + (m & 3)];
      xs136[i] = sx * (136.0f / 256.0f);
    }
    {
      // logits of the router rows [e0, e0 + ne): warp = (row, part of the columns); x' = 256 x,
      // so the dot product is 256 times the wanted one, exactly
      const int ncol = d / 4;
      const int nparts = ne > 0 ? max(1, kFzWarps / ne) : 1;
      const int my_e = warp % max(ne, 1), my_p = warp / max(ne, 1);
      const bool r_on = ne > 0 && my_p < nparts;
      if (ne > 0) ok = tc::mbar_wait_warp(&wr_full, 0, &s_abort, kFzConsumerSleep);
      if (ok && r_on) {
        const int cb = (int)((long long)ncol * my_p / nparts), ce = (int)((long long)ncol * (my_p + 1) / nparts);
        const float4* wr = reinterpret_cast<const float4*>(wr_s) + (size_t)my_e * ncol;
        float acc[kFzMaxT];
#pragma unroll
        for (int t = 0; t < kFzMaxT; ++t) acc[t] = 0.f;
        #pragma unroll 1
        for (int cc = cb + lane; cc < ce; cc += 32) {
          const float4 wv = wr[cc];
          const int g = cc >> 3, m4 = cc & 7;
#pragma unroll
          for (int t = 0; t < kFzMaxT; ++t) {
            if (t < T) {
              const float4 xv = xq[((size_t)t * 8 + m4) * G + g];
              acc[t] = fmaf(wv.x, xv.x, acc[t]);
              acc[t] = fmaf(wv.y, xv.y, acc[t]);
              acc[t] = fmaf(wv.z, xv.z, acc[t]);
              acc[t] = fmaf(wv.w, xv.w, acc[t]);
            }
          }
        }
#pragma unroll
        for (int t = 0; t < kFzMaxT; ++t) {
          if (t < T) {
            const float v = warp_sum(acc[t]);
            if (lane == 0) lpart[warp * kFzMaxT + t] = v;
          }
        }
      }
      if (!ok && lane == 0) s_abort = 1;
      consumers_sync();
      if (ok)
        #pragma unroll 1
        for (int i = ctid; i < ne * T; i += kFzWarps * 32) {
          const int le = i / T, t = i - le * T;
          float v = 0.f;
          #pragma unroll 1
          for (int p = 0; p < nparts; ++p) v += lpart[(p * ne + le) * kFzMaxT + t];
          a.logits[(size_t)t * E + e0 + le] = v * (1.0f / 256.0f) + (a.bias ? a.bias[e0 + le] : 0.f);
        }
      consumers_sync();
      if (ctid == 0) grid_arrive(a.grid_bar);  // always arrive: the other CTAs must not wait on this one
    }

    // ---- the shared expert's columns of this CTA while the other CTAs finish their logits
    if (sh_on) {
      const bool okw = tc::mbar_wait_warp(&sh_full, 0, &s_abort, kFzConsumerSleep);
      ok = consumers_all(ok && okw && !s_abort);
      if (ok) run_stage<NG>(a, sh_stg, L, kFzUnit, -1, T, perm_s, w_s, xq, xs136, hbuf[0], y_s, warp, lane, ctid);
    }
    if (ctid == 0) s_ok = (!s_abort && grid_wait(a.grid_bar, bar_base + nc, &s_abort)) ? 1 : 0;
    consumers_sync();
    ok = consumers_all(ok && s_ok && !s_abort);
    if (!ok && ctid == 0) s_abort = 1;  // the producer stops waiting for the routing

    // ---- phase 2: selection (one warp per token) and dispatch, repeated by every CTA
    if (ok) {
      // the logits as order-preserving keys, [T][32 * ceil(E / 32)] (0 = no expert), in ring stage 0
      // (free until the routed stages are issued); all loads in flight together
      const int EP = (E + 31) & ~31;
      uint32_t* keys = reinterpret_cast<uint32_t*>(ring);
#pragma unroll 4
      for (int i = ctid; i < T * EP; i += kFzWarps * 32) {
        const int t = i / EP, e = i - t * EP;
        keys[i] = e < E ? topk_order_key(__ldcg(a.logits + (size_t)t * E + e)) : 0u;
      }
      consumers_sync();
      if (warp < T) {
        int my_i;
        float my_w;
        topk_warp(keys + (size_t)warp * EP, E, K, my_i, my_w);
        if (lane < K) {
          idx_s[warp * K + lane] = my_i;
          w_s[warp * K + lane] = my_w;
        }
      }
      consumers_sync();
      if (c == 0)
        #pragma unroll 1
        for (int i = ctid; i < T * K; i += kFzWarps * 32) {
          a.idx[i] = idx_s[i];
          a.w[i] = w_s[i];
        }
      {
        // dispatch by counting, one thread per assignment i (n <= 256): its place in the stable
        // counting sort is the number of smaller (expert, i) keys; the distinct experts below its
        // own give its slot
        const int n = T * K;
        int e_i = 0, start = 0, cnt_i = 0, first = 0;
        if (ctid < n) {
          e_i = idx_s[ctid];
          int pos = 0, before = 0;
          #pragma unroll 1
          for (int j = 0; j < n; ++j) {
            const int ej = idx_s[j];
            start += ej < e_i;
            cnt_i += ej == e_i;
            pos += ej < e_i || (ej == e_i && j < ctid);
            before += ej == e_i && j < ctid;
          }
          perm_s[pos] = ctid;
          first = before == 0;
          s_srt[ctid] = first;
        }
        consumers_sync();
        if (ctid < n && first) {
          int slot = 0;
          #pragma unroll 1
          for (int j = 0; j < n; ++j) slot += s_srt[j] && idx_s[j] < e_i;
          slot_s[slot] = make_int4(e_i, start, cnt_i, 0);
        }
        if (ctid == 0) {
          int na = 0;
          #pragma unroll 1
          for (int j = 0; j < n; ++j) na += s_srt[j];
          s_nact = na;
        }
        consumers_sync();
        if (c == 0) {
          // the full outputs: offs[e] = assignments with an expert below e
          const int na = s_nact;
          #pragma unroll 1
          for (int e = ctid; e <= E; e += kFzWarps * 32) {
            int o = 0, ce = 0;
            #pragma unroll 1
            for (int q = 0; q < n; ++q) {
              o += idx_s[q] < e;
              ce += idx_s[q] == e;
            }
            a.offs[e] = o;
            if (e < E) a.counts[e] = ce;
          }
          #pragma unroll 1
          for (int q = ctid; q < na; q += kFzWarps * 32) {
            a.active[q] = slot_s[q].x;
            a.slots[q] = slot_s[q];
          }
          #pragma unroll 1
          for (int q = ctid; q < n; q += kFzWarps * 32) a.perm[q] = perm_s[q];
          if (ctid == 0) {
            *a.n_active = na;
            if (a.stat) *a.stat = na;
          }
        }
      }
      if (ctid == 0) tc::mbar_arrive(&route_ready);  // the producer may now stream routed experts
    }

    // ---- phase 3: this CTA's routed units through the ring
    if (ok) {
      const long long U = (long long)s_nact * fu;
      UnitRange ur{(int)(U * c / nc), (int)(U * (c + 1) / nc)};
      int s, col, n, k = 0;
      while (next_stage(ur, fu, s, col, n)) {
        const int st = k % NS;
        const bool okw = tc::mbar_wait_warp(&full[st], (k / NS) & 1, &s_abort, kFzConsumerSleep);
        ok = consumers_all(okw && !s_abort);
        if (!ok) break;
        const int4 sl = slot_s[s];
        run_stage<NG>(a, ring + (size_t)st * SB, L, n, sl.y, sl.z, perm_s, w_s, xq, xs136, hbuf[k & 1], y_s, warp,
                      lane, ctid);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[st]);
        ++k;
      }
    }
    if (!ok && ctid == 0) s_abort = 1;

    // ---- the partial output of this CTA, then the second grid barrier
    consumers_sync();
    if (ok) {
      float4* pp = reinterpret_cast<float4*>(a.part + (size_t)c * T * d);
      const float4* ys = reinterpret_cast<const float4*>(y_s);
      #pragma unroll 1
      for (int i = ctid; i < T * QD; i += kFzWarps * 32) pp[i] = ys[i];
    }
    consumers_sync();
    if (ctid == 0) {
      grid_arrive(a.grid_bar);  // always arrive: the other CTAs must not wait on this one
      s_ok = (!s_abort && grid_wait(a.grid_bar, bar_base + 2ull * nc, &s_abort)) ? 1 : 0;
    }
    consumers_sync();
    ok = consumers_all(ok && s_ok && !s_abort);
    if (!ok && ctid == 0) s_abort = 1;

    // ---- phase 4: rows [4 q0, 4 q1) of y = sum of the partials in CTA order (+ residual)
    if (ok) {
      const int nq = q1 - q0;
      #pragma unroll 1
      for (int it = warp; it < T * nq; it += kFzWarps) {
        const int t = it / nq, qd = q0 + (it - t * nq);
        // all of the lane's loads in flight at once (gridDim.x <= 32 * kFzReduceLoads)
        float4 pv[kFzReduceLoads];
#pragma unroll
        for (int i = 0; i < kFzReduceLoads; ++i) {
          const int cc = lane + 32 * i;
          pv[i] = cc < nc ? __ldcg(reinterpret_cast<const float4*>(a.part + ((size_t)cc * T + t) * d) + qd)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kFzReduceLoads; ++i) {
          v[0] += pv[i].x;
          v[1] += pv[i].y;
          v[2] += pv[i].z;
          v[3] += pv[i].w;
        }
        const float sum = warp_sum_multi<4>(v);  // component i in the lanes with (lane >> 3) == i
        if ((lane & 7) == 0) {
          const size_t o = (size_t)t * d + 4 * qd + (lane >> 3);
          float yv = sum;
          if (a.resid) yv = load_act(a.resid, a.act, o) + yv;
          store_act(a.y, a.act, o, yv);
        }
      }
    } else if (ctid == 0) {
      atomicOr(a.status, kStatusTimeout);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) {
    // copies still in flight must land before the CTA's shared memory goes away
    volatile int never = 0;
    const int issued = s_issued;
    for (int kk = issued - 1; kk >= 0 && kk >= issued - NS; --kk)  // the last copy of every stage
      tc::mbar_wait(&full[kk % NS], (kk / NS) & 1, &never, 2000000000ll);
    if (ne > 0) tc::mbar_wait(&wr_full, 0, &never, 2000000000ll);
    if (sh_on) tc::mbar_wait(&sh_full, 0, &never, 2000000000ll);
  }
}

// ------------------------------------------------------------------ K-blocked copy of the down planes
// out_q[e][b][r] = the 4 code bytes of columns 8b .. 8b+7 of row r (row-major [E][d][f/2] input);
// out_s[e][g][r] = the scale of group g of row r.  A word keeps the input's nibble order.
__global__ void repack_down_kernel(const uint8_t* dn_q, const __half* dn_s, int n_exp, int d, int f, uint32_t* out_q,
                                   __half* out_s) {
  const size_t fu = (size_t)f / kFzUnit, fg = (size_t)f / 32;
  const size_t nq = (size_t)n_exp * fu * d, nsc = (size_t)n_exp * fg * d;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nq; i += stride) {
    const size_t r = i % d, eb = i / d, b = eb % fu, e = eb / fu;
    out_q[i] = *reinterpret_cast<const uint32_t*>(dn_q + (e * d + r) * (f / 2) + 4 * b);
  }
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nsc; i += stride) {
    const size_t r = i % d, eg = i / d, g = eg % fg, e = eg / fg;
    out_s[i] = dn_s[(e * d + r) * fg + g];
  }
}

cudaError_t repack_down_blocked(const void* dn_q, const void* dn_s, int n_exp, int d, int f, void* out_q, void* out_s,
                                cudaStream_t st) {
  repack_down_kernel<<<1024, 256, 0, st>>>(static_cast<const uint8_t*>(dn_q), static_cast<const __half*>(dn_s), n_exp,
                                           d, f, static_cast<uint32_t*>(out_q), static_cast<__half*>(out_s));
  return cudaGetLastError();
}

// ------------------------------------------------------------------ self-test of the bounded waits
// One CTA: thread 0 waits on an mbarrier nobody arrives at and on a barrier counter nobody bumps,
// each with a small budget, exactly as the layer kernels wait.  Bit 0 of *result: the mbarrier
// wait gave up; bit 1: the counter wait gave up; bit 2: a wait returned success (a bug).
__global__ void bounded_wait_selftest_kernel(unsigned long long* counter, long long budget, unsigned* result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int never;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    never = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned r = 0;
    if (!tc::mbar_wait(&bar, 0, &never, budget)) r |= 1u; else r |= 4u;
    // the counter never reaches this target; the poll limit bounds the wait
    const unsigned long long target = ld_acquire_gpu(counter) + (1ull << 40);
    bool ok = true;
    for (unsigned n = 0; ok && ld_acquire_gpu(counter) < target; ++n) {
      if (n > (unsigned)(budget >> 6)) ok = false;
      __nanosleep(32);
    }
    r |= ok ? 4u : 2u;
    *result = r;
    if (r & 3u) atomicOr(result + 1, kStatusTimeout);
  }
}

cudaError_t launch_bounded_wait_selftest(unsigned long long* counter, long long budget, unsigned* result,
                                         cudaStream_t st) {
  bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(counter, budget, result);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ host side
constexpr int kFzStaticSlack = 8192;  // static shared memory of the kernel and the driver's share

struct FusedPlan {
  int ns, stage_bytes, smem;
};

static size_t up16(size_t n) { return (n + 15) & ~size_t(15); }

static FusedPlan fused_plan(int T, int d, int f, int E, int K) {
  (void)f;
  (void)E;
  FusedPlan p{};
  p.stage_bytes = (int)((stage_layout(d).bytes + 127u) & ~127u);
  const size_t G = (size_t)d / 32;
  const size_t fixed = up16((size_t)T * d * 4) + up16((size_t)T * G * 4) + up16((size_t)T * d * 4) +
                       up16((size_t)T * K * 16) + 3 * up16((size_t)T * K * 4);
  const long long room = (long long)kFzSmemMax - kFzStaticSlack - (long long)fixed;
  p.ns = room > 0 ? (int)std::min<long long>(kFzMaxStages, room / p.stage_bytes) : 0;
  p.smem = (int)((size_t)p.ns * p.stage_bytes + fixed);
  return p;
}

static int g_fz_sms = 0;

template <int NG>
static const void* fused_fn() {
  return (const void*)decode_layer_kernel<NG>;
}

cudaError_t fused_kernels_init(int num_sms) {
  g_fz_sms = num_sms;
  const void* fns[3] = {fused_fn<1>(), fused_fn<2>(), fused_fn<4>()};
  for (const void* fn : fns) {
    cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kFzSmemMax - kFzStaticSlack);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Whether the one-launch layer serves this shape (int4 weights) with up to T tokens.
bool fused_shape_ok(int T, int d, int f, int E, int K) {
  const int nc = g_fz_sms;
  if (nc <= 0 || nc > 32 * kFzReduceLoads || T < 1 || T > kFzMaxT) return false;
  if (d % 256 || d > 4096 || f % 32 || f > 1024 || E > kMaxE || K > kMaxK) return false;
  if (f / kFzUnit > nc) return false;         // at most one shared-expert unit per CTA
  if (T * K > kFzWarps * 32) return false;    // dispatch: one thread per assignment
  const FusedPlan p = fused_plan(T, d, f, E, K);
  if (p.ns < 2) return false;                 // the router rows and the shared stage use stages 0 and 1
  if ((size_t)T * ((E + 31) & ~31) * 4 > (size_t)p.stage_bytes) return false;  // the selection's scratch
  return (size_t)((E + nc - 1) / nc) * d * 4 <= (size_t)p.stage_bytes;
}

// Bytes of the K-blocked down copy of n_exp experts: codes, then scales (256-byte aligned parts).
size_t fused_down_copy_bytes(int n_exp, int d, int f) {
  const size_t q = ((size_t)n_exp * d * (f / 2) + 255) & ~size_t(255);
  const size_t s = ((size_t)n_exp * d * (f / 16) + 255) & ~size_t(255);
  return q + s;
}

cudaError_t launch_decode_fused(const RouteArgs& r, const ExpertArgs& x, const FusedExtra& fx, cudaStream_t st) {
  FusedArgs a;
  a.x = r.x;
  a.act = r.act;
  a.T = r.T;
  a.d = r.d;
  a.E = r.E;
  a.K = r.K;
  a.f = x.f;
  a.has_shared = x.has_shared;
  a.prenorm = r.prenorm;
  a.eps = r.eps;
  a.xnorm = r.xnorm;
  a.Wr = r.Wr;
  a.bias = r.bias;
  a.logits = r.logits;
  a.idx = r.idx;
  a.w = r.w;
  a.counts = r.counts;
  a.offs = r.offs;
  a.perm = r.perm;
  a.active = r.active;
  a.n_active = r.n_active;
  a.stat = r.stat;
  a.slots = r.slots;
  a.gu_q = static_cast<const uint8_t*>(x.gu_q);
  a.gu_s = x.gu_s;
  a.dnb_q = static_cast<const uint32_t*>(fx.dnb_q);
  a.dnb_s = static_cast<const __half*>(fx.dnb_s);
  a.sh_gu_q = static_cast<const uint8_t*>(x.sh_gu_q);
  a.sh_gu_s = x.sh_gu_s;
  a.sh_dnb_q = static_cast<const uint32_t*>(fx.sh_dnb_q);
  a.sh_dnb_s = static_cast<const __half*>(fx.sh_dnb_s);
  a.part = fx.part;
  a.y = x.y;
  a.resid = x.resid;
  a.grid_bar = fx.grid_bar;
  a.status = r.status;
  const FusedPlan p = fused_plan(r.T, r.d, x.f, r.E, r.K);
  a.ns = p.ns;
  a.stage_bytes = p.stage_bytes;
  const int G = r.d / 32;
  const void* fn = G <= 32 ? fused_fn<1>() : G <= 64 ? fused_fn<2>() : fused_fn<4>();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g_fz_sms);
  cfg.blockDim = dim3(kFzThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  // One CTA per SM (shared memory and registers allow no second), grid = #SMs, and nothing else
  // in the stream runs beside it, so all CTAs are resident; the grid barriers are bounded anyway.
  // The launch may overlap the tail of the previous kernel in the stream (its prologue only reads
  // weights); griddepcontrol.wait orders everything else.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[1] = {&a};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace moe
