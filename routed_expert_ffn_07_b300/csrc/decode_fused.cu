// Decode / verify layer in one launch (sm_103a): router logits, softmax + top-K, dispatch, the
// gate/up and down projections of the selected and shared experts on tensor cores, and the
// fixed-order combine.
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
//            into #CTA contiguous ranges.  A CTA streams its units with one bulk copy per stage
//            (plus the stage's down scales) from the layer's decode-layout copy into a ring of
//            shared-memory stages and runs, per stage, gate/up as m16n8k16 tensor-core tiles
//            (16 rows = 8 gate + 8 up rows of a unit, N = the slot's tokens), h = w silu(g) u in
//            fp16, and the down share of those columns for all d outputs as m16n8k8 tiles into
//            fp32 accumulators that stay in registers; each CTA ends with a partial [T][d]; [grid barrier]
//   phase 4  each CTA sums the #CTA partials of its d / #CTA output rows in CTA order (a fixed
//            order: the run is bit-reproducible), adds the optional residual and writes y.
//
// Tensor-core operands: int4 codes become fp16 q exactly (two bit operations and one f16x2
// subtract per pair), x is fp16 (bf16 activations are exact in fp16 inside its range) and
// w * h is rounded once to fp16; every group of 32 codes is summed in fp32 and scaled by its
// fp16 group scale in fp32.  Every wait is bounded; on timeout the CTA records MOE status
// "timeout", stops issuing and waits (bounded) for its copies in flight before exiting.
#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace moe {

constexpr int kFzWarps = 16;                     // consumer warps
constexpr int kFzThreads = (kFzWarps + 1) * 32;  // + one producer warp
constexpr int kFzMaxT = 8;                       // tokens: the N of the tensor-core tiles
constexpr int kFzMaxStages = 8;
constexpr int kFzUnit = 8;                       // columns per work unit
constexpr int kFzStageUnits = 2;                 // units per stage (inside one 32-column group)
constexpr int kFzSmemMax = 227 * 1024;
constexpr int kFzReduceLoads = 8;                // final sum: up to 32 * 8 CTAs
constexpr unsigned kFzSpinLimit = 1u << 24;      // grid-barrier polls, at least 32 ns apart
constexpr unsigned kFzProducerSleep = 200;        // ns between polls of the producer's waits
constexpr unsigned kFzConsumerSleep = 64;         // ns between polls of a waiting consumer warp

// ------------------------------------------------------------------ decode layout
// The one-launch layer reads its own copy of each layer's experts, written by moe_set_layer in
// the order of its tensor-core fragments (same bytes as the row-major planes; codes stored as
// offset binary o = q + 8).  Per expert, f/8 unit blocks of dl_unit_bytes(d) each, unit u =
// columns 8u .. 8u+7:
//   gate/up part, per k-tile kt < d/128 (128 columns of K), 1152 bytes:
//     codes [half 2][lane 32][j 4] u32 (a warp's 16-byte loads of one half are contiguous): lane =
//       4g + t; half 0 = gate row 8u + g, half 1 = up row f + 8u + g; the word = the 8 codes of
//       columns 32 (4 kt + j) + 8t .. + 7 of that row (code i in bits 4i .. 4i + 3);
//     scales [g 8][half 2][j 4] fp16 at byte 1024: group 4 kt + j of those rows;
//   down part, 4d bytes, [pair p < d/32][lane 32] u32: rows 32p .. 32p + 31 of the down matrix,
//     columns 8u + 2t (bits 0-3, 4-7, 8-11, 12-15) and 8u + 2t + 1 (bits 16-19 .. 28-31) of rows
//     32p + g, 32p + g + 8, 32p + 16 + g, 32p + 24 + g.
// The down scales follow all unit blocks: per expert [group f/32][warp 16][g 8][tile i < d/256]
// [r 2] fp16 = the scale of down row w d/16 + 16 i + g + 8 r.
__host__ __device__ inline size_t dl_gu_bytes(int d) { return (size_t)(d / 128) * 1152; }
__host__ __device__ inline size_t dl_unit_bytes(int d) { return dl_gu_bytes(d) + (size_t)d * 4; }
__host__ __device__ inline size_t dl_expert_bytes(int d, int f) { return (size_t)(f / kFzUnit) * dl_unit_bytes(d); }
__host__ __device__ inline size_t dl_scale_bytes(int d, int f) { return (size_t)(f / 32) * d * 2; }

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
  const uint8_t* dl;       // routed experts, decode layout: [E] expert blocks
  const uint8_t* dls;      // their down scales: [E][dl_scale_bytes]
  const uint8_t* sh_dl;    // the shared expert, same layouts
  const uint8_t* sh_dls;
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
  // release at GPU scope; cumulative, so it also orders the writes of the CTA's other threads that
  // precede it through the CTA barrier the caller passed
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

// ------------------------------------------------------------------ tensor-core helpers
// D += A B for one m16n8k16 (A 16x16 row-major fp16, B 16x8 fp16, fp32 accumulators) and one
// m16n8k8 tile, in the register fragments of the PTX mma.sync description: lane = 4g + t holds
// A rows g and g + 8, B column g, C rows g and g + 8 at columns 2t and 2t + 1.
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_1688(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// Two offset-binary int4 codes of a word as the fp16 pair (q, q'), q = o - 8, exact: q_lo takes
// the codes in bits 0-3 and 16-19 (1024 + o through the exponent of 1024, minus 1032), q_hi those
// in bits 4-7 and 20-23 (1024 + 16 o, times 1/16, minus 72).
__device__ __forceinline__ uint32_t q_lo(uint32_t w) {
  const uint32_t p = (w & 0x000F000Fu) | 0x64006400u;
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(p), "r"(0x64086408u));  // 1032
  return r;
}
__device__ __forceinline__ uint32_t q_hi(uint32_t w) {
  const uint32_t p = (w & 0x00F000F0u) | 0x64006400u;
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(p), "r"(0x2C002C00u), "r"(0xD480D480u));  // 1/16, -72
  return r;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);  // lo in the low 16 bits
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float half_of(uint32_t v, int hi) {
  return __half2float(__ushort_as_half((unsigned short)(hi ? (v >> 16) : (v & 0xFFFFu))));
}

// A CTA's routed work: units [pos, end) of kFzUnit columns, numbered slot-major (slot * f/8 + u).
// Stages are cut at slot boundaries and at kFzStageUnits-unit windows (inside one 32-column
// scale group of the down weights).
struct UnitRange {
  int pos, end;
};
__device__ __forceinline__ bool next_stage(UnitRange& r, int fu, int& s, int& u0, int& nu) {
  if (r.pos >= r.end) return false;
  s = r.pos / fu;
  const int u = r.pos - s * fu;
  const int ue = min(min((u / kFzStageUnits + 1) * kFzStageUnits, fu), u + (r.end - r.pos));
  u0 = u;
  nu = ue - u;
  r.pos += nu;
  return true;
}

// The two bulk copies of a stage: units [u0, u0 + nu) of one expert (its unit blocks at dl, its
// down scales at dls) into dst; the scales of the units' group go after kFzStageUnits blocks.
__device__ __forceinline__ void issue_stage(uint8_t* dst, const uint8_t* dl, const uint8_t* dls, int u0, int nu,
                                            int d, uint64_t* bar) {
  const size_t ub = dl_unit_bytes(d);
  const uint32_t nb = (uint32_t)(nu * ub), sb = (uint32_t)(2 * d);
  tc::mbar_arrive_expect_tx(bar, nb + sb);
  tc::bulk_g2s(dst, dl + (size_t)u0 * ub, nb, bar);
  tc::bulk_g2s(dst + kFzStageUnits * ub, dls + (size_t)(u0 / 4) * 2 * d, sb, bar);
}

// Gate/up of a stage: warp w takes the items i = w + 16 m < nu * d/128 (unit i % nu, k-tile
// i / nu) and leaves its fp32 partial tile in pgu[w][lane]: rows g (gate of column 8u + g) and
// g + 8 (up), slot-local tokens 2t and 2t + 1.  xtok: the global token of slot-local token g
// (lane >> 2), or -1 past the slot's tokens; xh: x as fp16 fragments [T][d/32][t 4][4 pairs].
__device__ __forceinline__ void gu_stage(const uint8_t* stg, int nu, int d, int xtok, const uint4* xh, float4* pgu,
                                         int warp, int lane) {
  const int KT = d / 128, G = d / 32, t = lane & 3;
  const size_t ub = dl_unit_bytes(d);
  const int items = nu * KT;
  if (warp >= items) return;
  const int u = warp % nu;
  float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int i = warp; i < items; i += kFzWarps) {
    const int kt = i / nu;
    const uint8_t* blk = stg + u * ub + (size_t)kt * 1152;
    const uint4 wg = *reinterpret_cast<const uint4*>(blk + lane * 16);
    const uint4 wu = *reinterpret_cast<const uint4*>(blk + 512 + lane * 16);
    const uint4 sc = *reinterpret_cast<const uint4*>(blk + 1024 + (lane >> 2) * 16);
    uint4 xb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      xb[j] = xtok >= 0 ? xh[((size_t)xtok * G + 4 * kt + j) * 4 + t] : make_uint4(0u, 0u, 0u, 0u);
    // the four groups' tiles first (independent), their scales after
    float dg[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w0 = j == 0 ? wg.x : j == 1 ? wg.y : j == 2 ? wg.z : wg.w;
      const uint32_t w1 = j == 0 ? wu.x : j == 1 ? wu.y : j == 2 ? wu.z : wu.w;
      dg[j][0] = dg[j][1] = dg[j][2] = dg[j][3] = 0.f;
      // k-step 0: codes 0, 4 (K slots 2t, 2t+1) and 1, 5 (2t+8, 2t+9); k-step 1: codes 2, 6 and 3, 7
      mma_16816(dg[j], q_lo(w0), q_lo(w1), q_hi(w0), q_hi(w1), xb[j].x, xb[j].y);
      mma_16816(dg[j], q_lo(w0 >> 8), q_lo(w1 >> 8), q_hi(w0 >> 8), q_hi(w1 >> 8), xb[j].z, xb[j].w);
    }
    const float2 g01 = __half22float2(*reinterpret_cast<const __half2*>(&sc.x));  // [half][j] fp16
    const float2 g23 = __half22float2(*reinterpret_cast<const __half2*>(&sc.y));
    const float2 u01 = __half22float2(*reinterpret_cast<const __half2*>(&sc.z));
    const float2 u23 = __half22float2(*reinterpret_cast<const __half2*>(&sc.w));
    const float sg[4] = {g01.x, g01.y, g23.x, g23.y}, su[4] = {u01.x, u01.y, u23.x, u23.y};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      c[0] = fmaf(sg[j], dg[j][0], c[0]);
      c[1] = fmaf(sg[j], dg[j][1], c[1]);
      c[2] = fmaf(su[j], dg[j][2], c[2]);
      c[3] = fmaf(su[j], dg[j][3], c[3]);
    }
  }
  pgu[warp * 32 + lane] = make_float4(c[0], c[1], c[2], c[3]);
}

// h of a stage, once the gate/up partials are in: thread (u, n, col) of n_u * 64 writes
// hb[u][n][col] = w silu(gate) up as fp16 for global token n and column 8u + col, where the
// slot-local token j of token n holds the weight w (perm_s[pb + j], w_s); 0 for tokens outside
// the slot.  pb < 0: the shared expert, slot-local token = global token < nt, weight 1.  The
// partials of a unit are summed over its warps in warp order.
__device__ __forceinline__ void h_stage(int nu, int d, int pb, int nt, int K, const int* perm_s, const float* w_s,
                                        const float4* pgu, __half* hb, int ctid) {
  if (ctid >= nu * 64) return;
  const int u = ctid >> 6, n = (ctid >> 3) & 7, col = ctid & 7;
  int j = -1;
  float wt = 1.f;
  if (pb < 0) {
    if (n < nt) j = n;
  } else {
#pragma unroll 1
    for (int q = 0; q < nt; ++q)
      if (perm_s[pb + q] / K == n) {
        j = q;
        wt = w_s[perm_s[pb + q]];
      }
  }
  float hv = 0.f;
  if (j >= 0) {
    const int items = nu * (d / 128);
    const int ln = col * 4 + (j >> 1);
    float g = 0.f, up = 0.f;
#pragma unroll 1
    for (int w = u; w < kFzWarps && w < items; w += nu) {
      const float4 p = pgu[w * 32 + ln];
      g += (j & 1) ? p.y : p.x;
      up += (j & 1) ? p.w : p.z;
    }
    hv = wt * (silu(g) * up);
  }
  hb[(u * 8 + n) * 8 + col] = __float2half_rn(hv);
}

// Down share of a stage for the warp's TPW row tiles (rows w d/16 + 16 i + g, + 8): D over the
// stage's (at most two) units as one K = 16 tile, all loads first, then C += s D in fp32.
template <int TPW>
__device__ __forceinline__ void dn_stage(const uint8_t* stg, int nu, int d, const __half* hb, float (&C)[TPW][4],
                                          int warp, int lane) {
  const size_t ub = dl_unit_bytes(d), gb = dl_gu_bytes(d);
  const int g = lane >> 2, t = lane & 3;
  float D[TPW][4];
#pragma unroll
  for (int i = 0; i < TPW; ++i) D[i][0] = D[i][1] = D[i][2] = D[i][3] = 0.f;
  uint32_t w[2][TPW / 2], b[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    b[u] = u < nu ? *reinterpret_cast<const uint32_t*>(hb + (u * 8 + g) * 8 + 2 * t) : 0u;
    const uint32_t* dw = reinterpret_cast<const uint32_t*>(stg + u * ub + gb) + (size_t)warp * (TPW / 2) * 32 + lane;
#pragma unroll
    for (int ip = 0; ip < TPW / 2; ++ip) w[u][ip] = u < nu ? dw[ip * 32] : 0x88888888u;
  }
  // one m16n8k16 per tile: K slots 0-7 are unit 0's columns, 8-15 unit 1's (codes -8 and h 0 when
  // the stage has one unit)
#pragma unroll
  for (int ip = 0; ip < TPW / 2; ++ip) {
    mma_16816(D[2 * ip], q_lo(w[0][ip]), q_hi(w[0][ip]), q_lo(w[1][ip]), q_hi(w[1][ip]), b[0], b[1]);
    mma_16816(D[2 * ip + 1], q_lo(w[0][ip] >> 8), q_hi(w[0][ip] >> 8), q_lo(w[1][ip] >> 8), q_hi(w[1][ip] >> 8), b[0],
              b[1]);
  }
  const uint32_t* sp = reinterpret_cast<const uint32_t*>(stg + kFzStageUnits * ub) + ((size_t)warp * 8 + g) * TPW;
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    const uint32_t s = sp[i];
    const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&s));
    C[i][0] = fmaf(sf.x, D[i][0], C[i][0]);
    C[i][1] = fmaf(sf.x, D[i][1], C[i][1]);
    C[i][2] = fmaf(sf.y, D[i][2], C[i][2]);
    C[i][3] = fmaf(sf.y, D[i][3], C[i][3]);
  }
}
// One stage: gate/up partials, h, down.  Uniform over the consumer threads (two consumers_sync).
template <int TPW>
__device__ __forceinline__ void run_stage(const uint8_t* stg, int nu, int d, int pb, int nt, int K, const int* perm_s,
                                          const float* w_s, const uint4* xh, float4* pgu, __half* hb,
                                          float (&C)[TPW][4], int warp, int lane, int ctid) {
  const int gl = lane >> 2;
  const int xtok = gl < nt ? (pb >= 0 ? perm_s[pb + gl] / K : gl) : -1;
  gu_stage(stg, nu, d, xtok, xh, pgu, warp, lane);
  consumers_sync();
  h_stage(nu, d, pb, nt, K, perm_s, w_s, pgu, hb, ctid);
  consumers_sync();
  dn_stage<TPW>(stg, nu, d, hb, C, warp, lane);
}

template <int TPW>
__global__ void __launch_bounds__(kFzThreads, 1) decode_layer_kernel(const FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int T = a.T, d = a.d, E = a.E, K = a.K, f = a.f, G = d / 32;
  const int nc = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = a.ns, SB = a.stage_bytes;
  const int fu = f / kFzUnit, QD = d / 4;
  const size_t eb = dl_expert_bytes(d, f), sbytes = dl_scale_bytes(d, f);

  // this CTA's fixed shares
  const int e0 = (int)((long long)E * c / nc), ne = (int)((long long)E * (c + 1) / nc) - e0;  // router rows
  const int su0 = (int)((long long)fu * c / nc), su1 = (int)((long long)fu * (c + 1) / nc);  // shared units (<= 1)
  const int q0 = (int)((long long)QD * c / nc), q1 = (int)((long long)QD * (c + 1) / nc);    // output row quads
  const bool sh_on = a.has_shared && su1 > su0;

  // shared memory carve (all offsets 16-byte multiples); the router rows use ring stage 1, the
  // shared-expert stage and the selection's keys ring stage 0: all are done with before the
  // routed stages are issued
  uint8_t* ring = smem_raw;
  float* x32 = reinterpret_cast<float*>(ring + (size_t)NS * SB);     // [T][d] x (optionally normalised)
  uint4* xh = reinterpret_cast<uint4*>(x32 + (size_t)T * d);          // [T][G][4][4 fp16 pairs]
  float4* pgu = reinterpret_cast<float4*>(xh + (size_t)T * G * 4);   // [16 warps][32 lanes]
  int4* slot_s = reinterpret_cast<int4*>(pgu + kFzWarps * 32);       // [T*K]
  int* perm_s = reinterpret_cast<int*>(slot_s + T * K);
  int* idx_s = perm_s + T * K;
  float* w_s = reinterpret_cast<float*>(idx_s + T * K);
  const float* wr_s = reinterpret_cast<const float*>(ring + SB);
  uint8_t* sh_stg = ring;

  __shared__ __align__(8) uint64_t full[kFzMaxStages], empty[kFzMaxStages], wr_full, sh_full, route_ready;
  __shared__ __align__(8) uint64_t logits_done, bar1_done;
  __shared__ unsigned long long s_bar_base;
  __shared__ volatile int s_ok1;
  __shared__ __align__(16) __half hb[kFzStageUnits * 8 * 8];
  __shared__ float lpart[kFzWarps * kFzMaxT];
  __shared__ int s_srt[kFzMaxT * kMaxK];
  __shared__ float inv_s[kFzMaxT];
  __shared__ volatile int s_abort;
  __shared__ int s_nact, s_issued, s_ok, s_ncand;
  __shared__ uint32_t s_wmax[kFzWarps], s_tau;
  __shared__ float s_zp[kFzWarps], s_m;
  __shared__ uint2 s_sel[kMaxK];

  // This launch may start while the previous kernel in the stream is still finishing
  // (programmatic dependent launch): everything before griddepcontrol.wait touches only this CTA's
  // shared memory and read-only weights; activations, workspace and the barrier counter come after.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], kFzWarps);
    }
    tc::mbar_init(&wr_full, 1);
    tc::mbar_init(&sh_full, 1);
    tc::mbar_init(&route_ready, 1);
    tc::mbar_init(&logits_done, 1);
    tc::mbar_init(&bar1_done, 1);
    s_ok1 = 0;
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
      if (sh_on) issue_stage(sh_stg, a.sh_dl, a.sh_dls, su0, 1, d, &sh_full);
      // the first grid barrier on the consumers' behalf: they go on with the shared expert while the
      // release of their logits and the polling run here
      const bool got = tc::mbar_wait_sleepy(&logits_done, 0, &s_abort, 32);
      grid_arrive(a.grid_bar);  // always arrive: the other CTAs must not wait on this one
      s_ok1 = (got && !s_abort && grid_wait(a.grid_bar, s_bar_base + nc, &s_abort)) ? 1 : 0;
      tc::mbar_arrive(&bar1_done);
      bool ok = tc::mbar_wait_sleepy(&route_ready, 0, &s_abort, 32);
      int k = 0;
      if (ok) {
        const long long U = (long long)s_nact * fu;
        UnitRange ur{(int)(U * c / nc), (int)(U * (c + 1) / nc)};
        int s, u0, nu;
        while (next_stage(ur, fu, s, u0, nu)) {
          const int st = k % NS;
          if (!tc::mbar_wait_sleepy(&empty[st], ((k / NS) & 1) ^ 1u, &s_abort, kFzProducerSleep)) {
            ok = false;
            break;
          }
          const int e = slot_s[s].x;
          issue_stage(ring + (size_t)st * SB, a.dl + (size_t)e * eb, a.dls + (size_t)e * sbytes, u0, nu, d, &full[st]);
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
    float C[TPW][4];  // this warp's down rows w d/16 + 16 i + g (+ 8), tokens 2t, 2t + 1
#pragma unroll
    for (int i = 0; i < TPW; ++i) C[i][0] = C[i][1] = C[i][2] = C[i][3] = 0.f;

    asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous kernel's writes are visible
    // the barrier counter's base: the previous launch's barriers are complete and fewer than
    // gridDim.x arrivals of this launch's first barrier can precede this read
    unsigned long long bar_base = 0;
    if (ctid == 0) {
      bar_base = ld_acquire_gpu(a.grid_bar) / nc * nc;
      s_bar_base = bar_base;  // published to the producer with the logits_done arrival
    }

    // ---- phase 1: x (optionally RMS-normalised) in fp32 and as fp16 fragments, the logits
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
      float4* xf = reinterpret_cast<float4*>(x32 + (size_t)cc * 8);
      xf[0] = make_float4(v[0], v[1], v[2], v[3]);
      xf[1] = make_float4(v[4], v[5], v[6], v[7]);
      // fragment order of columns 8w .. 8w+7 of group g: pairs (0,4), (1,5), (2,6), (3,7)
      const int g = kk >> 5, w = (kk & 31) >> 3;
      uint4 hv;
      hv.x = pack_h2(v[0], v[4]);
      hv.y = pack_h2(v[1], v[5]);
      hv.z = pack_h2(v[2], v[6]);
      hv.w = pack_h2(v[3], v[7]);
      xh[((size_t)ti * G + g) * 4 + w] = hv;
    }
    consumers_sync();
    {
      // logits of the router rows [e0, e0 + ne): warp = (row, part of the columns)
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
#pragma unroll 2
        for (int cc = cb + lane; cc < ce; cc += 32) {
          const float4 wv = wr[cc];
#pragma unroll
          for (int t = 0; t < kFzMaxT; ++t) {
            if (t < T) {
              const float4 xv = reinterpret_cast<const float4*>(x32 + (size_t)t * d)[cc];
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
          a.logits[(size_t)t * E + e0 + le] = v + (a.bias ? a.bias[e0 + le] : 0.f);
        }
      consumers_sync();
      if (ctid == 0) tc::mbar_arrive(&logits_done);  // the producer arrives at the grid barrier
    }

    // ---- the shared expert's unit of this CTA while the other CTAs finish their logits
    if (sh_on) {
      const bool okw = tc::mbar_wait_warp(&sh_full, 0, &s_abort, kFzConsumerSleep);
      ok = consumers_all(ok && okw && !s_abort);
      if (ok) run_stage<TPW>(sh_stg, 1, d, -1, T, K, perm_s, w_s, xh, pgu, hb, C, warp, lane, ctid);
    }
    const bool okb = tc::mbar_wait_warp(&bar1_done, 0, &s_abort, kFzConsumerSleep);
    consumers_sync();
    ok = consumers_all(ok && okb && s_ok1 && !s_abort);
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
      // then, token by token, all consumer threads at once: the K-th largest of the 16 warp maxima
      // is a lower bound of the K-th largest key (the K largest warp maxima are K distinct keys), so
      // the keys at or above it hold the selection; each candidate is ranked against the others
      // (larger key, then lower expert) and rank k < K is the k-th choice.  Weights: exp(l - max)
      // over Z (all E, summed per warp and then over the warps in order), renormalised over the K
      // kept in ascending k.  (K > 16: every expert is a candidate.)
      uint2* cand = reinterpret_cast<uint2*>(keys + (size_t)T * EP);  // [E] (key, expert)
      if (T > 2) {
        // several tokens: one warp per token instead (the same choices)
        if (warp < T) {
          int my_i;
          float my_w;
          topk_warp_fast(keys + (size_t)warp * EP, E, K, cand + (size_t)warp * 64, my_i, my_w);
          if (lane < K) {
            idx_s[warp * K + lane] = my_i;
            w_s[warp * K + lane] = my_w;
          }
        }
        consumers_sync();
      }
#pragma unroll 1
      for (int t = 0; t < (T > 2 ? 0 : T); ++t) {
        const uint32_t* kt = keys + (size_t)t * EP;
        const int ea = ctid, eb = ctid + kFzWarps * 32;
        const uint32_t k0 = ea < E ? kt[ea] : 0u, k1 = eb < E ? kt[eb] : 0u;
        const uint32_t wm = __reduce_max_sync(0xffffffffu, max(k0, k1));
        if (lane == 0) s_wmax[warp] = wm;
        if (ctid == 0) s_ncand = 0;
        consumers_sync();
        if (warp == 0) {
          const uint32_t v = lane < kFzWarps ? s_wmax[lane] : 0u;
          int rk = 0;
#pragma unroll
          for (int l = 0; l < kFzWarps; ++l) {
            const uint32_t o = __shfl_sync(0xffffffffu, v, l);
            rk += (o > v) || (o == v && l < lane);
          }
          const uint32_t tau = K <= kFzWarps ? __reduce_max_sync(0xffffffffu, (lane < kFzWarps && rk == K - 1) ? v : 0u) : 0u;
          const uint32_t mx = __reduce_max_sync(0xffffffffu, v);
          if (lane == 0) {
            s_tau = tau;
            s_m = topk_key_value(mx);
          }
        }
        consumers_sync();
        const uint32_t tau = s_tau;
        const float mlog = s_m;
        float zp = 0.f;
        if (k0 != 0u) zp += expf(topk_key_value(k0) - mlog);
        if (k1 != 0u) zp += expf(topk_key_value(k1) - mlog);
        zp = warp_sum(zp);
        if (lane == 0) s_zp[warp] = zp;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t kk = h ? k1 : k0;
          const bool is_c = kk != 0u && kk >= tau;
          const unsigned bal = __ballot_sync(0xffffffffu, is_c);
          int basep = 0;
          if (lane == 0 && bal) basep = atomicAdd(&s_ncand, __popc(bal));
          basep = __shfl_sync(0xffffffffu, basep, 0);
          if (is_c) cand[basep + __popc(bal & ((1u << lane) - 1u))] = make_uint2(kk, (uint32_t)(h ? eb : ea));
        }
        consumers_sync();
        const int ncd = s_ncand;
#pragma unroll 1
        for (int ci = ctid; ci < ncd; ci += kFzWarps * 32) {
          const uint2 me = cand[ci];
          int rank = 0;
#pragma unroll 4
          for (int q = 0; q < ncd; ++q) {
            const uint2 o = cand[q];
            rank += (o.x > me.x) || (o.x == me.x && o.y < me.y);
          }
          if (rank < K) {
            s_sel[rank] = me;
          }
        }
        consumers_sync();
        if (warp == 0) {
          float z = 0.f;
#pragma unroll
          for (int w2 = 0; w2 < kFzWarps; ++w2) z += s_zp[w2];
          const uint2 sel = lane < K ? s_sel[lane] : make_uint2(0u, 0u);
          const float p = lane < K ? expf(topk_key_value(sel.x) - mlog) / z : 0.f;
          float psum = 0.f;
#pragma unroll 1
          for (int k = 0; k < K; ++k) psum += __shfl_sync(0xffffffffu, p, k);
          if (lane < K) {
            idx_s[t * K + lane] = (int)sel.y;
            w_s[t * K + lane] = p / psum;
          }
        }
        consumers_sync();
      }
      if (c == 0)
        #pragma unroll 1
        for (int i = ctid; i < T * K; i += kFzWarps * 32) {
          a.idx[i] = idx_s[i];
          a.w[i] = w_s[i];
        }
      {
        // dispatch by counting, one thread per assignment i (n <= 256): its place in the stable
        // counting sort is the number of smaller (expert, i) keys; the distinct experts below its
        // own give its slot.  One token: its K experts are distinct, so place = slot.
        const int n = T * K;
        if (T == 1) {
          if (ctid < n) {
            const int e_i = idx_s[ctid];
            int pos = 0;
#pragma unroll 4
            for (int j = 0; j < n; ++j) pos += idx_s[j] < e_i;
            perm_s[pos] = ctid;
            slot_s[pos] = make_int4(e_i, pos, 1, 0);
          }
          if (ctid == 0) s_nact = n;
          consumers_sync();
        } else {
          int e_i = 0, start = 0, cnt_i = 0, first = 0;
          if (ctid < n) {
            e_i = idx_s[ctid];
            int pos = 0, before = 0;
#pragma unroll 4
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
#pragma unroll 4
            for (int j = 0; j < n; ++j) slot += s_srt[j] && idx_s[j] < e_i;
            slot_s[slot] = make_int4(e_i, start, cnt_i, 0);
          }
          if (ctid == 0) {
            int na = 0;
#pragma unroll 4
            for (int j = 0; j < n; ++j) na += s_srt[j];
            s_nact = na;
          }
          consumers_sync();
        }
      }
      if (ctid == 0) tc::mbar_arrive(&route_ready);  // the producer may now stream routed experts
      if (c == 0) {
        // the full outputs: offs[e] = assignments with an expert below e
        const int n = T * K, na = s_nact;
#pragma unroll 1
        for (int e = ctid; e <= E; e += kFzWarps * 32) {
          int o = 0, ce = 0;
#pragma unroll 4
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

    // ---- phase 3: this CTA's routed units through the ring
    if (ok) {
      const long long U = (long long)s_nact * fu;
      UnitRange ur{(int)(U * c / nc), (int)(U * (c + 1) / nc)};
      int s, u0, nu, k = 0;
      while (next_stage(ur, fu, s, u0, nu)) {
        const int st = k % NS;
        const bool okw = tc::mbar_wait_warp(&full[st], (k / NS) & 1, &s_abort, kFzConsumerSleep);
        ok = consumers_all(okw && !s_abort);
        if (!ok) break;
        const int4 sl = slot_s[s];
        run_stage<TPW>(ring + (size_t)st * SB, nu, d, sl.y, sl.z, K, perm_s, w_s, xh, pgu, hb, C, warp, lane, ctid);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[st]);
        ++k;
      }
    }
    if (!ok && ctid == 0) s_abort = 1;

    // ---- the partial output of this CTA, then the second grid barrier
    if (ok) {
      const int g = lane >> 2, t = lane & 3;
      float* pc = a.part + (size_t)c * T * d;
#pragma unroll
      for (int i = 0; i < TPW; ++i) {
        const int r0 = warp * (d / 16) + 16 * i + g;
        if (2 * t < T) {
          pc[(size_t)(2 * t) * d + r0] = C[i][0];
          pc[(size_t)(2 * t) * d + r0 + 8] = C[i][2];
        }
        if (2 * t + 1 < T) {
          pc[(size_t)(2 * t + 1) * d + r0] = C[i][1];
          pc[(size_t)(2 * t + 1) * d + r0 + 8] = C[i][3];
        }
      }
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

// ------------------------------------------------------------------ decode layout from the row-major planes
// gu_q [n][2f][d/2], gu_s [n][2f][d/32], dn_q [n][d][f/2], dn_s [n][d][f/32] (n experts) -> out:
// n expert blocks of dl_expert_bytes, then n down-scale blocks of dl_scale_bytes.
__global__ void dl_repack_kernel(const uint8_t* gu_q, const __half* gu_s, const uint8_t* dn_q, const __half* dn_s,
                                 int n_exp, int d, int f, uint8_t* out) {
  const int KT = d / 128, G = d / 32, fu = f / kFzUnit, TPW = d / 256;
  const size_t ub = dl_unit_bytes(d), eb = dl_expert_bytes(d, f), gb = dl_gu_bytes(d);
  const size_t stride = (size_t)gridDim.x * blockDim.x, i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  // gate/up codes: (e, u, kt, lane, half, j)
  const size_t n_gu = (size_t)n_exp * fu * KT * 256;
  for (size_t i = i0; i < n_gu; i += stride) {
    const int j = (int)(i & 3), h = (int)((i >> 2) & 1), lane = (int)((i >> 3) & 31);
    size_t r = i >> 8;
    const int kt = (int)(r % KT);
    r /= KT;
    const int u = (int)(r % fu), e = (int)(r / fu);
    const int g = lane >> 2, t = lane & 3;
    const size_t row = (size_t)e * 2 * f + (h ? f : 0) + 8 * u + g;
    const uint32_t w = *reinterpret_cast<const uint32_t*>(gu_q + row * (d / 2) + (4 * kt + j) * 16 + 4 * t);
    *reinterpret_cast<uint32_t*>(out + e * eb + u * ub + (size_t)kt * 1152 + h * 512 + lane * 16 + j * 4) =
        w ^ 0x88888888u;
  }
  // gate/up scales: (e, u, kt, g, half, j)
  const size_t n_gs = (size_t)n_exp * fu * KT * 64;
  for (size_t i = i0; i < n_gs; i += stride) {
    const int j = (int)(i & 3), h = (int)((i >> 2) & 1), g = (int)((i >> 3) & 7);
    size_t r = i >> 6;
    const int kt = (int)(r % KT);
    r /= KT;
    const int u = (int)(r % fu), e = (int)(r / fu);
    const size_t row = (size_t)e * 2 * f + (h ? f : 0) + 8 * u + g;
    *reinterpret_cast<__half*>(out + e * eb + u * ub + (size_t)kt * 1152 + 1024 + (g * 8 + h * 4 + j) * 2) =
        gu_s[row * G + 4 * kt + j];
  }
  // down codes: (e, u, pair, lane)
  const size_t n_dn = (size_t)n_exp * fu * (d / 32) * 32;
  for (size_t i = i0; i < n_dn; i += stride) {
    const int lane = (int)(i & 31);
    size_t r = i >> 5;
    const int p = (int)(r % (d / 32));
    r /= (d / 32);
    const int u = (int)(r % fu), e = (int)(r / fu);
    const int g = lane >> 2, t = lane & 3;
    uint32_t w = 0;
#pragma unroll
    for (int tile = 0; tile < 2; ++tile)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const size_t row = (size_t)e * d + 32 * p + 16 * tile + g + 8 * hr;
          const int col = 8 * u + 2 * t + cc;
          const uint8_t byte = dn_q[row * (f / 2) + col / 2];
          const uint32_t o = (uint32_t)(((col & 1) ? (byte >> 4) : (byte & 15)) ^ 8);
          w |= o << (4 * hr + 8 * tile + 16 * cc);
        }
    *reinterpret_cast<uint32_t*>(out + e * eb + u * ub + gb + ((size_t)p * 32 + lane) * 4) = w;
  }
  // down scales: (e, group, warp, g, tile, r)
  __half* os = reinterpret_cast<__half*>(out + (size_t)n_exp * eb);
  const size_t n_ds = (size_t)n_exp * (f / 32) * d;
  for (size_t i = i0; i < n_ds; i += stride) {
    const int rr = (int)(i & 1);
    size_t r = i >> 1;
    const int ti = (int)(r % TPW);
    r /= TPW;
    const int g = (int)(r & 7);
    r >>= 3;
    const int w = (int)(r & 15);
    r >>= 4;
    const int grp = (int)(r % (f / 32)), e = (int)(r / (f / 32));
    const size_t row = (size_t)w * (d / 16) + 16 * ti + g + 8 * rr;
    os[i] = dn_s[((size_t)e * d + row) * (f / 32) + grp];
  }
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
  p.stage_bytes = (int)((kFzStageUnits * dl_unit_bytes(d) + 2 * (size_t)d + 127) & ~size_t(127));
  const size_t fixed = up16((size_t)T * d * 4) + up16((size_t)T * d * 2) + (size_t)kFzWarps * 32 * 16 +
                       up16((size_t)T * K * 16) + 3 * up16((size_t)T * K * 4);
  const long long room = (long long)kFzSmemMax - kFzStaticSlack - (long long)fixed;
  p.ns = room > 0 ? (int)std::min<long long>(kFzMaxStages, room / p.stage_bytes) : 0;
  p.smem = (int)((size_t)p.ns * p.stage_bytes + fixed);
  return p;
}

static int g_fz_sms = 0;

template <int TPW>
static const void* fused_fn() {
  return (const void*)decode_layer_kernel<TPW>;
}

static const void* fused_fn_for(int d) {
  switch (d / 256) {
    case 2: return fused_fn<2>();
    case 4: return fused_fn<4>();
    case 6: return fused_fn<6>();
    default: return fused_fn<8>();
  }
}

cudaError_t fused_kernels_init(int num_sms) {
  g_fz_sms = num_sms;
  const void* fns[4] = {fused_fn<2>(), fused_fn<4>(), fused_fn<6>(), fused_fn<8>()};
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
  if (d % 512 || d > 2048 || f % 32 || f > 1024 || E > kMaxE || K > kMaxK) return false;
  if (f / kFzUnit > nc) return false;         // at most one shared-expert unit per CTA
  if (T * K > kFzWarps * 32) return false;    // dispatch: one thread per assignment
  const FusedPlan p = fused_plan(T, d, f, E, K);
  if (p.ns < 2) return false;                 // the router rows and the shared stage use stages 0 and 1
  if ((size_t)T * ((E + 31) & ~31) * 4 + (size_t)std::max(E, T * 64) * 8 > (size_t)p.stage_bytes)
    return false;  // the selection's scratch
  if (E > 2 * kFzWarps * 32) return false;    // selection: two keys per consumer thread
  return (size_t)((E + nc - 1) / nc) * d * 4 <= (size_t)p.stage_bytes;
}

// Bytes of the decode-layout copy of n_exp experts (unit blocks, then down scales).
size_t fused_layout_bytes(int n_exp, int d, int f) {
  return (size_t)n_exp * (dl_expert_bytes(d, f) + dl_scale_bytes(d, f));
}

cudaError_t fused_repack(const void* gu_q, const void* gu_s, const void* dn_q, const void* dn_s, int n_exp, int d,
                         int f, void* out, cudaStream_t st) {
  dl_repack_kernel<<<2048, 256, 0, st>>>(static_cast<const uint8_t*>(gu_q), static_cast<const __half*>(gu_s),
                                         static_cast<const uint8_t*>(dn_q), static_cast<const __half*>(dn_s), n_exp, d,
                                         f, static_cast<uint8_t*>(out));
  return cudaGetLastError();
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
  a.dl = static_cast<const uint8_t*>(fx.dl);
  a.dls = static_cast<const uint8_t*>(fx.dl) + (size_t)r.E * dl_expert_bytes(r.d, x.f);
  a.sh_dl = static_cast<const uint8_t*>(fx.sh_dl);
  a.sh_dls = fx.sh_dl ? static_cast<const uint8_t*>(fx.sh_dl) + dl_expert_bytes(r.d, x.f) : nullptr;
  a.part = fx.part;
  a.y = x.y;
  a.resid = x.resid;
  a.grid_bar = fx.grid_bar;
  a.status = r.status;
  const FusedPlan p = fused_plan(r.T, r.d, x.f, r.E, r.K);
  a.ns = p.ns;
  a.stage_bytes = p.stage_bytes;
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
  return cudaLaunchKernelExC(&cfg, fused_fn_for(r.d), args);
}

}  // namespace moe
