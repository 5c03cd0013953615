// Decode / verify layer in one launch (sm_103a): router logits, softmax + top-K, dispatch, the
// gate/up and down GEMVs of the selected and shared experts, and the fixed-order combine.
//
// A decode step streams the bytes of the experts its few tokens chose and little else
// ('Strata はなぜ少ない VRAM でも速いのか' (modeldock.net), section '1 トークン、三者の分担';
// verifying 1 + 3 drafted tokens adds only the experts the drafts pick, section
// '予測してから検証する').  With every expert in HBM the cost that remains besides those bytes is
// the chain router -> selection -> experts -> down -> combine.  Here that chain runs inside one
// persistent kernel (one CTA per SM, all co-resident: cooperative launch) with two grid-wide
// barriers instead of five kernel boundaries and a single-block selection tail:
//
//   phase 1  every CTA scores its slice of the E experts for all T tokens (fp32 router rows held
//            in registers, issued before anything else) and stores the logits;     [grid arrive]
//            meanwhile it computes its share of the shared expert's gate/up rows, whose weights
//            were requested at kernel start (they do not depend on the routing);   [grid wait]
//   phase 2  every CTA reads all logits and repeats the selection and the dispatch in shared
//            memory (identical, deterministic); CTA 0 publishes them;
//   phase 3  the routed (expert, f) pairs are split evenly over the CTAs; one producer warp
//            streams each CTA's gate/up rows (and then its down rows) with bulk copies into a
//            ring of shared-memory stages; 16 consumer warps compute h = silu(g) * u;  [grid barrier]
//   phase 4  each CTA owns d/#CTA output rows: it computes those rows of every selected expert's
//            down projection for every token routed to it (weights already in shared memory),
//            then combines them per token in fixed order (ascending k, shared expert last) with
//            the optional residual, and writes y.
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
constexpr int kFzPairs = 16;                     // gate/up pairs per ring chunk: one per consumer warp
constexpr int kFzMaxT = 8;
constexpr int kFzMaxStages = 8;
constexpr int kFzSmemMax = 227 * 1024;
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
  const uint8_t* gu_q;
  const __half* gu_s;
  const uint8_t* dn_q;
  const __half* dn_s;
  const uint8_t* sh_gu_q;
  const __half* sh_gu_s;
  const uint8_t* sh_dn_q;
  const __half* sh_dn_s;
  float* h;             // [(T*K + T)][f]
  void* y;
  const void* resid;
  unsigned long long* grid_bar;  // grid-barrier arrival counter (only ever increases)
  unsigned* status;
  int ns;               // ring stages
  int stage_bytes;
  int shg_rows;         // row stride of the shared gate/up area (max pairs per CTA)
  int dn_rows_max;      // max down rows per CTA
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
#pragma unroll
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

// h[asg][i0 + p] = silu(gate_p . x) * (up_p . x), p < np <= NP, for the n tokens of one slot (the
// assignments at perm_s[pbase..], or all T tokens of the shared expert).  Gate rows at gq +
// p*qrow, up rows at uq + p*qrow, their scales at gs + p*G / us + p*G (shared memory).
template <int NG, int TB, int NP>
__device__ __forceinline__ void quad_h(const FusedArgs& a, const uint8_t* gq, const uint8_t* uq, const __half* gs,
                                       const __half* us, size_t qrow, int i0, int np, int n, int pbase, bool shared,
                                       const int* perm_s, const float4* xq, const float* xs136, int lane) {
  const int G = a.d / 32;
  for (int t0 = 0; t0 < n; t0 += TB) {
    int tok[TB];
#pragma unroll
    for (int tt = 0; tt < TB; ++tt) {
      const int ti = t0 + tt < n ? t0 + tt : t0;
      tok[tt] = shared ? ti : perm_s[pbase + ti] / a.K;
    }
    // pairs per pass: all NP for one token, half as many for two (register budget)
    constexpr int NPC = TB == 1 ? NP : (NP > 1 ? NP / 2 : 1);
    constexpr int NV = 2 * NPC * TB;                 // values reduced together: gate rows, then up rows
    constexpr int SH = NV == 8 ? 2 : NV == 4 ? 3 : 4;  // value i's total sits in lanes with (lane >> SH) == i
#pragma unroll
    for (int p0 = 0; p0 < NP; p0 += NPC) {
      float acc[2 * NPC][TB];
      const int npc = min(NPC, np - p0);
      pairs_dot<NG, TB, NPC>(gq + p0 * qrow, uq + p0 * qrow, gs + (size_t)p0 * G, us + (size_t)p0 * G, qrow,
                             npc > 0 ? npc : 1, G, xq, xs136, tok, acc, lane);
      float vals[NV];
#pragma unroll
      for (int r = 0; r < 2 * NPC; ++r)
#pragma unroll
        for (int tt = 0; tt < TB; ++tt) vals[r * TB + tt] = acc[r][tt];
      const float g = warp_sum_multi<NV>(vals);
      const float u = __shfl_down_sync(0xffffffffu, g, 16);  // the up row of the same pair and token
      const int vi = lane >> SH;                              // < NV / 2 for lanes < 16
      const int p = p0 + vi / TB, tt = vi % TB;
      if (lane < 16 && (lane & ((1 << SH) - 1)) == 0 && p - p0 < npc && t0 + tt < n) {
        const int as = shared ? a.T * a.K + (t0 + tt) : perm_s[pbase + t0 + tt];
        a.h[(size_t)as * a.f + i0 + p] = silu(g) * u;
      }
    }
  }
}

// Down rows [r_beg, r_end) of one expert (codes at q, scales at sc, row stride f/2 bytes and f/32
// scales, in shared memory) for the tokens [t_beg, t_end) of one slot:
// P[asg][r] = sum_f W[r][f] h[asg][f].  Lane = one 32-column group of h (f <= 1024); rows in
// batches of eight, each batch reduced over the warp in one multi-value reduction.  h is read
// through L1: each lane's 128 contiguous bytes are one line, fetched once.
__device__ __forceinline__ void dn_slot(const FusedArgs& a, const uint8_t* q, const __half* sc, int r_beg, int r_end,
                                        int t_beg, int t_end, int pbase, bool shared, const int* perm_s, float* P,
                                        int lane) {
  const int f = a.f, Gf = f / 32;
  const bool on = lane < Gf;
  for (int ti = t_beg; ti < t_end; ++ti) {
    const int as = shared ? a.T * a.K + ti : perm_s[pbase + ti];
    float4 hv[8];
    const float4* hp = reinterpret_cast<const float4*>(a.h + (size_t)as * f + (on ? lane : 0) * 32);
#pragma unroll
    for (int m = 0; m < 8; ++m) hv[m] = on ? __ldca(hp + m) : make_float4(0.f, 0.f, 0.f, 0.f);
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
    for (int r0 = r_beg; r0 < r_end; r0 += 8) {
      float pr[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = r0 + i;
        float pv = 0.f;
        if (on && r < r_end) {
          const uint4 w = *reinterpret_cast<const uint4*>(q + (size_t)r * (f / 2) + lane * 16);
#pragma unroll
          for (int wd = 0; wd < 4; ++wd) {
            const float4 xa = hv[2 * wd], xb = hv[2 * wd + 1];
            const uint32_t w32 = wd == 0 ? w.x : wd == 1 ? w.y : wd == 2 ? w.z : w.w;
            const uint32_t lo = (w32 & 0x0F0F0F0Fu) ^ 0x08080808u, hi = ((w32 >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
            pv = fmaf(v_lo(lo, 0), xa.x, pv);
            pv = fmaf(v_lo(hi, 0), xa.y, pv);
            pv = fmaf(v_lo(lo, 1), xa.z, pv);
            pv = fmaf(v_lo(hi, 1), xa.w, pv);
            pv = fmaf(v_lo(lo, 2), xb.x, pv);
            pv = fmaf(v_lo(hi, 2), xb.y, pv);
            pv = fmaf(v_lo(lo, 3), xb.z, pv);
            pv = fmaf(v_lo(hi, 3), xb.w, pv);
          }
          pv = __half2float(sc[(size_t)r * Gf + lane]) * (pv - h136);
        }
        pr[i] = pv;
      }
      const float o = warp_sum_multi<8>(pr);
      const int r = r0 + (lane >> 2);
      if ((lane & 3) == 0 && r < r_end) P[(size_t)as * a.dn_rows_max + r] = o;
    }
  }
}

// The next ring chunk of routed gate/up pairs: pairs [pos, end) numbered slot-major (slot * f + i),
// cut at slot boundaries and at kFzPairs.
struct PairRange {
  int pos, end;
};
__device__ __forceinline__ bool next_pairs(PairRange& r, int f, int& s, int& i0, int& n) {
  if (r.pos >= r.end) return false;
  s = r.pos / f;
  i0 = r.pos - s * f;
  n = min(kFzPairs, min(r.end - r.pos, f - i0));
  r.pos += n;
  return true;
}

// Ring chunk k is consumed by consumer group k % kFzGroups (kFzWarps / kFzGroups warps each), so
// that several chunks are in work at once and each warp reuses every x' load for four pairs.  Each
// group owns its own stages (stage g, g + kFzGroups, ...), filled and drained in its chunk order:
// every mbarrier is then waited on in phase order, never a phase ahead (a parity wait one phase
// ahead would return at once).
constexpr int kFzGroups = 4;
constexpr int kFzGroupWarps = kFzWarps / kFzGroups;
constexpr int kFzDnSlots = kFzGroupWarps;  // routed experts per down-projection ring chunk
__device__ __forceinline__ int ring_stage(int k, int sg) { return k % kFzGroups + kFzGroups * ((k / kFzGroups) % sg); }
__device__ __forceinline__ uint32_t ring_phase(int k, int sg) { return (uint32_t)((k / kFzGroups) / sg) & 1u; }

template <int NG, int TB>
__global__ void __launch_bounds__(kFzThreads, 1) decode_layer_kernel(const FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int T = a.T, d = a.d, E = a.E, K = a.K, f = a.f, G = d / 32, Gf = f / 32;
  const int nc = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int SB = a.stage_bytes, NS = a.ns, SG = NS / kFzGroups;  // NS is a multiple of kFzGroups
  const size_t qrow = (size_t)d / 2, srow = (size_t)G * 2;  // gate/up row bytes: codes, scales
  const size_t dq = (size_t)f / 2, ds = (size_t)Gf * 2;      // down row bytes: codes, scales
  const int DR = a.dn_rows_max;

  // this CTA's fixed shares
  const int sh0 = (int)((long long)f * c / nc), sh1 = (int)((long long)f * (c + 1) / nc);  // shared pairs
  const int j0 = (int)((long long)d * c / nc), nr = (int)((long long)d * (c + 1) / nc) - j0;  // down rows
  const int e0 = (int)((long long)E * c / nc), ne = (int)((long long)E * (c + 1) / nc) - e0;  // router rows

  // shared memory carve (all offsets 16-byte multiples)
  uint8_t* ring = smem_raw;
  uint8_t* shg = ring + (size_t)NS * SB;
  const int SR = a.shg_rows;
  uint8_t* shd = shg + (size_t)SR * 2 * (qrow + srow);
  float4* xq = reinterpret_cast<float4*>(shd + (size_t)DR * (dq + ds));
  float* xs136 = reinterpret_cast<float*>(xq + (size_t)T * 8 * G);
  float* part = xs136 + (size_t)T * G;                       // [16][kFzMaxT]
  float* P = part + kFzWarps * kFzMaxT;                      // [T*K + T][DR]
  int4* slot_s = reinterpret_cast<int4*>(P + (((size_t)(T * K + T) * DR + 3) & ~size_t(3)));
  int* perm_s = reinterpret_cast<int*>(slot_s + E);
  int* idx_s = perm_s + T * K;
  float* w_s = reinterpret_cast<float*>(idx_s + T * K);

  __shared__ __align__(8) uint64_t full[kFzMaxStages], empty[kFzMaxStages], shg_full, shd_full, route_ready;
  __shared__ uint64_t s_tkc[kFzWarps * kMaxK];
  __shared__ float s_tkf[2 * kFzWarps];
  __shared__ int s_srt[kFzMaxT * kMaxK];
  __shared__ volatile int s_abort;
  __shared__ int s_nact, s_issued, s_ok;
  __shared__ float inv_s[kFzMaxT];

  // This launch may start while the previous layer's kernel is still finishing (programmatic
  // dependent launch): everything before griddepcontrol.wait touches only this CTA's shared memory
  // and read-only weights; the activations, the workspace and the barrier counter come after it.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], kFzGroupWarps);
    }
    tc::mbar_init(&shg_full, 1);
    tc::mbar_init(&shd_full, 1);
    tc::mbar_init(&route_ready, 1);
    s_abort = 0;
    s_issued = 0;
    s_ok = 1;
    tc::fence_mbar_init();
  }
  __syncthreads();
  const bool sh_gu_on = a.has_shared && sh1 > sh0;
  const bool sh_dn_on = a.has_shared && nr > 0;

  if (warp == kFzWarps) {
    // ================================================================ producer
    if (lane == 0) {
      // the shared expert's rows of this CTA do not depend on the routing: request them first
      if (sh_gu_on) {
        const int n = sh1 - sh0;
        tc::mbar_arrive_expect_tx(&shg_full, (uint32_t)(2 * n * (qrow + srow)));
        tc::bulk_g2s(shg, a.sh_gu_q + (size_t)sh0 * qrow, (uint32_t)(n * qrow), &shg_full);
        tc::bulk_g2s(shg + SR * qrow, a.sh_gu_q + (size_t)(f + sh0) * qrow, (uint32_t)(n * qrow), &shg_full);
        tc::bulk_g2s(shg + 2 * SR * qrow, a.sh_gu_s + (size_t)sh0 * G, (uint32_t)(n * srow), &shg_full);
        tc::bulk_g2s(shg + 2 * SR * qrow + SR * srow, a.sh_gu_s + (size_t)(f + sh0) * G, (uint32_t)(n * srow),
                     &shg_full);
      }
      if (sh_dn_on) {
        tc::mbar_arrive_expect_tx(&shd_full, (uint32_t)(nr * (dq + ds)));
        tc::bulk_g2s(shd, a.sh_dn_q + (size_t)j0 * dq, (uint32_t)(nr * dq), &shd_full);
        tc::bulk_g2s(shd + nr * dq, a.sh_dn_s + (size_t)j0 * Gf, (uint32_t)(nr * ds), &shd_full);
      }
      bool ok = tc::mbar_wait_sleepy(&route_ready, 0, &s_abort, kFzProducerSleep);
      int k = 0;
      if (ok) {
        const int n_act = s_nact;

        const long long U = (long long)n_act * f;
        PairRange pr{(int)(U * c / nc), (int)(U * (c + 1) / nc)};
        int s, i0, n;
        while (ok && next_pairs(pr, f, s, i0, n)) {
          const int st = ring_stage(k, SG);
          if (!tc::mbar_wait_sleepy(&empty[st], ring_phase(k, SG) ^ 1u, &s_abort, kFzProducerSleep)) { ok = false; break; }
          const int e = slot_s[s].x;
          uint8_t* dst = ring + (size_t)st * SB;
          const size_t rg = (size_t)e * 2 * f + i0, ru = rg + f;
          tc::mbar_arrive_expect_tx(&full[st], (uint32_t)(2 * n * (qrow + srow)));
          tc::bulk_g2s(dst, a.gu_q + rg * qrow, (uint32_t)(n * qrow), &full[st]);
          tc::bulk_g2s(dst + kFzPairs * qrow, a.gu_q + ru * qrow, (uint32_t)(n * qrow), &full[st]);
          tc::bulk_g2s(dst + 2 * kFzPairs * qrow, a.gu_s + rg * G, (uint32_t)(n * srow), &full[st]);
          tc::bulk_g2s(dst + 2 * kFzPairs * qrow + kFzPairs * srow, a.gu_s + ru * G, (uint32_t)(n * srow), &full[st]);
          s_issued = ++k;
        }
        // the down rows are needed only after the second barrier: start their way into L2 now (after
        // the gate/up requests), so their copies into the ring, which wait for the gate/up stages,
        // are short
        for (int jj = 0; ok && jj < n_act && nr > 0; ++jj) {
          const int e = slot_s[jj].x;
          tc::bulk_prefetch_l2(a.dn_q + ((size_t)e * d + j0) * dq, (uint32_t)(nr * dq));
          tc::bulk_prefetch_l2(a.dn_s + ((size_t)e * d + j0) * Gf, (uint32_t)(nr * ds));
        }
        // then this CTA's down rows of every routed expert, kFzDnSlots experts per chunk
        for (int p0 = 0; ok && nr > 0 && p0 < n_act; p0 += kFzDnSlots) {
          const int st = ring_stage(k, SG);
          if (!tc::mbar_wait_sleepy(&empty[st], ring_phase(k, SG) ^ 1u, &s_abort, kFzProducerSleep)) { ok = false; break; }
          const int cntp = min(kFzDnSlots, n_act - p0);
          uint8_t* dst = ring + (size_t)st * SB;
          tc::mbar_arrive_expect_tx(&full[st], (uint32_t)(cntp * nr * (dq + ds)));
          for (int jj = 0; jj < cntp; ++jj) {
            const int e = slot_s[p0 + jj].x;
            uint8_t* sd = dst + (size_t)jj * DR * (dq + ds);
            tc::bulk_g2s(sd, a.dn_q + ((size_t)e * d + j0) * dq, (uint32_t)(nr * dq), &full[st]);
            tc::bulk_g2s(sd + DR * dq, a.dn_s + ((size_t)e * d + j0) * Gf, (uint32_t)(nr * ds), &full[st]);
          }
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
    const int grp = warp / kFzGroupWarps, wg = warp % kFzGroupWarps;
    bool ok = true;
    // ---- phase 1: router rows of experts [e0, e0 + ne), all tokens
    const int ncol = d / 4;                               // float4 columns per row
    const int nparts = ne > 0 ? max(1, kFzWarps / ne) : 1;
    const int my_e = warp % max(ne, 1), my_p = warp / max(ne, 1);
    const bool r_on = ne > 0 && my_p < nparts;
    const int cb = r_on ? (int)((long long)ncol * my_p / nparts) : 0;
    const int ce = r_on ? (int)((long long)ncol * (my_p + 1) / nparts) : 0;
    const float4* wr = reinterpret_cast<const float4*>(a.Wr + (size_t)(e0 + (r_on ? my_e : 0)) * d);
    float4 wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int cc = cb + lane + 32 * i;
      wv[i] = cc < ce ? __ldg(wr + cc) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous kernel's writes are visible
    // the barrier counter's base: the previous launch's barriers are complete and fewer than
    // gridDim.x arrivals of this launch's first barrier can precede this read
    unsigned long long bar_base = 0;
    if (ctid == 0) bar_base = ld_acquire_gpu(a.grid_bar) / gridDim.x * gridDim.x;
    if (a.prenorm) {
      for (int t = warp; t < T; t += kFzWarps) {
        float ss = 0.f;
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
    for (int i = ctid; i < T * G; i += kFzWarps * 32) {
      const int ti = i / G, g = i - ti * G;
      const float* xb = reinterpret_cast<const float*>(xq) + (size_t)ti * 8 * G * 4;
      float sx = 0.f;
      for (int m = 0; m < 32; ++m) sx += xb[((m >> 2) * G + g) * 4 + (m & 3)];
      xs136[i] = sx * (136.0f / 256.0f);
    }
    // logits: x' = 256 x, so the dot product is 256 times the wanted one, exactly
    {
      float acc[kFzMaxT];
#pragma unroll
      for (int t = 0; t < kFzMaxT; ++t) acc[t] = 0.f;
      for (int cbase = cb; cbase < ce; cbase += 32 * 8) {
        if (cbase > cb) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int cc = cbase + lane + 32 * i;
            wv[i] = cc < ce ? __ldg(wr + cc) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int cc = cbase + lane + 32 * i;
          if (cc >= ce) continue;
          const int g = cc >> 3, m4 = cc & 7;
#pragma unroll
          for (int t = 0; t < kFzMaxT; ++t) {
            if (t < T) {
              const float4 xv = xq[((size_t)t * 8 + m4) * G + g];
              acc[t] = fmaf(wv[i].x, xv.x, acc[t]);
              acc[t] = fmaf(wv[i].y, xv.y, acc[t]);
              acc[t] = fmaf(wv[i].z, xv.z, acc[t]);
              acc[t] = fmaf(wv[i].w, xv.w, acc[t]);
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kFzMaxT; ++t) {
        if (t < T) {
          const float v = warp_sum(acc[t]);
          if (lane == 0) part[warp * kFzMaxT + t] = v;
        }
      }
    }
    consumers_sync();
    for (int i = ctid; i < ne * T; i += kFzWarps * 32) {
      const int le = i / T, t = i - le * T;
      float v = 0.f;
      for (int p = 0; p < nparts; ++p) v += part[(p * ne + le) * kFzMaxT + t];
      a.logits[(size_t)t * E + e0 + le] = v * (1.0f / 256.0f) + (a.bias ? a.bias[e0 + le] : 0.f);
    }
    consumers_sync();
    if (ctid == 0) grid_arrive(a.grid_bar);

    // ---- shared expert gate/up while the other CTAs finish their logits
    if (sh_gu_on) {
      ok = tc::mbar_wait_warp(&shg_full, 0, &s_abort, kFzConsumerSleep);
      const int n = sh1 - sh0;
      // one pair per warp: this runs while the barrier waits, so spread it out
      for (int p0 = warp; ok && p0 < n; p0 += kFzWarps)
        quad_h<NG, TB, 1>(a, shg + p0 * qrow, shg + SR * qrow + p0 * qrow,
                          reinterpret_cast<const __half*>(shg + 2 * SR * qrow) + (size_t)p0 * G,
                          reinterpret_cast<const __half*>(shg + 2 * SR * qrow + SR * srow) + (size_t)p0 * G, qrow,
                          sh0 + p0, 1, T, 0, true, perm_s, xq, xs136, lane);
    }
    if (ctid == 0) s_ok = grid_wait(a.grid_bar, bar_base + nc, &s_abort) ? 1 : 0;
    consumers_sync();
    ok = consumers_all(ok && s_ok && !s_abort);
    if (!ok && ctid == 0) s_abort = 1;  // the producer stops waiting for the routing

    // ---- phase 2: selection and dispatch, repeated by every CTA
    int k = 0;
    if (ok) {
      topk_group(a.logits, T, E, K, kFzWarps, warp, s_tkf, s_tkc, idx_s, w_s, [] { consumers_sync(); });
      if (c == 0)
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
          for (int j = 0; j < n; ++j) slot += s_srt[j] && idx_s[j] < e_i;
          slot_s[slot] = make_int4(e_i, start, cnt_i, 0);
        }
        if (ctid == 0) {
          int na = 0;
          for (int j = 0; j < n; ++j) na += s_srt[j];
          s_nact = na;
        }
        consumers_sync();
        if (c == 0) {
          // the full outputs: offs[e] = assignments with an expert below e
          const int na = s_nact;
          for (int e = ctid; e <= E; e += kFzWarps * 32) {
            int o = 0, ce = 0;
            for (int q = 0; q < n; ++q) {
              o += idx_s[q] < e;
              ce += idx_s[q] == e;
            }
            a.offs[e] = o;
            if (e < E) a.counts[e] = ce;
          }
          for (int q = ctid; q < na; q += kFzWarps * 32) {
            a.active[q] = slot_s[q].x;
            a.slots[q] = slot_s[q];
          }
          for (int q = ctid; q < n; q += kFzWarps * 32) a.perm[q] = perm_s[q];
          if (ctid == 0) {
            *a.n_active = na;
            if (a.stat) *a.stat = na;
          }
        }
      }
      if (ctid == 0) tc::mbar_arrive(&route_ready);  // the producer may now stream routed experts
    }
    const int n_act = ok ? s_nact : 0;

    // ---- phase 3: routed gate/up pairs through the ring; chunk k goes to group k % kFzGroups
    if (ok) {
      const long long U = (long long)n_act * f;
      PairRange pr{(int)(U * c / nc), (int)(U * (c + 1) / nc)};
      int s, i0, n;
      while (next_pairs(pr, f, s, i0, n)) {
        if (k % kFzGroups == grp) {
          const int st = ring_stage(k, SG);
          ok = tc::mbar_wait_warp(&full[st], ring_phase(k, SG), &s_abort, kFzConsumerSleep);
          if (!ok) break;
          const int p0 = 4 * wg;
          if (p0 < n) {
            const uint8_t* base = ring + (size_t)st * SB;
            const int4 sl = slot_s[s];
            quad_h<NG, TB, 4>(a, base + p0 * qrow, base + kFzPairs * qrow + p0 * qrow,
                           reinterpret_cast<const __half*>(base + 2 * kFzPairs * qrow) + (size_t)p0 * G,
                           reinterpret_cast<const __half*>(base + 2 * kFzPairs * qrow + kFzPairs * srow) + (size_t)p0 * G,
                           qrow, i0 + p0, min(4, n - p0), sl.z, sl.y, false, perm_s, xq, xs136, lane);
          }
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&empty[st]);
        }
        ++k;
      }
    }
    if (!ok && lane == 0) s_abort = 1;
    consumers_sync();
    if (ctid == 0) {
      grid_arrive(a.grid_bar);  // always arrive: the other CTAs must not wait on this one
      s_ok = (!s_abort && grid_wait(a.grid_bar, bar_base + 2ull * nc, &s_abort)) ? 1 : 0;
    }
    consumers_sync();
    ok = consumers_all(ok && s_ok && !s_abort);
    if (!ok && ctid == 0) s_abort = 1;

    // ---- phase 4: this CTA's down rows of every expert, then the combine
    {
      if (ok && sh_dn_on && grp == kFzGroups - 1) {
        // the shared expert: one warp per token of the last group
        ok = tc::mbar_wait_warp(&shd_full, 0, &s_abort, kFzConsumerSleep);
        for (int t = wg; ok && t < T; t += kFzGroupWarps)
          dn_slot(a, shd, reinterpret_cast<const __half*>(shd + nr * dq), 0, nr, t, t + 1, 0, true, perm_s, P, lane);
      }
      for (int p0 = 0; ok && nr > 0 && p0 < n_act; p0 += kFzDnSlots, ++k) {
        if (k % kFzGroups != grp) continue;
        const int st = ring_stage(k, SG);
        ok = tc::mbar_wait_warp(&full[st], ring_phase(k, SG), &s_abort, kFzConsumerSleep);
        if (!ok) break;
        const int cntp = min(kFzDnSlots, n_act - p0);
        if (wg < cntp) {
          const int4 sl = slot_s[p0 + wg];
          const uint8_t* q = ring + (size_t)st * SB + (size_t)wg * DR * (dq + ds);
          dn_slot(a, q, reinterpret_cast<const __half*>(q + DR * dq), 0, nr, 0, sl.z, sl.y, false, perm_s, P, lane);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[st]);
      }
    }
    if (!ok && lane == 0) s_abort = 1;
    ok = consumers_all(ok && !s_abort);
    if (ok) {
      // fixed-order combine: ascending k, shared expert last, optional residual, one rounding
      for (int i = ctid; i < T * nr; i += kFzWarps * 32) {
        const int t = i / nr, r = i - t * nr;
        float yv = 0.f;
        for (int kk = 0; kk < K; ++kk) yv = fmaf(w_s[t * K + kk], P[(size_t)(t * K + kk) * DR + r], yv);
        if (a.has_shared) yv += P[(size_t)(T * K + t) * DR + r];
        const size_t o = (size_t)t * d + j0 + r;
        if (a.resid) yv = load_act(a.resid, a.act, o) + yv;
        store_act(a.y, a.act, o, yv);
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
    for (int kk = issued - 1; kk >= 0 && kk >= issued - NS; --kk)  // the last chunk of every stage
      tc::mbar_wait(&full[ring_stage(kk, SG)], ring_phase(kk, SG), &never, 2000000000ll);
    if (sh_gu_on) tc::mbar_wait(&shg_full, 0, &never, 2000000000ll);
    if (sh_dn_on) tc::mbar_wait(&shd_full, 0, &never, 2000000000ll);
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

// ------------------------------------------------------------------ host side
struct FusedPlan {
  int ns, stage_bytes, shg_rows, dn_rows_max;
  size_t smem;
};

constexpr int kFzStaticSlack = 8192;  // static shared memory of the kernel and the driver's share

static FusedPlan fused_plan(int T, int d, int f, int E, int K, int nsm) {
  FusedPlan p{};
  const int G = d / 32, Gf = f / 32;
  p.stage_bytes = kFzPairs * 2 * (d / 2 + G * 2);
  p.shg_rows = (f + nsm - 1) / nsm;
  p.dn_rows_max = (d + nsm - 1) / nsm;
  size_t fixed = (size_t)p.shg_rows * 2 * (d / 2 + G * 2) + (size_t)p.dn_rows_max * (f / 2 + Gf * 2);
  fixed += (size_t)T * d * 4 + (size_t)T * G * 4 + kFzWarps * kFzMaxT * 4;
  fixed += ((size_t)(T * K + T) * p.dn_rows_max * 4 + 15) & ~size_t(15);
  fixed += (size_t)E * 16 + (size_t)T * K * 12 + 64;
  const long long room = (long long)kFzSmemMax - (long long)fixed - kFzStaticSlack;
  p.ns = room > 0 ? (int)std::min<long long>(kFzMaxStages, room / p.stage_bytes) : 0;
  p.ns -= p.ns % kFzGroups;  // whole stages per consumer group
  p.smem = fixed + (size_t)p.ns * p.stage_bytes;
  return p;
}

static int g_fz_sms = 0;

template <int NG, int TB>
static const void* fused_fn() {
  return (const void*)decode_layer_kernel<NG, TB>;
}

cudaError_t fused_kernels_init(int num_sms) {
  g_fz_sms = num_sms;
  const void* fns[6] = {fused_fn<1, 1>(), fused_fn<2, 1>(), fused_fn<4, 1>(),
                        fused_fn<1, 2>(), fused_fn<2, 2>(), fused_fn<4, 2>()};
  for (const void* fn : fns) {
    cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kFzSmemMax - kFzStaticSlack);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Whether the fused decode path serves this shape (int4 weights) with up to T tokens.
bool fused_shape_ok(int T, int d, int f, int E, int K) {
  if (g_fz_sms <= 0 || T < 1 || T > kFzMaxT) return false;
  if (d % 256 || f % 256 || f > 1024 || d > 4096 || E > kMaxE || K > kMaxK) return false;
  if (E > kTopkLanes * 32 * (kFzWarps / T)) return false;  // the selection's per-lane register budget
  const FusedPlan p = fused_plan(T, d, f, E, K, g_fz_sms);
  if (p.ns < kFzGroups) return false;
  return (size_t)kFzDnSlots * p.dn_rows_max * (f / 2 + f / 16) <= (size_t)p.stage_bytes;
}

cudaError_t launch_decode_fused(const RouteArgs& r, const ExpertArgs& x, unsigned long long* grid_bar,
                                cudaStream_t st) {
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
  a.dn_q = static_cast<const uint8_t*>(x.dn_q);
  a.dn_s = x.dn_s;
  a.sh_gu_q = static_cast<const uint8_t*>(x.sh_gu_q);
  a.sh_gu_s = x.sh_gu_s;
  a.sh_dn_q = static_cast<const uint8_t*>(x.sh_dn_q);
  a.sh_dn_s = x.sh_dn_s;
  a.h = x.h;
  a.y = x.y;
  a.resid = x.resid;
  a.grid_bar = grid_bar;
  a.status = r.status;
  const FusedPlan p = fused_plan(r.T, r.d, x.f, r.E, r.K, g_fz_sms);
  a.ns = p.ns;
  a.stage_bytes = p.stage_bytes;
  a.shg_rows = p.shg_rows;
  a.dn_rows_max = p.dn_rows_max;
  const int G = r.d / 32;
  const bool one = r.T == 1;
  const void* fn = G <= 32 ? (one ? fused_fn<1, 1>() : fused_fn<1, 2>())
                 : G <= 64 ? (one ? fused_fn<2, 1>() : fused_fn<2, 2>())
                           : (one ? fused_fn<4, 1>() : fused_fn<4, 2>());
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
