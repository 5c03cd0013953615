// Decode / verify layer in one launch (sm_103a): router logits, softmax + top-K, dispatch, the
// gate/up and down projections of the selected and shared experts on tensor cores, and the
// fixed-order combine, reading the experts' row-major int4 planes directly.
//
// A decode step streams the bytes of the experts its few tokens chose and little else
// ('Strata はなぜ少ない VRAM でも速いのか' (modeldock.net), section '1 トークン、三者の分担';
// verifying 1 + 3 drafted tokens adds only the experts the drafts pick, section
// '予測してから検証する').  With every expert in HBM what remains besides those bytes is the chain
// router -> selection -> experts -> combine, so it runs in one kernel of one CTA per SM (16
// consumer warps in 4 teams of 4, one producer warp that issues the TMA copies):
//
//   prologue  (may overlap the previous kernel) the CTA's router rows and, when the CTA's first
//             gate/up unit belongs to the shared expert, that unit start streaming in;
//   phase 1   x (optionally RMS-normalised) becomes fp16 tensor-core fragments in shared memory;
//             the CTA scores its E / #CTA experts for all T tokens and publishes every logit as
//             one 64-bit word (launch epoch << 32 | order-preserving key);
//   phase 2   every CTA reads all T x E words, re-reading those whose tag is not yet this launch's,
//             and repeats the selection and the dispatch (identical, deterministic); CTA 0
//             publishes them;
//   phase 3   gate/up.  The slots (the shared expert first, then the distinct routed experts in
//             ascending order) are cut into units of 8 columns of f; unit g goes to CTA g mod
//             #CTA.  A unit (8 gate + 8 up rows x d) arrives as one 128-byte-swizzled TMA box plus
//             its scales; a team of 4 warps runs it as m16n8k16 tensor-core tiles (N = the slot's
//             tokens), sums its 4 warps' partial tiles in a fixed order, and publishes
//             h = w silu(gate) up (fp16, routing weight folded in) for its 8 columns as 64-bit
//             words (launch epoch << 32 | two fp16), one strong store each;
//   phase 4   down.  CTA c owns output rows [d c / #CTA, d (c + 1) / #CTA).  For every slot in
//             order the producer streams the slot's down rows of those outputs (TMA) as soon as a
//             stage is free; a team (one warp, with <= 16 items) copies the slot's h rows into the
//             stage, re-reading words whose tag is not yet this launch's, and multiplies them (N =
//             all T tokens; other tokens contribute zeros) into fp32 register accumulators kept
//             across the slots.  The 16 warps' partial sums are added in warp order and the
//             residual is added: y is written once, each element by one CTA.
//
// Nothing waits on a counter or a grid barrier: a word's tag tells its reader that the word is this
// launch's (a word is written and read as one single-copy-atomic access).
//
// Tensor-core operands: int4 codes become fp16 q exactly, x is fp16 (bf16 activations are exact in
// fp16 inside its range) and w * h is rounded once to fp16; every 32-code group is summed in fp32
// and scaled by its fp16 group scale in fp32.  Every wait is bounded; on timeout the CTA records
// MOE status "timeout", writes NaN to its rows of y, stops issuing, and waits (bounded) for its
// copies in flight before exiting.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace moe {

constexpr int kDlWarps = 16;                     // consumer warps
constexpr int kDlThreads = (kDlWarps + 1) * 32;  // + one producer warp
constexpr int kDlTeams = 4;                      // gate/up teams
constexpr int kDlTeamWarps = kDlWarps / kDlTeams;
constexpr int kDlMaxT = 16;                      // tokens: two n8 tiles
constexpr int kDlMaxStages = 16;
constexpr int kDlSmemMax = 227 * 1024;
constexpr int kDlStaticSlack = 12 * 1024;        // static shared memory, alignment and reserve
constexpr int kDlRowsMax = 16;                   // down rows per CTA: one m16 tile
constexpr int kDlUnit = 8;                       // f columns per gate/up unit
constexpr unsigned kDlSpinLimit = 1u << 24;      // polls of a tagged word, >= 32 ns apart
constexpr unsigned kDlProducerSleep = 128;       // ns between polls of the producer's waits
constexpr unsigned kDlConsumerSleep = 32;        // ns between polls of a waiting consumer warp
constexpr int kDlXPad = 4;                       // 16-byte blocks of padding per row of x fragments

// TMA descriptors of one layer (routed planes, then the shared expert's).
//   gu_q: 4-d view of the [rows][d/2] gate/up codes: (128 bytes, row, 128-byte chunk of the row,
//         gate|up), box (128, 8, d/256, 2) = one unit (8 gate rows + the matching 8 up rows), laid
//         out in shared memory as [gate|up][chunk][row][128 B] with the 128-byte swizzle;
//   gu_s: (d/32 scales, row, gate|up), box (d/32, 8, 2), unswizzled [gate|up][row][d/32];
//   dn_q: the down codes of `rows_box` consecutive rows: (128 bytes, row, chunk) box
//         (128, rows_box, f/256) -> [chunk][row][128 B] when dn_swap, else (128 bytes, chunk, row)
//         -> [row][chunk][128 B]; 128-byte swizzle either way;
//   dn_s: (f/32 scales, row), box (f/32, rows_box).
struct DlMaps {
  CUtensorMap gu_q, gu_s, dn_q, dn_s;
  CUtensorMap sh_gu_q, sh_gu_s, sh_dn_q, sh_dn_s;
};

struct DlArgs {
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
  unsigned long long* usage;
  unsigned long long* hw;        // [T (shared) + T*K][f/2]: (epoch << 32) | two fp16 of w silu(g) u, fragment order
  void* y;
  const void* resid;
  unsigned long long* lgt;       // [T][E] published logits: (launch epoch << 32) | order-preserving key
  unsigned long long* launches;  // every CTA of every launch adds 1 when it ends
  unsigned* status;
  int ns;                        // ring stages
  int stage_bytes;
  int rows_box;                  // down rows per TMA box (>= the rows of any CTA)
  int dn_swap;                   // down box layout, see DlMaps
  unsigned long long* timeline;  // [#CTA][kDlEvents] globaltimer stamps (ns), or null
};

// In-kernel timeline (tracing): one globaltimer stamp per CTA and event when enabled.
enum DlEvent {
  kEvStart = 0,        // kernel entered
  kEvDepWait,          // griddepcontrol.wait passed
  kEvLogits,           // logits stored
  kEvUnitComputed,     // first routed unit: warp 0 of its team finished its tensor-core loop
  kEvRouted,           // selection and dispatch done
  kEvFirstUnit,        // first gate/up unit's bytes landed (team 0)
  kEvUnitsDone,        // all of the CTA's gate/up units done
  kEvFirstDown,        // first down item's weights landed
  kEvDownDone,         // all down items done
  kEvEnd,              // y written
  kEvLastUnitIssued,   // producer: last gate/up unit issued
  kEvFirstDownIssued,  // producer: first down item's weights issued
  kEvLastDownIssued,   // producer: last down item's weights issued
  kEvFirstUnitIssued,  // producer: first gate/up unit issued after the routing
  kClkStart = 14,      // SM clock (clock64) at kernel entry
  kClkEnd = 15,        // SM clock when y is written
  kEvXStaged,          // x staged as fragments
  kEvRouterRows,       // router rows landed
  kEvKeys,             // selection keys loaded
  kEvSelected,         // top-K chosen
  kEvDispatched,       // dispatch done
  kEvProducerRouted,   // producer learned the routing
  kEvUnitReduced,      // first routed unit: its team's partial tiles are in shared memory
  kEvFirstDownDone,    // first down item done (its h rows were complete)
  kEvProducerGo,       // producer: routing broadcast to its warp, issue loop starts
  kEvGatherStart,      // consumers start reading the published logits
  kEvFirstRoutedLanded,  // first routed gate/up unit's bytes landed
  kEvFirstRoutedDone,    // first routed gate/up unit's h published
  kEvLastDownDone,       // the last slot's down item done
  kEvSecondLanded,       // the same team's next gate/up unit: its bytes landed (the team saw them)
  kEvSecondComputed,     // ... its tensor-core loop finished (warp 0 of the team)
  kEvSecondDone,         // ... its h published
  kDlEvents = 32
};
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define DL_STAMP(ev) \
  do { \
    if (a.timeline) a.timeline[(size_t)blockIdx.x * kDlEvents + (ev)] = gtimer(); \
  } while (0)
#define DL_CLOCK(ev) \
  do { \
    if (a.timeline) a.timeline[(size_t)blockIdx.x * kDlEvents + (ev)] = (unsigned long long)clock64(); \
  } while (0)

// ------------------------------------------------------------------ epoch-tagged words
// Two strong (relaxed, GPU scope) 64-bit loads as one vector access (each word single-copy atomic).
__device__ __forceinline__ void ld_relaxed_gpu_v2(const unsigned long long* p, unsigned long long& a,
                                                  unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
// Strong (relaxed, GPU scope) load: a poll of a word that another SM writes must be a strong
// operation to be sure to see the new value.
__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_gpu(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ------------------------------------------------------------------ shared-memory accesses
// Explicit shared-space loads and stores by 32-bit shared address.  The units' code reaches the
// kernel's dynamic shared memory through pointers kept in their shared context, which the compiler
// cannot prove to be shared, and generic loads from shared memory cost several times an ld.shared
// on this part; the hot paths use these instead.
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ int lds_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ int lds_s8(uint32_t a) {
  int v;
  asm volatile("ld.shared.s8 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_h2f(uint32_t a) {  // one fp16 value, widened
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return __half2float(__ushort_as_half(v));
}
__device__ __forceinline__ void sts_f4(uint32_t a, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}
__device__ __forceinline__ void sts_v2(uint32_t a, uint2 v) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ int lds_acquire_s32(uint32_t a) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_release_s32(uint32_t a, int v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Named barriers: 1 = the 512 consumer threads, 2 + team = the 128 threads of a gate/up team,
// 6 = the routing group (below).
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kDlWarps * 32) : "memory"); }
__device__ __forceinline__ bool consumers_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kDlWarps * 32)
      : "memory");
  return r != 0;
}
// Barrier 6: the routing group (the consumer threads [512 - n, 512)), n a multiple of 32.
__device__ __forceinline__ void group_sync(int n) { asm volatile("bar.sync 6, %0;" ::"r"(n) : "memory"); }
__device__ __forceinline__ bool group_all(int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 6, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void team_sync(int team) {
  asm volatile("bar.sync %0, %1;" ::"r"(2 + team), "n"(kDlTeamWarps * 32) : "memory");
}
__device__ __forceinline__ bool team_all(int team, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(2 + team), "n"(kDlTeamWarps * 32)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ tensor-core helpers
// D += A B for one m16n8k16 (A 16x16 row-major fp16, B 16x8 fp16, fp32 accumulators), in the
// register fragments of the PTX mma.sync description: lane = 4g + t holds A rows g and g + 8 (K
// slots 2t, 2t+1 in a0/a1, 2t+8, 2t+9 in a2/a3), B column g (K slots 2t, 2t+1 in b0, 2t+8, 2t+9
// in b1), C rows g and g + 8 at columns 2t and 2t + 1.
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Four 8x8 matrices of 16-bit elements from shared memory: lane 8m + r gives the address of row r
// of matrix m; lane 4g + t receives, in register m, the two elements (bytes 4t .. 4t+3) of row g of
// matrix m.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// The stored codes are two's complement nibbles n (q = n - 16 [n >= 8]); o = n ^ 8 = q + 8 is the
// offset-binary code.  q_lo: the codes in bits 0-3 and 16-19 of w as the fp16 pair (q, q'): one
// LOP3 builds 1024 + o under the exponent of 1024 -- mask ? (w ^ k) : k, truth table 0x6A, with
// k = 0x64086408: inside the mask k's bit 3 flips the nibble, outside it k supplies the exponent
// bits -- and one subtraction of 1032.
// q_hi: the codes in bits 4-7 and 20-23: 1024 + 16 o, times 1/16, minus 72.  Both exact.
__device__ __forceinline__ uint32_t q_lo(uint32_t w) {
  uint32_t p, r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(p) : "r"(w), "r"(0x000F000Fu), "r"(0x64086408u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(p), "r"(0x64086408u));  // 1032
  return r;
}
__device__ __forceinline__ uint32_t q_hi(uint32_t w) {
  uint32_t p, r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(p) : "r"(w), "r"(0x00F000F0u), "r"(0x64806480u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(p), "r"(0x2C002C00u), "r"(0xD480D480u));  // 1/16, -72
  return r;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);  // lo in the low 16 bits
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte offset of 16-byte sub-block `sub` of 128-byte line `line` of a tile written by TMA with the
// 128-byte swizzle (tile base 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(uint32_t line, uint32_t sub) { return line * 128u + ((sub ^ (line & 7u)) << 4); }

// One 32-code group of a tile: two k16 MMAs on the words wa (A rows g) and wb (rows g + 8) against
// the x / h fragment pairs b (pairs of columns (0,4), (1,5), (2,6), (3,7) of the lane's 8 columns).
__device__ __forceinline__ void mma_group(float (&dg)[4], uint32_t wa, uint32_t wb, const uint4& b) {
  dg[0] = dg[1] = dg[2] = dg[3] = 0.f;
  mma_16816(dg, q_lo(wa), q_lo(wb), q_hi(wa), q_hi(wb), b.x, b.y);
  mma_16816(dg, q_lo(wa >> 8), q_lo(wb >> 8), q_hi(wa >> 8), q_hi(wb >> 8), b.z, b.w);
}

__device__ __forceinline__ uint32_t max16(const uint32_t (&k)[16]) {  // a balanced tree
  uint32_t m8[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) m8[j] = max(k[2 * j], k[2 * j + 1]);
  const uint32_t a = max(max(m8[0], m8[1]), max(m8[2], m8[3])), b = max(max(m8[4], m8[5]), max(m8[6], m8[7]));
  return max(a, b);
}

// Top-K of one token by all 16 consumer warps (T = 1, E <= 512, K <= 16): warp w holds keys
// 32 w + lane.  The K-th largest of the 16 warp maxima is a lower bound of the K-th largest key (the
// K largest warp maxima are K keys), so the keys at or above it hold the selection; when there are
// at most 64 of them, warp w ranks candidates w, w + 16, ... against all the others (larger key,
// then lower expert: one ballot per half of the candidate list) and rank r < K is the r-th choice,
// written to sel[r].  Returns false (uniformly) when there were more candidates (many equal
// logits): the caller then selects with one warp.  Ends with the group barrier.
__device__ __forceinline__ bool topk_select_cta(const uint32_t* key, int EP, int K, int gw, int lane, int gt,
                                                uint32_t* wmax, uint2* cand, int* ncand, uint2* sel, int gn) {
  const uint32_t k = gt < EP ? key[gt] : 0u;
  const uint32_t wm = __reduce_max_sync(0xffffffffu, k);
  if (lane == 0) wmax[gw] = wm;
  if (gt == 0) *ncand = 0;
  group_sync(gn);
  const uint32_t mv = lane < kDlWarps ? wmax[lane] : 0u;
  int rk = 0;  // rank of this lane's warp maximum among the 16, ties to the lower warp
#pragma unroll
  for (int j = 0; j < kDlWarps; ++j) {
    const uint32_t o = __shfl_sync(0xffffffffu, mv, j);
    rk += (o > mv) || (o == mv && j < lane);
  }
  const uint32_t tau = __reduce_max_sync(0xffffffffu, lane < kDlWarps && rk == K - 1 ? mv : 0u);
  const bool is_c = k != 0u && k >= tau;
  const unsigned bal = __ballot_sync(0xffffffffu, is_c);
  int base = 0;
  if (lane == 0 && bal) base = atomicAdd(ncand, __popc(bal));
  base = __shfl_sync(0xffffffffu, base, 0);
  if (is_c) {
    const int pos = base + __popc(bal & ((1u << lane) - 1u));
    if (pos < 64) cand[pos] = make_uint2(k, (uint32_t)gt);
  }
  group_sync(gn);
  const int nc = *ncand;
  if (nc > 64) return false;
  const uint2 c0 = lane < nc ? cand[lane] : make_uint2(0u, 0u);
  const uint2 c1 = lane + 32 < nc ? cand[lane + 32] : make_uint2(0u, 0u);
#pragma unroll 1
  for (int m = gw; m < nc; m += kDlWarps) {
    const uint2 me = cand[m];
    const bool g0 = lane < nc && (c0.x > me.x || (c0.x == me.x && c0.y < me.y));
    const bool g1 = lane + 32 < nc && (c1.x > me.x || (c1.x == me.x && c1.y < me.y));
    const int rank = __popc(__ballot_sync(0xffffffffu, g0)) + __popc(__ballot_sync(0xffffffffu, g1));
    if (rank < K && lane == 0) sel[rank] = me;
  }
  group_sync(gn);
  return true;
}

// Top-K of one token by one warp from its keys in shared memory (key[e] = order-preserving key of
// logit e, never 0; 0 past E; E <= 512): lane l holds keys l + 32 j in registers and its maximum.
// Round r takes the largest remaining key (a warp max-reduction) and, among the lanes holding it,
// the lowest expert index (a min-reduction over each holder's lowest j), i.e. larger logit first,
// ties to the lower expert; the holder clears it.  Weights: exp(l - l_max) renormalised over the K
// kept (the full softmax's normaliser cancels).  Lane k < K returns the k-th expert and its weight.
__device__ __forceinline__ void topk_select_warp(const uint32_t* key, int E, int K, int& my_i, float& my_w) {
  const int lane = threadIdx.x & 31;
  const int nj = (E + 31) >> 5;
  uint32_t k[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) k[j] = j < nj ? key[j * 32 + lane] : 0u;
  uint32_t lm = max16(k);
  uint32_t my_key = 0u, top_key = 0u;
  my_i = 0;
#pragma unroll 1
  for (int r = 0; r < K; ++r) {
    const uint32_t mx = __reduce_max_sync(0xffffffffu, lm);
    uint32_t hit = 0u;  // bit j: k[j] holds the maximum (independent tests, an OR tree)
#pragma unroll
    for (int j = 0; j < 16; ++j) hit |= (k[j] == mx ? 1u : 0u) << j;
    const int jm = __ffs(hit) - 1;
    const uint32_t win = __reduce_min_sync(0xffffffffu, hit ? (uint32_t)(jm * 32 + lane) : 0xFFFFFFFFu);
    if (r == 0) top_key = mx;
    if (lane == r) {
      my_key = mx;
      my_i = (int)win;
    }
    if ((int)(win & 31u) == lane) {
#pragma unroll
      for (int j = 0; j < 16; ++j) k[j] = j == jm ? 0u : k[j];
      lm = max16(k);
    }
  }
  const float top = topk_key_value(top_key);
  const float p = lane < K ? expf(topk_key_value(my_key) - top) : 0.f;
  const float psum = warp_sum(p);
  my_w = lane < K ? p / psum : 0.f;
}

// What a gate/up unit needs to know about the launch and the CTA (one copy in shared memory).
struct UnitCtx {
  uint8_t* ring;
  const uint4* xh;        // [T][XS] x fragments
  float4* pgu;            // [16 warps][NT][32] partial tiles
  uint32_t ring_a, xh_a, pgu_a, perm_a, w_a, tpos_a;  // the same regions as shared addresses
  uint32_t avail_a;  // shared int: ring items whose copies the producer has issued (down items)
  const int4* slot_s;     // routed slots {expert, start, count, 0}
  const int* perm_s;
  const float* w_s;
  uint64_t* full;
  uint64_t* empty;
  volatile int* abort;
  unsigned long long* hw;   // [T + T*K][f/2] h, two fp16 columns per word under the launch's epoch tag
  unsigned long long ep_tag;  // this launch's epoch << 32
  unsigned long long* timeline;
  int NS, SB, XS, CH, d, f, fu, T, K, HS, c, nc, gu_code_bytes;
  int i0;  // the first routed unit's item index (timeline only)
  // down items
  const signed char* tpos;  // [slot][kDlMaxT] slot-local position of every token (-1: not in the slot)
  int RB, CHd, GF, dn_swap, dn_scale_off, dn_h_off;
};

// One gate/up unit (item i of this CTA) by the 4 warps of team `team`: wait for its bytes, run its
// 16 rows x d as m16n8k16 tiles over this warp's quarter of d, free the stage, sum the team's 4
// partial tiles in warp order, and publish h = w silu(gate) up (fp16) of its 8 columns and tokens.
// Returns false when a wait gave up (uniform over the team).
template <int NT>
__device__ __forceinline__ bool gu_unit(const UnitCtx& u, int i, int team, int tw, int lane) {
  const int g8 = lane >> 2, t4 = lane & 3;
  const int st = i % u.NS;
  // the unit's slot and tokens, while its bytes may still be landing
  const int g = u.c + i * u.nc, s = g / u.fu, un = g - s * u.fu;
  int n_s, start = 0;
  if (s < u.HS) {
    n_s = u.T;
  } else {
    const int4 sl = u.slot_s[s - u.HS];
    n_s = sl.z;
    start = sl.y;
  }
  // B fragments: the lane's column g8 of n-tile j is slot-local token 8 j + g8
  int xrow[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int n = 8 * j + g8;
    xrow[j] = n < n_s ? (s < u.HS ? n : lds_s32(u.perm_a + 4u * (start + n)) / u.K) * u.XS : -1;
  }
  // the epilogue's routing weights (warps tw < NT): slot-local tokens 8 tw + 2 (lane % 4) (+ 1)
  float wt[2] = {1.f, 1.f};
  if (tw < NT && s >= u.HS) {
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      const int n = 8 * tw + 2 * (lane & 3) + o;
      if (n < n_s) wt[o] = lds_f32(u.w_a + 4u * lds_s32(u.perm_a + 4u * (start + n)));
    }
  }
  const bool okw = tc::mbar_wait_warp(&u.full[st], (i / u.NS) & 1, u.abort, kDlConsumerSleep);
  if (!team_all(team, okw && !*u.abort)) return false;
  if (tw == 0 && lane == 0 && u.timeline) {
    if (i == 0) u.timeline[(size_t)u.c * kDlEvents + kEvFirstUnit] = gtimer();
    if (i == u.i0) u.timeline[(size_t)u.c * kDlEvents + kEvFirstRoutedLanded] = gtimer();
    if (i == u.i0 + kDlTeams) u.timeline[(size_t)u.c * kDlEvents + kEvSecondLanded] = gtimer();
  }
  const uint8_t* stg = u.ring + (size_t)st * u.SB;
  const uint32_t sbase = tc::smem_u32(stg);
  const int CH = u.CH, d = u.d;
  float C[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) C[j][0] = C[j][1] = C[j][2] = C[j][3] = 0.f;
  const int cb = tw * CH / kDlTeamWarps, cend = (tw + 1) * CH / kDlTeamWarps;  // this warp's chunks of K
  const uint32_t scl = sbase + (uint32_t)u.gu_code_bytes;  // [gate|up][8][d/32] fp16
  const int mi = lane >> 3, rr = lane & 7;
#pragma unroll 1
  for (int ch = cb; ch < cend; ++ch) {
    const uint4 sgv = lds_v4(scl + 2u * (uint32_t)(g8 * (d / 32) + ch * 8));
    const uint4 suv = lds_v4(scl + 2u * (uint32_t)((8 + g8) * (d / 32) + ch * 8));
    const uint32_t sgw[4] = {sgv.x, sgv.y, sgv.z, sgv.w}, suw[4] = {suv.x, suv.y, suv.z, suv.w};
    const uint32_t line = (uint32_t)(((mi & 1) * CH + ch) * 8 + rr);
#pragma unroll
    for (int jj = 0; jj < 8; jj += 2) {
      // matrices (gate, group jj), (up, jj), (gate, jj + 1), (up, jj + 1) of this chunk
      uint32_t wg0, wu0, wg1, wu1;
      ldsm_x4(sbase + swz(line, (uint32_t)(jj + (mi >> 1))), wg0, wu0, wg1, wu1);
      const float2 sg = __half22float2(*reinterpret_cast<const __half2*>(&sgw[jj >> 1]));
      const float2 su = __half22float2(*reinterpret_cast<const __half2*>(&suw[jj >> 1]));
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int J = ch * 8 + jj + h2;  // group of 32 columns of d
        const float sgf = h2 ? sg.y : sg.x, suf = h2 ? su.y : su.x;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const uint4 xb = xrow[j] >= 0 ? lds_v4(u.xh_a + 16u * (uint32_t)(xrow[j] + 4 * J + t4)) : make_uint4(0u, 0u, 0u, 0u);
          float dg[4];
          mma_group(dg, h2 ? wg1 : wg0, h2 ? wu1 : wu0, xb);
          C[j][0] = fmaf(sgf, dg[0], C[j][0]);
          C[j][1] = fmaf(sgf, dg[1], C[j][1]);
          C[j][2] = fmaf(suf, dg[2], C[j][2]);
          C[j][3] = fmaf(suf, dg[3], C[j][3]);
        }
      }
    }
  }
  __syncwarp();
  if (lane == 0) tc::mbar_arrive_cnt(&u.empty[st], kDlWarps / kDlTeamWarps);  // the stage is free
  if (tw == 0 && lane == 0 && u.timeline && i == u.i0) u.timeline[(size_t)u.c * kDlEvents + kEvUnitComputed] = gtimer();
  if (tw == 0 && lane == 0 && u.timeline && i == u.i0 + kDlTeams)
    u.timeline[(size_t)u.c * kDlEvents + kEvSecondComputed] = gtimer();
  const uint32_t my_p = u.pgu_a + 16u * (uint32_t)((team * kDlTeamWarps + tw) * NT * 32);
#pragma unroll
  for (int j = 0; j < NT; ++j) sts_f4(my_p + 16u * (uint32_t)(j * 32 + lane), make_float4(C[j][0], C[j][1], C[j][2], C[j][3]));
  team_sync(team);
  if (tw == 0 && lane == 0 && u.timeline && i == u.i0) u.timeline[(size_t)u.c * kDlEvents + kEvUnitReduced] = gtimer();
  // team thread (j, ln): column ln / 4 of the unit, slot-local tokens 8 j + 2 (ln % 4) (+ 1); the
  // team's 4 partial tiles are summed in warp order.  The words of h pair the unit's columns c and
  // c + 4 (fragment positions 2c, 2c + 1); each is published under the launch's epoch tag with one
  // strong store, so a reader that sees the tag sees the values.
  const int tt = tw * 32 + lane;
  if (tt < NT * 32) {  // whole warps
    const int j = tt >> 5, ln = tt & 31;
    const int col = ln >> 2, n0 = 8 * j + 2 * (ln & 3);
    float4 sum = lds_f4(u.pgu_a + 16u * (uint32_t)(((team * kDlTeamWarps) * NT + j) * 32 + ln));
#pragma unroll
    for (int q = 1; q < kDlTeamWarps; ++q) {
      const float4 pp = lds_f4(u.pgu_a + 16u * (uint32_t)(((team * kDlTeamWarps + q) * NT + j) * 32 + ln));
      sum.x += pp.x;
      sum.y += pp.y;
      sum.z += pp.z;
      sum.w += pp.w;
    }
    float hv[2];
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      const float gte = o ? sum.y : sum.x, upv = o ? sum.w : sum.z;
      // silu with the fast exponential and division: h is rounded to fp16 right after
      hv[o] = wt[o] * (__fdividef(gte, 1.0f + __expf(-gte)) * upv);
    }
    const float hp0 = __shfl_xor_sync(0xffffffffu, hv[0], 16), hp1 = __shfl_xor_sync(0xffffffffu, hv[1], 16);
    if (col < 4) {
#pragma unroll
      for (int o = 0; o < 2; ++o) {
        const int n = n0 + o;
        if (n < n_s) {
          const size_t row = s < u.HS ? (size_t)n : (size_t)u.HS * u.T + start + n;
          const uint32_t pair = pack_h2(o ? hv[1] : hv[0], o ? hp1 : hp0);
          st_relaxed_gpu(u.hw + row * (u.f / 2) + 4 * un + col, u.ep_tag | pair);
        }
      }
    }
  }
  if (tw == 0 && lane == 0 && u.timeline && i == u.i0) u.timeline[(size_t)u.c * kDlEvents + kEvFirstRoutedDone] = gtimer();
  if (tw == 0 && lane == 0 && u.timeline && i == u.i0 + kDlTeams)
    u.timeline[(size_t)u.c * kDlEvents + kEvSecondDone] = gtimer();
  return true;
}

// One down item (slot s, item k of this CTA) by the 4 warps of team `team`: wait for the slot's down
// rows of this CTA's outputs, copy the slot's h rows from their epoch-tagged words into the stage
// (polling words whose tag is not yet this launch's), and add this warp's quarter of the slot's
// 32-column groups into the warp's accumulators D (rows g / g + 8 of the CTA's output tile, all T
// tokens as N; a token not in the slot contributes zeros); free the stage.  With two token tiles
// (T > 8) an item covers at most 8 of the slot's tokens, slot-local 8 half .. 8 half + 7, so that a
// stage holds the h rows of 8 tokens at most.  Returns false when a wait gave up.
template <int NT>
__device__ __forceinline__ bool down_item(const UnitCtx& u, int k, int s, int half, int team, int tw, int lane,
                                          float (&D)[NT][4]) {
  const int g8 = lane >> 2, t4 = lane & 3;
  const int st = k % u.NS;
  const bool okw = tc::mbar_wait_warp(&u.full[st], (k / u.NS) & 1, u.abort, kDlConsumerSleep);
  if (!team_all(team, okw && !*u.abort)) return false;
  uint8_t* stg = u.ring + (size_t)st * u.SB;
  {
    // the stage is this item's (its weights landed, so its previous item is done with it)
    int n_s, hrow0;
    if (s < u.HS) {
      n_s = u.T;
      hrow0 = 0;
    } else {
      const int4 sl = u.slot_s[s - u.HS];
      n_s = sl.z;
      hrow0 = u.HS * u.T + sl.y;
    }
    if constexpr (NT == 2) {  // the item's half of the slot: slot-local tokens 8 half .. 8 half + 7
      n_s = half ? n_s - 8 : min(n_s, 8);
      hrow0 += 8 * half;
    }
    const unsigned ept = (unsigned)(u.ep_tag >> 32);
    const unsigned long long* src = u.hw + (size_t)hrow0 * (u.f / 2);
    const uint32_t hdst = tc::smem_u32(stg) + (uint32_t)u.dn_h_off;  // [n_s][f/4] pairs of words' payloads
    const int npair = n_s * (u.f / 4), tt = tw * 32 + lane;
    bool okh = true;
#pragma unroll 1
    for (int base = 0; okh && base < npair; base += 4 * kDlTeamWarps * 32) {
      unsigned long long w[8];
      int pending = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int pi = base + tt + q * kDlTeamWarps * 32;
        if (pi < npair)
          ld_relaxed_gpu_v2(src + 2 * pi, w[2 * q], w[2 * q + 1]);
        else
          w[2 * q] = w[2 * q + 1] = u.ep_tag;
        pending += ((unsigned)(w[2 * q] >> 32) != ept) + ((unsigned)(w[2 * q + 1] >> 32) != ept);
      }
      unsigned polls = 0;
      while (pending) {
        if (++polls > kDlSpinLimit || *u.abort) {
          okh = false;
          break;
        }
        __nanosleep(32);
        pending = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int pi = base + tt + q * kDlTeamWarps * 32;
          if ((unsigned)(w[2 * q] >> 32) != ept || (unsigned)(w[2 * q + 1] >> 32) != ept) {
            ld_relaxed_gpu_v2(src + 2 * pi, w[2 * q], w[2 * q + 1]);
            pending += ((unsigned)(w[2 * q] >> 32) != ept) + ((unsigned)(w[2 * q + 1] >> 32) != ept);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int pi = base + tt + q * kDlTeamWarps * 32;
        if (pi < npair) sts_v2(hdst + 8u * (uint32_t)pi, make_uint2((uint32_t)w[2 * q], (uint32_t)w[2 * q + 1]));
      }
    }
    // (also the team barrier that makes the h rows visible to the team)
    if (!team_all(team, okh && !*u.abort)) return false;
  }
  const uint32_t sbase = tc::smem_u32(stg);
  const uint32_t dsc = sbase + (uint32_t)u.dn_scale_off;  // [RB][GF] fp16
  const uint32_t hrows = sbase + (uint32_t)u.dn_h_off;    // [n_s][f/8] 16-byte blocks
  const uint32_t tp = u.tpos_a + (uint32_t)(s * kDlMaxT);
  const int RB = u.RB, GF = u.GF;
  int hpos[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int n = 8 * j + g8;
    if constexpr (NT == 2) {  // the token's row among the item's staged rows, or -1
      const int pr = n < u.T ? lds_s8(tp + (uint32_t)n) - 8 * half : -1;
      hpos[j] = pr >= 0 && pr < 8 ? pr * (u.f / 8) : -1;
    } else {
      hpos[j] = n < u.T ? lds_s8(tp + (uint32_t)n) * (u.f / 8) : -1;
    }
  }
  const int rga = min(g8, RB - 1), rgb = min(g8 + 8, RB - 1);
  const int rrow = min((lane & 7) + 8 * ((lane >> 3) & 1), RB - 1);  // ldmatrix row address of this lane
  const int jb = tw * GF / kDlTeamWarps, je = (tw + 1) * GF / kDlTeamWarps;
#pragma unroll 2
  for (int jg = jb; jg < je; ++jg) {
    const int chd = jg >> 3, sub = jg & 7;
    const uint32_t line = u.dn_swap ? (uint32_t)(chd * RB + rrow) : (uint32_t)(rrow * u.CHd + chd);
    uint32_t wa, wb;
    ldsm_x2(sbase + swz(line, (uint32_t)sub), wa, wb);
    const float sa = lds_h2f(dsc + 2u * (uint32_t)(rga * GF + jg)), sb = lds_h2f(dsc + 2u * (uint32_t)(rgb * GF + jg));
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const uint4 hb = hpos[j] >= 0 ? lds_v4(hrows + 16u * (uint32_t)(hpos[j] + 4 * jg + t4)) : make_uint4(0u, 0u, 0u, 0u);
      float dd[4];
      mma_group(dd, wa, wb, hb);
      D[j][0] = fmaf(sa, dd[0], D[j][0]);
      D[j][1] = fmaf(sa, dd[1], D[j][1]);
      D[j][2] = fmaf(sb, dd[2], D[j][2]);
      D[j][3] = fmaf(sb, dd[3], D[j][3]);
    }
  }
  __syncwarp();
  if (lane == 0) tc::mbar_arrive_cnt(&u.empty[st], kDlWarps / kDlTeamWarps);  // the stage is free
  return true;
}

// The same down item taken by one warp alone, over all of the slot's groups (used when a CTA has
// at most 16 down items, so that they all run at once): wait for the slot's down rows of this
// CTA's outputs, copy the slot's h rows from their epoch-tagged words into the stage (polling words
// whose tag is not yet this launch's), and add all of the slot's 32-column groups into the warp's
// accumulators D (rows g / g + 8 of the CTA's output tile, all T tokens as N; a token not in the
// slot contributes zeros); free the stage.  With two token tiles (T > 8) an item covers at most 8 of
// the slot's tokens, slot-local 8 half .. 8 half + 7, so that a stage holds the h rows of 8 tokens
// at most.  Returns false (uniformly over the warp) when a wait gave up.
template <int NT>
__device__ __forceinline__ bool down_item_warp(const UnitCtx& u, int k, int s, int half, int lane,
                                               float (&D)[NT][4]) {
  const int g8 = lane >> 2, t4 = lane & 3;
  const int st = k % u.NS;
  // A parity wait tells a phase only from the one before it: a warp that came to this item early
  // could see the stage's previous phase (item k - NS) still pending and take it for this one.  Once
  // the producer has issued item k, item k - NS is consumed and its phase complete.
  {
    int ready = 1;
    if (lane == 0) {
      unsigned polls = 0;
      while (lds_acquire_s32(u.avail_a) <= k) {
        if (++polls > kDlSpinLimit || *u.abort) {
          ready = 0;
          break;
        }
        __nanosleep(32);
      }
    }
    if (!__shfl_sync(0xffffffffu, ready, 0)) return false;
  }
  // every lane polls the barrier, so every lane acquires the landed rows
  if (!tc::mbar_wait_all(&u.full[st], (k / u.NS) & 1, u.abort)) return false;
  if (__any_sync(0xffffffffu, *u.abort != 0)) return false;
  uint8_t* stg = u.ring + (size_t)st * u.SB;
  {
    // the stage is this item's (its weights landed, so its previous item is done with it)
    int n_s, hrow0;
    if (s < u.HS) {
      n_s = u.T;
      hrow0 = 0;
    } else {
      const int4 sl = u.slot_s[s - u.HS];
      n_s = sl.z;
      hrow0 = u.HS * u.T + sl.y;
    }
    if constexpr (NT == 2) {  // the item's half of the slot: slot-local tokens 8 half .. 8 half + 7
      n_s = half ? n_s - 8 : min(n_s, 8);
      hrow0 += 8 * half;
    }
    const unsigned ept = (unsigned)(u.ep_tag >> 32);
    const unsigned long long* src = u.hw + (size_t)hrow0 * (u.f / 2);
    const uint32_t hdst = tc::smem_u32(stg) + (uint32_t)u.dn_h_off;  // [n_s][f/4] pairs of words' payloads
    const int npair = n_s * (u.f / 4);
    bool okh = true;
#pragma unroll 1
    for (int base = 0; okh && base < npair; base += 4 * 32) {
      unsigned long long w[8];
      int pending = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int pi = base + lane + q * 32;
        if (pi < npair)
          ld_relaxed_gpu_v2(src + 2 * pi, w[2 * q], w[2 * q + 1]);
        else
          w[2 * q] = w[2 * q + 1] = u.ep_tag;
        pending += ((unsigned)(w[2 * q] >> 32) != ept) + ((unsigned)(w[2 * q + 1] >> 32) != ept);
      }
      unsigned polls = 0;
      while (pending) {
        if (++polls > kDlSpinLimit || *u.abort) {
          okh = false;
          break;
        }
        __nanosleep(32);
        pending = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int pi = base + lane + q * 32;
          if ((unsigned)(w[2 * q] >> 32) != ept || (unsigned)(w[2 * q + 1] >> 32) != ept) {
            ld_relaxed_gpu_v2(src + 2 * pi, w[2 * q], w[2 * q + 1]);
            pending += ((unsigned)(w[2 * q] >> 32) != ept) + ((unsigned)(w[2 * q + 1] >> 32) != ept);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int pi = base + lane + q * 32;
        if (pi < npair) sts_v2(hdst + 8u * (uint32_t)pi, make_uint2((uint32_t)w[2 * q], (uint32_t)w[2 * q + 1]));
      }
    }
    if (!__all_sync(0xffffffffu, okh && !*u.abort)) return false;
    __syncwarp();  // the h rows are visible to the warp
  }
  const uint32_t sbase = tc::smem_u32(stg);
  const uint32_t dsc = sbase + (uint32_t)u.dn_scale_off;  // [RB][GF] fp16
  const uint32_t hrows = sbase + (uint32_t)u.dn_h_off;    // [n_s][f/8] 16-byte blocks
  const uint32_t tp = u.tpos_a + (uint32_t)(s * kDlMaxT);
  const int RB = u.RB, GF = u.GF;
  int hpos[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int n = 8 * j + g8;
    if constexpr (NT == 2) {  // the token's row among the item's staged rows, or -1
      const int pr = n < u.T ? lds_s8(tp + (uint32_t)n) - 8 * half : -1;
      hpos[j] = pr >= 0 && pr < 8 ? pr * (u.f / 8) : -1;
    } else {
      hpos[j] = n < u.T ? lds_s8(tp + (uint32_t)n) * (u.f / 8) : -1;
    }
  }
  const int rga = min(g8, RB - 1), rgb = min(g8 + 8, RB - 1);
  const int rrow = min((lane & 7) + 8 * ((lane >> 3) & 1), RB - 1);  // ldmatrix row address of this lane
#pragma unroll 2
  for (int jg = 0; jg < GF; ++jg) {
    const int chd = jg >> 3, sub = jg & 7;
    const uint32_t line = u.dn_swap ? (uint32_t)(chd * RB + rrow) : (uint32_t)(rrow * u.CHd + chd);
    uint32_t wa, wb;
    ldsm_x2(sbase + swz(line, (uint32_t)sub), wa, wb);
    const float sa = lds_h2f(dsc + 2u * (uint32_t)(rga * GF + jg)), sb = lds_h2f(dsc + 2u * (uint32_t)(rgb * GF + jg));
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const uint4 hb = hpos[j] >= 0 ? lds_v4(hrows + 16u * (uint32_t)(hpos[j] + 4 * jg + t4)) : make_uint4(0u, 0u, 0u, 0u);
      float dd[4];
      mma_group(dd, wa, wb, hb);
      D[j][0] = fmaf(sa, dd[0], D[j][0]);
      D[j][1] = fmaf(sa, dd[1], D[j][1]);
      D[j][2] = fmaf(sb, dd[2], D[j][2]);
      D[j][3] = fmaf(sb, dd[3], D[j][3]);
    }
  }
  __syncwarp();
  if (lane == 0) tc::mbar_arrive_cnt(&u.empty[st], kDlWarps);  // the stage is free (one warp)
  return true;
}

// ------------------------------------------------------------------ the kernel
template <int NT>  // n8 token tiles: 1 (T <= 8) or 2 (T <= 16)
__global__ void __launch_bounds__(kDlThreads, 1) decode_layer_kernel(const DlArgs a, const __grid_constant__ DlMaps m) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);  // 1024-byte aligned
  const int T = a.T, d = a.d, E = a.E, K = a.K, f = a.f;
  const int nc = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = a.ns, SB = a.stage_bytes, RB = a.rows_box;
  const int fu = f / kDlUnit;          // units per slot (unit g of the CTA plan: slot g / fu)
  const int CH = d / 256;              // 128-byte chunks of a gate/up row
  const int CHd = f / 256;             // 128-byte chunks of a down row
  const int GF = f / 32;               // scale groups of a down row
  const int NB = d / 8;                // 8-column blocks of x
  const int XS = NB + kDlXPad;         // row stride of the x fragments (conflict-free B loads)
  const int HS = a.has_shared ? 1 : 0;
  const int gu_code_bytes = CH * 2048;                       // 2 halves x CH chunks x 8 rows x 128 B
  const int dn_code_bytes = RB * CHd * 128;
  const int dn_scale_off = (dn_code_bytes + 127) & ~127;
  const int dn_h_off = (dn_scale_off + RB * GF * 2 + 127) & ~127;

  // this CTA's fixed shares
  const int e0 = (int)((long long)E * c / nc), ne = (int)((long long)E * (c + 1) / nc) - e0;  // router rows
  const int r0 = (int)((long long)d * c / nc), nr = (int)((long long)d * (c + 1) / nc) - r0;  // down rows

  // shared memory: ring | xh | pgu | slot tables
  uint8_t* ring = smem;
  uint4* xh = reinterpret_cast<uint4*>(ring + (size_t)NS * SB);           // [T][XS] fp16 fragment blocks
  float4* pgu = reinterpret_cast<float4*>(xh + (size_t)T * XS);          // [16 warps][NT][32] partial tiles
  int4* slot_s = reinterpret_cast<int4*>(pgu + kDlWarps * NT * 32);      // [T*K] {expert, start, count, 0}
  signed char* tpos = reinterpret_cast<signed char*>(slot_s + T * K);    // [T*K + 1][kDlMaxT]: slot-local position
  int* perm_s = reinterpret_cast<int*>(tpos + (size_t)(T * K + 1) * kDlMaxT);  // [T*K]
  int* idx_s = perm_s + T * K;                                           // [T*K]
  float* w_s = reinterpret_cast<float*>(idx_s + T * K);                  // [T*K]
  // the router rows, then the selection's keys, use ring stages 1 and 2: both are done with before
  // the routed units are issued
  uint8_t* scratch = ring + SB;
  const float* wr_s = reinterpret_cast<const float*>(scratch);

  __shared__ __align__(8) uint64_t full[kDlMaxStages], empty[kDlMaxStages], wr_full, route_ready;
  __shared__ UnitCtx uc_s;
  __shared__ uint32_t s_bits[32], s_bpre[32];  // dispatch: bitmap of the selected experts, its prefix counts
  __shared__ uint32_t s_wmax[kDlWarps];          // one-token selection: the warps' maximum keys,
  __shared__ uint2 s_cand[64], s_sel[kDlWarps];  // the candidates (key, expert) and the ranked choices
  __shared__ int s_ncand;
  __shared__ volatile int s_abort;
  __shared__ unsigned s_ep;
  __shared__ int s_nact, s_issued, s_avail;
  __shared__ int s_big[64], s_nbig;  // T > 8: the slots with more than 8 tokens (their second down items)
  __shared__ float lpart[kDlWarps * kDlMaxT];
  __shared__ float inv_s[kDlMaxT];
  __shared__ float bias_s[kDlRowsMax];                 // this CTA's router bias entries
  __shared__ float resid_s[kDlMaxT * kDlRowsMax];      // the residual of this CTA's output rows

  // This launch may start while the previous kernel in the stream is still finishing
  // (programmatic dependent launch): before griddepcontrol.wait only this CTA's shared memory and
  // read-only weights are touched.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    // bring every line of the launch's argument block into this SM's constant cache now (the
    // later phases each touch other fields; a miss there would sit on their critical path)
    const unsigned long long touch = reinterpret_cast<uintptr_t>(a.x) ^ reinterpret_cast<uintptr_t>(a.idx) ^
                                     reinterpret_cast<uintptr_t>(a.slots) ^ reinterpret_cast<uintptr_t>(a.usage) ^
                                     reinterpret_cast<uintptr_t>(a.y) ^ reinterpret_cast<uintptr_t>(a.lgt) ^
                                     reinterpret_cast<uintptr_t>(a.timeline) ^ (unsigned long long)a.ns;
    asm volatile("" ::"l"(touch));
    DL_STAMP(kEvStart);
    DL_CLOCK(kClkStart);
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], kDlWarps);
    }
    tc::mbar_init(&wr_full, 1);
    tc::mbar_init(&route_ready, 1);
    s_abort = 0;
    s_issued = 0;
    s_avail = 0;
    s_nbig = 0;
    UnitCtx& u = uc_s;
    u.ring = ring;
    u.xh = xh;
    u.pgu = pgu;
    u.ring_a = tc::smem_u32(ring);
    u.xh_a = tc::smem_u32(xh);
    u.pgu_a = tc::smem_u32(pgu);
    u.perm_a = tc::smem_u32(perm_s);
    u.w_a = tc::smem_u32(w_s);
    u.tpos_a = tc::smem_u32(tpos);
    u.avail_a = tc::smem_u32(&s_avail);
    u.slot_s = slot_s;
    u.perm_s = perm_s;
    u.w_s = w_s;
    u.full = full;
    u.empty = empty;
    u.abort = &s_abort;
    u.hw = a.hw;
    u.timeline = a.timeline;
    u.NS = NS;
    u.SB = SB;
    u.XS = XS;
    u.CH = CH;
    u.d = d;
    u.f = f;
    u.fu = fu;
    u.T = T;
    u.K = K;
    u.HS = HS;
    u.c = c;
    u.nc = nc;
    u.gu_code_bytes = gu_code_bytes;
    u.i0 = (HS && c < fu) ? 1 : 0;
    u.tpos = tpos;
    u.RB = RB;
    u.CHd = CHd;
    u.GF = GF;
    u.dn_swap = a.dn_swap;
    u.dn_scale_off = dn_scale_off;
    u.dn_h_off = dn_h_off;
    tc::fence_mbar_init();
  }
  __syncthreads();

  // ---- the unit plan (identical in the producer and the consumers): unit g = c + i * nc
  const bool first_is_shared = HS && c < fu;
  UnitCtx* uc = &uc_s;

  if (warp == kDlWarps) {
    // ================================================================ producer
    // The whole warp runs the control flow (converged: a lane that loops alone while the others
    // wait at a warp-synchronous point runs far slower); lane 0 issues the copies.
    const int k = first_is_shared ? 1 : 0;  // items issued before the routing is known
    bool ok = true;
    if (lane == 0) {
      // warm the routed experts' descriptors in the TMA unit: a small L2 prefetch through each (the
      // rows of expert 0 that this CTA would read; harmless if unused)
      tc::tma_prefetch_l2_4d(&m.gu_q, 0, 0, 0, 0);
      tc::tma_prefetch_l2_3d(&m.gu_s, 0, 0, 0);
      if (a.dn_swap)
        tc::tma_prefetch_l2_3d(&m.dn_q, 0, r0, 0);
      else
        tc::tma_prefetch_l2_3d(&m.dn_q, 0, 0, r0);
      tc::tma_prefetch_l2_2d(&m.dn_s, 0, r0);
      if (ne > 0) {
        tc::mbar_arrive_expect_tx(&wr_full, (uint32_t)(ne * d * 4));
        tc::bulk_g2s(scratch, a.Wr + (size_t)e0 * d, (uint32_t)(ne * d * 4), &wr_full);
      }
      if (first_is_shared) {
        tc::mbar_arrive_expect_tx(&full[0], (uint32_t)(gu_code_bytes + 2 * 8 * (d / 32) * 2));
        tc::tma_load_4d(ring, &m.sh_gu_q, 0, 8 * c, 0, 0, &full[0]);
        tc::tma_load_3d(ring + gu_code_bytes, &m.sh_gu_s, 0, 8 * c, 0, &full[0]);
        s_issued = 1;
      }
    }
    __syncwarp();
    ok = tc::mbar_wait_sleepy(&route_ready, 0, &s_abort, 32);
    ok = __all_sync(0xffffffffu, ok);
    const int nact = ok ? s_nact : 0;
    if (lane == 0) DL_STAMP(kEvProducerRouted);
    const int nslots = HS + nact;
    const int nitems = nslots + (NT == 2 && ok ? s_nbig : 0);  // down items
    const int total_units = nslots * fu;
    const int nG = total_units > c ? (total_units - c + nc - 1) / nc : 0;
    if (lane == 0) DL_STAMP(kEvProducerGo);
    // gate/up units in order; a stage is waited for only once the ring wraps
    {
      const uint32_t gu_bytes = (uint32_t)(gu_code_bytes + 2 * 8 * (d / 32) * 2);
      int st = k % NS, ph = (k / NS) & 1;
      int g = c + k * nc, sl = g / fu, u = g - sl * fu;
      const int step_s = nc / fu, step_u = nc - step_s * fu;  // g += nc in (slot, unit) coordinates
      int i = k;
#pragma unroll 1
      for (; i < nG; ++i) {
        if (i >= NS && !__all_sync(0xffffffffu, tc::mbar_wait_sleepy(&empty[st], ph ^ 1u, &s_abort, kDlProducerSleep))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* dst = ring + (size_t)st * SB;
          tc::mbar_arrive_expect_tx(&full[st], gu_bytes);
          if (sl < HS) {
            tc::tma_load_4d(dst, &m.sh_gu_q, 0, 8 * u, 0, 0, &full[st]);
            tc::tma_load_3d(dst + gu_code_bytes, &m.sh_gu_s, 0, 8 * u, 0, &full[st]);
          } else {
            const int row = slot_s[sl - HS].x * 2 * f + 8 * u;
            tc::tma_load_4d(dst, &m.gu_q, 0, row, 0, 0, &full[st]);
            tc::tma_load_3d(dst + gu_code_bytes, &m.gu_s, 0, row, 0, &full[st]);
          }
          if (i == k) DL_STAMP(kEvFirstUnitIssued);
        }
        if (++st == NS) {
          st = 0;
          ph ^= 1;
        }
        sl += step_s;
        u += step_u;
        if (u >= fu) {
          u -= fu;
          ++sl;
        }
      }
      if (lane == 0) {
        s_issued = i;
        DL_STAMP(kEvLastUnitIssued);
      }
    }
    __syncwarp();
    // down items: the weights of slot s's down rows (this CTA's outputs) as soon as a ring stage is
    // free; the slots' h rows are read by the teams themselves
    {
      int q = 0;
#pragma unroll 1
      for (; ok && q < nitems; ++q) {
        const int item = nG + q, st = item % NS;
        const int sq = q < nslots ? q : s_big[q - nslots];  // the item's slot
        if (item >= NS &&
            !__all_sync(0xffffffffu, tc::mbar_wait_sleepy(&empty[st], ((item / NS) & 1) ^ 1u, &s_abort, kDlProducerSleep))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const CUtensorMap *mq, *ms;
          int drow;
          if (sq < HS) {
            mq = &m.sh_dn_q;
            ms = &m.sh_dn_s;
            drow = r0;
          } else {
            mq = &m.dn_q;
            ms = &m.dn_s;
            drow = slot_s[sq - HS].x * d + r0;
          }
          uint8_t* dst = ring + (size_t)st * SB;
          tc::mbar_arrive_expect_tx(&full[st], (uint32_t)(dn_code_bytes + RB * GF * 2));
          if (a.dn_swap)
            tc::tma_load_3d(dst, mq, 0, drow, 0, &full[st]);
          else
            tc::tma_load_3d(dst, mq, 0, 0, drow, &full[st]);
          tc::tma_load_2d(dst + dn_scale_off, ms, 0, drow, &full[st]);
          sts_release_s32(tc::smem_u32(&s_avail), item + 1);  // item's copies are issued
          if (q == 0) DL_STAMP(kEvFirstDownIssued);
          if (q == nitems - 1) DL_STAMP(kEvLastDownIssued);
        }
      }
      if (lane == 0) s_issued = nG + q;
    }
    if (!ok && lane == 0) {
      atomicOr(a.status, kStatusTimeout);
      s_abort = 1;
    }
    __syncwarp();
  } else {
    // ================================================================ consumers
    const int ctid = threadIdx.x;
    const int team = warp / kDlTeamWarps, tw = warp % kDlTeamWarps;
    bool ok = true;

    // the router bias rows are weights: read before the previous kernel has finished
    if (a.bias && ctid < ne) bias_s[ctid] = __ldg(a.bias + e0 + ctid);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous kernel's writes are visible
    // ctid 0 reads the launch state while the others load x; the barrier after the x staging
    // publishes it
    if (ctid == 0) {
      DL_STAMP(kEvDepWait);
      // this launch's epoch: 1 + the number of complete launches.  Every CTA adds 1 to the counter
      // when it ends; the previous launch is complete and fewer than gridDim.x additions of this
      // launch can precede this read (this CTA's own is not among them), so the quotient is exact.
      // A launch that gave up leaves the status word's timeout bit set: then this one gives up too
      // (its y is NaN) until moe_get_device_status has reported it and reset the state.
      const unsigned ep = (unsigned)(__ldcg(a.launches) / (unsigned long long)nc) + 1u, stw = __ldcg(a.status);
      if (stw & kStatusTimeout) s_abort = 1;
      s_ep = ep;
      uc_s.ep_tag = (unsigned long long)ep << 32;
    }

    // ---- phase 1: x (optionally RMS-normalised) as fp16 fragments, then the logits
    if (a.prenorm) {
#pragma unroll 1
      for (int t = warp; t < T; t += kDlWarps) {
        float ss = 0.f;
#pragma unroll 4
        for (int cc = lane; cc < NB; cc += 32) {
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
    {
      // all of a thread's x loads in flight at once (at most 8 per thread: T * d / 8 <= 4096)
      uint4 xraw[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int cc = ctid + q * kDlWarps * 32;
        if (cc < T * NB) xraw[q] = __ldg(reinterpret_cast<const uint4*>(a.x) + cc);
      }
#pragma unroll 1
      for (int q = 0; q < 8; ++q) {
        const int cc = ctid + q * kDlWarps * 32;
        if (cc >= T * NB) break;
        const uint4 xr = q == 0 ? xraw[0] : q == 1 ? xraw[1] : q == 2 ? xraw[2] : q == 3 ? xraw[3]
                       : q == 4 ? xraw[4] : q == 5 ? xraw[5] : q == 6 ? xraw[6] : xraw[7];
        const uint32_t wv[4] = {xr.x, xr.y, xr.z, xr.w};
        float v[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // bf16 pairs
          v[2 * j] = __uint_as_float(wv[j] << 16);
          v[2 * j + 1] = __uint_as_float(wv[j] & 0xFFFF0000u);
        }
        const int ti = cc / NB, b = cc - ti * NB;
        if (a.prenorm) {
#pragma unroll
          for (int qq = 0; qq < 8; ++qq) {
            v[qq] = round_act(a.act, v[qq] * inv_s[ti]);
            if (c == 0) store_act(a.xnorm, a.act, (size_t)cc * 8 + qq, v[qq]);
          }
        }
        // fragment order of the 8 columns: pairs (0,4), (1,5), (2,6), (3,7)
        xh[(size_t)ti * XS + b] =
            make_uint4(pack_h2(v[0], v[4]), pack_h2(v[1], v[5]), pack_h2(v[2], v[6]), pack_h2(v[3], v[7]));
      }
      // the residual of this CTA's output rows, for the end
      if (a.resid)
        for (int i = ctid; i < T * nr; i += kDlWarps * 32) {
          const int n = i / nr, r = i - n * nr;
          resid_s[i] = load_act(a.resid, a.act, (size_t)n * d + r0 + r);
        }
    }
    consumers_sync();
    const unsigned long long ep_tag = (unsigned long long)s_ep << 32;
    ok = !s_abort;
    if (ctid == 0) DL_STAMP(kEvXStaged);
    {
      // logits of the router rows [e0, e0 + ne): warp = (row, part of the columns), tokens 4 at a time
      const int nparts = ne > 0 ? max(1, kDlWarps / ne) : 1;
      const int my_e = warp % max(ne, 1), my_pt = warp / max(ne, 1);
      const bool r_on = ne > 0 && my_pt < nparts;
      if (ne > 0) ok = tc::mbar_wait_warp(&wr_full, 0, &s_abort, kDlConsumerSleep);
      if (ctid == 0) DL_STAMP(kEvRouterRows);
      if (ok && r_on) {
        const int bb = (int)((long long)NB * my_pt / nparts), be = (int)((long long)NB * (my_pt + 1) / nparts);
        const uint32_t wr = tc::smem_u32(wr_s) + (uint32_t)(my_e * d * 4);
        const uint32_t xa = tc::smem_u32(xh);
#pragma unroll 1
        for (int t0 = 0; t0 < T; t0 += 4) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
          for (int b = bb + lane; b < be; b += 32) {
            const float4 wa = lds_f4(wr + 32u * (uint32_t)b), wb = lds_f4(wr + 32u * (uint32_t)b + 16u);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (t0 + q >= T) break;  // (warp-uniform)
              const int t = t0 + q;
              const uint4 xv = lds_v4(xa + 16u * (uint32_t)(t * XS + b));
              const float2 p0 = __half22float2(*reinterpret_cast<const __half2*>(&xv.x));  // x0, x4
              const float2 p1 = __half22float2(*reinterpret_cast<const __half2*>(&xv.y));  // x1, x5
              const float2 p2 = __half22float2(*reinterpret_cast<const __half2*>(&xv.z));  // x2, x6
              const float2 p3 = __half22float2(*reinterpret_cast<const __half2*>(&xv.w));  // x3, x7
              float sacc = acc[q];
              sacc = fmaf(wa.x, p0.x, sacc);
              sacc = fmaf(wa.y, p1.x, sacc);
              sacc = fmaf(wa.z, p2.x, sacc);
              sacc = fmaf(wa.w, p3.x, sacc);
              sacc = fmaf(wb.x, p0.y, sacc);
              sacc = fmaf(wb.y, p1.y, sacc);
              sacc = fmaf(wb.z, p2.y, sacc);
              sacc = fmaf(wb.w, p3.y, sacc);
              acc[q] = sacc;
            }
          }
          const float v = warp_sum_multi<4>(acc);  // token t0 + q in the lanes with (lane >> 3) == q
          if ((lane & 7) == 0 && t0 + (lane >> 3) < T) lpart[warp * kDlMaxT + t0 + (lane >> 3)] = v;
        }
      }
      ok = consumers_all(ok && !s_abort);
      if (ok)
#pragma unroll 1
        for (int i = ctid; i < ne * T; i += kDlWarps * 32) {
          const int le = i / T, t = i - le * T;
          float v = 0.f;
#pragma unroll 1
          for (int p = 0; p < nparts; ++p) v += lpart[(p * ne + le) * kDlMaxT + t];
          // published as one 64-bit word (epoch, key): a reader sees both or neither
          st_relaxed_gpu(a.lgt + (size_t)t * E + e0 + le, ep_tag | topk_order_key(v + (a.bias ? bias_s[le] : 0.f)));
        }
      consumers_sync();
      if (ctid == 0) DL_STAMP(kEvLogits);
    }

    // ---- team 0 runs the shared expert's unit of this CTA (routing-independent) while the other
    // teams (the routing group) gather the logits, select and dispatch; it joins them afterwards
    const bool t0_busy = false;
    const int gb = t0_busy ? kDlTeamWarps * 32 : 0;  // the routing group: threads [gb, 512)
    const int gn = kDlWarps * 32 - gb;
    if (t0_busy && team == 0) {
      if (ok) ok = gu_unit<NT>(*uc, 0, 0, tw, lane);
    } else {
      // ---- phase 2: the routing group gathers all logits of this launch (polling their epoch
      // tags), then repeats the selection and the dispatch
      const int gt = ctid - gb, gw = gt >> 5, gnw = gn >> 5;
      if (gt == 0) DL_STAMP(kEvGatherStart);
      const int EP = (E + 31) & ~31;
      uint32_t* keys = reinterpret_cast<uint32_t*>(scratch);  // [T][EP] order-preserving keys, 0 = none
      if (ok) {
        // rounds of 8 words per thread, all loads of a round in flight, then re-poll the stale ones
        const unsigned ept = (unsigned)(ep_tag >> 32);
#pragma unroll 1
        for (int base = 0; ok && base < T * EP; base += 8 * gn) {
          unsigned long long wv[8];
          int pending = 0;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int i = base + gt + q * gn;
            const int t = i / EP, e = i - t * EP;
            wv[q] = (i < T * EP && e < E) ? ld_relaxed_gpu(a.lgt + (size_t)t * E + e) : ep_tag;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) pending += (unsigned)(wv[q] >> 32) != ept;
          unsigned polls = 0;
          while (pending) {
            if (++polls > kDlSpinLimit || s_abort) break;
            __nanosleep(16);
            pending = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              if ((unsigned)(wv[q] >> 32) != ept) {
                const int i = base + gt + q * gn;
                const int t = i / EP, e = i - t * EP;
                wv[q] = ld_relaxed_gpu(a.lgt + (size_t)t * E + e);
                pending += (unsigned)(wv[q] >> 32) != ept;
              }
            }
          }
          ok = pending == 0;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int i = base + gt + q * gn;
            if (i < T * EP) keys[i] = (i - (i / EP) * EP) < E ? (uint32_t)wv[q] : 0u;
          }
        }
      }
      // the dispatch's expert bitmap and the slot-local position table start cleared
      if (gt < 32) s_bits[gt] = 0u;
      for (int i = gt; i < HS + T * K; i += gn)
        reinterpret_cast<uint4*>(tpos)[i] = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
      ok = group_all(gn, ok && !s_abort);
      if (!ok && gt == 0) {
        atomicOr(a.status, kStatusTimeout);
        s_abort = 1;
      }
      if (gt == 0) DL_STAMP(kEvKeys);
      if (ok) {
        // one token and all 16 warps: a threshold from the warp maxima, then every candidate ranked
        // by a warp (at most 64 candidates; otherwise the one-warp selection below)
        bool cta_done = false;
        if (T == 1 && E <= kDlWarps * 32 && gn == kDlWarps * 32 && K <= kDlWarps)
          cta_done = topk_select_cta(keys, EP, K, gw, lane, gt, s_wmax, s_cand, &s_ncand, s_sel, gn);
        if (cta_done) {
          if (gw == 0) {
            const uint2 mine = lane < K ? s_sel[lane] : make_uint2(0u, 0u);
            const float top = topk_key_value(s_sel[0].x);
            const float p = lane < K ? expf(topk_key_value(mine.x) - top) : 0.f;
            const float psum = warp_sum(p);
            if (lane < K) {
              idx_s[lane] = (int)mine.y;
              w_s[lane] = p / psum;
              atomicOr(&s_bits[mine.y >> 5], 1u << (mine.y & 31));
            }
          }
        } else {
          // one warp per token
#pragma unroll 1
          for (int t = gw; t < T; t += gnw) {
            int my_i;
            float my_w;
            if (E <= 512)
              topk_select_warp(keys + (size_t)t * EP, E, K, my_i, my_w);
            else
              topk_warp(keys + (size_t)t * EP, E, K, my_i, my_w);
            if (lane < K) {
              idx_s[t * K + lane] = my_i;
              w_s[t * K + lane] = my_w;
              atomicOr(&s_bits[my_i >> 5], 1u << (my_i & 31));
            }
          }
        }
        group_sync(gn);
        if (gt == 0) DL_STAMP(kEvSelected);
        const int n = T * K;
        if (T == 1 && E <= 1024) {
          // one token: its K experts are distinct, so expert e's slot (= its place in the stable
          // sort) is the number of selected experts below e, read off the selection bitmap with a
          // prefix count over its words (lane w: word w; 32 words cover E <= 1024)
          if (gw == 0) {
            const uint32_t bw = s_bits[lane];
            const int pc = __popc(bw);
            int incl = pc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int y = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += y;
            }
            const int e_i = lane < K ? idx_s[lane] : 0;
            const int wpre = __shfl_sync(0xffffffffu, incl - pc, e_i >> 5);
            const uint32_t wbits = __shfl_sync(0xffffffffu, bw, e_i >> 5);
            if (lane < K) {
              const int slot = wpre + __popc(wbits & ((1u << (e_i & 31)) - 1u));
              perm_s[slot] = lane;
              slot_s[slot] = make_int4(e_i, slot, 1, 0);
              tpos[(HS + slot) * kDlMaxT] = (signed char)0;
            }
            if (HS && lane == 0) tpos[0] = (signed char)0;
            if (lane == 0) s_nact = K;
          }
        } else if (n <= 32) {
          // few assignments: one warp does the whole dispatch with shuffles.  Lane i = assignment i:
          // its place in the stable counting sort (assignments with a smaller expert, plus the
          // earlier ones with its expert), its slot (distinct experts below its own), its position in
          // the slot.
          if (gw == 0) {
            const int e_i = lane < n ? idx_s[lane] : 0x7fffffff;
            int start = 0, cnt_i = 0, before = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int ej = __shfl_sync(0xffffffffu, e_i, j);
              start += ej < e_i;
              cnt_i += ej == e_i;
              before += ej == e_i && j < lane;
            }
            const bool first = lane < n && before == 0;
            const unsigned fm = __ballot_sync(0xffffffffu, first);
            int slot = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) slot += ((fm >> j) & 1u) && __shfl_sync(0xffffffffu, e_i, j) < e_i;
            if (lane < n) {
              perm_s[start + before] = lane;
              if (first) slot_s[slot] = make_int4(e_i, start, cnt_i, 0);
              tpos[(HS + slot) * kDlMaxT + lane / K] = (signed char)before;
            }
            if (HS && lane < T) tpos[lane] = (signed char)lane;
            if (lane == 0) s_nact = __popc(fm);
          }
        } else {
          if (gw == 0) {
            // slot of expert e = number of selected experts below e: per-word prefix of the bitmap
            const uint32_t bw = s_bits[lane];
            const int pc = __popc(bw);
            int incl = pc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int y = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += y;
            }
            s_bpre[lane] = incl - pc;
            if (lane == 31) s_nact = incl;
          }
          group_sync(gn);
#pragma unroll 1
          for (int ai = gt; ai < n; ai += gn) {
            // assignment ai: its place in the stable counting sort by expert, its slot, its position
            // among the slot's tokens (tokens ascend with the assignment number)
            const int e_i = idx_s[ai];
            int start = 0, cnt_i = 0, before = 0;
#pragma unroll 4
            for (int j = 0; j < n; ++j) {
              const int ej = idx_s[j];
              start += ej < e_i;
              cnt_i += ej == e_i;
              before += ej == e_i && j < ai;
            }
            perm_s[start + before] = ai;
            const int slot = s_bpre[e_i >> 5] + __popc(s_bits[e_i >> 5] & ((1u << (e_i & 31)) - 1u));
            if (before == 0) slot_s[slot] = make_int4(e_i, start, cnt_i, 0);
            tpos[(HS + slot) * kDlMaxT + ai / K] = (signed char)before;
          }
          if (HS && gt < T) tpos[gt] = (signed char)gt;
        }
        // the keys are done with: the producer's bulk copies may overwrite them
        tc::fence_proxy_async_smem();
        group_sync(gn);
        if (NT == 2 && gw == 0) {
          // the slots with more than 8 tokens, ascending: each has a second down item (tokens 8..)
          const int ns_all = HS + s_nact;
          int nb = 0;
#pragma unroll 1
          for (int b = 0; b < ns_all; b += 32) {
            const int sl = b + lane;
            const bool big = sl < ns_all && (sl < HS ? T : slot_s[sl - HS].z) > 8;
            const unsigned bm = __ballot_sync(0xffffffffu, big);
            if (big) s_big[nb + __popc(bm & ((1u << lane) - 1u))] = sl;
            nb += __popc(bm);
          }
          if (lane == 0) s_nbig = nb;
          __syncwarp();
        }
        if (gt == 0) {
          DL_STAMP(kEvDispatched);
          DL_STAMP(kEvRouted);
          tc::mbar_arrive(&route_ready);
        }
        // the full outputs (every CTA holds the same routing): offs[e] = assignments with an expert
        // below e, counts and the usage histogram for this CTA's share of the experts (offs[E] by the
        // last CTA); idx, w, perm, the distinct experts and the slots by CTA 0
        {
          const int eb = (int)((long long)E * c / nc);
          const int ee = (int)((long long)E * (c + 1) / nc) + (c == nc - 1 ? 1 : 0);
#pragma unroll 1
          for (int e = eb + gt; e < ee; e += gn) {
            int o = 0, ce = 0;
#pragma unroll 4
            for (int q = 0; q < n; ++q) {
              o += idx_s[q] < e;
              ce += idx_s[q] == e;
            }
            a.offs[e] = o;
            if (e < E) a.counts[e] = ce;
            if (e < E && ce && a.usage) a.usage[e] += (unsigned long long)ce;
          }
        }
        if (c == 0) {
          const int na = s_nact;
#pragma unroll 1
          for (int i = gt; i < n; i += gn) {
            a.idx[i] = idx_s[i];
            a.w[i] = w_s[i];
            a.perm[i] = perm_s[i];
          }
#pragma unroll 1
          for (int q = gt; q < na; q += gn) {
            a.active[q] = slot_s[q].x;
            a.slots[q] = slot_s[q];
          }
          if (gt == 0) {
            *a.n_active = na;
            if (a.stat) *a.stat = na;
          }
        }
      }
    }
    // team 0 joins: the routing (or its failure) is known to all consumers
    ok = consumers_all(ok && !s_abort);
    if (!ok && ctid == 0) {
      atomicOr(a.status, kStatusTimeout);
      s_abort = 1;
    }

    const int nslots = HS + (ok ? s_nact : 0);
    const int nitems = nslots + (NT == 2 && ok ? s_nbig : 0);  // down items: every slot, then second halves
    const int total_units = nslots * fu;
    const int nG = total_units > c ? (total_units - c + nc - 1) / nc : 0;

    // ---- phase 3: this CTA's items in order -- its gate/up units, then the down items of every
    // slot; team (k % 4) takes item k.  A team finishes all its gate/up units before any of its down
    // items, so the slots' h rows (everywhere) do not wait on a down item.  With at most 16 down
    // items (one token) each is taken by one warp instead (warp q takes down item q), all at once.
    float D[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) D[j][0] = D[j][1] = D[j][2] = D[j][3] = 0.f;
    const bool warp_items = nitems <= kDlWarps;
#pragma unroll 1
    for (int k = team; ok && k < nG + (warp_items ? 0 : nitems); k += kDlTeams) {
      if (k < nG) {
        ok = gu_unit<NT>(*uc, k, team, tw, lane);
        if (k + kDlTeams >= nG && tw == 0 && lane == 0) DL_STAMP(kEvUnitsDone);  // this team's last unit
      } else {
        if (k - nG < kDlTeams && tw == 0 && lane == 0 && team == 0) DL_STAMP(kEvFirstDown);
        const int q = k - nG;
        ok = down_item<NT>(*uc, k, q < nslots ? q : s_big[q - nslots], q < nslots ? 0 : 1, team, tw, lane, D);
        if (tw == 0 && lane == 0) {
          if (k == nG) DL_STAMP(kEvFirstDownDone);
          if (k == nG + nitems - 1) DL_STAMP(kEvLastDownDone);
        }
      }
    }
    if (warp_items && ok && warp < nitems) {
      const int q = warp;
      if (q == 0 && lane == 0) DL_STAMP(kEvFirstDown);
      ok = down_item_warp<NT>(*uc, nG + q, q < nslots ? q : s_big[q - nslots], q < nslots ? 0 : 1, lane, D);
      if (lane == 0) {
        if (q == 0) DL_STAMP(kEvFirstDownDone);
        if (q == nitems - 1) DL_STAMP(kEvLastDownDone);
      }
    }
    ok = consumers_all(ok && !s_abort);
    if (!ok && ctid == 0) s_abort = 1;  // the producer stops issuing
    if (ctid == 0) DL_STAMP(kEvDownDone);

    // ---- y rows [r0, r0 + nr): the 16 warps' partial sums in warp order (+ residual)
    const uint32_t pgu_a = tc::smem_u32(pgu);
#pragma unroll
    for (int j = 0; j < NT; ++j)
      sts_f4(pgu_a + 16u * (uint32_t)((warp * NT + j) * 32 + lane), make_float4(D[j][0], D[j][1], D[j][2], D[j][3]));
    consumers_sync();
    for (int i = ctid; i < nr * T; i += kDlWarps * 32) {
      const int n = i / nr, r = i - n * nr;
      const int j = n >> 3, nn = n & 7;
      const int ln = (r & 7) * 4 + (nn >> 1), comp = (r >> 3) * 2 + (nn & 1);
      float v = 0.f;
      const uint32_t pb = pgu_a + (uint32_t)((j * 32 + ln) * 16 + comp * 4);
#pragma unroll
      for (int q = 0; q < kDlWarps; ++q) v += lds_f32(pb + (uint32_t)(q * NT * 32 * 16));
      const size_t o = (size_t)n * d + r0 + r;
      if (ok) {
        if (a.resid) v = resid_s[n * nr + r] + v;
      } else {
        v = __int_as_float(0x7fc00000);  // NaN: this CTA gave up, its rows are not a result
      }
      store_act(a.y, a.act, o, v);
    }
    if (!ok && ctid == 0) {
      atomicOr(a.status, kStatusTimeout);
      s_abort = 1;
    }
    consumers_sync();
    if (ctid == 0) {
      DL_STAMP(kEvEnd);
      DL_CLOCK(kClkEnd);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd(a.launches, 1ull);  // this CTA is done with the launch's epoch
  if (threadIdx.x == 0 && s_abort) {
    // copies still in flight must land before the CTA's shared memory goes away
    volatile int never = 0;
    const int issued = s_issued;
    for (int kk = issued - 1; kk >= 0 && kk >= issued - NS; --kk)  // the last copy of every stage
      tc::mbar_wait(&full[kk % NS], (kk / NS) & 1, &never, 2000000000ll);
    if (ne > 0) tc::mbar_wait(&wr_full, 0, &never, 2000000000ll);
  }
}

// ------------------------------------------------------------------ self-test of the bounded waits
// One CTA: thread 0 waits on an mbarrier nobody arrives at and for a tag nobody writes on a word,
// each with a small budget, exactly as the layer kernel waits.  Bit 0 of *result: the mbarrier
// wait gave up; bit 1: the tagged-word wait gave up; bit 2: a wait returned success (a bug).
__global__ void bounded_wait_selftest_kernel(unsigned long long* word, long long budget, unsigned* result) {
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
    // the word never carries this tag (nothing writes it); the poll limit bounds the wait
    const unsigned tag = (unsigned)(ld_relaxed_gpu(word) >> 32) + 1u;
    bool ok = true;
    for (unsigned n = 0; ok && (unsigned)(ld_relaxed_gpu(word) >> 32) != tag; ++n) {
      if (n > (unsigned)(budget >> 6)) ok = false;
      __nanosleep(32);
    }
    r |= ok ? 4u : 2u;
    *result = r;
    if (r & 3u) atomicOr(result + 1, kStatusTimeout);
  }
}

// The self-test's word and result, file-scope device memory (no allocation).
__device__ unsigned long long g_selftest_word;
__device__ unsigned g_selftest_result[2];

cudaError_t launch_bounded_wait_selftest(long long budget, unsigned* result_host, cudaStream_t st) {
  void* wp = nullptr;
  void* rp = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&wp, g_selftest_word);
  if (e == cudaSuccess) e = cudaGetSymbolAddress(&rp, g_selftest_result);
  if (e == cudaSuccess) e = cudaMemsetAsync(wp, 0, sizeof(unsigned long long), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(rp, 0, 2 * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(static_cast<unsigned long long*>(wp), budget,
                                                 static_cast<unsigned*>(rp));
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyAsync(result_host, rp, 2 * sizeof(unsigned), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e;
}

// ------------------------------------------------------------------ host side
struct DlPlan {
  int ns, stage_bytes, smem, rows_box;
};

static size_t up16(size_t n) { return (n + 15) & ~size_t(15); }

static int rows_box_for(int d, int nsm) { return (d + nsm - 1) / nsm; }

static DlPlan dl_plan(int T, int d, int f, int E, int K, int nsm) {
  DlPlan p{};
  p.rows_box = rows_box_for(d, nsm);
  const int RB = p.rows_box;
  const size_t gu = (size_t)(d / 256) * 2048 + 2 * 8 * (d / 32) * 2;
  const size_t dn_codes = (size_t)RB * (f / 2);
  // a down item stages the h rows of at most 8 tokens (a slot with more tokens is two items)
  const size_t dn = ((((dn_codes + 127) & ~size_t(127)) + (size_t)RB * (f / 32) * 2 + 127) & ~size_t(127)) +
                    (size_t)std::min(T, 8) * f * 2;
  p.stage_bytes = (int)((std::max(gu, dn) + 1023) & ~size_t(1023));
  const int NT = T > 8 ? 2 : 1;
  const size_t fixed = 1024 /* alignment */ + (size_t)T * (d / 8 + kDlXPad) * 16 + (size_t)kDlWarps * NT * 32 * 16 +
                       up16((size_t)T * K * 16) + 3 * up16((size_t)T * K * 4) + up16((size_t)(T * K + 1) * kDlMaxT);
  const long long room = (long long)kDlSmemMax - kDlStaticSlack - (long long)fixed;
  p.ns = room > 0 ? (int)std::min<long long>(kDlMaxStages, room / p.stage_bytes) : 0;
  p.smem = (int)((size_t)p.ns * p.stage_bytes + fixed);
  return p;
}

static PFN_cuTensorMapEncodeTiled_v12000 g_dl_encode = nullptr;

template <int NT>
static const void* dl_fn() {
  return (const void*)decode_layer_kernel<NT>;
}

cudaError_t decode_kernels_init() {
  if (!g_dl_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_dl_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const void* fns[2] = {dl_fn<1>(), dl_fn<2>()};
  for (const void* fn : fns) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kDlSmemMax - kDlStaticSlack);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Whether the one-launch layer serves this shape (INT4 weights, bf16 activations) with T tokens on
// nsm SMs, all resident at once.
bool decode_shape_ok(int T, int d, int f, int E, int K, int nsm) {
  if (nsm <= 0 || T < 1 || T > kDlMaxT) return false;
  if ((d != 1024 && d != 2048) || f % 256 || f > 2048 || E > kMaxE || K > kMaxK) return false;
  if (T * K > kDlWarps * 32 || E > 2 * kDlWarps * 32) return false;  // dispatch / selection thread maps
  if (rows_box_for(d, nsm) > kDlRowsMax || (E + nsm - 1) / nsm > kDlRowsMax) return false;
  const DlPlan p = dl_plan(T, d, f, E, K, nsm);
  if (p.ns < 3) return false;  // stage 0 (first unit) + stages 1-2 (router rows, then the selection's keys)
  if ((size_t)((E + nsm - 1) / nsm) * d * 4 > 2 * (size_t)p.stage_bytes) return false;
  if ((size_t)T * ((E + 31) & ~31) * 4 > 2 * (size_t)p.stage_bytes) return false;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, T > 8 ? dl_fn<2>() : dl_fn<1>(), kDlThreads, p.smem) !=
          cudaSuccess ||
      occ < 1) {
    cudaGetLastError();
    return false;
  }
  return true;
}

size_t decode_maps_bytes() { return sizeof(DlMaps); }

static cudaError_t encode(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int rank, const cuuint64_t* dims,
                          const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  const cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_dl_encode(m, dt, rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static cudaError_t expert_maps(CUtensorMap* gq, CUtensorMap* gs, CUtensorMap* dq, CUtensorMap* ds, int n_exp, int d,
                               int f, int RB, int dn_swap, const void* gu_q, const void* gu_s, const void* dn_q,
                               const void* dn_s) {
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cudaError_t e;
  {
    const cuuint64_t dims[4] = {128, (cuuint64_t)n_exp * 2 * f, (cuuint64_t)d / 256, 2};
    const cuuint64_t str[3] = {(cuuint64_t)d / 2, 128, (cuuint64_t)f * d / 2};
    const cuuint32_t box[4] = {128, 8, (cuuint32_t)d / 256, 2};
    if ((e = encode(gq, gu_q, U8, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)d / 32, (cuuint64_t)n_exp * 2 * f, 2};
    const cuuint64_t str[2] = {(cuuint64_t)d / 32 * 2, (cuuint64_t)f * (d / 32) * 2};
    const cuuint32_t box[3] = {(cuuint32_t)d / 32, 8, 2};
    if ((e = encode(gs, gu_s, F16, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess) return e;
  }
  if (dn_swap) {
    const cuuint64_t dims[3] = {128, (cuuint64_t)n_exp * d, (cuuint64_t)f / 256};
    const cuuint64_t str[2] = {(cuuint64_t)f / 2, 128};
    const cuuint32_t box[3] = {128, (cuuint32_t)RB, (cuuint32_t)f / 256};
    if ((e = encode(dq, dn_q, U8, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
  } else {
    const cuuint64_t dims[3] = {128, (cuuint64_t)f / 256, (cuuint64_t)n_exp * d};
    const cuuint64_t str[2] = {128, (cuuint64_t)f / 2};
    const cuuint32_t box[3] = {128, (cuuint32_t)f / 256, (cuuint32_t)RB};
    if ((e = encode(dq, dn_q, U8, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)f / 32, (cuuint64_t)n_exp * d};
    const cuuint64_t str[1] = {(cuuint64_t)f / 32 * 2};
    const cuuint32_t box[2] = {(cuuint32_t)f / 32, (cuuint32_t)RB};
    if ((e = encode(ds, dn_s, F16, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// The down box is [chunk][row] when the row's chunk count is even (rows then differ in the
// swizzle's line bits), [row][chunk] when it is odd.
static int dn_swap_for(int f) { return ((f / 256) & 1) ? 0 : 1; }

cudaError_t decode_build_maps(void* maps, int E, int d, int f, int nsm, int has_shared, const void* gu_q,
                              const void* gu_s, const void* dn_q, const void* dn_s, const void* sh_gu_q,
                              const void* sh_gu_s, const void* sh_dn_q, const void* sh_dn_s) {
  if (!g_dl_encode) return cudaErrorNotSupported;
  DlMaps* mp = static_cast<DlMaps*>(maps);
  const int RB = rows_box_for(d, nsm), sw = dn_swap_for(f);
  cudaError_t e = expert_maps(&mp->gu_q, &mp->gu_s, &mp->dn_q, &mp->dn_s, E, d, f, RB, sw, gu_q, gu_s, dn_q, dn_s);
  if (e != cudaSuccess) return e;
  if (!has_shared) {  // the maps must be valid even when unused
    sh_gu_q = gu_q;
    sh_gu_s = gu_s;
    sh_dn_q = dn_q;
    sh_dn_s = dn_s;
  }
  return expert_maps(&mp->sh_gu_q, &mp->sh_gu_s, &mp->sh_dn_q, &mp->sh_dn_s, 1, d, f, RB, sw, sh_gu_q, sh_gu_s,
                     sh_dn_q, sh_dn_s);
}

int decode_timeline_events() { return kDlEvents; }

cudaError_t launch_decode_layer(const RouteArgs& r, const ExpertArgs& x, const void* maps, unsigned long long* hw,
                                unsigned long long* lgt, unsigned long long* launches, int nsm,
                                unsigned long long* timeline, cudaStream_t st) {
  DlArgs a;
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
  a.idx = r.idx;
  a.w = r.w;
  a.counts = r.counts;
  a.offs = r.offs;
  a.perm = r.perm;
  a.active = r.active;
  a.n_active = r.n_active;
  a.stat = r.stat;
  a.slots = r.slots;
  a.usage = r.usage;
  a.hw = hw;
  a.y = x.y;
  a.resid = x.resid;
  a.lgt = lgt;
  a.launches = launches;
  a.status = r.status;
  const DlPlan p = dl_plan(r.T, r.d, x.f, r.E, r.K, nsm);
  a.ns = p.ns;
  a.stage_bytes = p.stage_bytes;
  a.rows_box = p.rows_box;
  a.dn_swap = dn_swap_for(x.f);
  a.timeline = timeline;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nsm);
  cfg.blockDim = dim3(kDlThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  // One CTA per SM (the shared-memory plan allows no second), grid = #SMs (checked resident with
  // the occupancy query when the handle is created); every wait is bounded anyway.  The launch may
  // overlap the tail of the previous kernel in the stream (its prologue only reads weights);
  // griddepcontrol.wait orders everything else.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const DlMaps& mp = *static_cast<const DlMaps*>(maps);
  void* args[2] = {&a, const_cast<DlMaps*>(&mp)};
  return cudaLaunchKernelExC(&cfg, r.T > 8 ? dl_fn<2>() : dl_fn<1>(), args);
}

}  // namespace moe
