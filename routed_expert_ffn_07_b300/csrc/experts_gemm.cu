// Prefill experts: token-grouped GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// A prefill chunk of thousands of tokens routes to almost every expert of every layer, so each
// expert's weights are streamed once and shared by all tokens of the chunk that chose it ('Strata
// はなぜ少ない VRAM でも速いのか' (modeldock.net), section '長いプロンプトを読む：大きなまとまりで流す').
// Here the tokens of each expert form one or more tiles of <= 128 rows (sorted by the dispatch),
// and every tile is a dense contraction:
//   GEMM1 (gate/up): [128 f rows of W_gate | W_up] x [tile tokens]^T over d -> h = silu(g) * u
//   GEMM2 (down)   : [128 d rows of W_down] x [tile h rows]^T over f        -> w_a * o, per assignment
//   combine        : y_t = sum_k (w_{t,k} o_{t,k}) + o_shared,t  (fixed order, fp32)
//
// Per CTA (one per SM, persistent over work items = (tile, 128-row block)):
//   warp 0     : allocates 512 TMEM columns; one thread issues tcgen05.mma (A from TMEM, B from SMEM)
//   warp 1     : one thread issues the TMA loads of the int4 weights (128 rows x 128 bytes = 256 K
//                per stage, 128B swizzle) and of each item's fp16 scales
//   warp 18    : one thread issues the TMA loads of the tile's activation rows (128 rows x 64
//                columns per stage, 128B swizzle)
//   warps 2-17 : dequantise int4 -> fp16 (q * scale, one rounding) straight into TMEM (tcgen05.st),
//                then the epilogue (tcgen05.ld of the fp32 accumulators).  Warp w reaches TMEM lanes
//                32*(w%4).. of the 128 weight rows.  Two teams of eight warps take alternate pipeline
//                stages, so two stages are being dequantised at once; inside a team the warps split
//                the stage's K columns (and the two matrices of the gate/up GEMM).  All sixteen warps
//                share the epilogue, four groups of 32 token columns.
// The activation rows of each expert are contiguous because a staging kernel first writes the
// chunk's tokens in dispatch order (fp16, K-permuted), so every B tile is one TMA box.
// The weights are the MMA M side (128 rows), the tile's tokens the N side (16..128, padded to 16),
// so ~80-token groups are not padded to 128.  The dequantised A operand never touches shared
// memory, which keeps SMEM traffic to the B tiles.  mbarrier pipelines: SMEM stages (TMA + cp.async
// -> MMA / dequant), TMEM A stages (dequant -> MMA), accumulators (MMA -> epilogue).  Every wait
// is bounded: on timeout the CTA records MOE status "timeout", stops all roles and frees TMEM.
//
// Operand precision: A = fp16(q * s) (exact product, one rounding), B = fp16 activations (bf16
// inputs are exact in fp16 within its normal range; h is rounded once to fp16); fp32 accumulation.
// Values outside the fp16 range set the status word.  Within each 8-column block the K order of
// both operands is permuted the same way, (0,4,1,5,2,6,3,7), which is what the dequantiser
// produces without extra byte shuffles.
#include <cudaTypedefs.h>

#include <cstdlib>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {

constexpr int kGemmThreads = 608;  // warps: 0 MMA, 1 TMA (weights), 2-17 dequant + epilogue, 18 TMA (activations)
constexpr int kDqWarps = 16;
constexpr int kBWarp = 18;
constexpr int kDqWarp0 = 2;
constexpr int kNT = 128;            // max token rows per tile (MMA N)
constexpr int kBM = 128;            // weight rows per A matrix (MMA M)
constexpr int kKS = 64;             // K per MMA / activation stage
constexpr int kKA = 256;            // K per weight stage (128-byte int4 rows)
constexpr int kSub = kKA / kKS;     // MMA stages per weight stage
constexpr int kAStages = 3;         // weight stages in SMEM (int4 rows + their fp16 scales)
constexpr int kScB = kKA / 32 * 2;  // scale bytes per weight row per weight stage (8 groups)
constexpr int kBPrefetch = 16;      // gate/up: activation stages prefetched into L2 ahead of the loads
// activation stages in SMEM and dequantised A stages in TMEM, per kind (0 gate/up, 1 down)
template <int KIND> struct Stages {
  static constexpr int NA = KIND == 0 ? 2 : 1;   // A matrices per tile
  static constexpr int B = KIND == 0 ? 7 : 10;   // activation stages: deep, the TMA latency is long
  static constexpr int J = KIND == 0 ? 4 : 8;    // TMEM A stages (NA*32 columns each, 256 columns in all)
};
struct GemmMaps {
  CUtensorMap gu_q, gu_s, sh_gu_q, sh_gu_s, dn_q, dn_s, sh_dn_q, sh_dn_s;
};

// Maps of the workspace activation buffers (fixed per handle).
struct GemmActMaps {
  CUtensorMap xs, hs;
};

struct GemmWs {
  __half* x16;          // [T*K + T][d] fp16, K-permuted, rows in dispatch order
  __half* h16;          // [T*K + T][f] fp16, K-permuted
  __nv_bfloat16* P;     // [T*K + T][d] weighted per-assignment partials
  int32_t* n_tiles;     // [1]
  int32_t* tile_group;  // [max_tiles]
  int32_t* tile_row;
  int32_t* tile_n;
};

struct GemmArgs {
  int T, d, f, E, K, n_assign, has_shared;
  const int32_t* perm;
  const float* topk_w;
  __half* h16;
  __nv_bfloat16* P;
  const int32_t* n_tiles;
  const int32_t* tile_group;
  const int32_t* tile_row;
  const int32_t* tile_n;
  unsigned* status;
};

__device__ __forceinline__ int inv_perm8(int i) { return (i & 3) * 2 + (i >> 2); }  // 0,2,4,6,1,3,5,7

// 32 int4 values (16 bytes) -> 16 words of fp16 pairs (q*s), in the order (0,4),(1,5),(2,6),(3,7) per word.
__device__ __forceinline__ void dequant32(const uint4 q, const __half2 s2, uint32_t* v) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  const __half2 m1032 = __float2half2_rn(-1032.f);
  const __half2 sixteenth = __float2half2_rn(0.0625f);
  const __half2 m72 = __float2half2_rn(-72.f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t x = w[i], x8 = x >> 8;
    uint32_t a0 = (x & 0x000F000Fu) ^ 0x64086408u;
    uint32_t a1 = (x & 0x00F000F0u) ^ 0x64806480u;
    uint32_t a2 = (x8 & 0x000F000Fu) ^ 0x64086408u;
    uint32_t a3 = (x8 & 0x00F000F0u) ^ 0x64806480u;
    __half2 h0 = __hadd2(*reinterpret_cast<__half2*>(&a0), m1032);
    __half2 h1 = __hfma2(*reinterpret_cast<__half2*>(&a1), sixteenth, m72);
    __half2 h2 = __hadd2(*reinterpret_cast<__half2*>(&a2), m1032);
    __half2 h3 = __hfma2(*reinterpret_cast<__half2*>(&a3), sixteenth, m72);
    h0 = __hmul2(h0, s2);
    h1 = __hmul2(h1, s2);
    h2 = __hmul2(h2, s2);
    h3 = __hmul2(h3, s2);
    v[4 * i + 0] = *reinterpret_cast<uint32_t*>(&h0);
    v[4 * i + 1] = *reinterpret_cast<uint32_t*>(&h1);
    v[4 * i + 2] = *reinterpret_cast<uint32_t*>(&h2);
    v[4 * i + 3] = *reinterpret_cast<uint32_t*>(&h3);
  }
}

// 16 int4 values (8 bytes) -> 8 words of fp16 pairs, same order as dequant32.
__device__ __forceinline__ void dequant16(const uint2 q, const __half2 s2, uint32_t* v) {
  uint32_t t[16];
  dequant32(make_uint4(q.x, q.y, 0u, 0u), s2, t);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = t[i];
}

__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

template <int KIND>  // 0: gate/up + SwiGLU, 1: down + weighted partials
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const GemmArgs g, const __grid_constant__ CUtensorMap mq_r, const __grid_constant__ CUtensorMap ms_r,
                const __grid_constant__ CUtensorMap mq_s, const __grid_constant__ CUtensorMap ms_s,
                const __grid_constant__ CUtensorMap mb) {
  constexpr int NA = Stages<KIND>::NA;
  constexpr int NB = KIND == 0 ? 1 : 2;  // accumulator buffers
  constexpr int BS = Stages<KIND>::B;
  constexpr int J = Stages<KIND>::J;
  static_assert(J <= BS && 256 + J * NA * 32 <= 512, "TMEM budget");
  const int Kdim = KIND == 0 ? g.d : g.f;
  const int KS = Kdim / kKS;
  const int nblk = (KIND == 0 ? g.f : g.d) / kBM;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;                               // BS x [128 rows x 128 B] fp16
  uint8_t* sA = sB + BS * kNT * 128;                // kAStages x NA x [128 rows x 128 B] int4
  uint8_t* sS = sA + kAStages * NA * kBM * 128;     // kAStages x NA x [128 rows x 8 fp16]
  // fa/ea: weight stages; fb: activation stages; tfull: stage gs dequantised into TMEM A stage
  // gs % J; sdone: the MMAs of stage gs finished,
  // which frees activation slot gs % BS and (J stages later) TMEM A stage gs % J
  __shared__ __align__(8) uint64_t fa[kAStages], ea[kAStages], fb[BS], tfull[BS], sdone[BS], acc_full[2],
      acc_empty[2], fin;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      tc::mbar_init(&fa[s], 1);
      tc::mbar_init(&ea[s], kDqWarps);  // every dequant warp, after its last sub-stage of the weight stage
    }
    for (int s = 0; s < BS; ++s) {
      tc::mbar_init(&fb[s], 1);
      tc::mbar_init(&tfull[s], kDqWarps / 2);
      tc::mbar_init(&sdone[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], kDqWarps);
    }
    tc::mbar_init(&fin, 1);
    s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int n_items = *g.n_tiles * nblk;
  auto give_up = [&]() {
    atomicOr(g.status, kStatusTimeout);
    s_abort = 1;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs this loop converged (all values warp-uniform); one elected lane issues.
    uint32_t gs = 0, it = 0;
    bool ok = true;
    const uint32_t leader = tc::elect_one();
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
      const int tile = item / nblk;
      const int nmma = (g.tile_n[tile] + 15) & ~15;
      const uint32_t idesc = tc::idesc_f16_f32(128, nmma);
      const int b = it % NB;
      if (!tc::mbar_wait_all(&acc_empty[b], ((it / NB) & 1) ^ 1, &s_abort)) { ok = false; break; }
      tc::tc_fence_after();
      const uint32_t dcol0 = KIND == 0 ? 0u : (uint32_t)b * 128u;
      for (int s = 0; s < KS; ++s, ++gs) {
        const int slot = gs % BS;
        const uint32_t ph = (gs / BS) & 1;
        // the stage's activations landed (fb) and every dequant warp of its team stored its part of
        // A (tfull); the whole warp polls each barrier
        if (!tc::mbar_wait_all(&fb[slot], ph, &s_abort) || !tc::mbar_wait_all(&tfull[slot], ph, &s_abort)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint64_t bd0 = tc::sdesc_sw128(tc::smem_u32(sB + slot * kNT * 128));
        const uint32_t a0 = tmem + 256 + (gs % J) * (NA * 32);
#pragma unroll
        for (int kk = 0; kk < kKS / 16; ++kk) {
#pragma unroll
          for (int m = 0; m < NA; ++m)
            tc::mma_ts_pred(tmem + dcol0 + (KIND == 0 ? m * 128 : 0), a0 + m * 32 + kk * 8, bd0 + (uint64_t)(kk * 2),
                            idesc, (s > 0 || kk > 0) ? 1u : 0u, leader);
        }
        tc::mma_commit_pred(&sdone[slot], leader);
      }
      if (!ok) break;
      tc::mma_commit_pred(&acc_full[b], leader);
    }
    if (!ok && lane == 0) give_up();
    __syncwarp();
    tc::mma_commit_elect(&fin);  // completes when every MMA issued above has finished
    if (lane == 0) {
      volatile int never = 0;
      tc::mbar_wait(&fin, 0, &never, 2000000000ll);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- TMA producer (weights)
    if (lane == 0) {
      tc::prefetch_tmap(&mq_r);
      tc::prefetch_tmap(&ms_r);
      tc::prefetch_tmap(&mq_s);
      tc::prefetch_tmap(&ms_s);
      uint32_t as = 0, it = 0;
      bool ok = true;
      const int rows_per_expert = KIND == 0 ? 2 * g.f : g.d;
      const int KAS = Kdim / kKA;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
        const int tile = item / nblk, blk = item % nblk;
        const int grp = g.tile_group[tile];
        const bool sh = grp >= g.E;
        const CUtensorMap* mq = sh ? &mq_s : &mq_r;
        const CUtensorMap* ms = sh ? &ms_s : &ms_r;
        const int r0 = (sh ? 0 : grp * rows_per_expert) + blk * kBM;
        for (int a = 0; a < KAS; ++a, ++as) {
          const int slot = as % kAStages;
          if (!tc::mbar_wait(&ea[slot], ((as / kAStages) & 1) ^ 1, &s_abort)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&fa[slot], NA * kBM * (128 + kScB));
#pragma unroll
          for (int m = 0; m < NA; ++m) {
            tc::tma_load_2d(sA + (slot * NA + m) * kBM * 128, mq, a * 128, r0 + m * g.f, &fa[slot]);
            tc::tma_load_2d(sS + (slot * NA + m) * kBM * kScB, ms, a * (kKA / 32), r0 + m * g.f, &fa[slot]);
          }
        }
      }
      if (!ok) give_up();
    }
    __syncwarp();
  } else if (warp == kBWarp) {
    // ---------------------------------------------------------------- TMA producer (activations)
    if (lane == 0) {
      tc::prefetch_tmap(&mb);
      uint32_t gs = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int tile = item / nblk;
        const int brow = g.tile_row[tile];
        for (int s = 0; s < KS; ++s, ++gs) {
          const int slot = gs % BS;
          if (!tc::mbar_wait(&sdone[slot], ((gs / BS) & 1) ^ 1, &s_abort)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&fb[slot], kNT * 128);
          tc::tma_load_2d(sB + slot * kNT * 128, &mb, s * kKS, brow, &fb[slot]);
          // the activation tile kBPrefetch stages ahead into L2, so that its load (issued once a slot
          // frees) finds it there: the slots alone look too few stages ahead to hide the HBM latency
          int s2 = s + kBPrefetch, item2 = item;
          while (s2 >= KS) {
            s2 -= KS;
            item2 += gridDim.x;
          }
          if (KIND == 0 && item2 < n_items) tc::tma_prefetch_l2_2d(&mb, s2 * kKS, g.tile_row[item2 / nblk]);
        }
      }
      if (!ok) give_up();
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- dequant + epilogue
    const int q = warp & 3;                      // TMEM lane quarter
    const int grp = (warp - kDqWarp0) >> 2;      // 0..3 (epilogue token-column group)
    const int team = grp >> 1;                   // stages with gs % 2 == team
    const int sub = grp & 1;                     // gate/up: matrix; down: 16-byte chunk of the stage
    const int m = KIND == 0 ? sub : 0;
    const int row = q * 32 + lane;
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    const int swz = row & 7;  // 128-byte swizzle of the int4 rows: 16-byte chunk c sits at c ^ (row % 8)
    // Epilogue of one finished item: accumulators -> registers, release them to the MMA, then the
    // math and the global stores.  (a, w) of this thread's token column (down GEMM) were loaded
    // when the item started.
    auto epilogue = [&](int item, uint32_t eit, int ea_id, float ew) -> bool {
      const int tile = item / nblk, blk = item % nblk;
      const int n = g.tile_n[tile], row0 = g.tile_row[tile];
      const int b = eit % NB;
      if (!tc::mbar_wait_warp(&acc_full[b], (eit / NB) & 1, &s_abort)) return false;
      tc::tc_fence_after();
      const int cb = grp * 32;
      if (KIND == 0) {
        // h = silu(gate) * up for 32 token columns, in two halves of 16 to bound register use
        __half hv[32];
        bool range_bad = false;
        if (cb < n) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t gv[16], uv[16];
            tc::tmem_ld16(tmem + lane_base + cb + hh * 16, gv);
            tc::tmem_ld16(tmem + lane_base + 128 + cb + hh * 16, uv);
            tc::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const float h = silu_fast(__uint_as_float(gv[jj])) * __uint_as_float(uv[jj]);
              range_bad |= !(fabsf(h) <= 65504.f) && cb + hh * 16 + jj < n;
              hv[hh * 16 + jj] = __float2half_rn(h);
            }
          }
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acc_empty[b]);
        if (cb < n) {
          const int fidx = blk * kBM + row;
          const int fpos = (fidx & ~7) | inv_perm8(fidx & 7);
          __half* hp = g.h16 + (size_t)(row0 + cb) * g.f + fpos;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            if (cb + jj < n) hp[(size_t)jj * g.f] = hv[jj];
          if (range_bad) atomicOr(g.status, kStatusRange);
        }
      } else {
        uint32_t ov[32];
        if (cb < n) {
          tc::tmem_ld32(tmem + lane_base + b * 128 + cb, ov);
          tc::tmem_wait_ld();
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acc_empty[b]);
        if (cb < n) {
          const int jrow = blk * kBM + row;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int a_jj = __shfl_sync(0xffffffffu, ea_id, jj);
            const float w_jj = __shfl_sync(0xffffffffu, ew, jj);
            if (cb + jj < n) g.P[(size_t)a_jj * g.d + jrow] = __float2bfloat16_rn(w_jj * __uint_as_float(ov[jj]));
          }
        }
      }
      return true;
    };

    uint32_t gs = 0, it = 0;
    bool ok = true;
    // the finished item whose epilogue is still due: it runs once the dequant is `lag` stages into
    // the next item, by which time the item's MMAs are (nearly) done and the MMA has stages queued.
    // With one accumulator buffer the lag must not exceed J, or the dequant would wait on TMEM A
    // stages that only the next item's MMAs (blocked on this epilogue) can free.
    const uint32_t lag = (uint32_t)min(J, KS - 1);  // KS - 1: the epilogue always falls inside the next item
    int p_item = -1, p_a = 0;
    uint32_t p_it = 0, p_end = 0;
    float p_w = 0.f;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
      const int tile = item / nblk;
      int c_a = 0;
      float c_w = 0.f;
      if (KIND == 1) {
        // assignment id and weight of this thread's token column, for the epilogue
        const int n = g.tile_n[tile], rr = g.tile_row[tile] + grp * 32 + lane;
        if (grp * 32 + lane < n) {
          c_a = rr < g.n_assign ? g.perm[rr] : g.T * g.K + (rr - g.n_assign);
          c_w = rr < g.n_assign ? g.topk_w[c_a] : 1.f;
        }
      }
      for (int s = 0; s < KS; ++s, ++gs) {
        if (p_item >= 0 && gs >= p_end + lag) {
          if (!epilogue(p_item, p_it, p_a, p_w)) { ok = false; break; }
          p_item = -1;
        }
        if ((int)(gs & 1) != team) continue;
        const uint32_t as = gs / kSub;  // weight stage (continuous across items: K % 256 == 0)
        const int sub_k = gs % kSub;   // which 64-K part of it
        const int aslot = as % kAStages, slot = gs % BS, j = gs % J;
        // TMEM A stage j is free once the MMAs of stage gs - J have finished
        if (!tc::mbar_wait(&fa[aslot], (as / kAStages) & 1, &s_abort) ||
            (gs >= (uint32_t)J && !tc::mbar_wait(&sdone[(gs - J) % BS], ((gs - J) / BS) & 1, &s_abort))) {
          ok = false;
          break;
        }
        const uint8_t* arow = sA + ((aslot * NA + m) * kBM + row) * 128;
        // this row's two scales of the stage's 64 K (groups 2*sub_k, 2*sub_k + 1 of the weight stage)
        const uint32_t sc2 = *reinterpret_cast<const uint32_t*>(sS + ((aslot * NA + m) * kBM + row) * kScB + sub_k * 4);
        const __half2 scp = *reinterpret_cast<const __half2*>(&sc2);
        if (KIND == 0) {
          // the whole 64-K stage of matrix m: two 16-byte chunks
          uint32_t v[32];
          const uint4 q0 = *reinterpret_cast<const uint4*>(arow + (((2 * sub_k) ^ swz) << 4));
          const uint4 q1 = *reinterpret_cast<const uint4*>(arow + (((2 * sub_k + 1) ^ swz) << 4));
          dequant32(q0, __low2half2(scp), v);
          dequant32(q1, __high2half2(scp), v + 16);
          tc::tmem_st32(tmem + lane_base + 256 + j * (NA * 32) + m * 32, v);
        } else {
          // one 16-byte chunk (32 K) of the stage
          uint32_t v[16];
          const uint4 qq = *reinterpret_cast<const uint4*>(arow + (((2 * sub_k + sub) ^ swz) << 4));
          dequant32(qq, sub ? __high2half2(scp) : __low2half2(scp), v);
          tc::tmem_st16(tmem + lane_base + 256 + j * 32 + sub * 16, v);
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&tfull[slot]);
          if (sub_k >= kSub - 2) tc::mbar_arrive(&ea[aslot]);  // this warp's last part of the weight stage
        }
        __syncwarp();
      }
      if (!ok) break;
      p_item = item;
      p_it = it;
      p_end = gs;
      p_a = c_a;
      p_w = c_w;
    }
    if (ok && p_item >= 0) ok = epilogue(p_item, p_it, p_a, p_w);
    if (!ok) give_up();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ helper kernels
// Activations of the routed rows in dispatch order, fp16, K-permuted within 8-column blocks:
// row r < T*K holds token perm[r] / K, row T*K + t holds token t (shared expert).  One thread per
// 8-column block; flags values outside the fp16 range.
__global__ void xgather_kernel(const void* x, int act, const int32_t* perm, __half* xs, int T, int K, int d,
                               int has_shared, unsigned* status) {
  const int rows = T * K + (has_shared ? T : 0);
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)rows * d / 8) return;
  const int r = (int)(i / (d / 8)), c = (int)(i % (d / 8));
  const int tok = r < T * K ? perm[r] / K : r - T * K;
  float v[8];
  load8_act(x, act, (size_t)tok * d + c * 8, v);
  const int sig[8] = {0, 4, 1, 5, 2, 6, 3, 7};
  __align__(16) __half o[8];
  bool bad = false;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const float t = v[sig[p]];
    bad |= !(fabsf(t) <= 65504.f);
    o[p] = __float2half_rn(t);
  }
  *reinterpret_cast<uint4*>(xs + (size_t)r * d + c * 8) = *reinterpret_cast<const uint4*>(o);
  if (bad) atomicOr(status, kStatusRange);
}

// Tiles of <= 128 sorted rows: each active expert in ascending order, then the shared expert.
// One block of 1024 threads: a thread per slot (looping when there are more), block prefix sum of
// the tiles per slot, then every slot writes its own tiles.
__global__ void __launch_bounds__(1024) plan_tiles_kernel(const int4* slots, const int32_t* n_active, int E, int T,
                                                          int K, int has_shared, int32_t* n_tiles, int32_t* tg,
                                                          int32_t* tr, int32_t* tn) {
  __shared__ int wsum[32];
  __shared__ int carry;
  const int na = *n_active;
  const int ns = na + (has_shared ? 1 : 0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < ns; base += blockDim.x) {
    const int s = base + threadIdx.x;
    int e = 0, r0 = 0, c = 0;
    if (s < na) {
      const int4 sl = slots[s];
      e = sl.x;
      r0 = sl.y;
      c = sl.z;
    } else if (s < ns) {
      e = E;
      r0 = T * K;
      c = T;
    }
    const int nt = (c + kNT - 1) / kNT;
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = wsum[lane];
      int wi = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      wsum[lane] = wi - v;
    }
    __syncthreads();
    const int first = carry + wsum[warp] + incl - nt;
    for (int i = 0; i < nt; ++i) {
      tg[first + i] = e;
      tr[first + i] = r0 + i * kNT;
      tn[first + i] = min(kNT, c - i * kNT);
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = first + nt;
    __syncthreads();
  }
  if (threadIdx.x == 0) *n_tiles = carry;
}

// y[t] = sum_k P[t*K + k] + P[T*K + t] (+ resid), fp32, fixed order; 8 columns per thread.
__global__ void combine_kernel(const __nv_bfloat16* P, int T, int d, int K, int has_shared, const void* resid,
                               void* y, int act) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)T * d / 8) return;
  const int t = (int)(i / (d / 8));
  const int c0 = (int)(i % (d / 8)) * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int k = 0; k < K + (has_shared ? 1 : 0); ++k) {
    const size_t row = k < K ? (size_t)t * K + k : (size_t)T * K + t;
    const uint4 u = *reinterpret_cast<const uint4*>(P + row * d + c0);
    const __nv_bfloat16* pv = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
    for (int p = 0; p < 8; ++p) acc[p] += __bfloat162float(pv[p]);
  }
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const size_t o = (size_t)t * d + c0 + p;
    float v = acc[p];
    if (resid) v = load_act(resid, act, o) + v;
    store_act(y, act, o, v);
  }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

constexpr int kGemmSmemMax = 226 * 1024;

template <int KIND>
constexpr size_t gemm_smem_bytes() {
  return 1024 + (size_t)Stages<KIND>::B * kNT * 128 + (size_t)kAStages * Stages<KIND>::NA * kBM * (128 + kScB);
}
static_assert(gemm_smem_bytes<0>() <= kGemmSmemMax && gemm_smem_bytes<1>() <= kGemmSmemMax, "shared memory");

cudaError_t gemm_kernels_init() {
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cudaError_t e =
      cudaFuncSetAttribute(gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm_smem_bytes<0>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm_smem_bytes<1>());
}

bool gemm_shape_ok(int d, int f) {
  return d % kKA == 0 && f % kKA == 0;
}

size_t gemm_workspace_bytes(int T, int d, int f, int E, int K) {
  const size_t rows = (size_t)T * K + T;
  const size_t max_tiles = (size_t)(T * K) / kNT + E + (T + kNT - 1) / kNT + 2;
  auto up = [](size_t n) { return (n + 255) & ~size_t(255); };
  return up(rows * d * 2) + up(rows * f * 2) + up(rows * d * 2) + up(4) + 3 * up(max_tiles * 4) +
         up(sizeof(GemmActMaps) + 64);
}

static GemmWs carve(void* ws, int T, int d, int f, int E, int K) {
  const size_t rows = (size_t)T * K + T;
  const size_t max_tiles = (size_t)(T * K) / kNT + E + (T + kNT - 1) / kNT + 2;
  auto up = [](size_t n) { return (n + 255) & ~size_t(255); };
  char* p = static_cast<char*>(ws);
  GemmWs w;
  w.x16 = reinterpret_cast<__half*>(p); p += up(rows * d * 2);
  w.h16 = reinterpret_cast<__half*>(p); p += up(rows * f * 2);
  w.P = reinterpret_cast<__nv_bfloat16*>(p); p += up(rows * d * 2);
  w.n_tiles = reinterpret_cast<int32_t*>(p); p += up(4);
  w.tile_group = reinterpret_cast<int32_t*>(p); p += up(max_tiles * 4);
  w.tile_row = reinterpret_cast<int32_t*>(p); p += up(max_tiles * 4);
  w.tile_n = reinterpret_cast<int32_t*>(p);
  return w;
}

static cudaError_t make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t rows,
                            uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor maps of one layer's int4 planes (box: 128 rows x 128 bytes = 256 K, 128-byte swizzle) and
// fp16 scale planes (box: 128 rows x the 8 scales of the same 256 K, no swizzle).
cudaError_t gemm_build_maps(void* maps, int E, int d, int f, int has_shared, const void* gu_q, const void* gu_s,
                            const void* dn_q, const void* dn_s, const void* sh_gu_q, const void* sh_gu_s,
                            const void* sh_dn_q, const void* sh_dn_s) {
  if (!g_encode) return cudaErrorNotSupported;
  GemmMaps* mp = static_cast<GemmMaps*>(maps);
  const int Gd = d / 32, Gf = f / 32;
  const CUtensorMapSwizzle sgu = CU_TENSOR_MAP_SWIZZLE_NONE, sdn = CU_TENSOR_MAP_SWIZZLE_NONE;
  const uint32_t sbox = kScB / 2;
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cudaError_t e;
  if ((e = make_map(&mp->gu_q, gu_q, U8, d / 2, (uint64_t)E * 2 * f, d / 2, kKA / 2, kBM, CU_TENSOR_MAP_SWIZZLE_128B))) return e;
  if ((e = make_map(&mp->gu_s, gu_s, F16, Gd, (uint64_t)E * 2 * f, Gd * 2, sbox, kBM, sgu))) return e;
  if ((e = make_map(&mp->dn_q, dn_q, U8, f / 2, (uint64_t)E * d, f / 2, kKA / 2, kBM, CU_TENSOR_MAP_SWIZZLE_128B))) return e;
  if ((e = make_map(&mp->dn_s, dn_s, F16, Gf, (uint64_t)E * d, Gf * 2, sbox, kBM, sdn))) return e;
  const void* sgq = has_shared ? sh_gu_q : gu_q;  // maps must be valid even when unused
  const void* sgs = has_shared ? sh_gu_s : gu_s;
  const void* sdq = has_shared ? sh_dn_q : dn_q;
  const void* sds = has_shared ? sh_dn_s : dn_s;
  if ((e = make_map(&mp->sh_gu_q, sgq, U8, d / 2, 2 * f, d / 2, kKA / 2, kBM, CU_TENSOR_MAP_SWIZZLE_128B))) return e;
  if ((e = make_map(&mp->sh_gu_s, sgs, F16, Gd, 2 * f, Gd * 2, sbox, kBM, sgu))) return e;
  if ((e = make_map(&mp->sh_dn_q, sdq, U8, f / 2, d, f / 2, kKA / 2, kBM, CU_TENSOR_MAP_SWIZZLE_128B))) return e;
  if ((e = make_map(&mp->sh_dn_s, sds, F16, Gf, d, Gf * 2, sbox, kBM, sdn))) return e;
  return cudaSuccess;
}

// Tensor maps of the workspace's sorted activation rows (GEMM1 B) and h rows (GEMM2 B):
// box 128 rows x 64 fp16 columns, 128-byte swizzle.
cudaError_t gemm_build_act_maps(void* ws, int T, int d, int f, int E, int K, void* out) {
  if (!g_encode) return cudaErrorNotSupported;
  GemmWs w = carve(ws, T, d, f, E, K);
  GemmActMaps* am = static_cast<GemmActMaps*>(out);
  const uint64_t rows = (uint64_t)T * K + T;
  cudaError_t e = make_map(&am->xs, w.x16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, d, rows, (uint64_t)d * 2, kKS, kNT,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  return make_map(&am->hs, w.h16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, f, rows, (uint64_t)f * 2, kKS, kNT,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

size_t gemm_act_maps_bytes() { return sizeof(GemmActMaps); }

void* gemm_maps_new() { return aligned_alloc(64, (sizeof(GemmMaps) + 63) & ~size_t(63)); }
void gemm_maps_free(void* p) { free(p); }

// Launches: sorted fp16 activations, tile plan, GEMM1, [mid event], GEMM2, [mid2 event], combine.
cudaError_t launch_experts_gemm(const ExpertArgs& a, const void* maps_v, const void* act_maps_v, void* ws,
                                cudaStream_t st, cudaEvent_t mid, cudaEvent_t mid2) {
  const GemmMaps& mp = *static_cast<const GemmMaps*>(maps_v);
  const GemmActMaps& am = *static_cast<const GemmActMaps*>(act_maps_v);
  const int T = a.T, d = a.d, f = a.f, E = a.E, K = a.K;
  GemmWs w = carve(ws, a.max_tokens, d, f, E, K);  // layout fixed by max_tokens (the TMA maps point into it)
  const size_t rows = (size_t)T * K + (a.has_shared ? T : 0);
  const size_t nch = rows * d / 8;
  xgather_kernel<<<(unsigned)((nch + 255) / 256), 256, 0, st>>>(a.x, a.act, a.perm, w.x16, T, K, d, a.has_shared,
                                                                a.status);
  plan_tiles_kernel<<<1, 1024, 0, st>>>(a.slots, a.n_active, E, T, K, a.has_shared, w.n_tiles, w.tile_group,
                                        w.tile_row, w.tile_n);
  GemmArgs g;
  g.T = T;
  g.d = d;
  g.f = f;
  g.E = E;
  g.K = K;
  g.n_assign = T * K;
  g.has_shared = a.has_shared;
  g.perm = a.perm;
  g.topk_w = a.topk_w;
  g.h16 = w.h16;
  g.P = w.P;
  g.n_tiles = w.n_tiles;
  g.tile_group = w.tile_group;
  g.tile_row = w.tile_row;
  g.tile_n = w.tile_n;
  g.status = a.status;
  gemm_kernel<0><<<a.num_sms, kGemmThreads, gemm_smem_bytes<0>(), st>>>(g, mp.gu_q, mp.gu_s, mp.sh_gu_q, mp.sh_gu_s,
                                                                        am.xs);
  if (mid) record_timing_event(mid, st);
  gemm_kernel<1><<<a.num_sms, kGemmThreads, gemm_smem_bytes<1>(), st>>>(g, mp.dn_q, mp.dn_s, mp.sh_dn_q, mp.sh_dn_s,
                                                                        am.hs);
  if (mid2) record_timing_event(mid2, st);
  const size_t nblk8 = (size_t)T * d / 8;
  combine_kernel<<<(unsigned)((nblk8 + 255) / 256), 256, 0, st>>>(w.P, T, d, K, a.has_shared, a.resid, a.y, a.act);
  return cudaGetLastError();
}

}  // namespace moe
