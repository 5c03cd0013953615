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
//   warp 1     : one thread issues TMA loads of the int4 weight tiles and their fp16 scales
//   warps 2-3  : gather the tile's activation rows into 128B-swizzled SMEM with cp.async
//   warps 4-11 : dequantise int4 -> fp16 (q * scale, one rounding) straight into TMEM (tcgen05.st),
//                then the epilogue (tcgen05.ld of the fp32 accumulators)
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

constexpr int kGemmThreads = 384;
constexpr int kNT = 128;            // max token rows per tile (MMA N)
constexpr int kBM = 128;            // weight rows per A matrix (MMA M)
constexpr int kKS = 64;             // K per pipeline stage
constexpr int kStages = 6;          // SMEM stages
constexpr int kLoaders = 64;        // threads of warps 2-3
constexpr int kLag = 4;             // cp.async stages in flight per loader before it signals
constexpr unsigned kStatusRange = 4u;

struct GemmMaps {
  CUtensorMap gu_q, gu_s, sh_gu_q, sh_gu_s, dn_q, dn_s, sh_dn_q, sh_dn_s;
  int gu_s_sw128, dn_s_sw128;
};

struct GemmWs {
  __half* x16;          // [T][d] fp16, K-permuted
  __half* h16;          // [T*K + T][f] fp16, K-permuted
  __nv_bfloat16* P;     // [T*K + T][d] weighted per-assignment partials
  int32_t* n_tiles;     // [1]
  int32_t* tile_group;  // [max_tiles]
  int32_t* tile_row;
  int32_t* tile_n;
};

struct GemmArgs {
  int T, d, f, E, K, n_assign, has_shared, sc_sw128;
  const int32_t* perm;
  const float* topk_w;
  const __half* x16;
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

__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

template <int KIND>  // 0: gate/up + SwiGLU, 1: down + weighted partials
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const GemmArgs g, const __grid_constant__ CUtensorMap mq_r, const __grid_constant__ CUtensorMap ms_r,
                const __grid_constant__ CUtensorMap mq_s, const __grid_constant__ CUtensorMap ms_s) {
  constexpr int NA = KIND == 0 ? 2 : 1;  // A matrices per tile
  constexpr int NB = KIND == 0 ? 1 : 2;  // accumulator buffers
  constexpr int J = KIND == 0 ? 4 : 8;   // TMEM A stages
  const int Kdim = KIND == 0 ? g.d : g.f;
  const int KS = Kdim / kKS;
  const int G = Kdim / 32;
  const int nblk = (KIND == 0 ? g.f : g.d) / kBM;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;                               // kStages x [128 rows x 128 B]
  uint8_t* sA = sB + kStages * kNT * 128;           // kStages x NA x [128 rows x 32 B] int4
  uint8_t* sS = sA + kStages * NA * kBM * 32;       // 2 x NA x [128 rows x G fp16]
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], tfull[8], tempty[8], acc_full[2], acc_empty[2],
      sc_empty[2], fin, info_full[2], info_empty[2];
  __shared__ int info_a[2][kNT];    // down epilogue: assignment id of each tile row
  __shared__ float info_w[2][kNT];  // and its routing weight
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1 + kLoaders);
      tc::mbar_init(&empty[s], 1 + 8);
    }
    for (int j = 0; j < J; ++j) {
      tc::mbar_init(&tfull[j], 8);
      tc::mbar_init(&tempty[j], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], 8);
      tc::mbar_init(&sc_empty[b], 8);
    }
    tc::mbar_init(&fin, 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&info_full[b], kLoaders);
      tc::mbar_init(&info_empty[b], 8);
    }
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
    if (lane == 0) {
      uint32_t gs = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
        const int tile = item / nblk;
        const int nmma = (g.tile_n[tile] + 15) & ~15;
        const uint32_t idesc = tc::idesc_f16_f32(128, nmma);
        const int b = it % NB;
        if (!tc::mbar_wait(&acc_empty[b], ((it / NB) & 1) ^ 1, &s_abort)) { ok = false; break; }
        tc::tc_fence_after();
        for (int s = 0; s < KS; ++s, ++gs) {
          const int slot = gs % kStages, j = gs % J;
          if (!tc::mbar_wait(&full[slot], (gs / kStages) & 1, &s_abort) ||
              !tc::mbar_wait(&tfull[j], (gs / J) & 1, &s_abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t bbase = tc::smem_u32(sB + slot * kNT * 128);
#pragma unroll
          for (int kk = 0; kk < kKS / 16; ++kk) {
            const uint64_t bd = tc::sdesc_sw128(bbase + kk * 32);
#pragma unroll
            for (int m = 0; m < NA; ++m) {
              const uint32_t dcol = KIND == 0 ? m * 128 : b * 128;
              const uint32_t acol = 256 + j * (NA * 32) + m * 32 + kk * 8;
              tc::mma_ts(tmem + dcol, tmem + acol, bd, idesc, (s > 0 || kk > 0) ? 1u : 0u);
            }
          }
          tc::mma_commit(&empty[slot]);
          tc::mma_commit(&tempty[j]);
        }
        if (!ok) break;
        tc::mma_commit(&acc_full[b]);
      }
      if (!ok) give_up();
      tc::mma_commit(&fin);  // completes when every MMA issued above has finished
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
      uint32_t gs = 0, it = 0;
      bool ok = true;
      const int rows_per_expert = KIND == 0 ? 2 * g.f : g.d;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
        const int tile = item / nblk, blk = item % nblk;
        const int grp = g.tile_group[tile];
        const bool sh = grp >= g.E;
        const CUtensorMap* mq = sh ? &mq_s : &mq_r;
        const CUtensorMap* ms = sh ? &ms_s : &ms_r;
        const int r0 = (sh ? 0 : grp * rows_per_expert) + blk * kBM;
        const int sb = it & 1;
        for (int s = 0; s < KS; ++s, ++gs) {
          const int slot = gs % kStages;
          if (!tc::mbar_wait(&empty[slot], ((gs / kStages) & 1) ^ 1, &s_abort)) { ok = false; break; }
          uint32_t bytes = NA * kBM * 32;
          if (s == 0) {
            if (!tc::mbar_wait(&sc_empty[sb], ((it >> 1) & 1) ^ 1, &s_abort)) { ok = false; break; }
            bytes += NA * kBM * G * 2;
          }
          tc::mbar_arrive_expect_tx(&full[slot], bytes);
#pragma unroll
          for (int m = 0; m < NA; ++m) {
            tc::tma_load_2d(sA + (slot * NA + m) * kBM * 32, mq, s * 32, r0 + m * g.f, &full[slot]);
            if (s == 0) tc::tma_load_2d(sS + (sb * NA + m) * kBM * G * 2, ms, 0, r0 + m * g.f, &full[slot]);
          }
        }
      }
      if (!ok) give_up();
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---------------------------------------------------------------- B gather (cp.async)
    const int lt = threadIdx.x - 64;
    uint32_t gs = 0, sig = 0, it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
      const int tile = item / nblk;
      const int n = g.tile_n[tile], nmma = (n + 15) & ~15, row0 = g.tile_row[tile];
      const int grp = g.tile_group[tile];
      if (KIND == 1) {
        // assignment ids and weights of the tile's rows, for this item's epilogue
        const int ib = it & 1;
        if (!tc::mbar_wait(&info_empty[ib], ((it >> 1) & 1) ^ 1, &s_abort)) { ok = false; break; }
        for (int r = lt; r < n; r += kLoaders) {
          const int rr = row0 + r;
          const int as = rr < g.n_assign ? g.perm[rr] : g.T * g.K + (rr - g.n_assign);
          info_a[ib][r] = as;
          info_w[ib][r] = rr < g.n_assign ? g.topk_w[as] : 1.f;
        }
        tc::mbar_arrive(&info_full[ib]);
      }
      const __half* src[2];
      bool valid[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = lt + 64 * i;
        valid[i] = r < n;
        src[i] = g.x16;
        if (valid[i]) {
          if (KIND == 0) {
            const int tok = grp < g.E ? g.perm[row0 + r] / g.K : row0 + r - g.n_assign;
            src[i] = g.x16 + (size_t)tok * g.d;
          } else {
            src[i] = g.h16 + (size_t)(row0 + r) * g.f;
          }
        }
      }
      for (int s = 0; s < KS; ++s, ++gs) {
        const int slot = gs % kStages;
        if (!tc::mbar_wait(&empty[slot], ((gs / kStages) & 1) ^ 1, &s_abort)) { ok = false; break; }
        const uint32_t base = tc::smem_u32(sB + slot * kNT * 128);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = lt + 64 * i;
          if (r < nmma) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t dst = base + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
              tc::cp_async16(dst, valid[i] ? src[i] + s * kKS + c * 8 : g.x16, valid[i] ? 16u : 0u);
            }
          }
        }
        tc::cp_async_commit();
        if (gs + 1 - sig > (uint32_t)kLag) {
          tc::cp_async_wait<kLag>();
          tc::fence_proxy_async_smem();
          while (gs + 1 - sig > (uint32_t)kLag) {
            tc::mbar_arrive(&full[sig % kStages]);
            ++sig;
          }
        }
      }
    }
    tc::cp_async_wait<0>();
    tc::fence_proxy_async_smem();
    while (sig < gs) {
      tc::mbar_arrive(&full[sig % kStages]);
      ++sig;
    }
    if (!ok) give_up();
  } else {
    // ---------------------------------------------------------------- dequant + epilogue
    const int q = warp & 3;
    const int m = (warp - 4) >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    const int swz = (row >> 2) & 1;  // 32-byte swizzle of the int4 tiles: 16-byte chunk c sits at c ^ bit 7 of the address
    uint32_t gs = 0, it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
      const int tile = item / nblk, blk = item % nblk;
      const int n = g.tile_n[tile], row0 = g.tile_row[tile];
      const int sb = it & 1;
      const uint8_t* srow = sS + ((sb * NA + (KIND == 0 ? m : 0)) * kBM + row) * G * 2;
      for (int s = 0; s < KS; ++s, ++gs) {
        const int slot = gs % kStages, j = gs % J;
        if (!tc::mbar_wait(&full[slot], (gs / kStages) & 1, &s_abort) ||
            !tc::mbar_wait(&tempty[j], ((gs / J) & 1) ^ 1, &s_abort)) {
          ok = false;
          break;
        }
        const uint8_t* arow = sA + ((slot * NA + (KIND == 0 ? m : 0)) * kBM + row) * 32;
        auto scale_at = [&](int grp_idx) -> __half2 {
          const int o = grp_idx * 2;
          const int off = g.sc_sw128 ? ((((o >> 4) ^ (row & 7)) << 4) | (o & 15)) : o;
          const __half s1 = *reinterpret_cast<const __half*>(srow + off);
          return __halves2half2(s1, s1);
        };
        if (KIND == 0) {
          uint32_t v[32];
          const uint4 q0 = *reinterpret_cast<const uint4*>(arow + ((0 ^ swz) << 4));
          const uint4 q1 = *reinterpret_cast<const uint4*>(arow + ((1 ^ swz) << 4));
          dequant32(q0, scale_at(2 * s), v);
          dequant32(q1, scale_at(2 * s + 1), v + 16);
          tc::tmem_st32(tmem + lane_base + 256 + j * (NA * 32) + m * 32, v);
        } else {
          uint32_t v[16];
          const uint4 qq = *reinterpret_cast<const uint4*>(arow + ((m ^ swz) << 4));
          dequant32(qq, scale_at(2 * s + m), v);
          tc::tmem_st16(tmem + lane_base + 256 + j * 32 + m * 16, v);
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&tfull[j]);
          tc::mbar_arrive(&empty[slot]);
          if (s == KS - 1) tc::mbar_arrive(&sc_empty[sb]);
        }
      }
      if (!ok) break;
      // epilogue
      const int b = it % NB;
      if (!tc::mbar_wait(&acc_full[b], (it / NB) & 1, &s_abort)) { ok = false; break; }
      if (KIND == 1 && !tc::mbar_wait(&info_full[it & 1], (it >> 1) & 1, &s_abort)) { ok = false; break; }
      tc::tc_fence_after();
      bool range_bad = false;
      for (int cb = m * 64; cb < m * 64 + 64 && cb < n; cb += 32) {
        if (KIND == 0) {
          uint32_t gv[32], uv[32];
          tc::tmem_ld32(tmem + lane_base + cb, gv);
          tc::tmem_ld32(tmem + lane_base + 128 + cb, uv);
          tc::tmem_wait_ld();
          const int fidx = blk * kBM + row;
          const int fpos = (fidx & ~7) | inv_perm8(fidx & 7);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int nn = cb + jj;
            if (nn < n) {
              const float hv = silu_fast(__uint_as_float(gv[jj])) * __uint_as_float(uv[jj]);
              range_bad |= !(fabsf(hv) <= 65504.f);
              g.h16[(size_t)(row0 + nn) * g.f + fpos] = __float2half_rn(hv);
            }
          }
        } else {
          uint32_t ov[32];
          tc::tmem_ld32(tmem + lane_base + b * 128 + cb, ov);
          tc::tmem_wait_ld();
          const int jrow = blk * kBM + row;
          const int ib = it & 1;
#pragma unroll 8
          for (int jj = 0; jj < 32; ++jj) {
            const int nn = cb + jj;
            if (nn < n)
              g.P[(size_t)info_a[ib][nn] * g.d + jrow] = __float2bfloat16_rn(info_w[ib][nn] * __uint_as_float(ov[jj]));
          }
        }
      }
      if (range_bad) atomicOr(g.status, kStatusRange);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&acc_empty[b]);
        if (KIND == 1) tc::mbar_arrive(&info_empty[it & 1]);
      }
    }
    if (!ok) give_up();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ helper kernels
// x (act type) -> fp16, K-permuted within 8-column blocks; flags values outside the fp16 range.
__global__ void xconv_kernel(const void* x, int act, __half* x16, int T, int d, unsigned* status) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // one 8-column block
  if (i >= (size_t)T * d / 8) return;
  float v[8];
#pragma unroll
  for (int p = 0; p < 8; ++p) v[p] = load_act(x, act, i * 8 + p);
  const int sig[8] = {0, 4, 1, 5, 2, 6, 3, 7};
  __align__(16) __half o[8];
  bool bad = false;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const float t = v[sig[p]];
    bad |= !(fabsf(t) <= 65504.f);
    o[p] = __float2half_rn(t);
  }
  *reinterpret_cast<uint4*>(x16 + i * 8) = *reinterpret_cast<const uint4*>(o);
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
static int g_sms = 148;

constexpr int kGemmSmemMax = 220 * 1024;

static size_t gemm_smem_bytes(int kind, int d, int f) {
  const int NA = kind == 0 ? 2 : 1;
  const int G = (kind == 0 ? d : f) / 32;
  return 1024 + (size_t)kStages * kNT * 128 + (size_t)kStages * NA * kBM * 32 + (size_t)2 * NA * kBM * G * 2;
}

cudaError_t gemm_kernels_init(int num_sms) {
  g_sms = num_sms;
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  // the largest dynamic size any supported shape needs (d <= 8192, f <= 8192 keep it under the limit)
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemMax);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemMax);
}

bool gemm_shape_ok(int d, int f) {
  return d % 256 == 0 && f % 256 == 0 && d / 32 <= 256 && f / 32 <= 256 &&
         gemm_smem_bytes(0, d, f) <= kGemmSmemMax && gemm_smem_bytes(1, d, f) <= kGemmSmemMax;
}

size_t gemm_workspace_bytes(int T, int d, int f, int E, int K) {
  const size_t rows = (size_t)T * K + T;
  const size_t max_tiles = (size_t)(T * K) / kNT + E + (T + kNT - 1) / kNT + 2;
  auto up = [](size_t n) { return (n + 255) & ~size_t(255); };
  return up((size_t)T * d * 2) + up(rows * f * 2) + up(rows * d * 2) + up(4) + 3 * up(max_tiles * 4);
}

static GemmWs carve(void* ws, int T, int d, int f, int E, int K) {
  const size_t rows = (size_t)T * K + T;
  const size_t max_tiles = (size_t)(T * K) / kNT + E + (T + kNT - 1) / kNT + 2;
  auto up = [](size_t n) { return (n + 255) & ~size_t(255); };
  char* p = static_cast<char*>(ws);
  GemmWs w;
  w.x16 = reinterpret_cast<__half*>(p); p += up((size_t)T * d * 2);
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

// Tensor maps of one layer's int4 planes (box: 128 rows x 32 bytes) and fp16 scale planes
// (box: 128 rows x the whole row of scales).
cudaError_t gemm_build_maps(void* maps, int E, int d, int f, int has_shared, const void* gu_q, const void* gu_s,
                            const void* dn_q, const void* dn_s, const void* sh_gu_q, const void* sh_gu_s,
                            const void* sh_dn_q, const void* sh_dn_s) {
  if (!g_encode) return cudaErrorNotSupported;
  GemmMaps* mp = static_cast<GemmMaps*>(maps);
  const int Gd = d / 32, Gf = f / 32;
  const CUtensorMapSwizzle sgu = Gd * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUtensorMapSwizzle sdn = Gf * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  mp->gu_s_sw128 = sgu == CU_TENSOR_MAP_SWIZZLE_128B;
  mp->dn_s_sw128 = sdn == CU_TENSOR_MAP_SWIZZLE_128B;
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cudaError_t e;
  if ((e = make_map(&mp->gu_q, gu_q, U8, d / 2, (uint64_t)E * 2 * f, d / 2, 32, kBM, CU_TENSOR_MAP_SWIZZLE_32B))) return e;
  if ((e = make_map(&mp->gu_s, gu_s, F16, Gd, (uint64_t)E * 2 * f, Gd * 2, Gd, kBM, sgu))) return e;
  if ((e = make_map(&mp->dn_q, dn_q, U8, f / 2, (uint64_t)E * d, f / 2, 32, kBM, CU_TENSOR_MAP_SWIZZLE_32B))) return e;
  if ((e = make_map(&mp->dn_s, dn_s, F16, Gf, (uint64_t)E * d, Gf * 2, Gf, kBM, sdn))) return e;
  const void* sgq = has_shared ? sh_gu_q : gu_q;  // maps must be valid even when unused
  const void* sgs = has_shared ? sh_gu_s : gu_s;
  const void* sdq = has_shared ? sh_dn_q : dn_q;
  const void* sds = has_shared ? sh_dn_s : dn_s;
  if ((e = make_map(&mp->sh_gu_q, sgq, U8, d / 2, 2 * f, d / 2, 32, kBM, CU_TENSOR_MAP_SWIZZLE_32B))) return e;
  if ((e = make_map(&mp->sh_gu_s, sgs, F16, Gd, 2 * f, Gd * 2, Gd, kBM, sgu))) return e;
  if ((e = make_map(&mp->sh_dn_q, sdq, U8, f / 2, d, f / 2, 32, kBM, CU_TENSOR_MAP_SWIZZLE_32B))) return e;
  if ((e = make_map(&mp->sh_dn_s, sds, F16, Gf, d, Gf * 2, Gf, kBM, sdn))) return e;
  return cudaSuccess;
}

void* gemm_maps_new() { return aligned_alloc(64, (sizeof(GemmMaps) + 63) & ~size_t(63)); }
void gemm_maps_free(void* p) { free(p); }

// Launches: x -> fp16, tile plan, GEMM1, [mid event], GEMM2, combine.
cudaError_t launch_experts_gemm(const ExpertArgs& a, const void* maps_v, void* ws, cudaStream_t st, cudaEvent_t mid,
                                cudaEvent_t mid2) {
  const GemmMaps& mp = *static_cast<const GemmMaps*>(maps_v);
  const int T = a.T, d = a.d, f = a.f, E = a.E, K = a.K;
  GemmWs w = carve(ws, T, d, f, E, K);
  const size_t nblk8 = (size_t)T * d / 8;
  xconv_kernel<<<(unsigned)((nblk8 + 255) / 256), 256, 0, st>>>(a.x, a.act, w.x16, T, d, a.status);
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
  g.x16 = w.x16;
  g.h16 = w.h16;
  g.P = w.P;
  g.n_tiles = w.n_tiles;
  g.tile_group = w.tile_group;
  g.tile_row = w.tile_row;
  g.tile_n = w.tile_n;
  g.status = a.status;
  g.sc_sw128 = mp.gu_s_sw128;
  gemm_kernel<0><<<g_sms, kGemmThreads, gemm_smem_bytes(0, d, f), st>>>(g, mp.gu_q, mp.gu_s, mp.sh_gu_q, mp.sh_gu_s);
  if (mid) record_timing_event(mid, st);
  g.sc_sw128 = mp.dn_s_sw128;
  gemm_kernel<1><<<g_sms, kGemmThreads, gemm_smem_bytes(1, d, f), st>>>(g, mp.dn_q, mp.dn_s, mp.sh_dn_q, mp.sh_dn_s);
  if (mid2) record_timing_event(mid2, st);
  combine_kernel<<<(unsigned)((nblk8 + 255) / 256), 256, 0, st>>>(w.P, T, d, K, a.has_shared, a.resid, a.y, a.act);
  return cudaGetLastError();
}

}  // namespace moe
