// Router, top-K selection and token->expert dispatch (sm_103a).
//
// The router scores every expert of the layer for every token and keeps the 10 best per token
// ('Strata はなぜ少ない VRAM でも速いのか' (modeldock.net), section '問題：1,250 億パラメータと
// 12 GB'); the chosen expert numbers are handed on to whoever computes the experts (same page,
// section '1 トークン、三者の分担', where they go to a page-locked "doorbell" for the CPU).  Here
// every expert is in HBM, so the hand-off is a device-side dispatch: a per-expert histogram, an
// exclusive prefix sum and a stable counting sort of the assignments, plus the ascending list of
// distinct experts, all deterministic.
//
// Arithmetic: logits in fp32 (FMA, fixed per-lane order + fixed shuffle tree), softmax over all E
// logits with expf, K rounds of warp arg-max (larger logit first, ties to the lower index), the
// kept probabilities renormalised.  Selection compares fp32 logits.
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace moe {

// Block-wide exclusive scan of vals[0..n) in shared memory, n <= 4 * blockDim.x, blockDim a
// multiple of 32 and <= 1024.  Returns the total on every thread.
__device__ int block_exclusive_scan(int* vals, int n, int* scratch /* >= 33 ints */) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int per = (n + blockDim.x - 1) / blockDim.x;  // <= 4
  int loc[4];
  int s = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = tid * per + i;
    loc[i] = (i < per && j < n) ? vals[j] : 0;
    s += loc[i];
  }
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < nwarps ? scratch[lane] : 0;
    int wi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    scratch[lane] = wi - v;          // exclusive prefix of warp totals
    if (lane == 31) scratch[32] = wi; // grand total
  }
  __syncthreads();
  int run = scratch[warp] + incl - s;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = tid * per + i;
    if (i < per && j < n) {
      vals[j] = run;
      run += loc[i];
    }
  }
  const int total = scratch[32];
  __syncthreads();
  return total;
}

// Softmax over E logits (in shared memory, one warp), the K largest (ties: lower index), weights
// renormalised over the kept K.  Writes idx/w for the token (global).  sidx / sp: K-entry scratch.
__device__ void topk_warp(const float* lg, int E, int K, int32_t* out_idx, float* out_w, int32_t* sidx,
                          float* sp) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int e = lane; e < E; e += 32) m = fmaxf(m, lg[e]);
  m = warp_max(m);
  float z = 0.f;
  for (int e = lane; e < E; e += 32) z += expf(lg[e] - m);
  z = warp_sum(z);
  uint32_t taken = 0u;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    int j = 0;
    for (int e = lane; e < E; e += 32, ++j) {
      if ((taken >> j) & 1u) continue;
      const float v = lg[e];
      if (bi == 0x7fffffff || v > bv) {
        bv = v;
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) {
      sidx[k] = bi;
      sp[k] = expf(bv - m) / z;
    }
  }
  __syncwarp();
  if (lane < K) {
    float s = 0.f;
    for (int k = 0; k < K; ++k) s += sp[k];
    out_idx[lane] = sidx[lane];
    out_w[lane] = sp[lane] / s;
  }
  __syncwarp();
}

// ------------------------------------------------------------------ small T (fused, one launch)
// grid = ceil(E / 4) blocks of 256 threads; two warps score one expert (half a row each) for all T
// tokens; the last block to finish (ticket) runs softmax/top-K for every token (logits held in
// registers, one warp per token) and the dispatch, entirely from shared memory.
// Dynamic shared memory: T*d floats (activations).
__global__ void __launch_bounds__(256) route_small_kernel(RouteArgs a) {
  extern __shared__ float smem[];
  float* xs = smem;                         // [T][d]
  __shared__ float part[kRouterExpertsPerBlock][2][kSmallT];
  __shared__ int32_t idx_s[kSmallT * kMaxK];
  __shared__ int cnt[kMaxE], offv[kMaxE], flag[kMaxE];
  __shared__ float inv_s[kSmallT];
  __shared__ int scratch[40];
  __shared__ int is_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, d = a.d, E = a.E, K = a.K;

  const int e = blockIdx.x * kRouterExpertsPerBlock + (warp >> 1);
  const int half = warp & 1;
  const int nc = d >> 2;
  const int hc = (nc + 1) >> 1;
  const int cbeg = half ? hc : 0, cend = half ? nc : hc;
  const float4* wr = reinterpret_cast<const float4*>(a.Wr + (size_t)(e < E ? e : 0) * d);
  // the router row does not depend on x: start its loads before the activations are staged
  float4 wv[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int c = cbeg + lane + 32 * i;
    wv[i] = (e < E && c < cend) ? __ldg(wr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int nch = T * d / 8;  // 8-activation chunks, loaded 16 bytes at a time
  if (a.prenorm) {
    // sum of squares per token: one warp per token, a lane's chunks loaded together
    for (int t = warp; t < T; t += kRouterWarps) {
      float ss = 0.f;
      for (int c0 = 0; c0 < d / 8; c0 += 32 * 8) {
        float v[8][8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = c0 + lane + 32 * u;
          if (c < d / 8) load8_act(a.x, a.act, (size_t)t * d + c * 8, v[u]);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (c0 + lane + 32 * u < d / 8) {
#pragma unroll
            for (int q = 0; q < 8; ++q) ss = fmaf(v[u][q], v[u][q], ss);
          }
        }
      }
      ss = warp_sum(ss);
      if (lane == 0) inv_s[t] = 1.0f / sqrtf(ss / (float)d + a.eps);
    }
    __syncthreads();
  }
  for (int c0 = tid; c0 < nch; c0 += 4 * blockDim.x) {
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
        if (a.prenorm) {
          const float inv = inv_s[(c * 8) / d];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            v[u][q] = round_act(a.act, v[u][q] * inv);
            if (blockIdx.x == 0) store_act(a.xnorm, a.act, (size_t)c * 8 + q, v[u][q]);
          }
        }
        float4* xp = reinterpret_cast<float4*>(xs + (size_t)c * 8);
        xp[0] = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
        xp[1] = make_float4(v[u][4], v[u][5], v[u][6], v[u][7]);
      }
    }
  }
  __syncthreads();

  {
    float acc[kSmallT];
#pragma unroll
    for (int t = 0; t < kSmallT; ++t) acc[t] = 0.f;
    for (int c0 = cbeg; c0 < cend; c0 += 32 * 16) {
      if (c0 > cbeg) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = c0 + lane + 32 * i;
          wv[i] = (e < E && c < cend) ? __ldg(wr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = c0 + lane + 32 * i;
        if (c < cend) {
#pragma unroll
          for (int t = 0; t < kSmallT; ++t) {
            if (t < T) {
              const float4 xv = reinterpret_cast<const float4*>(xs + (size_t)t * d)[c];
              acc[t] = fmaf(wv[i].x, xv.x, acc[t]);
              acc[t] = fmaf(wv[i].y, xv.y, acc[t]);
              acc[t] = fmaf(wv[i].z, xv.z, acc[t]);
              acc[t] = fmaf(wv[i].w, xv.w, acc[t]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kSmallT; ++t) {
      if (t < T) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) part[warp >> 1][half][t] = v;
      }
    }
  }
  __syncthreads();
  if (tid < kRouterExpertsPerBlock * T) {
    const int le = tid / T, t = tid - le * T;
    const int ee = blockIdx.x * kRouterExpertsPerBlock + le;
    if (ee < E) a.logits[(size_t)t * E + ee] = (part[le][0][t] + part[le][1][t]) + (a.bias ? a.bias[ee] : 0.f);
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned tk = atomicAdd(a.ticket, 1u);
    is_last = (tk == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // ---- last block: softmax + top-K per token, one warp per token (logits held in registers).
  for (int i = tid; i < E; i += blockDim.x) cnt[i] = 0;
  for (int t = warp; t < T; t += kRouterWarps) {
    int my_i;
    float my_w;
    topk_token(a.logits + (size_t)t * E, E, K, my_i, my_w);
    if (lane < K) {
      a.idx[(size_t)t * K + lane] = my_i;
      a.w[(size_t)t * K + lane] = my_w;
      idx_s[t * K + lane] = my_i;
    }
  }
  __syncthreads();
  // ---- dispatch (shared memory only)
  const int n = T * K;
  for (int i = tid; i < n; i += blockDim.x) atomicAdd(&cnt[idx_s[i]], 1);
  __syncthreads();
  for (int i = tid; i < E; i += blockDim.x) {
    const int c = cnt[i];
    a.counts[i] = c;
    offv[i] = c;
    flag[i] = c > 0 ? 1 : 0;
    if (a.usage && c) a.usage[i] += (unsigned long long)c;
  }
  __syncthreads();
  const int total = block_exclusive_scan(offv, E, scratch);
  const int nact = block_exclusive_scan(flag, E, scratch);
  for (int i = tid; i < E; i += blockDim.x) {
    a.offs[i] = offv[i];
    if (cnt[i] > 0) {
      a.active[flag[i]] = i;
      a.slots[flag[i]] = make_int4(i, offv[i], cnt[i], 0);
    }
  }
  for (int i = tid; i < n; i += blockDim.x) {
    const int ei = idx_s[i];
    int r = 0;
    for (int j = 0; j < i; ++j) r += (idx_s[j] == ei);
    a.perm[offv[ei] + r] = i;
  }
  if (tid == 0) {
    a.offs[E] = total;
    *a.n_active = nact;
    if (a.stat) *a.stat = nact;
    *a.ticket = 0u;
  }
}

// ------------------------------------------------------------------ large T
// RMSNorm without weight, one warp per token: xnorm = round_act(x / sqrt(mean(x^2) + eps)).
__global__ void __launch_bounds__(256) rmsnorm_kernel(const void* x, void* xnorm, int act, int T, int d, float eps) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  float ss = 0.f;
  for (int j = lane; j < d; j += 32) {
    const float v = load_act(x, act, (size_t)t * d + j);
    ss += v * v;
  }
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / (float)d + eps);
  for (int j = lane; j < d; j += 32)
    store_act(xnorm, act, (size_t)t * d + j, load_act(x, act, (size_t)t * d + j) * inv);
}

// logits[T][E] = X[T][d] * Wr[E][d]^T (+ bias), fp32 FMA in ascending k per output.
// Register-blocked SIMT GEMM: CTA tile 128 tokens x 128 experts, k-step 8, 256 threads, 8 x 8
// outputs per thread held in registers (rows ty*4 + {0..3, 64..67}, columns tx*4 + {0..3, 64..67},
// so every shared-memory read is a conflict-free 16-byte load).  Both operands are staged k-major
// in shared memory, double-buffered; the next k-step's global loads are in flight while the current
// one is multiplied.  Activations are widened from bf16 as they are staged.
constexpr int kRlBM = 128, kRlBN = 128, kRlBK = 8;
__global__ void __launch_bounds__(256) router_logits_kernel(const void* x, int act, const float* Wr, const float* bias,
                                                            float* logits, int T, int d, int E) {
  __shared__ __align__(16) float As[2][kRlBK][kRlBM];
  __shared__ __align__(16) float Bs[2][kRlBK][kRlBN];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.y * kRlBM, e0 = blockIdx.x * kRlBN;
  // staging: thread tid loads row (tid >> 1) and 4 consecutive k (tid & 1) * 4 of each operand
  const int lr = tid >> 1, lk = (tid & 1) * 4;
  const int ta = t0 + lr, eb = e0 + lr;
  const bool a_on = ta < T, b_on = eb < E;
  float ra[4], rb[4];
  auto load = [&](int k0) {
    if (a_on) {
      if (act == kActBf16) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(x) + (size_t)ta * d + k0 + lk));
        ra[0] = __uint_as_float(u.x << 16);
        ra[1] = __uint_as_float(u.x & 0xFFFF0000u);
        ra[2] = __uint_as_float(u.y << 16);
        ra[3] = __uint_as_float(u.y & 0xFFFF0000u);
      } else {
        const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + (size_t)ta * d + k0 + lk));
        ra[0] = v.x; ra[1] = v.y; ra[2] = v.z; ra[3] = v.w;
      }
    } else {
      ra[0] = ra[1] = ra[2] = ra[3] = 0.f;
    }
    if (b_on) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(Wr + (size_t)eb * d + k0 + lk));
      rb[0] = v.x; rb[1] = v.y; rb[2] = v.z; rb[3] = v.w;
    } else {
      rb[0] = rb[1] = rb[2] = rb[3] = 0.f;
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      As[buf][lk + i][lr] = ra[i];
      Bs[buf][lk + i][lr] = rb[i];
    }
  };
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  load(0);
  store(0);
  __syncthreads();
  const int nk = d / kRlBK;
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) load((kt + 1) * kRlBK);
#pragma unroll
    for (int k = 0; k < kRlBK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4 + 64]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4 + 64]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (kt + 1 < nk) {
      store(buf ^ 1);
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + ty * 4 + (i & 3) + (i >> 2) * 64;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + tx * 4 + (j & 3) + (j >> 2) * 64;
      if (e < E) logits[(size_t)t * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
    }
  }
}

// logits[T][E] = X[T][d] Wr[E][d]^T (+ bias) for bf16 activations on fp16 tensor cores (mma.sync
// m16n8k16, fp32 accumulation).  X is one fp16 operand (bf16 values are exact in fp16 inside its
// range; |x| > 65504 sets the range status bit).  The fp32 router rows become two fp16 operands,
// hi = fp16(w) and lo = fp16((w - hi) 2^11), so that |w - hi - 2^-11 lo| <= 2^-22 |w| (up to fp16
// subnormals for |w| < 2^-3 of the smallest normal): logits = X hi^T + 2^-11 X lo^T, each product
// exact; every k16 partial product is added to fp32 running sums with round-to-nearest additions
// (fp32-level accuracy as the SIMT kernel above, in another order).
// CTA tile 128 tokens x 128 experts, k-step 32, 512 threads (16 warps of 32 x 32), operands staged
// through registers into padded shared rows (80 bytes: conflict-free ldmatrix), double-buffered.
constexpr int kRmBM = 128, kRmBN = 128, kRmBK = 32, kRmRow = kRmBK + 8;  // row stride in halves
constexpr size_t kRmSmem = (size_t)2 * 3 * kRmBM * kRmRow * 2;           // x, hi, lo; two buffers
__device__ __forceinline__ void rm_ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void rm_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__global__ void __launch_bounds__(512, 1) router_logits_mma_kernel(const __nv_bfloat16* x, const float* Wr,
                                                                   const float* bias, float* logits, int T, int d,
                                                                   int E, unsigned* status) {
  extern __shared__ __align__(16) uint8_t rm_smem[];
  __half* xs = reinterpret_cast<__half*>(rm_smem);  // [2][BM][kRmRow]
  __half* hs = xs + 2 * kRmBM * kRmRow;              // [2][BN][kRmRow]
  __half* ls = hs + 2 * kRmBN * kRmRow;              // [2][BN][kRmRow]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.y * kRmBM, e0 = blockIdx.x * kRmBN;
  // staging: thread tid takes row tid / 4 and k (tid % 4) * 8 .. + 7 of each operand
  const int lr = tid >> 2, lk = (tid & 3) * 8;
  const bool a_on = t0 + lr < T, b_on = e0 + lr < E;
  const __nv_bfloat16* xrow = x + (size_t)(t0 + lr) * d + lk;
  const float* wrow = Wr + (size_t)(e0 + lr) * d + lk;
  uint4 ra;
  float4 rb0, rb1;
  bool range_bad = false;
  auto load = [&](int k0) {
    ra = a_on ? __ldg(reinterpret_cast<const uint4*>(xrow + k0)) : make_uint4(0u, 0u, 0u, 0u);
    rb0 = b_on ? __ldg(reinterpret_cast<const float4*>(wrow + k0)) : make_float4(0.f, 0.f, 0.f, 0.f);
    rb1 = b_on ? __ldg(reinterpret_cast<const float4*>(wrow + k0 + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  auto store = [&](int buf) {
    const uint32_t xw[4] = {ra.x, ra.y, ra.z, ra.w};
    uint32_t xo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float v0 = __uint_as_float(xw[q] << 16), v1 = __uint_as_float(xw[q] & 0xFFFF0000u);
      range_bad |= !(fabsf(v0) <= 65504.f) || !(fabsf(v1) <= 65504.f);
      const __half2 h2 = __floats2half2_rn(v0, v1);
      xo[q] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(xs + ((size_t)buf * kRmBM + lr) * kRmRow + lk) = make_uint4(xo[0], xo[1], xo[2], xo[3]);
    const float wv[8] = {rb0.x, rb0.y, rb0.z, rb0.w, rb1.x, rb1.y, rb1.z, rb1.w};
    uint32_t ho[4], lo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half h0 = __float2half_rn(wv[2 * q]), h1 = __float2half_rn(wv[2 * q + 1]);
      const __half l0 = __float2half_rn((wv[2 * q] - __half2float(h0)) * 2048.f);
      const __half l1 = __float2half_rn((wv[2 * q + 1] - __half2float(h1)) * 2048.f);
      ho[q] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
      lo[q] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
    }
    *reinterpret_cast<uint4*>(hs + ((size_t)buf * kRmBN + lr) * kRmRow + lk) = make_uint4(ho[0], ho[1], ho[2], ho[3]);
    *reinterpret_cast<uint4*>(ls + ((size_t)buf * kRmBN + lr) * kRmRow + lk) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  };
  const int wm = warp >> 2, wn = warp & 3;  // warp tile: tokens wm*32 .. +31, experts wn*32 .. +31
  float ch[2][4][4], cl[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) ch[i][j][q] = cl[i][j][q] = 0.f;
  // ldmatrix lane addresses (element offsets within a buffer)
  const int a_off = (wm * 32 + (lane & 15)) * kRmRow + (lane >> 4) * 8;
  const int b_off = (wn * 32 + ((lane >> 4) << 3) + (lane & 7)) * kRmRow + ((lane >> 3) & 1) * 8;
  const uint32_t xs_u = tc::smem_u32(xs), hs_u = tc::smem_u32(hs), ls_u = tc::smem_u32(ls);
  load(0);
  store(0);
  __syncthreads();
  const int nk = d / kRmBK;
#pragma unroll 1
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) load((kt + 1) * kRmBK);
    const uint32_t xb = xs_u + (uint32_t)(buf * kRmBM * kRmRow) * 2, hb = hs_u + (uint32_t)(buf * kRmBN * kRmRow) * 2,
                   lb = ls_u + (uint32_t)(buf * kRmBN * kRmRow) * 2;
#pragma unroll
    for (int kk = 0; kk < kRmBK; kk += 16) {
      uint32_t a[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
        rm_ldsm_x4(xb + (uint32_t)(a_off + i * 16 * kRmRow + kk) * 2, a[i][0], a[i][1], a[i][2], a[i][3]);
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {  // pairs of n8 tiles
        uint32_t bh[4], bl[4];
        rm_ldsm_x4(hb + (uint32_t)(b_off + jp * 16 * kRmRow + kk) * 2, bh[0], bh[1], bh[2], bh[3]);
        rm_ldsm_x4(lb + (uint32_t)(b_off + jp * 16 * kRmRow + kk) * 2, bl[0], bl[1], bl[2], bl[3]);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          // each k16 product from zero, then added in fp32 (round to nearest): the tensor core's own
          // accumulation covers 16 terms only
          float p[4][4] = {};
          rm_mma(p[0], a[i][0], a[i][1], a[i][2], a[i][3], bh[0], bh[1]);
          rm_mma(p[1], a[i][0], a[i][1], a[i][2], a[i][3], bh[2], bh[3]);
          rm_mma(p[2], a[i][0], a[i][1], a[i][2], a[i][3], bl[0], bl[1]);
          rm_mma(p[3], a[i][0], a[i][1], a[i][2], a[i][3], bl[2], bl[3]);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            ch[i][2 * jp][q] += p[0][q];
            ch[i][2 * jp + 1][q] += p[1][q];
            cl[i][2 * jp][q] += p[2][q];
            cl[i][2 * jp + 1][q] += p[3][q];
          }
        }
      }
    }
    if (kt + 1 < nk) {
      // the other buffer was last read in the previous step, before its closing barrier
      store(buf ^ 1);
      __syncthreads();
    }
  }
  if (range_bad) atomicOr(status, kStatusRange);
  const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t = t0 + wm * 32 + i * 16 + g + 8 * h;
        if (t >= T) continue;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int e = e0 + wn * 32 + j * 8 + 2 * t4 + c;
          if (e < E)
            logits[(size_t)t * E + e] =
                ch[i][j][2 * h + c] + cl[i][j][2 * h + c] * (1.0f / 2048.f) + (bias ? bias[e] : 0.f);
        }
      }
}

// Top-K for T tokens, one warp per token.  Dynamic shared memory: 8*E floats.
__global__ void __launch_bounds__(256) topk_kernel(RouteArgs a) {
  extern __shared__ float smem[];
  __shared__ int32_t sidx[kRouterWarps][kMaxK];
  __shared__ float sp[kRouterWarps][kMaxK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kRouterWarps + warp;
  if (t >= a.T) return;
  float* lg = smem + (size_t)warp * a.E;
  for (int j = lane; j < a.E; j += 32) lg[j] = a.logits[(size_t)t * a.E + j];
  __syncwarp();
  topk_warp(lg, a.E, a.K, a.idx + (size_t)t * a.K, a.w + (size_t)t * a.K, sidx[warp], sp[warp]);
}

constexpr int kDispatchBlock = 256;  // assignments per block of the large-T dispatch

// Per-block histogram of expert ids: blockhist[b][e].
__global__ void __launch_bounds__(kDispatchBlock) dispatch_hist_kernel(RouteArgs a) {
  __shared__ int cnt[kMaxE];
  const int n = a.T * a.K;
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int i = blockIdx.x * kDispatchBlock + threadIdx.x;
  if (i < n) {
    const int e = a.idx[i];
    if (e >= 0 && e < a.E)
      atomicAdd(&cnt[e], 1);
    else
      atomicOr(a.status, kStatusBadIndex);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) a.blockhist[(size_t)blockIdx.x * a.E + e] = cnt[e];
}

// One block of 1024 threads: counts, offs, per-block bases (in place in blockhist), active list.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(RouteArgs a, int nblocks) {
  __shared__ int vals[kMaxE];
  __shared__ int scratch[40];
  const int E = a.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
    for (int b = 0; b < nblocks; ++b) s += a.blockhist[(size_t)b * E + e];
    a.counts[e] = s;
    vals[e] = s;
    if (a.usage && s) a.usage[e] += (unsigned long long)s;
  }
  __syncthreads();
  const int total = block_exclusive_scan(vals, E, scratch);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    a.offs[e] = vals[e];
    int run = vals[e];
    for (int b = 0; b < nblocks; ++b) {
      const int c = a.blockhist[(size_t)b * E + e];
      a.blockhist[(size_t)b * E + e] = run;
      run += c;
    }
  }
  if (threadIdx.x == 0) a.offs[E] = total;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) vals[e] = a.counts[e] > 0 ? 1 : 0;
  __syncthreads();
  const int nact = block_exclusive_scan(vals, E, scratch);
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (a.counts[e] > 0) {
      a.active[vals[e]] = e;
      a.slots[vals[e]] = make_int4(e, a.offs[e], a.counts[e], 0);
    }
  if (threadIdx.x == 0) {
    *a.n_active = nact;
    if (a.stat) *a.stat = nact;
  }
}

// Stable scatter: assignment i goes to base[b][e] + (rank among earlier same-expert ones in block b).
__global__ void __launch_bounds__(kDispatchBlock) dispatch_scatter_kernel(RouteArgs a) {
  __shared__ int32_t ids[kDispatchBlock];
  const int n = a.T * a.K;
  const int i0 = blockIdx.x * kDispatchBlock;
  const int i = i0 + threadIdx.x;
  ids[threadIdx.x] = (i < n) ? a.idx[i] : -1;
  __syncthreads();
  if (i >= n) return;
  const int e = ids[threadIdx.x];
  if (e < 0 || e >= a.E) return;
  int r = 0;
  for (int j = 0; j < (int)threadIdx.x; ++j) r += (ids[j] == e);
  a.perm[a.blockhist[(size_t)blockIdx.x * a.E + e] + r] = i;
}

// ------------------------------------------------------------------ host-side launchers
size_t route_small_smem(int T, int d, int E) { return (size_t)T * d * sizeof(float); }

cudaError_t launch_route(const RouteArgs& a, int nblocks_dispatch, cudaStream_t st) {
  if (a.T <= kSmallT && (size_t)a.T * a.d * 4 <= 160 * 1024) {
    const size_t sm = route_small_smem(a.T, a.d, a.E);
    const int grid = (a.E + kRouterExpertsPerBlock - 1) / kRouterExpertsPerBlock;
    route_small_kernel<<<grid, 256, sm, st>>>(a);
    return cudaGetLastError();
  }
  const void* xin = a.x;
  if (a.prenorm) {
    rmsnorm_kernel<<<(a.T + 7) / 8, 256, 0, st>>>(a.x, a.xnorm, a.act, a.T, a.d, a.eps);
    xin = a.xnorm;
  }
  if (a.act == kActBf16 && a.d % kRmBK == 0) {
    dim3 g((a.E + kRmBN - 1) / kRmBN, (a.T + kRmBM - 1) / kRmBM);
    router_logits_mma_kernel<<<g, 512, kRmSmem, st>>>(static_cast<const __nv_bfloat16*>(xin), a.Wr, a.bias,
                                                      a.logits, a.T, a.d, a.E, a.status);
  } else {
    dim3 g((a.E + kRlBN - 1) / kRlBN, (a.T + kRlBM - 1) / kRlBM);
    router_logits_kernel<<<g, 256, 0, st>>>(xin, a.act, a.Wr, a.bias, a.logits, a.T, a.d, a.E);
  }
  topk_kernel<<<(a.T + kRouterWarps - 1) / kRouterWarps, 256, (size_t)kRouterWarps * a.E * sizeof(float), st>>>(a);
  dispatch_hist_kernel<<<nblocks_dispatch, kDispatchBlock, 0, st>>>(a);
  dispatch_scan_kernel<<<1, 1024, 0, st>>>(a, nblocks_dispatch);
  dispatch_scatter_kernel<<<nblocks_dispatch, kDispatchBlock, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t route_kernels_init() {
  cudaError_t e = cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(router_logits_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRmSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
}

// ------------------------------------------------------------------ routing without allocation
// Scratch of moe_route_noalloc: one file-scope device array, shared by every call on a device.
// Layout (bytes): logits [16][1024] fp32 | idx [16*32] | w [16*32] | perm [16*32] | counts [1024] |
// offs [1025] | active [1024] | slots [1024] int4 | n_active | ticket | status.
namespace {
constexpr int kNaMaxT = kSmallT, kNaMaxE = kMaxE, kNaMaxK = kMaxK;
constexpr size_t kNaLogits = 0;
constexpr size_t kNaIdx = kNaLogits + (size_t)kNaMaxT * kNaMaxE * 4;
constexpr size_t kNaW = kNaIdx + (size_t)kNaMaxT * kNaMaxK * 4;
constexpr size_t kNaPerm = kNaW + (size_t)kNaMaxT * kNaMaxK * 4;
constexpr size_t kNaCounts = kNaPerm + (size_t)kNaMaxT * kNaMaxK * 4;
constexpr size_t kNaOffs = kNaCounts + (size_t)kNaMaxE * 4;
constexpr size_t kNaActive = kNaOffs + 256 * (((size_t)(kNaMaxE + 1) * 4 + 255) / 256);
constexpr size_t kNaSlots = kNaActive + (size_t)kNaMaxE * 4;
constexpr size_t kNaNActive = kNaSlots + (size_t)kNaMaxE * 16;
constexpr size_t kNaTicket = kNaNActive + 256;
constexpr size_t kNaStatus = kNaTicket + 256;
constexpr size_t kNaBytes = kNaStatus + 256;  // 121,600 bytes
}  // namespace

static __device__ __align__(256) unsigned char g_route_scratch[kNaBytes];

void set_last_cuda_error(cudaError_t e);

}  // namespace moe

extern "C" moe_status moe_route_noalloc(const float* router_w, const float* router_b, const void* x, int act, int T,
                                        int d, int E, int K, int32_t* topk_idx, float* topk_w, int32_t* expert_offs,
                                        int32_t* perm, void* stream) {
  using namespace moe;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!router_w || !x || !a16(router_w) || !a16(x) || (router_b && !a16(router_b))) return MOE_ERR_INVALID_ARG;
  if (act != MOE_ACT_BF16 && act != MOE_ACT_F32) return MOE_ERR_INVALID_ARG;
  if (T < 1 || d < 8 || d % 8 || E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
  // beyond the fixed scratch: at most 16 tokens, 1024 experts, top-32, and T*d*4 <= 160 KB
  if (T > kNaMaxT || E > kNaMaxE || K > kNaMaxK || (size_t)T * d * 4 > 160 * 1024) return MOE_ERR_UNSUPPORTED;

  // per-device set-up: the device address of the scratch array (and kernel attributes)
  static std::mutex mu;
  static void* base[64] = {};
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) {
    set_last_cuda_error(ce);
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  unsigned char* sc;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!base[dev]) {
      void* p = nullptr;
      ce = cudaGetSymbolAddress(&p, g_route_scratch);
      if (ce == cudaSuccess) ce = route_kernels_init();
      if (ce != cudaSuccess || !p) {
        set_last_cuda_error(ce);
        return MOE_ERR_CUDA;
      }
      base[dev] = p;
    }
    sc = static_cast<unsigned char*>(base[dev]);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RouteArgs a;
  a.x = x;
  a.act = act;
  a.T = T;
  a.d = d;
  a.E = E;
  a.K = K;
  a.Wr = router_w;
  a.bias = router_b;
  a.prenorm = 0;
  a.eps = 0.f;
  a.xnorm = nullptr;
  a.logits = reinterpret_cast<float*>(sc + kNaLogits);
  a.idx = topk_idx ? topk_idx : reinterpret_cast<int32_t*>(sc + kNaIdx);
  a.w = topk_w ? topk_w : reinterpret_cast<float*>(sc + kNaW);
  a.perm = perm ? perm : reinterpret_cast<int32_t*>(sc + kNaPerm);
  a.counts = reinterpret_cast<int32_t*>(sc + kNaCounts);
  a.offs = expert_offs ? expert_offs : reinterpret_cast<int32_t*>(sc + kNaOffs);
  a.active = reinterpret_cast<int32_t*>(sc + kNaActive);
  a.slots = reinterpret_cast<int4*>(sc + kNaSlots);
  a.n_active = reinterpret_cast<int32_t*>(sc + kNaNActive);
  a.stat = nullptr;
  a.blockhist = nullptr;
  a.ticket = reinterpret_cast<unsigned*>(sc + kNaTicket);
  a.status = reinterpret_cast<unsigned*>(sc + kNaStatus);
  a.usage = nullptr;
  // the last-block ticket must start at zero
  ce = cudaMemsetAsync(a.ticket, 0, sizeof(unsigned), st);
  if (ce == cudaSuccess) ce = launch_route(a, 1, st);
  if (ce != cudaSuccess) {
    set_last_cuda_error(ce);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
