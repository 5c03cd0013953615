// Softmax + top-K selection of one token's router logits by one warp (sm_103a).
//
// The router keeps the K largest of the E logits ('Strata はなぜ少ない VRAM でも速いのか'
// (modeldock.net), section '問題：1,250 億パラメータと 12 GB'): ties go to the lower expert index,
// and the kept softmax probabilities are renormalised to sum to one.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace moe {

// Descending bitonic sort of the first N entries of kv (N a power of two), fully unrolled.
template <int N>
__device__ __forceinline__ void bitonic_desc(uint64_t (&kv)[32]) {
#pragma unroll
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t x0 = kv[i], x1 = kv[ixj];
          const bool sw = ((i & k) == 0) ? (x0 < x1) : (x0 > x1);
          kv[i] = sw ? x1 : x0;
          kv[ixj] = sw ? x0 : x1;
        }
      }
    }
  }
}

// One warp, one token, E <= 1024 logits at lg (global memory, read through L2).  Each lane holds
// the keys of its experts lane, lane+32, ... sorted once (order-preserving key of the logit in
// the high word, 31 - j in the low word so equal logits keep the lower expert first); each of the
// K rounds takes the warp maximum of the lanes' heads with two redux reductions (largest key, then
// lowest expert index among equal keys).  Lane k < K returns the k-th expert and its weight
// exp(l - max) / Z renormalised over the K kept (summed in ascending k).
__device__ __forceinline__ void topk_token(const float* lg, int E, int K, int& my_i, float& my_w) {
  const int lane = threadIdx.x & 31;
  uint64_t kv[32];
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int ej = lane + 32 * j;
    const float v = ej < E ? __ldcg(lg + ej) : -INFINITY;
    m = fmaxf(m, v);
    const uint32_t u = __float_as_uint(v);
    const uint32_t key = ej < E ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
    kv[j] = ((uint64_t)key << 32) | (uint32_t)(31 - j);
  }
  m = warp_max(m);
  float z = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int ej = lane + 32 * j;
    if (ej < E) z += expf(__ldcg(lg + ej) - m);
  }
  z = warp_sum(z);
  if (E <= 512)
    bitonic_desc<16>(kv);
  else
    bitonic_desc<32>(kv);
  int head = 0;
  my_i = 0;
  for (int k = 0; k < K; ++k) {
    uint64_t hk = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j == head) hk = kv[j];
    const uint32_t key = (uint32_t)(hk >> 32);
    const uint32_t best = __reduce_max_sync(0xffffffffu, key);
    const int e_mine = lane + 32 * (31 - (int)(hk & 31u));
    const uint32_t cand = (key == best && key != 0u) ? (uint32_t)e_mine : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    if (lane == (int)(win & 31u)) ++head;
    if (lane == k) my_i = (int)win;
  }
  float my_p = 0.f;
  if (lane < K) my_p = expf(__ldcg(lg + my_i) - m) / z;
  float psum = 0.f;
  for (int k = 0; k < K; ++k) psum += __shfl_sync(0xffffffffu, my_p, k);
  my_w = lane < K ? my_p / psum : 0.f;
}

// Order-preserving u32 key of a logit (larger logit, larger key; never 0) and its inverse.
__device__ __forceinline__ uint32_t topk_order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float topk_key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// The same selection and weights as topk_token, in compact code for kernels where it runs once per
// launch, from keys already in shared memory: s_key[32 j + lane] = topk_order_key(logit of expert
// lane + 32 j), 0 past E (E <= 1024); taken keys are overwritten.  Each lane keeps its best and
// second-best untaken key (order: larger key, then lower expert); a round takes the warp's best
// with two redux reductions, and only a lane that wins a second time rescans its experts.
__device__ __forceinline__ void topk_warp(uint32_t* s_key, int E, int K, int& my_i, float& my_w) {
  const int lane = threadIdx.x & 31;
  const int nj = (E + 31) >> 5;
  uint32_t b1 = 0u, b2 = 0u;
  int j1 = 0, j2 = 0;
#pragma unroll 4
  for (int j = 0; j < nj; ++j) {
    const uint32_t key = s_key[j * 32 + lane];
    if (key > b1) {
      b2 = b1;
      j2 = j1;
      b1 = key;
      j1 = j;
    } else if (key > b2) {
      b2 = key;
      j2 = j;
    }
  }
  const float m = topk_key_value(__reduce_max_sync(0xffffffffu, b1));
  float z = 0.f;
#pragma unroll 4
  for (int j = 0; j < nj; ++j) {
    const uint32_t key = s_key[j * 32 + lane];
    if (key != 0u) z += expf(topk_key_value(key) - m);
  }
  z = warp_sum(z);
  bool have2 = true;
  uint32_t my_key = 0u;
  my_i = 0;
#pragma unroll 1
  for (int k = 0; k < K; ++k) {
    const uint32_t best = __reduce_max_sync(0xffffffffu, b1);
    const uint32_t cand = (b1 == best && b1 != 0u) ? (uint32_t)(lane + 32 * j1) : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    if (lane == k) {
      my_i = (int)win;
      my_key = best;
    }
    if (lane == (int)(win & 31u)) {
      s_key[j1 * 32 + lane] = 0u;  // taken
      if (have2) {
        b1 = b2;
        j1 = j2;
        have2 = false;
      } else {
        b1 = 0u;
        j1 = 0;
#pragma unroll 4
        for (int j = 0; j < nj; ++j) {
          const uint32_t key = s_key[j * 32 + lane];
          if (key > b1) {
            b1 = key;
            j1 = j;
          }
        }
      }
    }
    __syncwarp();
  }
  const float my_p = lane < K ? expf(topk_key_value(my_key) - m) / z : 0.f;
  float psum = 0.f;
#pragma unroll 1
  for (int k = 0; k < K; ++k) psum += __shfl_sync(0xffffffffu, my_p, k);
  my_w = lane < K ? my_p / psum : 0.f;
}

// The same selection and weights in fewer dependent steps.  The K-th largest of the 32 lane maxima
// is a lower bound of the K-th largest key (the K largest lane maxima are K distinct keys), so the
// keys at or above it hold the selection; when there are at most 32 of them each lane ranks one
// candidate against the others (larger key, then lower expert) and rank k < K is the k-th choice.
// Otherwise (many equal or clustered logits) it falls back to the rounds of topk_warp.
// s_cand: 64 uint2 of shared-memory scratch for this warp.
__device__ __forceinline__ void topk_warp_fast(uint32_t* s_key, int E, int K, uint2* s_cand, int& my_i, float& my_w) {
  const int lane = threadIdx.x & 31;
  const int nj = (E + 31) >> 5;
  uint32_t lm = 0u;
#pragma unroll 4
  for (int j = 0; j < nj; ++j) lm = max(lm, s_key[j * 32 + lane]);
  int rk = 0;  // rank of this lane's maximum among the lane maxima, ties to the lower lane
#pragma unroll
  for (int l = 0; l < 32; ++l) {
    const uint32_t o = __shfl_sync(0xffffffffu, lm, l);
    rk += (o > lm) || (o == lm && l < lane);
  }
  const uint32_t tau = __reduce_max_sync(0xffffffffu, rk == K - 1 ? lm : 0u);
  int cnt = 0;
#pragma unroll 4
  for (int j = 0; j < nj; ++j) {
    const uint32_t key = s_key[j * 32 + lane];
    cnt += key != 0u && key >= tau;
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (total > 32) {
    topk_warp(s_key, E, K, my_i, my_w);
    return;
  }
  const float m = topk_key_value(__reduce_max_sync(0xffffffffu, lm));
  float z = 0.f;
  int pos = incl - cnt;
#pragma unroll 4
  for (int j = 0; j < nj; ++j) {
    const uint32_t key = s_key[j * 32 + lane];
    if (key != 0u) z += expf(topk_key_value(key) - m);
    if (key != 0u && key >= tau) s_cand[pos++] = make_uint2(key, (uint32_t)(lane + 32 * j));
  }
  z = warp_sum(z);
  __syncwarp();
  const uint2 cd = lane < total ? s_cand[lane] : make_uint2(0u, 0xffffffffu);
  int rank = 0;
#pragma unroll
  for (int l = 0; l < 32; ++l) {
    const uint32_t ok = __shfl_sync(0xffffffffu, cd.x, l), oi = __shfl_sync(0xffffffffu, cd.y, l);
    rank += l < total && (ok > cd.x || (ok == cd.x && oi < cd.y));
  }
  if (lane < total && rank < K) s_cand[32 + rank] = cd;
  __syncwarp();
  uint32_t my_key = 0u;
  my_i = 0;
  if (lane < K) {
    const uint2 sel = s_cand[32 + lane];
    my_i = (int)sel.y;
    my_key = sel.x;
  }
  const float my_p = lane < K ? expf(topk_key_value(my_key) - m) / z : 0.f;
  float psum = 0.f;
#pragma unroll 1
  for (int k = 0; k < K; ++k) psum += __shfl_sync(0xffffffffu, my_p, k);
  my_w = lane < K ? my_p / psum : 0.f;
}

}  // namespace moe
