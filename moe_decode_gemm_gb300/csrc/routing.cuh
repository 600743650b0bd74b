// routing.cuh -- top-k expert selection with renormalised softmax gates, one
// warp per token. "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §3
// "改进 MoE 调度与重叠" (router scores select the experts).
#pragma once

#include "dg_common.cuh"

namespace dg {

// Order-preserving map of a float to uint32 (larger float, larger key). Keys
// start at 1: 0 marks an entry already taken (or past E), so every selected
// index is a real expert whatever the scores hold.
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f);
  const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return k > 1u ? k : 1u;
}

__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// The K largest of row[0..E) (E <= 1024, K <= 32, K <= E), ordered by (value
// desc, index asc), and gates g_j = exp(l_j - l_max) / sum_j' exp(l_j' - l_max)
// summed j' = 0..K-1, written to idx/gate[0..K) (and to the optional user
// copies). Called by all 32 lanes of a warp. A lane holds the scores
// e = lane + 32 j as keys in registers; each round takes every lane's best
// (its smallest index on ties), the warp's largest key and, among the lanes
// holding it, the smallest index. The scores are read from L2 (they were
// written by other SMs).
__device__ __forceinline__ void warp_topk_gates(const float* row, int E, int K, int lane, int* idx,
                                                float* gate, int32_t* idx_user, float* w_user) {
  const int per = (E + 31) >> 5;
  uint32_t kv[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int e = lane + 32 * j;
    kv[j] = (j < per && e < E) ? float_key(__ldcg(row + e)) : 0u;
  }
  float selv0 = 0.f, myv = 0.f;
  int mye = 0;
  for (int j = 0; j < K; ++j) {
    uint32_t bk = kv[0];
    int bj = 0;
#pragma unroll
    for (int jj = 1; jj < 32; ++jj)
      if (jj < per && kv[jj] > bk) {  // strict: the smallest jj (smallest index) on ties
        bk = kv[jj];
        bj = jj;
      }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t cand = (bk == kmax && kmax != 0u) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu;
    const uint32_t emin = __reduce_min_sync(0xffffffffu, cand);
    if ((int)(emin & 31) == lane) {
#pragma unroll
      for (int jj = 0; jj < 32; ++jj)
        if (jj == bj) kv[jj] = 0u;
    }
    const float wv = key_float(kmax);
    if (j == 0) selv0 = wv;
    if (lane == j) {
      myv = wv;
      mye = (int)emin;
    }
  }
  const float w = (lane < K) ? expf(myv - selv0) : 0.f;
  float denom = 0.f;
  for (int j = 0; j < K; ++j) denom += __shfl_sync(0xffffffffu, w, j);
  if (lane < K) {
    const float g = w / denom;
    idx[lane] = mye;
    gate[lane] = g;
    if (idx_user) idx_user[lane] = mye;
    if (w_user) w_user[lane] = g;
  }
}

}  // namespace dg
