// Per-token noaux_tc selection as a warp-level device function, shared by the stand-alone
// selection kernel and the fused decode kernel so both decide identically.
//   s = sigmoid(logit); b = s + bias (selection only)
//   group score = sum of the two largest b of each contiguous group of E/n_group experts
//   keep the topk_group best groups (ties -> lower group index)
//   top_k largest b among kept experts (ties -> lower expert index), slot order descending
//   w[j] = s[id_j] / sum_j s[id_j] * rsf
//   adaptive top-p (0 < top_p < 1): order the top_k by s (larger first, lower id on ties);
//   a slot stays while the s ranked before it sums below top_p * sum s (the first always);
//   dropped slots get id -1, weight 0, and the kept weights are renormalised to rsf
// (DeepSeek-V3-style sigmoid router with noaux_tc and routed_scaling_factor, "Show HN:
// Menjalankan GLM 5.2 di komputer lambat", section "Fitur utama yang diimplementasikan".)
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

// Warp-wide argmax of (value, index): larger value wins, equal values go to the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
    }
  }
}

// Whole warp calls. `b`, `s` are warp-private shared arrays of E floats. Writes ids[0..k)
// and weights[0..k) (lanes 0..k-1) and returns, on lane j < k, the id of slot j.
// Logits are read through L2 (they may have been written by other CTAs of this grid).
__device__ __forceinline__ int select_token(const float* logits_row, const float* bias, int E,
                                            int n_group, int topk_group, int top_k, float rsf,
                                            float top_p, float* b, float* s, int32_t* ids,
                                            float* weights, int* status) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < E; e += 32) {
    const float sc = sigmoidf_acc(__ldcg(logits_row + e));
    s[e] = sc;
    b[e] = sc + __ldg(bias + e);
  }
  __syncwarp();
  const int G = E / n_group;
  float gscore = -INFINITY;
  if (lane < n_group) {
    float m1 = -INFINITY, m2 = -INFINITY;
    for (int i = 0; i < G; ++i) {
      const float v = b[lane * G + i];
      if (v > m1) {
        m2 = m1;
        m1 = v;
      } else if (v > m2) {
        m2 = v;
      }
    }
    gscore = m1 + m2;
  }
  unsigned kept = 0;
  for (int r = 0; r < topk_group; ++r) {
    float v = gscore;
    int gi = lane < n_group ? lane : 0x7fffffff;
    warp_argmax(v, gi);
    kept |= 1u << gi;
    if (lane == gi) gscore = -INFINITY;
  }
  float wsum = 0.f;
  int my_id = -1;
  float my_s = 0.f;
  for (int j = 0; j < top_k; ++j) {
    float v = -INFINITY;
    int vi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float be = ((kept >> (e / G)) & 1u) ? b[e] : -INFINITY;
      if (be > v) {
        v = be;
        vi = e;
      }
    }
    warp_argmax(v, vi);
    if (vi < 0 || vi >= E) {   // fewer candidates than top_k: host validation forbids it
      raise_status(status, MOE_ERR_DEVICE_CHECK);
      vi = 0;
    }
    const float sv = s[vi];
    wsum += sv;
    if (lane == j) {
      my_id = vi;
      my_s = sv;
    }
    __syncwarp();
    if (lane == 0) b[vi] = -INFINITY;
    __syncwarp();
  }
  float norm = wsum;
  if (top_p > 0.f && top_p < 1.f) {
    // rank by s and the mass ranked before this slot, both added in slot order
    int rank = 0;
    float before = 0.f;
    for (int i = 0; i < top_k; ++i) {
      const float si = __shfl_sync(0xffffffffu, my_s, i);
      const int ii = __shfl_sync(0xffffffffu, my_id, i);
      const bool above = si > my_s || (si == my_s && ii < my_id);
      rank += above;
      if (above) before += si;
    }
    const bool keep = rank == 0 || before < top_p * wsum;
    norm = 0.f;
    for (int i = 0; i < top_k; ++i) {
      const int ki = __shfl_sync(0xffffffffu, (int)keep, i);
      const float si = __shfl_sync(0xffffffffu, my_s, i);
      if (ki) norm += si;
    }
    if (lane < top_k && !keep) {
      my_id = -1;
      my_s = 0.f;
    }
  }
  if (lane < top_k) {
    ids[lane] = my_id;
    weights[lane] = my_s / norm * rsf;
  }
  return my_id;
}

}  // namespace moe
