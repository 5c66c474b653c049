// Router of the routed experts (sm_103a).
//
// For each token [KTransformers page, «规则二»: the gate yields the top-k
// expert indices and weights]: the k largest of the E logits in descending
// order, equal logits taken lower index first, and weights renormalised over
// the chosen k: w_i = exp(l_i - l_max) / sum_j exp(l_j - l_max).  That is the
// softmax over all E logits (max subtracted, engine page §5.1) restricted to
// the k chosen and renormalised: the common factor cancels.  The choice is
// made on the fp32 logits themselves (exact comparisons); the softmax is
// monotonic, so it chooses the same experts as a comparison of probabilities.
//
// One warp per token; lane j holds logits j, j + 32, ... in registers.
#include <cstdint>
#include <cuda_runtime.h>

#include "q4_device.cuh"
#include "q4_kernels.h"

namespace q4 {

constexpr int kGateMaxPerLane = kGateMaxExperts / 32;

// (v, e) comes before (v2, e2): larger logit, or equal logit and lower index.
__device__ __forceinline__ bool gate_before(float v, int e, float v2, int e2) {
  return v > v2 || (v == v2 && e < e2);
}

__global__ void __launch_bounds__(128) q4_moe_gate_kernel(int32_t* topk_idx, float* topk_w,
                                                          const float* logits, int T, int E,
                                                          int topk, int32_t* shared_idx,
                                                          float* shared_w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* l = logits + static_cast<size_t>(t) * E;
  float v[kGateMaxPerLane];
#pragma unroll
  for (int j = 0; j < kGateMaxPerLane; ++j) {
    const int e = lane + 32 * j;
    v[j] = (e < E) ? l[e] : 0.f;
  }
  unsigned taken = 0u;   // bit j: logit lane + 32j already chosen
  float mine_v = 0.f;    // lane i (< topk) keeps the i-th choice
  int mine_e = 0;
  for (int k = 0; k < topk; ++k) {
    // this lane's best remaining logit
    float bv = 0.f;
    int be = -1;
#pragma unroll
    for (int j = 0; j < kGateMaxPerLane; ++j) {
      const int e = lane + 32 * j;
      if (e < E && !((taken >> j) & 1u) && (be < 0 || gate_before(v[j], e, bv, be))) {
        bv = v[j];
        be = e;
      }
    }
    // the warp's best: a fixed butterfly of comparisons
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (oe >= 0 && (be < 0 || gate_before(ov, oe, bv, be))) {
        bv = ov;
        be = oe;
      }
    }
    // every lane now holds the winner (E >= topk, so be >= 0)
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == k) {
      mine_v = bv;
      mine_e = be;
    }
  }
  // weights: exp relative to the largest chosen logit (lane 0's); every lane
  // sums the k values in choice order
  const float vmax = __shfl_sync(0xffffffffu, mine_v, 0);
  const float ex = (lane < topk) ? expf(mine_v - vmax) : 0.f;
  float sum = 0.f;
  for (int k = 0; k < topk; ++k) sum += __shfl_sync(0xffffffffu, ex, k);
  if (lane < topk) {
    topk_idx[static_cast<size_t>(t) * topk + lane] = mine_e;
    topk_w[static_cast<size_t>(t) * topk + lane] = ex / sum;
  }
  if (shared_idx && lane == 0) {
    shared_idx[t] = 0;
    shared_w[t] = 1.0f;
  }
}

cudaError_t launch_moe_gate(int32_t* topk_idx, float* topk_w, const float* logits, int T, int E,
                            int topk, int32_t* shared_idx, float* shared_w, cudaStream_t st) {
  const int warps = 4;
  const int grid = (T + warps - 1) / warps;
  (void)cudaGetLastError();   // report this launch's error, not an earlier one's
  q4_moe_gate_kernel<<<grid, warps * 32, 0, st>>>(topk_idx, topk_w, logits, T, E, topk,
                                                  shared_idx, shared_w);
  return cudaGetLastError();
}

}  // namespace q4
