// Forward load statistics of one MoE batch, the quantities the pages say to watch and the
// Switch balancing loss built from them:
//   f_e   = c_e / T            fraction of tokens routed to expert e (c_e: its assignments)
//   P_e   = (1/T) sum_t s_e(x_t), the mean score of expert e (softmax over all E, or sigmoid)
//   L_aux = alpha E sum_e f_e P_e
//   max/mean load = max_e c_e / (T k / E)
// (page "8.6 - Mixture of Experts (MoE)", section 3.1; page "Mixture-of-Experts Internals: A
// Systems Engineer's Field Manual", section 3.2; page "T2.6 What MoE changes", "Routing creates
// an assignment problem").
//
// Scores are summed per block of tokens (one warp per token, fixed order), then over the
// blocks in block order: no atomics, identical results from run to run.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

extern thread_local int g_launches;

namespace {

constexpr unsigned FULL = 0xffffffffu;

template <int EPL>
__global__ void __launch_bounds__(256) score_partial_kernel(const float* __restrict__ logits,
                                                            const float* __restrict__ lb, int T, int E, int scoring,
                                                            int tokens_per_block, float* __restrict__ partial) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8][EPL * 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * tokens_per_block;
  const int t1 = min(T, t0 + tokens_per_block);
  float acc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
  for (int t = t0 + warp; t < t1; t += 8) {
    float l[EPL];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      l[i] = 0.f;
      if (e < E) {
        l[i] = __ldg(logits + (size_t)t * E + e) + (lb ? __ldg(lb + e) : 0.f);
        m = fmaxf(m, l[i]);
      }
    }
    if (scoring == 1) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i < E) acc[i] += 1.0f / (1.0f + expf(-l[i]));
    } else {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
      float ex[EPL];
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        ex[i] = lane + 32 * i < E ? expf(l[i] - m) : 0.f;
        z += ex[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(FULL, z, o);
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i < E) acc[i] += ex[i] / z;
    }
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) red[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += 256) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += red[w][e];
    partial[(size_t)blockIdx.x * E + e] = s;
  }
}

__global__ void __launch_bounds__(1024) stats_final_kernel(const float* __restrict__ partial, int nblk,
                                                           const int32_t* __restrict__ counts, int T, int k, int E,
                                                           float alpha, float* __restrict__ f, float* __restrict__ P,
                                                           float* __restrict__ summary) {
  pdl_wait();
  pdl_trigger();
  __shared__ float prod[1024];
  __shared__ int cmax[1024];
  const int e = threadIdx.x;
  float pr = 0.f;
  int c = 0;
  if (e < E) {
    float s = 0.f;
    for (int b = 0; b < nblk; ++b) s += partial[(size_t)b * E + e];
    const float pe = s / (float)T;
    c = __ldg(counts + e);
    const float fe = (float)c / (float)T;
    f[e] = fe;
    P[e] = pe;
    pr = fe * pe;
  }
  prod[e] = pr;
  cmax[e] = c;
  __syncthreads();
  for (int h = 512; h > 0; h >>= 1) {
    if (e < h) {
      prod[e] += prod[e + h];
      cmax[e] = max(cmax[e], cmax[e + h]);
    }
    __syncthreads();
  }
  if (e == 0) {
    summary[0] = alpha * (float)E * prod[0];
    summary[1] = (float)cmax[0] * (float)E / (float)((long long)T * k);
  }
}

}  // namespace

int stats_num_blocks(int T) {
  const int tpb = max(8, (T + 295) / 296);
  return (T + tpb - 1) / tpb;
}

cudaError_t load_stats(const float* logits, const float* logit_bias, const int32_t* counts, int T, int k, int E,
                       int scoring, float alpha, float* partial, float* f, float* P, float* summary,
                       cudaStream_t st) {
  const int tpb = max(8, (T + 295) / 296);
  const int nblk = (T + tpb - 1) / tpb;
#define MOE_SCORE_PARTIAL(EPL)                                                                          \
  MOE_RETURN_ON_ERROR(launch_k(score_partial_kernel<EPL>, nblk, 256, 0, st, logits, logit_bias, T, E, scoring, tpb, \
                               partial))
  if (E <= 32) MOE_SCORE_PARTIAL(1);
  else if (E <= 64) MOE_SCORE_PARTIAL(2);
  else if (E <= 128) MOE_SCORE_PARTIAL(4);
  else if (E <= 256) MOE_SCORE_PARTIAL(8);
  else if (E <= 512) MOE_SCORE_PARTIAL(16);
  else MOE_SCORE_PARTIAL(32);
#undef MOE_SCORE_PARTIAL
  ++g_launches;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  MOE_RETURN_ON_ERROR(launch_k(stats_final_kernel, 1, 1024, 0, st, (const float*)partial, nblk, counts, T, k, E, alpha,
                               f, P, summary));
  ++g_launches;
  return cudaGetLastError();
}

}  // namespace moe
