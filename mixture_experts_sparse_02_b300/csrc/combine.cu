// Combine of the MoE layer: y[t] = sum_j g[t][j] * y_perm[inv_pos[t][j]] (+ shared[t]),
// summed in float32 in slot order j = 0..k-1 and rounded once to the output dtype
// (page "8.6 - Mixture of Experts (MoE)", sections 2 and 4.1; page "Mixture of Experts: What
// Actually Happens When a Token Hits the Router", Step 3: scatter results back).
// Each output element has exactly one writer: no atomics, run-to-run identical.
// HBM-bound: reads k float32 rows per token and writes one row.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

template <bool BF16>
__global__ void __launch_bounds__(256) combine_vec_kernel(const float4* __restrict__ y_perm,
                                                          const int32_t* __restrict__ inv_pos,
                                                          const float* __restrict__ gate,
                                                          const float4* __restrict__ ys, int T, int d4, int k,
                                                          long long rows_perm, void* __restrict__ y, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_pos[32];
  __shared__ float s_g[32];
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (threadIdx.x < k) {
      const int p = __ldg(inv_pos + (size_t)t * k + threadIdx.x);
      debug_bounds(p >= -1 && p < rows_perm, err);   // -1: a pair dropped at dispatch
      s_pos[threadIdx.x] = p;
      s_g[threadIdx.x] = __ldg(gate + (size_t)t * k + threadIdx.x);
    }
    __syncthreads();
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < k; ++j) {
        const int p = s_pos[j];
        if (p < 0 || p >= rows_perm) continue;   // a dropped pair, or a bad position (skipped)
        const float g = s_g[j];
        const float4 v = __ldg(y_perm + (size_t)p * d4 + c);
        acc.x = fmaf(g, v.x, acc.x);
        acc.y = fmaf(g, v.y, acc.y);
        acc.z = fmaf(g, v.z, acc.z);
        acc.w = fmaf(g, v.w, acc.w);
      }
      if (ys) {
        const float4 s = __ldg(ys + (size_t)t * d4 + c);
        acc.x += s.x; acc.y += s.y; acc.z += s.z; acc.w += s.w;
      }
      if (BF16) {
        uint2 o = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
        reinterpret_cast<uint2*>(y)[(size_t)t * d4 + c] = o;
      } else {
        reinterpret_cast<float4*>(y)[(size_t)t * d4 + c] = acc;
      }
    }
    __syncthreads();
  }
}

template <bool BF16>
__global__ void __launch_bounds__(256) combine_scalar_kernel(const float* __restrict__ y_perm,
                                                             const int32_t* __restrict__ inv_pos,
                                                             const float* __restrict__ gate,
                                                             const float* __restrict__ ys, int T, int d, int k,
                                                             long long rows_perm, void* __restrict__ y,
                                                             uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int p = __ldg(inv_pos + (size_t)t * k + j);
        if (c == threadIdx.x) debug_bounds(p >= -1 && p < rows_perm, err);
        if (p < 0 || p >= rows_perm) continue;
        acc = fmaf(__ldg(gate + (size_t)t * k + j), __ldg(y_perm + (size_t)p * d + c), acc);
      }
      if (ys) acc += __ldg(ys + (size_t)t * d + c);
      if (BF16)
        reinterpret_cast<__nv_bfloat16*>(y)[(size_t)t * d + c] = __float2bfloat16_rn(acc);
      else
        reinterpret_cast<float*>(y)[(size_t)t * d + c] = acc;
    }
  }
}

}  // namespace

cudaError_t combine(int dtype, const float* y_perm, const int32_t* inv_pos, const float* gate, const float* ys, int T,
                    int d, int k, void* y, uint32_t* err, cudaStream_t st) {
  const long long rows_perm = (long long)T * k;
  const unsigned blocks = (unsigned)(T < 148 * 32 ? T : 148 * 32);
  const bool vec = (d % 4 == 0) && ((uintptr_t)y_perm % 16 == 0) && (!ys || (uintptr_t)ys % 16 == 0) &&
                   ((uintptr_t)y % (dtype == 1 ? 8 : 16) == 0);
  if (vec) {
    if (dtype == 1)
      MOE_RETURN_ON_ERROR(launch_k(combine_vec_kernel<true>, blocks, 256, 0, st, (const float4*)y_perm, inv_pos, gate,
                         (const float4*)ys, T, d / 4, k, rows_perm, y, err));
    else
      MOE_RETURN_ON_ERROR(launch_k(combine_vec_kernel<false>, blocks, 256, 0, st, (const float4*)y_perm, inv_pos, gate,
                         (const float4*)ys, T, d / 4, k, rows_perm, y, err));
  } else {
    if (dtype == 1)
      MOE_RETURN_ON_ERROR(launch_k(combine_scalar_kernel<true>, blocks, 256, 0, st, y_perm, inv_pos, gate, ys, T, d, k, rows_perm, y, err));
    else
      MOE_RETURN_ON_ERROR(launch_k(combine_scalar_kernel<false>, blocks, 256, 0, st, y_perm, inv_pos, gate, ys, T, d, k, rows_perm,
                         y, err));
  }
  ++g_launches;
  return cudaGetLastError();
}

}  // namespace moe
