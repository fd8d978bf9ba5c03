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

// The same for k = 1 or 2, k known at compile time: every thread first issues the loads of its K
// slots for U = 8 / K column chunks (eight 16-byte loads in flight), then sums them.  The kernel
// above is bound by load latency there (Mixtral-shaped layer: 35 us for 134 MB, 61% of the DRAM
// bandwidth; this one takes 31 us); with k = 8 it is the faster of the two (Hunyuan-shaped
// 0.180 against 0.192 ms), so larger k keep it.  The sum is taken in the same slot order with the
// same fmaf chain: the results are bit for bit those of the kernel above.
template <bool BF16, int K>
__global__ void __launch_bounds__(256) combine_vec_k_kernel(const float4* __restrict__ y_perm,
                                                            const int32_t* __restrict__ inv_pos,
                                                            const float* __restrict__ gate,
                                                            const float4* __restrict__ ys, int T, int d4,
                                                            long long rows_perm, void* __restrict__ y,
                                                            uint32_t* err) {
  static_assert(K == 1 || K == 2, "k = 1 or 2");
  constexpr int U = 8 / K;
  pdl_wait();
  pdl_trigger();
  __shared__ int s_pos[K];
  __shared__ float s_g[K];
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (threadIdx.x < K) {
      const int p = __ldg(inv_pos + (size_t)t * K + threadIdx.x);
      debug_bounds(p >= -1 && p < rows_perm, err);   // -1: a pair dropped at dispatch
      s_pos[threadIdx.x] = p;
      s_g[threadIdx.x] = __ldg(gate + (size_t)t * K + threadIdx.x);
    }
    __syncthreads();
    int pos[K];
    float g[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      pos[j] = s_pos[j];
      g[j] = s_g[j];
      if (pos[j] >= rows_perm) pos[j] = -1;   // a bad position (skipped)
    }
    for (int c0 = threadIdx.x; c0 < d4; c0 += blockDim.x * U) {
      float4 v[K][U];
#pragma unroll
      for (int j = 0; j < K; ++j) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + u * blockDim.x;
          v[j][u] = (pos[j] >= 0 && c < d4) ? __ldg(y_perm + (size_t)pos[j] * d4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * blockDim.x;
        if (c >= d4) continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < K; ++j) {
          if (pos[j] < 0) continue;
          acc.x = fmaf(g[j], v[j][u].x, acc.x);
          acc.y = fmaf(g[j], v[j][u].y, acc.y);
          acc.z = fmaf(g[j], v[j][u].z, acc.z);
          acc.w = fmaf(g[j], v[j][u].w, acc.w);
        }
        if (ys) {
          const float4 sv = __ldg(ys + (size_t)t * d4 + c);
          acc.x += sv.x; acc.y += sv.y; acc.z += sv.z; acc.w += sv.w;
        }
        if (BF16) {
          uint2 o = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
          reinterpret_cast<uint2*>(y)[(size_t)t * d4 + c] = o;
        } else {
          reinterpret_cast<float4*>(y)[(size_t)t * d4 + c] = acc;
        }
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
  if (vec && k <= 2) {
#define MOE_COMBINE_K(BF, KK)                                                                              \
  MOE_RETURN_ON_ERROR(launch_k(combine_vec_k_kernel<BF, KK>, blocks, 256, 0, st, (const float4*)y_perm, inv_pos, \
                               gate, (const float4*)ys, T, d / 4, rows_perm, y, err))
#define MOE_COMBINE_KS(BF)                    \
  if (k == 1) {                               \
    MOE_COMBINE_K(BF, 1);                     \
  } else {                                    \
    MOE_COMBINE_K(BF, 2);                     \
  }
    if (dtype == 1) {
      MOE_COMBINE_KS(true)
    } else {
      MOE_COMBINE_KS(false)
    }
#undef MOE_COMBINE_KS
#undef MOE_COMBINE_K
  } else if (vec) {
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
