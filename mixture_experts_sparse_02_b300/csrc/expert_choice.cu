// Expert-choice routing: every expert takes its m best tokens instead of every token taking
// its k best experts (page "Mixture-of-Experts Internals: A Systems Engineer's Field Manual",
// section 5.1: each expert chooses its top-m tokens from the batch, exactly m per expert; page
// "Mixture-of-Experts, from the router to the all-to-all", "Load balancing": load is balanced
// by construction).  The token-to-expert scores are the softmax over each token's router
// logits; expert e weights its output for token t by s[t][e]; a token may be taken by any
// number of experts, including none.
//
//   ec_scores   one warp per token: s[t][:] = softmax(logits[t][:] + bias), in place.
//   ec_select   one block per expert: the m-th largest s[:, e] by a 4-pass radix select on the
//               float bits (scores are >= 0, so their bits order like unsigned integers), then
//               the tokens above it plus the first equal ones in token order, compacted in
//               token order: perm_tok[e m + r], gate[e m + r], pos_of[t][e] (-1 if not taken).
//   ec_combine  one block per token: y[t] = sum over e of gate * y_perm[pos_of[t][e]] in
//               expert order (+ shared experts), one rounding.
// No order-dependent atomics: identical results from run to run.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

extern thread_local int g_launches;

namespace {

constexpr unsigned FULL = 0xffffffffu;

template <int EPL>
__global__ void __launch_bounds__(256) ec_scores_kernel(float* __restrict__ s, const float* __restrict__ lb, int T,
                                                        int E) {
  pdl_wait();
  pdl_trigger();
  const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float* row = s + (size_t)t * E;
  float l[EPL];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    l[i] = -INFINITY;
    if (e < E) {
      l[i] = row[e] + (lb ? __ldg(lb + e) : 0.f);
      m = fmaxf(m, l[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    l[i] = lane + 32 * i < E ? expf(l[i] - m) : 0.f;
    z += l[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(FULL, z, o);
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i < E) row[lane + 32 * i] = l[i] / z;
}

// Block-wide exclusive scan of one int per thread (1024 threads); returns the prefix and
// the block total in *total.  Uses `wsum` (32 ints of shared memory).
__device__ __forceinline__ int block_exclusive_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int x = wsum[lane];
    int xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(FULL, xi, o);
      if (lane >= o) xi += n;
    }
    wsum[lane] = xi - x;
    if (lane == 31) wsum[32] = xi;
  }
  __syncthreads();
  const int r = incl - v + wsum[w];
  *total = wsum[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) ec_select_kernel(const float* __restrict__ s, int T, int E, int m,
                                                         int32_t* __restrict__ offsets, int32_t* __restrict__ perm_tok,
                                                         float* __restrict__ gate, int32_t* __restrict__ pos_of) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t keys[];   // [T]
  __shared__ int hist[256];
  __shared__ int wsum[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  const int e = blockIdx.x;
  const int tid = threadIdx.x;
  for (int t = tid; t < T; t += 1024) keys[t] = __float_as_uint(s[(size_t)t * E + e]);
  if (tid == 0) {
    s_prefix = 0;
    s_need = m;   // how many of the keys that match the prefix are still to be taken
  }
  __syncthreads();
  // radix select of the m-th largest key, 8 bits at a time from the top
  uint32_t mask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += 1024) hist[b] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int t = tid; t < T; t += 1024) {
      const uint32_t k = keys[t];
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int need = s_need, cum = 0, b = 255;
      for (; b > 0; --b) {
        if (cum + hist[b] >= need) break;
        cum += hist[b];
      }
      s_need = need - cum;   // keys with this digit still to be taken
      s_prefix = prefix | ((uint32_t)b << shift);
    }
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t kth = s_prefix;   // the m-th largest key
  const int need_eq = s_need;      // keys equal to it to take, the first ones in token order
  // take keys above kth, and the first need_eq keys equal to it; compact in token order
  int carry_eq = 0, carry_out = 0;
  for (int base = 0; base < T; base += 1024) {
    const int t = base + tid;
    const uint32_t k = t < T ? keys[t] : 0u;
    const bool eq = t < T && k == kth;
    int tot_eq;
    const int eq_rank = block_exclusive_scan(eq ? 1 : 0, wsum, &tot_eq) + carry_eq;
    const bool take = t < T && (k > kth || (eq && eq_rank < need_eq));
    int tot_take;
    const int r = block_exclusive_scan(take ? 1 : 0, wsum, &tot_take) + carry_out;
    if (t < T) {
      if (take) {
        const int p = e * m + r;
        perm_tok[p] = t;
        gate[p] = __uint_as_float(k);
        pos_of[(size_t)t * E + e] = p;
      } else {
        pos_of[(size_t)t * E + e] = -1;
      }
    }
    carry_eq += tot_eq;
    carry_out += tot_take;
  }
  if (tid == 0) {
    offsets[e] = e * m;
    if (e == E - 1) offsets[E] = E * m;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(256) ec_combine_kernel(const float4* __restrict__ y_perm,
                                                         const int32_t* __restrict__ pos_of,
                                                         const float* __restrict__ gate, const float4* __restrict__ ys,
                                                         int T, int E, int d4, long long rows_perm, void* __restrict__ y,
                                                         uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int sh[];   // [E] positions, then [E] gates, of the experts that took t
  int* s_pos = sh;
  float* s_g = reinterpret_cast<float*>(sh + E);
  __shared__ int s_cnt[9];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    // compact the experts that took t, in expert order
    int cnt_before = 0;
    for (int base = 0; base < E; base += 256) {
      const int e = base + threadIdx.x;
      int p = e < E ? __ldg(pos_of + (size_t)t * E + e) : -1;
      debug_bounds(p >= -1 && p < rows_perm, err);   // -1: expert e did not take t
      if (p >= rows_perm) p = -1;                      // a bad position is skipped
      const unsigned bal = __ballot_sync(FULL, p >= 0);
      if (lane == 0) s_cnt[warp] = __popc(bal);
      __syncthreads();
      if (threadIdx.x == 0) {
        int run = 0;
        for (int w = 0; w < 8; ++w) {
          const int c = s_cnt[w];
          s_cnt[w] = run;
          run += c;
        }
        s_cnt[8] = run;
      }
      __syncthreads();
      if (p >= 0) {
        const int r = cnt_before + s_cnt[warp] + __popc(bal & ((1u << lane) - 1u));
        s_pos[r] = p;
        s_g[r] = __ldg(gate + p);
      }
      cnt_before += s_cnt[8];
      __syncthreads();
    }
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < cnt_before; ++j) {
        const float g = s_g[j];
        const float4 v = __ldg(y_perm + (size_t)s_pos[j] * d4 + c);
        acc.x = fmaf(g, v.x, acc.x);
        acc.y = fmaf(g, v.y, acc.y);
        acc.z = fmaf(g, v.z, acc.z);
        acc.w = fmaf(g, v.w, acc.w);
      }
      if (ys) {
        const float4 sv = __ldg(ys + (size_t)t * d4 + c);
        acc.x += sv.x; acc.y += sv.y; acc.z += sv.z; acc.w += sv.w;
      }
      if (BF16) {
        reinterpret_cast<uint2*>(y)[(size_t)t * d4 + c] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
      } else {
        reinterpret_cast<float4*>(y)[(size_t)t * d4 + c] = acc;
      }
    }
    __syncthreads();
  }
}

}  // namespace

size_t ec_select_smem(int T) { return (size_t)T * sizeof(uint32_t); }

cudaError_t ec_route(float* scores, const float* logit_bias, int T, int E, int m, int32_t* offsets,
                     int32_t* perm_tok, float* gate, int32_t* pos_of, cudaStream_t st) {
  const unsigned blocks = (unsigned)(((long long)T * 32 + 255) / 256);
#define MOE_EC_SCORES(EPL) MOE_RETURN_ON_ERROR(launch_k(ec_scores_kernel<EPL>, blocks, 256, 0, st, scores, logit_bias, T, E))
  if (E <= 32) MOE_EC_SCORES(1);
  else if (E <= 64) MOE_EC_SCORES(2);
  else if (E <= 128) MOE_EC_SCORES(4);
  else if (E <= 256) MOE_EC_SCORES(8);
  else if (E <= 512) MOE_EC_SCORES(16);
  else MOE_EC_SCORES(32);
#undef MOE_EC_SCORES
  ++g_launches;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = ec_select_smem(T);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  MOE_RETURN_ON_ERROR(launch_k(ec_select_kernel, E, 1024, smem, st, (const float*)scores, T, E, m, offsets, perm_tok,
                               gate, pos_of));
  ++g_launches;
  return cudaGetLastError();
}

cudaError_t ec_combine(int dtype, const float* y_perm, const int32_t* pos_of, const float* gate, const float* ys,
                       int T, int E, int d, long long rows_perm, void* y, uint32_t* err, cudaStream_t st) {
  const unsigned blocks = (unsigned)(T < 148 * 16 ? T : 148 * 16);
  const size_t smem = (size_t)E * 8;
  if (dtype == 1)
    MOE_RETURN_ON_ERROR(launch_k(ec_combine_kernel<true>, blocks, 256, smem, st, (const float4*)y_perm, pos_of, gate,
                                 (const float4*)ys, T, E, d / 4, rows_perm, y, err));
  else
    MOE_RETURN_ON_ERROR(launch_k(ec_combine_kernel<false>, blocks, 256, smem, st, (const float4*)y_perm, pos_of, gate,
                                 (const float4*)ys, T, E, d / 4, rows_perm, y, err));
  ++g_launches;
  return cudaGetLastError();
}

}  // namespace moe
