// Router of the MoE layer: logits l = x W_g (+ logit_bias), top-k on l (+ sel_bias), gates.
//
// Page "8.6 - Mixture of Experts (MoE)", section 2: router(x) = x W_g, the k experts with the
// largest logits, gates normalised over the chosen k.  Page "Mixture-of-Experts Internals: A
// Systems Engineer's Field Manual", section 2.1 (softmax, top-k, renormalise) and 3.3 (bias
// for the choice only).  Page "Mixture-of-Experts, from the router to the all-to-all", "The
// router" (sigmoid scores normalised among the selected).
//
// Switch-style gates (softmax without renormalisation) need the full softmax denominator.
// Softmax gates renormalised over the chosen set only need the chosen logits:
// s_i / sum_{I} s_j = exp(l_i - m) / sum_{I} exp(l_j - m) for any m (the full-softmax
// denominator cancels), so the kernels take m = the largest chosen logit.
//
// Selection is a warp-wide argmax repeated k times, ties going to the lower expert id.
// Logits are float32, summed in a fixed order, so the result is run-to-run identical.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

extern thread_local int g_launches;

namespace {

constexpr unsigned FULL = 0xffffffffu;

// Warp argmax of (value, index): larger value wins, equal values go to the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(FULL, v, o);
    const int oi = __shfl_xor_sync(FULL, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

// The value the top-k is taken over.  Without a selection bias: the logit (softmax and
// sigmoid are monotone).  With a bias b used for choosing only: logit + b for softmax routing
// (page "Mixture-of-Experts Internals: A Systems Engineer's Field Manual", section 3.3) and
// sigmoid(logit) + b for sigmoid routing (page "Mixture-of-Experts, from the router to the
// all-to-all", "Load balancing"), in float32.
__device__ __forceinline__ float selection_key(float l, const float* __restrict__ sb, int e, int scoring) {
  if (!sb) return l;
  const float b = __ldg(sb + e);
  return scoring == 1 ? 1.0f / (1.0f + expf(-l)) + b : l + b;
}

// Lane L holds logits of experts L, L+32, ..., in l[EPL] (unbiased) and key[EPL] (selection
// keys).  Chooses k experts and writes idx/gate for token t.  Padding slots must carry
// key = -inf and an index >= E (excluded through `valid`).
template <int EPL>
__device__ __forceinline__ void select_and_gate(const float (&l)[EPL], float (&key)[EPL], int E, int k, int scoring,
                                                int t, int32_t* idx, float* gate) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i >= E) taken |= 1u << i;
  int my_idx = 0;
  float my_l = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (!(taken & (1u << i))) {
        const int e = lane + 32 * i;
        if (key[i] > bv || (key[i] == bv && e < bi)) { bv = key[i]; bi = e; }
      }
    }
    warp_argmax(bv, bi);
    const int owner = bi & 31, slot = bi >> 5;
    float wl = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (i == slot) wl = l[i];
    wl = __shfl_sync(FULL, wl, owner);
    if (lane == owner) taken |= 1u << slot;
    if (lane == j) { my_idx = bi; my_l = wl; }
  }
  float g;
  if (scoring == 0) {
    const float m = warp_max(lane < k ? my_l : -INFINITY);
    const float ex = lane < k ? expf(my_l - m) : 0.f;
    g = ex / warp_sum(ex);
  } else if (scoring == 2) {
    // Switch-style: the softmax probability over all E itself, not renormalised (page
    // "Mixture-of-Experts, from the router to the all-to-all", "The router": y = p_i(x) E_i(x))
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < E) m = fmaxf(m, l[i]);
    m = warp_max(m);
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < E) z += expf(l[i] - m);
    z = warp_sum(z);
    g = lane < k ? expf(my_l - m) / z : 0.f;
  } else {
    const float s = lane < k ? 1.0f / (1.0f + expf(-my_l)) : 0.f;
    g = s / warp_sum(s);
  }
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_idx;
    gate[(size_t)t * k + lane] = g;
  }
}

// One warp per token: logits on CUDA cores (lane-strided over d, then a butterfly sum), then
// top-k and gates.  E <= EM <= 32.
template <typename T, int EM>
__global__ void __launch_bounds__(256) route_fused_kernel(const T* __restrict__ x, const T* __restrict__ Wg,
                                                          const float* __restrict__ lb, const float* __restrict__ sb,
                                                          int Tn, int d, int E, int k, int scoring, int32_t* idx,
                                                          float* gate, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= Tn) return;
  const T* xr = x + (size_t)t * d;
  float acc[EM];
#pragma unroll
  for (int e = 0; e < EM; ++e) acc[e] = 0.f;
  for (int i = lane; i < d; i += 32) {
    const float xv = load_as_float(xr + i);
    const T* w = Wg + (size_t)i * E;
#pragma unroll
    for (int e = 0; e < EM; ++e)
      if (e < E) acc[e] = fmaf(xv, load_as_float(w + e), acc[e]);
  }
#pragma unroll
  for (int e = 0; e < EM; ++e) acc[e] = warp_sum(acc[e]);
  float l[1], key[1];
  l[0] = 0.f;
#pragma unroll
  for (int e = 0; e < EM; ++e)
    if (e == lane) l[0] = acc[e];
  key[0] = -INFINITY;
  if (lane < E) {
    if (lb) l[0] += __ldg(lb + lane);
    key[0] = selection_key(l[0], sb, lane, scoring);
    if (!isfinite(l[0]) || isnan(key[0])) {
      flag_error(err, ERR_ROUTE);
      if (isnan(key[0])) key[0] = -INFINITY;
    }
  }
  select_and_gate<1>(l, key, E, k, scoring, t, idx, gate);
}

// Sum NV per-lane partials over the 32 lanes of a warp by recursive halving: at each step a
// lane keeps one half of its values, adds the peer's copy of that half and sends the other
// half.  After min(5, log2 NV) steps lane L holds the complete sums of indices
// base(L) .. base(L) + NV/2^steps - 1; if NV < 32 the remaining steps are plain butterflies, so
// lanes that differ only in those low bits hold the same sums.  The order of additions is
// fixed, so the result is run-to-run identical.
template <int NV, int O>
__device__ __forceinline__ void halve_sum(float* v, int lane) {
  if constexpr (O >= 1) {
    if constexpr (NV >= 2) {
      constexpr int H = NV / 2;
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = up ? v[i] : v[i + H];
        const float keep = up ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(FULL, send, O);
      }
      halve_sum<H, O / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(FULL, v[0], O);
      halve_sum<1, O / 2>(v, lane);
    }
  }
}

// After halve_sum<NV, 16>: the first index a lane holds, and whether it is the lane that owns
// those sums (its low bits, over which only plain butterflies ran, are zero).  NV is a power of 2.
template <int NV>
__device__ __forceinline__ int halve_base(int lane, bool& owner) {
  constexpr int H = NV >= 32 ? 5 : NV >= 16 ? 4 : NV >= 8 ? 3 : NV >= 4 ? 2 : NV >= 2 ? 1 : 0;
  int base = 0;
#pragma unroll
  for (int s = 0; s < H; ++s)
    if (lane & (16 >> s)) base += NV >> (s + 1);
  owner = (lane & ((1 << (5 - H)) - 1)) == 0;
  return base;
}

__device__ __forceinline__ uint32_t u4_word(const uint4& v, int w) {
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// Element j of an array of 16-byte vectors holding bf16 (uint16_t) or float values.
template <typename T> __device__ __forceinline__ float vec_elem(const uint4* a, int j);
template <> __device__ __forceinline__ float vec_elem<uint16_t>(const uint4* a, int j) {
  const uint32_t w = u4_word(a[j >> 3], (j >> 1) & 3);
  return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
}
template <> __device__ __forceinline__ float vec_elem<float>(const uint4* a, int j) {
  return __uint_as_float(u4_word(a[j >> 2], j & 3));
}

// Fused router for E in {1, 2, 4, 8, 16, 32}: a block of 8 warps takes TW tokens.  Every lane
// reads 16-byte vectors of the TW token rows (VE elements of d each) and the VE matching rows
// of W_g, strided over the block, so many loads are in flight and W_g is read once per TW
// tokens.  The per-lane partial logits are summed over the warp (halve_sum) and then over the
// 8 warps in warp order through shared memory.  Warp t then selects and gates token t.
template <typename T, int E, int TW>
__global__ void __launch_bounds__(256) route_vec_kernel(const T* __restrict__ x, const T* __restrict__ Wg,
                                                        const float* __restrict__ lb, const float* __restrict__ sb,
                                                        int Tn, int d, int k, int scoring, int32_t* idx, float* gate,
                                                        uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  constexpr int VE = 16 / (int)sizeof(T);   // elements of d per 16-byte vector
  constexpr int NV = TW * E;                // partial logits per lane, index t * E + e
  constexpr int WG_VEC = E;                 // 16-byte vectors per VE rows of W_g (VE * E * sizeof(T) = 16 E)
  __shared__ float red[8][NV];
  __shared__ float logit[NV];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * TW;
  float acc[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) acc[i] = 0.f;
  const int nvec = d / VE;
  const uint4* xv4 = reinterpret_cast<const uint4*>(x);
  const uint4* wv4 = reinterpret_cast<const uint4*>(Wg);
  const size_t row_vecs = (size_t)nvec;
  constexpr int UNROLL = NV <= 32 ? 2 : 1;
#pragma unroll UNROLL
  for (int v = threadIdx.x; v < nvec; v += 256) {
    uint4 xr[TW];
#pragma unroll
    for (int t = 0; t < TW; ++t)
      xr[t] = (t0 + t < Tn) ? __ldg(xv4 + (size_t)(t0 + t) * row_vecs + v) : make_uint4(0, 0, 0, 0);
    if constexpr ((E * sizeof(T)) % 16 == 0) {
      // each of the VE rows of W_g is a whole number of 16-byte vectors: load row by row
      constexpr int RV = E * (int)sizeof(T) / 16;
#pragma unroll
      for (int r = 0; r < VE; ++r) {
        uint4 wr[RV];
#pragma unroll
        for (int i = 0; i < RV; ++i) wr[i] = __ldg(wv4 + ((size_t)v * VE + r) * RV + i);
        float xe[TW];
#pragma unroll
        for (int t = 0; t < TW; ++t) xe[t] = vec_elem<T>(xr, t * VE + r);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float w = vec_elem<T>(wr, e);
#pragma unroll
          for (int t = 0; t < TW; ++t) acc[t * E + e] = fmaf(xe[t], w, acc[t * E + e]);
        }
      }
    } else {
      // small E: the VE rows together are E 16-byte vectors
      uint4 wr[WG_VEC];
#pragma unroll
      for (int i = 0; i < WG_VEC; ++i) wr[i] = __ldg(wv4 + (size_t)v * WG_VEC + i);
#pragma unroll
      for (int r = 0; r < VE; ++r) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float w = vec_elem<T>(wr, r * E + e);
#pragma unroll
          for (int t = 0; t < TW; ++t) acc[t * E + e] = fmaf(vec_elem<T>(xr, t * VE + r), w, acc[t * E + e]);
        }
      }
    }
  }
  halve_sum<NV, 16>(acc, lane);
  constexpr int HN = NV >= 32 ? NV / 32 : 1;   // sums a lane holds after the halving
  bool owner;
  const int base = halve_base<NV>(lane, owner);
  if (owner) {
#pragma unroll
    for (int i = 0; i < HN; ++i) red[warp][base + i] = acc[i];
  }
  __syncthreads();
  if (threadIdx.x < NV) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += red[w][threadIdx.x];
    logit[threadIdx.x] = sum;
  }
  __syncthreads();
  if (warp < TW && t0 + warp < Tn) {
    float l[1], key[1];
    l[0] = 0.f;
    key[0] = -INFINITY;
    if (lane < E) {
      l[0] = logit[warp * E + lane];
      if (lb) l[0] += __ldg(lb + lane);
      key[0] = selection_key(l[0], sb, lane, scoring);
      if (!isfinite(l[0]) || isnan(key[0])) {
        flag_error(err, ERR_ROUTE);
        if (isnan(key[0])) key[0] = -INFINITY;
      }
    }
    select_and_gate<1>(l, key, E, k, scoring, t0 + warp, idx, gate);
  }
}

// One warp per token over precomputed float32 logits [T][E].
template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, const float* __restrict__ lb,
                                                         const float* __restrict__ sb, int Tn, int E, int k,
                                                         int scoring, int32_t* idx, float* gate, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= Tn) return;
  const float* lr = logits + (size_t)t * E;
  float l[EPL], key[EPL];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    l[i] = 0.f;
    key[i] = -INFINITY;
    if (e < E) {
      l[i] = __ldg(lr + e);
      if (lb) l[i] += __ldg(lb + e);
      key[i] = selection_key(l[i], sb, e, scoring);
      if (!isfinite(l[i]) || isnan(key[i])) {
        bad = true;
        if (isnan(key[i])) key[i] = -INFINITY;
      }
    }
  }
  if (bad) flag_error(err, ERR_ROUTE);
  select_and_gate<EPL>(l, key, E, k, scoring, t, idx, gate);
}

// Logits on CUDA cores: 64 tokens x 64 experts per block, 4 x 4 per thread.
template <typename T>
__global__ void __launch_bounds__(256) logits_simt_kernel(const T* __restrict__ x, const T* __restrict__ Wg, int Tn,
                                                          int d, int E, float* __restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  constexpr int BT = 64, BE = 64, BK = 16;
  __shared__ float xs[BK][BT + 4];
  __shared__ float ws[BK][BE + 4];
  const int t0 = blockIdx.y * BT, e0 = blockIdx.x * BE;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += BK) {
    for (int i = threadIdx.x; i < BT * BK; i += 256) {
      const int r = i / BK, kk = i % BK;
      const int tt = t0 + r, kx = k0 + kk;
      xs[kk][r] = (tt < Tn && kx < d) ? load_as_float(x + (size_t)tt * d + kx) : 0.f;
    }
    for (int i = threadIdx.x; i < BK * BE; i += 256) {
      const int kk = i / BE, c = i % BE;
      const int kx = k0 + kk, e = e0 + c;
      ws[kk][c] = (kx < d && e < E) ? load_as_float(Wg + (size_t)kx * E + e) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { av[i] = xs[kk][ty * 4 + i]; bv[i] = ws[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tt = t0 + ty * 4 + i, e = e0 + tx * 4 + j;
      if (tt < Tn && e < E) logits[(size_t)tt * E + e] = acc[i][j];
    }
}

// One step of the bias controller: an expert whose load is above its share T k / E has its
// selection bias lowered by gamma, one below raised by gamma (page "Mixture-of-Experts
// Internals: A Systems Engineer's Field Manual", section 3.3).  Loads are compared in integers.
__global__ void __launch_bounds__(256) update_sel_bias_kernel(const int32_t* __restrict__ counts, int E,
                                                              long long share, float gamma, float* sb) {
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const long long c = (long long)__ldg(counts + e) * E;
  float b = sb[e];
  if (c > share) b = __fsub_rn(b, gamma);
  else if (c < share) b = __fadd_rn(b, gamma);
  sb[e] = b;
}

}  // namespace

cudaError_t update_sel_bias(const int32_t* counts, int T, int k, int E, float gamma, float* sel_bias,
                            cudaStream_t st) {
  MOE_RETURN_ON_ERROR(launch_k(update_sel_bias_kernel, (E + 255) / 256, 256, 0, st, counts, E, (long long)T * k, gamma,
                               sel_bias));
  ++g_launches;
  return cudaGetLastError();
}

cudaError_t route_fused(int dtype, const void* x, const void* W_g, const float* logit_bias, const float* sel_bias,
                        int T, int d, int E, int k, int scoring, int32_t* idx, float* gate, uint32_t* err,
                        cudaStream_t st) {
  const int threads = 256;
  const int ve = dtype == 1 ? 8 : 4;
  const bool vec = d % ve == 0 && ((uintptr_t)x % 16) == 0 && ((uintptr_t)W_g % 16) == 0 && (E & (E - 1)) == 0;
  if (vec) {
    // tokens per block: enough to reuse each W_g vector, few enough to keep the partials in registers
    const int tw = E >= 32 ? 4 : E >= 8 ? 4 : 8;
    const unsigned blocks = (unsigned)((T + tw - 1) / tw);
#define MOE_ROUTE_VEC(TY, EE, TWW)                                                                           \
  MOE_RETURN_ON_ERROR(launch_k(route_vec_kernel<TY, EE, TWW>, blocks, threads, 0, st, (const TY*)x, (const TY*)W_g, \
                               logit_bias, sel_bias, T, d, k, scoring, idx, gate, err))
#define MOE_ROUTE_VEC_E(TY)                          \
  switch (E) {                                       \
    case 1: MOE_ROUTE_VEC(TY, 1, 8); break;          \
    case 2: MOE_ROUTE_VEC(TY, 2, 8); break;          \
    case 4: MOE_ROUTE_VEC(TY, 4, 8); break;          \
    case 8: MOE_ROUTE_VEC(TY, 8, 4); break;          \
    case 16: MOE_ROUTE_VEC(TY, 16, 4); break;        \
    default: MOE_ROUTE_VEC(TY, 32, 4); break;        \
  }
    if (dtype == 1) {
      MOE_ROUTE_VEC_E(uint16_t)
    } else {
      MOE_ROUTE_VEC_E(float)
    }
#undef MOE_ROUTE_VEC_E
#undef MOE_ROUTE_VEC
    ++g_launches;
    return cudaGetLastError();
  }
  const unsigned blocks = (unsigned)(((long long)T * 32 + threads - 1) / threads);
#define MOE_ROUTE_FUSED(TY, EM)                                                                             \
  MOE_RETURN_ON_ERROR(launch_k(route_fused_kernel<TY, EM>, blocks, threads, 0, st, (const TY*)x, (const TY*)W_g, \
                               logit_bias, sel_bias, T, d, E, k, scoring, idx, gate, err))
  if (dtype == 1) {
    if (E <= 8) MOE_ROUTE_FUSED(uint16_t, 8);
    else if (E <= 16) MOE_ROUTE_FUSED(uint16_t, 16);
    else MOE_ROUTE_FUSED(uint16_t, 32);
  } else {
    if (E <= 8) MOE_ROUTE_FUSED(float, 8);
    else if (E <= 16) MOE_ROUTE_FUSED(float, 16);
    else MOE_ROUTE_FUSED(float, 32);
  }
#undef MOE_ROUTE_FUSED
  ++g_launches;
  return cudaGetLastError();
}

cudaError_t route_logits_simt(int dtype, const void* x, const void* W_g, int T, int d, int E, float* logits,
                              cudaStream_t st) {
  dim3 grid((E + 63) / 64, (T + 63) / 64);
  if (dtype == 1)
    MOE_RETURN_ON_ERROR(launch_k(logits_simt_kernel<uint16_t>, grid, 256, 0, st, (const uint16_t*)x, (const uint16_t*)W_g,
                                 T, d, E, logits));
  else
    MOE_RETURN_ON_ERROR(launch_k(logits_simt_kernel<float>, grid, 256, 0, st, (const float*)x, (const float*)W_g, T, d, E,
                                 logits));
  ++g_launches;
  return cudaGetLastError();
}

cudaError_t route_topk(const float* logits, const float* logit_bias, const float* sel_bias, int T, int E, int k,
                       int scoring, int32_t* idx, float* gate, uint32_t* err, cudaStream_t st) {
  const int threads = 256;
  const unsigned blocks = (unsigned)(((long long)T * 32 + threads - 1) / threads);
#define MOE_TOPK(EPL)                                                                                       \
  MOE_RETURN_ON_ERROR(launch_k(route_topk_kernel<EPL>, blocks, threads, 0, st, (const float*)logits, logit_bias, \
                               sel_bias, T, E, k, scoring, idx, gate, err))
  if (E <= 32) MOE_TOPK(1);
  else if (E <= 64) MOE_TOPK(2);
  else if (E <= 128) MOE_TOPK(4);
  else if (E <= 256) MOE_TOPK(8);
  else if (E <= 512) MOE_TOPK(16);
  else MOE_TOPK(32);
#undef MOE_TOPK
  ++g_launches;
  return cudaGetLastError();
}

}  // namespace moe
