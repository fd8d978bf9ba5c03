// Grouped float32 GEMM on CUDA cores (FFMA) for the float32 dtype, where the tolerance
// (1e-4 relative) rules out TF32 tensor cores.  Same grouping as the tensor-core path: one
// group per expert over its block of permuted rows (page "Mixture of Experts: What Actually
// Happens When a Token Hits the Router", Step 3), SwiGLU epilogue h = (X W1) * SiLU(X W2)
// (page "8.6 - Mixture of Experts (MoE)", section 2) or a plain float32 store.
//
// 64 x 64 output tile per block, 16-deep K slices through shared memory, 4 x 4 per thread.
// The grid covers an upper bound of the row tiles (rows/64 + groups); a block finds its group
// by walking the offsets on the device and exits when it has none.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int BM = 64, BN = 64, BK = 16;

struct SimtArgs {
  const int* offsets;
  int G, M, K, N;
  long long w_stride_z;
  int b_z;
  float* out;
  int accumulate;
  int rows_cap;
  uint32_t* err;
};

template <int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const float* __restrict__ A, const float* __restrict__ W0,
                                                        const float* __restrict__ W1, const SimtArgs p) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[BK][BM + 4];
  __shared__ float B0s[BK][BN + 4];
  __shared__ float B1s[EPI == EPI_SWIGLU ? BK : 1][BN + 4];

  int y = blockIdx.y, g = 0, row0 = 0, row_end = 0;
  bool found = false;
  if (p.offsets) {
    for (g = 0; g < p.G; ++g) {
      int a0 = __ldg(p.offsets + g), a1 = __ldg(p.offsets + g + 1);
      a0 = min(max(a0, 0), p.rows_cap);
      a1 = min(max(a1, 0), p.rows_cap);
      const int rows = a1 - a0;
      const int mt = rows > 0 ? (rows + BM - 1) / BM : 0;
      if (y < mt) { row0 = a0 + y * BM; row_end = a1; found = true; break; }
      y -= mt;
    }
  } else if (y * BM < p.M) {
    row0 = y * BM;
    row_end = p.M;
    found = true;
  }
  if (!found) return;
  const long long z = p.offsets ? g : p.b_z;
  const float* w0 = W0 + z * p.w_stride_z;
  const float* w1 = (EPI == EPI_SWIGLU) ? W1 + z * p.w_stride_z : nullptr;
  const int n0 = blockIdx.x * BN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int K = p.K, N = p.N;

  float acc0[4][4] = {}, acc1[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = threadIdx.x; i < BM * BK; i += 256) {
      const int r = i / BK, kk = i % BK;
      const int row = row0 + r, kx = k0 + kk;
      As[kk][r] = (row < row_end && kx < K) ? __ldg(A + (size_t)row * K + kx) : 0.f;
    }
    for (int i = threadIdx.x; i < BK * BN; i += 256) {
      const int kk = i / BN, c = i % BN;
      const int kx = k0 + kk, nx = n0 + c;
      const bool in = kx < K && nx < N;
      B0s[kk][c] = in ? __ldg(w0 + (size_t)kx * N + nx) : 0.f;
      if (EPI == EPI_SWIGLU) B1s[kk][c] = in ? __ldg(w1 + (size_t)kx * N + nx) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], b0[4], b1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = As[kk][ty * 4 + i];
        b0[i] = B0s[kk][tx * 4 + i];
        if (EPI == EPI_SWIGLU) b1[i] = B1s[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc0[i][j] = fmaf(av[i], b0[j], acc0[i][j]);
          if (EPI == EPI_SWIGLU) acc1[i][j] = fmaf(av[i], b1[j], acc1[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = row0 + ty * 4 + i;
    if (row >= row_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx * 4 + j;
      if (col >= N) continue;
      float* dst = p.out + (size_t)row * N + col;
      if (EPI == EPI_SWIGLU) {
        const float v = acc1[i][j];
        *dst = acc0[i][j] * (v / (1.0f + expf(-v)));
      } else {
        *dst = p.accumulate ? *dst + acc0[i][j] : acc0[i][j];
      }
    }
  }
}

template <int EPI>
cudaError_t launch(const float* A, const float* W0, const float* W1, const SimtArgs& p, cudaStream_t st) {
  const long long row_tiles = p.offsets ? ((long long)p.rows_cap + BM - 1) / BM + p.G : ((long long)p.M + BM - 1) / BM;
  if (row_tiles <= 0) return cudaSuccess;
  dim3 grid((p.N + BN - 1) / BN, (unsigned)row_tiles);
  MOE_RETURN_ON_ERROR(launch_k(simt_gemm_kernel<EPI>, grid, 256, 0, st, A, W0, W1, p));
  ++g_launches;
  return cudaGetLastError();
}

}  // namespace

cudaError_t simt_swiglu_f32(const float* A, int rows_cap, int K, const float* W1, const float* W2, int N,
                            const int* offsets, int G, int M_dense, long long w_stride_z, int b_z, float* h,
                            uint32_t* err, cudaStream_t st) {
  SimtArgs p{offsets, G, M_dense, K, N, w_stride_z, b_z, h, 0, rows_cap, err};
  return launch<EPI_SWIGLU>(A, W1, W2, p, st);
}

cudaError_t simt_matmul_f32(const float* A, int rows_cap, int K, const float* W, int N, const int* offsets, int G,
                            int M_dense, long long w_stride_z, int b_z, float* out, int accumulate, uint32_t* err,
                            cudaStream_t st) {
  SimtArgs p{offsets, G, M_dense, K, N, w_stride_z, b_z, out, accumulate, rows_cap, err};
  return launch<EPI_F32>(A, W, nullptr, p, st);
}

}  // namespace moe
