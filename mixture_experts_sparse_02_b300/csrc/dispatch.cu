// Dispatch of the MoE layer: per-expert histogram, exclusive prefix sum, stable permutation
// and row gather (page "Mixture of Experts: What Actually Happens When a Token Hits the
// Router", Step 3: sort tokens by assigned expert into contiguous blocks per expert).  With a
// capacity of `cap` slots per expert, an expert keeps its first `cap` pairs in token order and
// the rest are dropped (page "8.6 - Mixture of Experts (MoE)", section 3.2; page "Mixture-of-
// Experts, from the router to the all-to-all", "Capacity and token dropping").
//
// The T*k (token, slot) pairs, in flattened order i = t*k + j, are cut into chunks of 256
// pairs, one chunk per warp.  No atomics anywhere, so counts, offsets and the permutation are
// identical from run to run:
//   hist     each warp counts its chunk per expert: __match_any_sync groups the lanes that
//            hold the same expert, and the lowest such lane adds the group size to the
//            warp's private histogram in shared memory.
//   scan     one block: per-expert totals, exclusive scan over experts (offsets), and each
//            chunk's starting position per expert (offsets[e] + pairs of e in earlier chunks).
//   permute  each warp replays its chunk: a pair's position is its chunk's running position
//            for that expert plus its rank among the lanes of the same expert in that round.
//            Pairs of one expert therefore keep ascending i.
//   scatter  x_perm[inv_pos[t][j]] = x[t], one warp per token: each token row is read once and
//            written to its k positions (expert-choice routing, which has no inv_pos, gathers
//            x_perm[p] = x[perm_tok[p]] by row instead).
// Batches of up to 16384 pairs over at most 256 experts take one single-block kernel for the
// first three steps instead (dispatch_small_kernel).
#include "common.cuh"
#include "internal.h"

namespace moe {

extern thread_local int g_launches;

namespace {

constexpr int CHUNK = 256;     // pairs per warp
constexpr int WARPS = 8;       // warps per block in hist / permute
constexpr unsigned FULL = 0xffffffffu;

__global__ void __launch_bounds__(WARPS * 32) hist_kernel(const int32_t* __restrict__ idx, long long N, int E,
                                                          int n_chunks, int32_t* __restrict__ chunk_counts,
                                                          uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * WARPS + warp;
  int* h = sh + warp * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  if (chunk >= n_chunks) return;
  const long long base = (long long)chunk * CHUNK;
  bool bad = false;
  for (int r = 0; r < CHUNK / 32; ++r) {
    const long long i = base + r * 32 + lane;
    int e = -1;
    if (i < N) {
      e = __ldg(idx + i);
      if (e < 0 || e >= E) { bad = true; e = -1; }
    }
    const unsigned m = __match_any_sync(FULL, e);
    if (e >= 0 && lane == __ffs(m) - 1) h[e] += __popc(m);
    __syncwarp();
  }
  if (bad) flag_error(err, ERR_EXPERT_ID);
  for (int e = lane; e < E; e += 32) chunk_counts[(size_t)chunk * E + e] = h[e];
}

// One block of 1024 threads.  Thread (e, s) owns expert e's column of the [n_chunks][E]
// count matrix over the chunk segment s (S segments per expert).
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ chunk_counts, int n_chunks, int E,
                                                    int S, int cap, int32_t* __restrict__ chunk_base,
                                                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  pdl_wait();
  pdl_trigger();
  __shared__ int part[1024];   // [S][E] segment sums, then exclusive segment bases
  __shared__ int tot[1024];    // per-expert totals, then offsets
  __shared__ int wsum[32];
  const int tid = threadIdx.x;
  const int e = tid % E, s = tid / E;
  const int seg = (n_chunks + S - 1) / S;
  const bool active = tid < E * S;
  const int c0 = s * seg, c1 = min(n_chunks, c0 + seg);
  if (active) {
    int acc = 0;
    for (int c = c0; c < c1; ++c) acc += chunk_counts[(size_t)c * E + e];
    part[s * E + e] = acc;
  }
  __syncthreads();
  if (tid < E) {
    int run = 0;
    for (int q = 0; q < S; ++q) {
      const int v = part[q * E + tid];
      part[q * E + tid] = run;
      run += v;
    }
    tot[tid] = min(run, cap);   // pairs the expert keeps; offsets are over kept pairs
    counts[tid] = run;          // the expert's load, before any dropping
  }
  __syncthreads();
  // exclusive scan of tot[0..E) (E <= 1024) across the block
  const int lane = tid & 31, w = tid >> 5;
  int v = tid < E ? tot[tid] : 0;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    int x = wsum[lane];
    int xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(FULL, xi, o);
      if (lane >= o) xi += n;
    }
    wsum[lane] = xi - x;
  }
  __syncthreads();
  const int excl = incl - v + wsum[w];
  __syncthreads();
  if (tid < E) {
    tot[tid] = excl;
    offsets[tid] = excl;
  }
  if (tid == E - 1) offsets[E] = excl + v;
  __syncthreads();
  if (active) {
    int run = tot[e] + part[s * E + e];
    for (int c = c0; c < c1; ++c) {
      chunk_base[(size_t)c * E + e] = run;
      run += chunk_counts[(size_t)c * E + e];
    }
  }
}

__global__ void __launch_bounds__(WARPS * 32) permute_kernel(const int32_t* __restrict__ idx, long long N, int k, int E,
                                                             int n_chunks, int cap, const int32_t* __restrict__ chunk_base,
                                                             const int32_t* __restrict__ offsets,
                                                             int32_t* __restrict__ perm_tok,
                                                             int32_t* __restrict__ inv_pos, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * WARPS + warp;
  if (chunk >= n_chunks) return;
  int* run = sh + warp * E;
  for (int e = lane; e < E; e += 32) run[e] = __ldg(chunk_base + (size_t)chunk * E + e);
  __syncwarp();
  const long long base = (long long)chunk * CHUNK;
  const unsigned lt = (1u << lane) - 1u;
  for (int r = 0; r < CHUNK / 32; ++r) {
    const long long i = base + r * 32 + lane;
    int e = -1;
    if (i < N) {
      e = __ldg(idx + i);
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned m = __match_any_sync(FULL, e);
    if (i < N) {
      if (e >= 0) {
        const int pos = run[e] + __popc(m & lt);
        debug_bounds(pos >= 0 && pos < N, err);
        if (pos - __ldg(offsets + e) < cap) {   // rank within the expert, in token order
          perm_tok[pos] = (int32_t)(i / k);
          inv_pos[i] = pos;
        } else {
          inv_pos[i] = -1;                        // the expert is full: the pair is dropped
        }
      } else {
        inv_pos[i] = -1;
      }
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) run[e] += __popc(m);
    __syncwarp();
  }
}

template <typename V>
__global__ void __launch_bounds__(256) gather_kernel(const V* __restrict__ x, const int32_t* __restrict__ perm_tok,
                                                     long long rows, const int32_t* __restrict__ rows_dev,
                                                     int vec_per_row, long long T, V* __restrict__ xp,
                                                     uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  if (rows_dev) {   // rows actually kept (offsets[E]); never more than the buffer holds
    const long long kept = __ldg(rows_dev);
    rows = kept < rows ? (kept > 0 ? kept : 0) : rows;
  }
  for (long long p = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; p < rows; p += warps) {
    const int t = __ldg(perm_tok + p);
    V* dst = xp + (size_t)p * vec_per_row;
    const bool in_range = t >= 0 && t < T;
    if (lane == 0) debug_bounds(in_range, err);
    if (!in_range) continue;   // only after an expert-id error (flagged), or a caller's bad perm_tok
    const V* src = x + (size_t)t * vec_per_row;
    for (int v = lane; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
  }
}

// Row scatter, the same x_perm by token: warp t reads token row t once, CH 16-byte vectors per
// lane at a time, and writes it to the positions of its kept pairs, inv_pos[t][0..k).  A gather
// by permuted row (above) reads each token's row k times, at scattered times, while the x_perm
// writes stream through L2 and evict it.
template <typename V, int CH>
__global__ void __launch_bounds__(256) scatter_kernel(const V* __restrict__ x, const int32_t* __restrict__ inv_pos,
                                                      long long T, int k, int vec_per_row, long long rows,
                                                      V* __restrict__ xp, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  for (long long t = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    int p = -1;   // lane j < k: the position of pair (t, j), or -1 (dropped)
    if (lane < k) {
      p = __ldg(inv_pos + t * k + lane);
      const bool in_range = p >= -1 && p < rows;
      debug_bounds(in_range, err);
      if (!in_range) p = -1;   // a caller's bad inv_pos (flagged in the bounds-checking build)
    }
    const V* src = x + (size_t)t * vec_per_row;
    // the trip count is the same for every lane (the shuffles below need the whole warp)
    for (int base = 0; base < vec_per_row; base += 32 * CH) {
      V buf[CH];
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int v = base + 32 * c + lane;
        if (v < vec_per_row) buf[c] = __ldg(src + v);
      }
      for (int j = 0; j < k; ++j) {
        const int pj = __shfl_sync(FULL, p, j);
        if (pj < 0) continue;
        V* dst = xp + (size_t)pj * vec_per_row;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int v = base + 32 * c + lane;
          if (v < vec_per_row) dst[v] = buf[c];
        }
      }
    }
  }
}

// Small batches (T k <= SMALL_PAIRS, E <= SMALL_E), as decode steps produce: the histogram,
// scan and permutation in one block of 1024 threads, with the same results as the three
// kernels above, and no atomics either.  Rounds of 1024 pairs in flattened order; warp w of
// a round takes its 32 pairs; a pair's rank within its expert is (pairs of the expert in
// earlier rounds) + (in earlier warps of the round) + (lanes of its warp before it with the
// same expert).
constexpr int SMALL_PAIRS = 16384;
constexpr int SMALL_E = 256;

__global__ void __launch_bounds__(1024) dispatch_small_kernel(const int32_t* __restrict__ idx, int N, int k, int E,
                                                              int cap, int32_t* __restrict__ counts,
                                                              int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ perm_tok,
                                                              int32_t* __restrict__ inv_pos, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int wc[32][SMALL_E];   // per-warp counts of a round, then their exclusive prefix over warps
  __shared__ int run[SMALL_E];      // per-expert totals, then pairs of each expert in earlier rounds
  __shared__ int off[SMALL_E + 1];
  __shared__ int wsum[33];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Histogram as in hist_kernel: each warp counts its pairs of every round in a private row of
  // wc (the lowest lane of each group of equal experts adds the group's size), then thread e
  // adds up expert e's column.
  for (int x = lane; x < E; x += 32) wc[warp][x] = 0;
  __syncwarp();
  bool bad = false;
  for (int base = 0; base < N; base += 1024) {
    const int i = base + tid;
    int e = -1;
    if (i < N) {
      e = __ldg(idx + i);
      if (e < 0 || e >= E) { bad = true; e = -1; }
    }
    const unsigned m = __match_any_sync(FULL, e);
    if (e >= 0 && lane == __ffs(m) - 1) wc[warp][e] += __popc(m);
    __syncwarp();
  }
  if (bad) flag_error(err, ERR_EXPERT_ID);
  __syncthreads();
  for (int x = tid; x < E; x += 1024) {
    int c = 0;
    for (int w = 0; w < 32; ++w) c += wc[w][x];
    run[x] = c;
  }
  __syncthreads();
  // exclusive scan of the kept counts over the experts (E <= 256 < 1024 threads)
  const int kept = tid < E ? min(run[tid], cap) : 0;
  int incl = kept;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
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
  const int excl = incl - kept + wsum[warp];
  if (tid < E) {
    counts[tid] = run[tid];
    off[tid] = excl;
    offsets[tid] = excl;
  }
  if (tid == 0) {
    off[E] = wsum[32];
    offsets[E] = wsum[32];
  }
  __syncthreads();
  for (int e = tid; e < E; e += 1024) run[e] = 0;
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int base = 0; base < N; base += 1024) {
    const int i = base + tid;
    int e = -1;
    if (i < N) {
      e = __ldg(idx + i);
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned m = __match_any_sync(FULL, e);
    for (int x = lane; x < E; x += 32) wc[warp][x] = 0;
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) wc[warp][e] = __popc(m);
    __syncthreads();
    for (int x = tid; x < E; x += 1024) {
      int r = run[x];
      for (int w = 0; w < 32; ++w) {
        const int c = wc[w][x];
        wc[w][x] = r;
        r += c;
      }
      run[x] = r;
    }
    __syncthreads();
    if (i < N) {
      int pos = -1;
      if (e >= 0) {
        const int rank = wc[warp][e] + __popc(m & lt);
        if (rank < cap) {
          pos = off[e] + rank;
          debug_bounds(pos < N, err);
          perm_tok[pos] = (int32_t)(i / k);
        }
      }
      inv_pos[i] = pos;
    }
    __syncthreads();
  }
}

}  // namespace

int dispatch_num_chunks(long long pairs) { return (int)((pairs + CHUNK - 1) / CHUNK); }

cudaError_t dispatch_indices(const int32_t* topk_idx, int T, int k, int E, int cap, int32_t* chunk_counts,
                             int32_t* chunk_base, int32_t* counts, int32_t* offsets, int32_t* perm_tok,
                             int32_t* inv_pos, uint32_t* err, cudaStream_t st, int* launches) {
  const long long N = (long long)T * k;
  if (N <= SMALL_PAIRS && E <= SMALL_E) {
    MOE_RETURN_ON_ERROR(launch_k(dispatch_small_kernel, 1, 1024, 0, st, topk_idx, (int)N, k, E, cap, counts, offsets,
                                 perm_tok, inv_pos, err));
    g_launches += 1;
    if (launches) *launches += 1;
    return cudaGetLastError();
  }
  const int n_chunks = dispatch_num_chunks(N);
  const unsigned blocks = (unsigned)((n_chunks + WARPS - 1) / WARPS);
  const size_t shm = (size_t)WARPS * E * sizeof(int);
  MOE_RETURN_ON_ERROR(launch_k(hist_kernel, blocks, WARPS * 32, shm, st, topk_idx, N, E, n_chunks, chunk_counts, err));
  int S = 1;
  while (S * 2 * E <= 1024 && S * 2 <= n_chunks) S *= 2;
  MOE_RETURN_ON_ERROR(launch_k(scan_kernel, 1, 1024, 0, st, chunk_counts, n_chunks, E, S, cap, chunk_base, counts,
                               offsets));
  MOE_RETURN_ON_ERROR(launch_k(permute_kernel, blocks, WARPS * 32, shm, st, topk_idx, N, k, E, n_chunks, cap,
                               chunk_base, offsets, perm_tok, inv_pos, err));
  g_launches += 3;
  if (launches) *launches += 3;
  return cudaGetLastError();
}

cudaError_t scatter_rows(const void* x, long long T, int k, const int32_t* inv_pos, long long rows, int d,
                         int elem_bytes, void* x_perm, uint32_t* err, cudaStream_t st) {
  const long long row_bytes = (long long)d * elem_bytes;
  const int threads = 256;
  const long long want = (T * 32 + threads - 1) / threads;
  const unsigned blocks = (unsigned)(want < 148LL * 16 ? want : 148LL * 16);
  if (row_bytes % 16 == 0 && ((uintptr_t)x % 16 == 0) && ((uintptr_t)x_perm % 16 == 0)) {
    MOE_RETURN_ON_ERROR(launch_k(scatter_kernel<uint4, 4>, blocks, threads, 0, st, (const uint4*)x, inv_pos, T, k,
                                 (int)(row_bytes / 16), rows, (uint4*)x_perm, err));
  } else if (row_bytes % 4 == 0) {
    MOE_RETURN_ON_ERROR(launch_k(scatter_kernel<uint32_t, 4>, blocks, threads, 0, st, (const uint32_t*)x, inv_pos, T,
                                 k, (int)(row_bytes / 4), rows, (uint32_t*)x_perm, err));
  } else {
    MOE_RETURN_ON_ERROR(launch_k(scatter_kernel<uint16_t, 4>, blocks, threads, 0, st, (const uint16_t*)x, inv_pos, T,
                                 k, (int)(row_bytes / 2), rows, (uint16_t*)x_perm, err));
  }
  ++g_launches;
  return cudaGetLastError();
}

cudaError_t gather_rows(const void* x, long long T, const int32_t* perm_tok, long long rows, const int32_t* rows_dev,
                        int d, int elem_bytes, void* x_perm, uint32_t* err, cudaStream_t st) {
  const long long row_bytes = (long long)d * elem_bytes;
  const int threads = 256;
  long long want = (rows * 32 + threads - 1) / threads;
  const unsigned blocks = (unsigned)(want < 148LL * 16 ? want : 148LL * 16);
  if (row_bytes % 16 == 0 && ((uintptr_t)x % 16 == 0) && ((uintptr_t)x_perm % 16 == 0)) {
    MOE_RETURN_ON_ERROR(launch_k(gather_kernel<uint4>, blocks, threads, 0, st, (const uint4*)x, perm_tok, rows, rows_dev,
                                 (int)(row_bytes / 16), T, (uint4*)x_perm, err));
  } else if (row_bytes % 4 == 0) {
    MOE_RETURN_ON_ERROR(launch_k(gather_kernel<uint32_t>, blocks, threads, 0, st, (const uint32_t*)x, perm_tok, rows,
                                 rows_dev, (int)(row_bytes / 4), T, (uint32_t*)x_perm, err));
  } else {
    MOE_RETURN_ON_ERROR(launch_k(gather_kernel<uint16_t>, blocks, threads, 0, st, (const uint16_t*)x, perm_tok, rows,
                                 rows_dev, (int)(row_bytes / 2), T, (uint16_t*)x_perm, err));
  }
  ++g_launches;
  return cudaGetLastError();
}

}  // namespace moe
