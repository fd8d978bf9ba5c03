// Internal launchers of libmoe (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Kernels launched by the current host thread since the last C-ABI entry (reset there).
extern thread_local int g_launches;

enum { EPI_SWIGLU = 0, EPI_F32 = 1 };

// Arguments of the grouped tensor-core GEMM kernel.
struct GemmArgs {
  const int* offsets;  // [G+1] row offsets of the groups (device); NULL: one group of M rows
  int G;
  int M;               // rows of the single group when offsets == NULL
  int K;               // reduction length
  int N;               // output columns
  int n_tiles;         // column tiles per group
  int b_z;             // B-matrix index (z) used when offsets == NULL
  void* out;           // output [rows_cap][ldo]
  long long ldo;
  int accumulate;      // EPI_F32: out += result
  int rows_cap;        // rows of A and of out; offsets beyond it are clamped and flagged
  uint32_t* err;       // device error word
  unsigned long long wait_limit_ns;  // bound of every pipeline wait
  int starve;          // test hook: the TMA producer issues no copies (the waits run out)
  int* tile_ctr;       // CTA-pair kernels: [2] ints of their dynamic tile scheduler (next tile,
                       // clusters finished), zero on entry and reset to zero by the kernel
};

// Test hook (moe_test_pipeline_fault): arm a starved pipeline with a short wait limit for the
// next grouped tensor-core GEMM launch of this process.
void arm_pipeline_fault(unsigned long long wait_limit_ns);

// ---- tensor-core (bf16) path
cudaError_t tc_swiglu(const void* A, long long rows_cap, int K, const void* W1, const void* W2, int Z, int N,
                      const int* offsets, int G, int M_dense, int b_z, void* h, uint32_t* err, cudaStream_t st);
cudaError_t tc_matmul_f32(const void* A, long long rows_cap, int K, const void* W, int Z, int N, const int* offsets,
                          int G, int M_dense, int b_z, float* out, long long ldo, int accumulate, uint32_t* err,
                          cudaStream_t st);

// ---- CUDA-core float32 path (the float32 dtype; no TF32)
cudaError_t simt_swiglu_f32(const float* A, int rows_cap, int K, const float* W1, const float* W2, int N,
                            const int* offsets, int G, int M_dense, long long w_stride_z, int b_z, float* h,
                            uint32_t* err, cudaStream_t st);
cudaError_t simt_matmul_f32(const float* A, int rows_cap, int K, const float* W, int N, const int* offsets, int G,
                            int M_dense, long long w_stride_z, int b_z, float* out, int accumulate, uint32_t* err,
                            cudaStream_t st);

// ---- router
// Fused logits + top-k + gates, one warp per token, for E <= 32.
cudaError_t route_fused(int dtype, const void* x, const void* W_g, const float* logit_bias, const float* sel_bias,
                        int T, int d, int E, int k, int scoring, int32_t* idx, float* gate, uint32_t* err,
                        cudaStream_t st);
// Logits [T][E] float32 on CUDA cores (any E).
cudaError_t route_logits_simt(int dtype, const void* x, const void* W_g, int T, int d, int E, float* logits,
                              cudaStream_t st);
// Top-k + gates from precomputed logits, one warp per token, E <= 1024.
cudaError_t route_topk(const float* logits, const float* logit_bias, const float* sel_bias, int T, int E, int k,
                       int scoring, int32_t* idx, float* gate, uint32_t* err, cudaStream_t st);

// One step of the selection-bias controller from the last batch's per-expert counts.
cudaError_t update_sel_bias(const int32_t* counts, int T, int k, int E, float gamma, float* sel_bias,
                            cudaStream_t st);

// ---- load statistics (f, P, L_aux, max/mean load) from float32 logits [T][E]
int stats_num_blocks(int T);
cudaError_t load_stats(const float* logits, const float* logit_bias, const int32_t* counts, int T, int k, int E,
                       int scoring, float alpha, float* partial, float* f, float* P, float* summary,
                       cudaStream_t st);

// ---- dispatch
int dispatch_num_chunks(long long pairs);
// cap: slots per expert (pairs beyond the first cap of an expert, in token order, are dropped:
// inv_pos = -1); a value >= T*k keeps everything.  counts = loads before dropping, offsets over
// the kept pairs.
cudaError_t dispatch_indices(const int32_t* topk_idx, int T, int k, int E, int cap, int32_t* chunk_counts,
                             int32_t* chunk_base, int32_t* counts, int32_t* offsets, int32_t* perm_tok,
                             int32_t* inv_pos, uint32_t* err, cudaStream_t st, int* launches);
// x_perm[inv_pos[t][j]] = x[t] for every kept pair (inv_pos >= 0); rows = the rows of x_perm.
cudaError_t scatter_rows(const void* x, long long T, int k, const int32_t* inv_pos, long long rows, int d,
                         int elem_bytes, void* x_perm, uint32_t* err, cudaStream_t st);
// rows_dev (optional, device): the number of rows to copy, bounded by `rows`.
cudaError_t gather_rows(const void* x, long long T, const int32_t* perm_tok, long long rows, const int32_t* rows_dev,
                        int d, int elem_bytes, void* x_perm, uint32_t* err, cudaStream_t st);

// ---- expert choice: scores [T][E] hold the router logits on entry and the per-token softmax
// on return; every expert takes its m best tokens (perm_tok / gate by position, pos_of [T][E])
size_t ec_select_smem(int T);
cudaError_t ec_route(float* scores, const float* logit_bias, int T, int E, int m, int32_t* offsets,
                     int32_t* perm_tok, float* gate, int32_t* pos_of, cudaStream_t st);
cudaError_t ec_combine(int dtype, const float* y_perm, const int32_t* pos_of, const float* gate, const float* ys,
                       int T, int E, int d, long long rows_perm, void* y, uint32_t* err, cudaStream_t st);

// ---- combine
cudaError_t combine(int dtype, const float* y_perm, const int32_t* inv_pos, const float* gate, const float* ys,
                    int T, int d, int k, void* y, uint32_t* err, cudaStream_t st);

}  // namespace moe
