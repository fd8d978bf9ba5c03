// C ABI of libmoe (declared in include/moe.h): argument checks, workspace layout, and the
// chain route -> dispatch -> experts -> combine of the MoE FFN forward pass.
//
// Route, dispatch, compute and combine are the four moves of one MoE layer on the page
// "Mixture-of-Experts, from the router to the all-to-all" (section "Expert parallelism and
// the all-to-all"); on one GPU both exchanges are local: dispatch is a permutation of rows
// and combine a gate-weighted gather back to token order.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "moe.h"

namespace moe {

thread_local int g_launches = 0;

// Device error word (one per device that loads the library).
static __device__ uint32_t g_error_word;

// Device address of g_error_word, looked up once per device with that device current (in host
// code the symbol's name is only a host-side stand-in).  The table is shared by every host
// thread, so the lookup and the cache are under a lock.
static uint32_t* error_word() {
  static std::mutex mu;
  static uint32_t* ptr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) ptr[dev] = static_cast<uint32_t*>(p);
  }
  return ptr[dev];
}

static size_t align_up(size_t v) { return (v + 255) & ~size_t(255); }

static int esize(const moe_config& c) { return c.dtype == MOE_BF16 ? 2 : 4; }

// Slots per expert: ceil(T k c / E) for a capacity factor c > 0 (page "8.6 - Mixture of
// Experts (MoE)", section 3.2: capacity = T k / E * c), computed in double as (T k) * c / E;
// without a capacity factor, T k (nothing is ever dropped).
static int capacity_slots(const moe_config& c) {
  const long long pairs = (long long)c.T * c.k;
  if (!(c.capacity_factor > 0.0f)) return (int)pairs;
  const double slots = ceil((double)pairs * (double)c.capacity_factor / (double)c.E);
  return slots >= (double)pairs ? (int)pairs : (int)slots;
}

// Expert choice: tokens each expert takes, m = ceil(T k c / E) (c = capacity factor, 1 when
// none is set), at most T (page "Mixture-of-Experts Internals: A Systems Engineer's Field
// Manual", section 5.1).
static bool expert_choice(const moe_config& c) { return c.scoring == MOE_EXPERT_CHOICE; }

static int ec_slots(const moe_config& c) {
  const long long pairs = (long long)c.T * c.k;
  const double f = c.capacity_factor > 0.0f ? (double)c.capacity_factor : 1.0;
  const double m = ceil((double)pairs * f / (double)c.E);
  return m >= (double)c.T ? c.T : (int)m;
}

// Rows of the permuted activations: the (token, expert) pairs (T k), or E m under expert choice.
static long long pairs_of(const moe_config& c) {
  return expert_choice(c) ? (long long)c.E * ec_slots(c) : (long long)c.T * c.k;
}

// Bytes of each scratch region.
struct Sizes {
  size_t logits, idx, gate, counts, offsets, chunk, perm, inv, x_perm, h, y_perm, hs, ys, x_io, y_io;
  size_t stats_logits, stats_partial;   // moe_load_stats: logits [T][E] f32, per-block score sums
};

static Sizes sizes(const moe_config& c) {
  Sizes s{};
  const size_t T = (size_t)c.T, N = (size_t)pairs_of(c);
  s.logits = (c.E > 32 || expert_choice(c)) ? align_up(T * c.E * 4) : 0;
  s.idx = align_up(N * 4);
  s.gate = align_up(N * 4);
  s.counts = align_up((size_t)c.E * 4);
  s.offsets = align_up(((size_t)c.E + 1) * 4);
  s.chunk = 2 * align_up((size_t)dispatch_num_chunks((long long)N) * c.E * 4);
  s.perm = align_up(N * 4);
  s.inv = expert_choice(c) ? align_up(T * c.E * 4) : align_up(N * 4);   // inv_pos, or pos_of [T][E]
  s.x_perm = align_up(N * c.d * esize(c));
  s.h = align_up(N * c.d_ff * esize(c));
  s.y_perm = align_up(N * c.d * 4);
  s.hs = c.n_shared > 0 ? align_up(T * c.d_ff_shared * esize(c)) : 0;
  s.ys = c.n_shared > 0 ? align_up(T * c.d * 4) : 0;
  s.x_io = align_up(T * c.d * esize(c));
  s.y_io = align_up(T * c.d * esize(c));
  s.stats_logits = align_up(T * c.E * 4);
  s.stats_partial = align_up((size_t)stats_num_blocks(c.T) * c.E * 4);
  return s;
}

static size_t max4(size_t a, size_t b, size_t c, size_t d) {
  size_t m = a > b ? a : b;
  m = m > c ? m : c;
  return m > d ? m : d;
}

// Workspace of moe_forward: persistent regions, then one region reused by the stages in turn
// (router logits | dispatch chunk tables | h | shared h + shared y).
struct FwdLayout {
  size_t idx, gate, counts, offsets, perm, inv, x_perm, y_perm, x_io, y_io, shared_region, total;
};

static FwdLayout fwd_layout(const moe_config& c) {
  const Sizes s = sizes(c);
  FwdLayout L{};
  size_t o = 0;
  L.idx = o; o += s.idx;
  L.gate = o; o += s.gate;
  L.counts = o; o += s.counts;
  L.offsets = o; o += s.offsets;
  L.perm = o; o += s.perm;
  L.inv = o; o += s.inv;
  L.x_perm = o; o += s.x_perm;
  L.y_perm = o; o += s.y_perm;
  L.x_io = o; o += s.x_io;
  L.y_io = o; o += s.y_io;
  L.shared_region = o;
  o += max4(s.logits, s.chunk, s.h, s.hs + s.ys);
  // moe_load_stats uses the workspace from its start
  L.total = o > s.stats_logits + s.stats_partial ? o : s.stats_logits + s.stats_partial;
  return L;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }
static bool aligned4(const void* p) { return ((uintptr_t)p & 3) == 0; }

static moe_status check_config(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d <= 0 || c->d_ff <= 0 || c->E <= 0 || c->k <= 0 || c->k > c->E) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->scoring != MOE_SOFTMAX_TOPK_RENORM && c->scoring != MOE_SIGMOID_TOPK_NORM &&
      c->scoring != MOE_SOFTMAX_TOPK_PLAIN && c->scoring != MOE_EXPERT_CHOICE)
    return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || (c->n_shared > 0 && c->d_ff_shared <= 0)) return MOE_ERR_INVALID_ARG;
  if (!isfinite(c->capacity_factor) || c->capacity_factor < 0.0f) return MOE_ERR_INVALID_ARG;
  if (c->E > 1024) return MOE_ERR_UNSUPPORTED;
  if (c->scoring == MOE_EXPERT_CHOICE) {
    // one block per expert holds the T scores of its column in shared memory
    if ((size_t)c->T * 4 > 200 * 1024) return MOE_ERR_UNSUPPORTED;
    if (c->dtype == MOE_F32 && c->d % 4) return MOE_ERR_UNSUPPORTED;
  } else if (c->k > 32) {
    return MOE_ERR_UNSUPPORTED;
  }
  const long long N = pairs_of(*c);
  if (N >= (1LL << 31) - 256 || (long long)c->T * c->k >= (1LL << 31) - 256) return MOE_ERR_UNSUPPORTED;
  if (c->dtype == MOE_BF16) {
    if (c->d % 8 || c->d_ff % 8) return MOE_ERR_UNSUPPORTED;
    if (c->n_shared > 0 && c->d_ff_shared % 8) return MOE_ERR_UNSUPPORTED;
  } else {
    // CUDA-core path: the grid covers rows / 64 + E row tiles in y.
    if (N / 64 + c->E + 1 > 65535 || (long long)c->T / 64 + 1 > 65535) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

static moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                          \
  do {                                         \
    const moe_status st__ = (expr);            \
    if (st__ != MOE_OK) return st__;           \
  } while (0)

#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

// ---------------------------------------------------------------- stages (checked inputs)

// Router logits [T][E] float32 (no bias): tensor cores for bf16 when E is a multiple of 8,
// CUDA cores otherwise.
static moe_status router_logits(const moe_config& c, const void* x, const void* W_g, float* logits, cudaStream_t st) {
  if (c.dtype == MOE_BF16 && c.E % 8 == 0 && aligned16(W_g))
    return cuda_status(tc_matmul_f32(x, c.T, c.d, W_g, 1, c.E, nullptr, 1, c.T, 0, logits, c.E, 0, error_word(), st));
  return cuda_status(route_logits_simt(c.dtype, x, W_g, c.T, c.d, c.E, logits, st));
}

static moe_status stage_route(const moe_config& c, const void* x, const void* W_g, const float* lb, const float* sb,
                              int32_t* idx, float* gate, float* logits, cudaStream_t st) {
  uint32_t* err = error_word();
  if (c.E <= 32) {
    return cuda_status(route_fused(c.dtype, x, W_g, lb, sb, c.T, c.d, c.E, c.k, c.scoring, idx, gate, err, st));
  }
  MOE_TRY(router_logits(c, x, W_g, logits, st));
  return cuda_status(route_topk(logits, lb, sb, c.T, c.E, c.k, c.scoring, idx, gate, err, st));
}

// Expert choice: logits -> per-token softmax (in place in `scores`) -> every expert's m tokens.
static moe_status stage_route_ec(const moe_config& c, const void* x, const void* W_g, const float* lb, float* scores,
                                 int32_t* offsets, int32_t* perm, float* gate, int32_t* pos_of, cudaStream_t st) {
  MOE_TRY(router_logits(c, x, W_g, scores, st));
  return cuda_status(ec_route(scores, lb, c.T, c.E, ec_slots(c), offsets, perm, gate, pos_of, st));
}

static moe_status stage_dispatch(const moe_config& c, const int32_t* idx, const void* x, int32_t* counts,
                                 int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm, int32_t* chunk_counts,
                                 int32_t* chunk_base, cudaStream_t st) {
  MOE_CUDA(dispatch_indices(idx, c.T, c.k, c.E, capacity_slots(c), chunk_counts, chunk_base, counts, offsets, perm,
                            inv, error_word(), st, nullptr));
  return cuda_status(scatter_rows(x, c.T, c.k, inv, pairs_of(c), c.d, esize(c), x_perm, error_word(), st));
}

static moe_status stage_w12(const moe_config& c, const void* x_perm, const int32_t* offsets, const void* W1,
                            const void* W2, void* h, cudaStream_t st) {
  const long long N = pairs_of(c);
  if (c.dtype == MOE_BF16)
    return cuda_status(tc_swiglu(x_perm, N, c.d, W1, W2, c.E, c.d_ff, offsets, c.E, 0, 0, h, error_word(), st));
  return cuda_status(simt_swiglu_f32((const float*)x_perm, (int)N, c.d, (const float*)W1, (const float*)W2, c.d_ff,
                                     offsets, c.E, 0, (long long)c.d * c.d_ff, 0, (float*)h, error_word(), st));
}

static moe_status stage_w3(const moe_config& c, const void* h, const int32_t* offsets, const void* W3, float* y_perm,
                           cudaStream_t st) {
  const long long N = pairs_of(c);
  if (c.dtype == MOE_BF16)
    return cuda_status(tc_matmul_f32(h, N, c.d_ff, W3, c.E, c.d, offsets, c.E, 0, 0, y_perm, c.d, 0, error_word(), st));
  return cuda_status(simt_matmul_f32((const float*)h, (int)N, c.d_ff, (const float*)W3, c.d, offsets, c.E, 0,
                                     (long long)c.d_ff * c.d, 0, y_perm, 0, error_word(), st));
}

static moe_status stage_shared(const moe_config& c, const void* x, const void* Ws1, const void* Ws2, const void* Ws3,
                               void* hs, float* ys, cudaStream_t st) {
  for (int s = 0; s < c.n_shared; ++s) {
    if (c.dtype == MOE_BF16) {
      MOE_CUDA(tc_swiglu(x, c.T, c.d, Ws1, Ws2, c.n_shared, c.d_ff_shared, nullptr, 1, c.T, s, hs, error_word(), st));
      MOE_CUDA(tc_matmul_f32(hs, c.T, c.d_ff_shared, Ws3, c.n_shared, c.d, nullptr, 1, c.T, s, ys, c.d, s > 0,
                             error_word(), st));
    } else {
      MOE_CUDA(simt_swiglu_f32((const float*)x, c.T, c.d, (const float*)Ws1, (const float*)Ws2, c.d_ff_shared, nullptr,
                               1, c.T, (long long)c.d * c.d_ff_shared, s, (float*)hs, error_word(), st));
      MOE_CUDA(simt_matmul_f32((const float*)hs, c.T, c.d_ff_shared, (const float*)Ws3, c.d, nullptr, 1, c.T,
                               (long long)c.d_ff_shared * c.d, s, ys, s > 0, error_word(), st));
    }
  }
  return MOE_OK;
}

static moe_status stage_combine(const moe_config& c, const float* y_perm, const int32_t* inv, const float* gate,
                                const float* ys, void* y, cudaStream_t st) {
  return cuda_status(combine(c.dtype, y_perm, inv, gate, ys, c.T, c.d, c.k, y, error_word(), st));
}

static moe_status stage_combine_ec(const moe_config& c, const float* y_perm, const int32_t* pos_of, const float* gate,
                                   const float* ys, void* y, cudaStream_t st) {
  return cuda_status(ec_combine(c.dtype, y_perm, pos_of, gate, ys, c.T, c.E, c.d, pairs_of(c), y, error_word(), st));
}

static moe_status check_weights(const moe_config& c, const void* W1, const void* W2, const void* W3) {
  if (!W1 || !W2 || !W3) return MOE_ERR_INVALID_ARG;
  if (!aligned16(W1) || !aligned16(W2) || !aligned16(W3)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

static moe_status check_shared(const moe_config& c, const void* Ws1, const void* Ws2, const void* Ws3) {
  if (c.n_shared == 0) return MOE_OK;
  if (!Ws1 || !Ws2 || !Ws3) return MOE_ERR_INVALID_ARG;
  if (!aligned16(Ws1) || !aligned16(Ws2) || !aligned16(Ws3)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

static moe_status forward_impl(const moe_config* cfg, const void* x, const void* W_g, const float* lb,
                               const float* sb, const void* W1, const void* W2, const void* W3, const void* Ws1,
                               const void* Ws2, const void* Ws3, void* y, int32_t* idx_out, int32_t* counts_out,
                               void* ws, size_t ws_bytes, cudaStream_t st, cudaEvent_t* ev) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (c.T == 0) return MOE_OK;
  if (!x || !W_g || !y || !aligned16(x) || !aligned16(y) || !aligned4(W_g)) return MOE_ERR_INVALID_ARG;
  if ((lb && !aligned4(lb)) || (sb && !aligned4(sb))) return MOE_ERR_INVALID_ARG;
  if ((idx_out && !aligned4(idx_out)) || (counts_out && !aligned4(counts_out))) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_weights(c, W1, W2, W3));
  MOE_TRY(check_shared(c, Ws1, Ws2, Ws3));
  if (expert_choice(c) && (sb || idx_out || counts_out)) return MOE_ERR_UNSUPPORTED;
  const FwdLayout L = fwd_layout(c);
  if (!ws || !aligned16(ws)) return ws ? MOE_ERR_INVALID_ARG : MOE_ERR_WORKSPACE;
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const Sizes s = sizes(c);
  int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(w + L.idx);
  float* gate = reinterpret_cast<float*>(w + L.gate);
  int32_t* counts = counts_out ? counts_out : reinterpret_cast<int32_t*>(w + L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(w + L.perm);
  int32_t* inv = reinterpret_cast<int32_t*>(w + L.inv);
  void* x_perm = w + L.x_perm;
  float* y_perm = reinterpret_cast<float*>(w + L.y_perm);
  uint8_t* R = w + L.shared_region;
  float* logits = reinterpret_cast<float*>(R);
  int32_t* chunk_counts = reinterpret_cast<int32_t*>(R);
  int32_t* chunk_base = reinterpret_cast<int32_t*>(R + s.chunk / 2);
  void* h = R;
  void* hs = R;
  float* ys = c.n_shared > 0 ? reinterpret_cast<float*>(R + s.hs) : nullptr;

  auto mark = [&](int i) -> moe_status {
    if (ev && ev[i]) return cuda_status(cudaEventRecord(ev[i], st));
    return MOE_OK;
  };
  const bool ec = expert_choice(c);
  MOE_TRY(mark(0));
  if (ec) {
    MOE_TRY(stage_route_ec(c, x, W_g, lb, logits, offsets, perm, gate, inv, st));
    MOE_TRY(mark(1));
    MOE_CUDA(gather_rows(x, c.T, perm, pairs_of(c), offsets + c.E, c.d, esize(c), x_perm, error_word(), st));
  } else {
    MOE_TRY(stage_route(c, x, W_g, lb, sb, idx, gate, logits, st));
    MOE_TRY(mark(1));
    MOE_TRY(stage_dispatch(c, idx, x, counts, offsets, perm, inv, x_perm, chunk_counts, chunk_base, st));
  }
  MOE_TRY(mark(2));
  MOE_TRY(stage_w12(c, x_perm, offsets, W1, W2, h, st));
  MOE_TRY(mark(3));
  MOE_TRY(stage_w3(c, h, offsets, W3, y_perm, st));
  MOE_TRY(mark(4));
  MOE_TRY(stage_shared(c, x, Ws1, Ws2, Ws3, hs, ys, st));
  MOE_TRY(mark(5));
  if (ec) {
    MOE_TRY(stage_combine_ec(c, y_perm, inv, gate, ys, y, st));
  } else {
    MOE_TRY(stage_combine(c, y_perm, inv, gate, ys, y, st));
  }
  MOE_TRY(mark(6));
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return fwd_layout(*cfg).total;
}

moe_status moe_route(const moe_config* cfg, const void* x, const void* W_g, const float* logit_bias,
                     const float* sel_bias, int32_t* topk_idx, float* topk_gate, void* ws, size_t ws_bytes,
                     moe_stream_t stream) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (expert_choice(c)) return MOE_ERR_UNSUPPORTED;   // see moe_route_expert_choice
  if (c.T == 0) return MOE_OK;
  if (!x || !W_g || !topk_idx || !topk_gate) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned4(W_g) || !aligned4(topk_idx) || !aligned4(topk_gate)) return MOE_ERR_INVALID_ARG;
  if ((logit_bias && !aligned4(logit_bias)) || (sel_bias && !aligned4(sel_bias))) return MOE_ERR_INVALID_ARG;
  const Sizes s = sizes(c);
  if (s.logits > 0) {
    if (!ws) return MOE_ERR_WORKSPACE;
    if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < s.logits) return MOE_ERR_WORKSPACE;
  }
  return stage_route(c, x, W_g, logit_bias, sel_bias, topk_idx, topk_gate, static_cast<float*>(ws),
                     (cudaStream_t)stream);
}

moe_status moe_load_stats(const moe_config* cfg, const void* x, const void* W_g, const float* logit_bias,
                          const int32_t* counts, float alpha, float* f, float* P, float* summary, void* ws,
                          size_t ws_bytes, moe_stream_t stream) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (c.T == 0) return MOE_ERR_INVALID_ARG;   // the statistics are means over the batch
  if (!x || !W_g || !counts || !f || !P || !summary) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned4(W_g) || !aligned4(counts) || !aligned4(f) || !aligned4(P) || !aligned4(summary))
    return MOE_ERR_INVALID_ARG;
  if (logit_bias && !aligned4(logit_bias)) return MOE_ERR_INVALID_ARG;
  if (!isfinite(alpha)) return MOE_ERR_INVALID_ARG;
  const Sizes s = sizes(c);
  if (!ws) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < s.stats_logits + s.stats_partial) return MOE_ERR_WORKSPACE;
  const cudaStream_t st = (cudaStream_t)stream;
  float* logits = static_cast<float*>(ws);
  float* partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + s.stats_logits);
  MOE_TRY(router_logits(c, x, W_g, logits, st));
  return cuda_status(load_stats(logits, logit_bias, counts, c.T, c.k, c.E, c.scoring, alpha, partial, f, P, summary,
                                st));
}

moe_status moe_update_sel_bias(const moe_config* cfg, const int32_t* counts, float gamma, float* sel_bias,
                               moe_stream_t stream) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  if (!counts || !sel_bias || !aligned4(counts) || !aligned4(sel_bias)) return MOE_ERR_INVALID_ARG;
  if (!(gamma >= 0.0f) || !isfinite(gamma)) return MOE_ERR_INVALID_ARG;
  return cuda_status(update_sel_bias(counts, cfg->T, cfg->k, cfg->E, gamma, sel_bias, (cudaStream_t)stream));
}

moe_status moe_dispatch(const moe_config* cfg, const int32_t* topk_idx, const void* x, int32_t* counts,
                        int32_t* offsets, int32_t* perm_tok, int32_t* inv_pos, void* x_perm, void* ws,
                        size_t ws_bytes, moe_stream_t stream) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (expert_choice(c)) return MOE_ERR_UNSUPPORTED;   // see moe_route_expert_choice
  if (c.T == 0) return MOE_OK;
  if (!topk_idx || !x || !counts || !offsets || !perm_tok || !inv_pos || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned4(topk_idx) || !aligned4(counts) || !aligned4(offsets) || !aligned4(perm_tok) || !aligned4(inv_pos) ||
      !aligned16(x) || !aligned16(x_perm))
    return MOE_ERR_INVALID_ARG;
  const Sizes s = sizes(c);
  if (!ws) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < s.chunk) return MOE_ERR_WORKSPACE;
  int32_t* chunk_counts = static_cast<int32_t*>(ws);
  int32_t* chunk_base = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + s.chunk / 2);
  return stage_dispatch(c, topk_idx, x, counts, offsets, perm_tok, inv_pos, x_perm, chunk_counts, chunk_base,
                        (cudaStream_t)stream);
}

moe_status moe_experts(const moe_config* cfg, const void* x_perm, const int32_t* offsets, const void* W1,
                       const void* W2, const void* W3, float* y_perm, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (c.T == 0) return MOE_OK;
  if (!x_perm || !offsets || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned4(offsets) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_weights(c, W1, W2, W3));
  const Sizes s = sizes(c);
  if (!ws) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < s.h) return MOE_ERR_WORKSPACE;
  const cudaStream_t st = (cudaStream_t)stream;
  MOE_TRY(stage_w12(c, x_perm, offsets, W1, W2, ws, st));
  return stage_w3(c, ws, offsets, W3, y_perm, st);
}

moe_status moe_combine(const moe_config* cfg, const float* y_perm, const int32_t* inv_pos, const float* topk_gate,
                       const void* x, const void* Ws1, const void* Ws2, const void* Ws3, void* y, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (expert_choice(c)) return MOE_ERR_UNSUPPORTED;   // see moe_route_expert_choice
  if (c.T == 0) return MOE_OK;
  if (!y_perm || !inv_pos || !topk_gate || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned4(inv_pos) || !aligned4(topk_gate) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  const cudaStream_t st = (cudaStream_t)stream;
  float* ys = nullptr;
  if (c.n_shared > 0) {
    if (!x || !aligned16(x)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_shared(c, Ws1, Ws2, Ws3));
    const Sizes s = sizes(c);
    if (!ws) return MOE_ERR_WORKSPACE;
    if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < s.hs + s.ys) return MOE_ERR_WORKSPACE;
    ys = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + s.hs);
    MOE_TRY(stage_shared(c, x, Ws1, Ws2, Ws3, ws, ys, st));
  }
  return stage_combine(c, y_perm, inv_pos, topk_gate, ys, y, st);
}

moe_status moe_route_expert_choice(const moe_config* cfg, const void* x, const void* W_g, const float* logit_bias,
                                   int32_t* offsets, int32_t* perm_tok, float* gate, int32_t* pos_of, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (!expert_choice(c)) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if (!x || !W_g || !offsets || !perm_tok || !gate || !pos_of) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned4(W_g) || !aligned4(offsets) || !aligned4(perm_tok) || !aligned4(gate) ||
      !aligned4(pos_of))
    return MOE_ERR_INVALID_ARG;
  if (logit_bias && !aligned4(logit_bias)) return MOE_ERR_INVALID_ARG;
  const Sizes s = sizes(c);
  if (!ws) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < s.logits) return MOE_ERR_WORKSPACE;
  return stage_route_ec(c, x, W_g, logit_bias, static_cast<float*>(ws), offsets, perm_tok, gate, pos_of,
                        (cudaStream_t)stream);
}

moe_status moe_combine_expert_choice(const moe_config* cfg, const float* y_perm, const float* gate,
                                     const int32_t* pos_of, const void* x, const void* Ws1, const void* Ws2,
                                     const void* Ws3, void* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (!expert_choice(c)) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if (!y_perm || !gate || !pos_of || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned4(gate) || !aligned4(pos_of) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  const cudaStream_t st = (cudaStream_t)stream;
  float* ys = nullptr;
  if (c.n_shared > 0) {
    if (!x || !aligned16(x)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_shared(c, Ws1, Ws2, Ws3));
    const Sizes s = sizes(c);
    if (!ws) return MOE_ERR_WORKSPACE;
    if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < s.hs + s.ys) return MOE_ERR_WORKSPACE;
    ys = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + s.hs);
    MOE_TRY(stage_shared(c, x, Ws1, Ws2, Ws3, ws, ys, st));
  }
  return stage_combine_ec(c, y_perm, pos_of, gate, ys, y, st);
}

moe_status moe_forward(const moe_config* cfg, const void* x, const void* W_g, const float* logit_bias,
                       const float* sel_bias, const void* W1, const void* W2, const void* W3, const void* Ws1,
                       const void* Ws2, const void* Ws3, void* y, int32_t* topk_idx_out, int32_t* counts_out,
                       void* ws, size_t ws_bytes, moe_stream_t stream) {
  return forward_impl(cfg, x, W_g, logit_bias, sel_bias, W1, W2, W3, Ws1, Ws2, Ws3, y, topk_idx_out, counts_out, ws,
                      ws_bytes, (cudaStream_t)stream, nullptr);
}

moe_status moe_forward_profiled(const moe_config* cfg, const void* x, const void* W_g, const float* logit_bias,
                                const float* sel_bias, const void* W1, const void* W2, const void* W3,
                                const void* Ws1, const void* Ws2, const void* Ws3, void* y, int32_t* topk_idx_out,
                                int32_t* counts_out, void* ws, size_t ws_bytes, moe_stream_t stream,
                                moe_event_t* events) {
  return forward_impl(cfg, x, W_g, logit_bias, sel_bias, W1, W2, W3, Ws1, Ws2, Ws3, y, topk_idx_out, counts_out, ws,
                      ws_bytes, (cudaStream_t)stream, reinterpret_cast<cudaEvent_t*>(events));
}

static moe_status forward_host_impl(const moe_config* cfg, const void* x_host, const void* W_g,
                                    const float* logit_bias, const float* sel_bias, const void* W1, const void* W2,
                                    const void* W3, const void* Ws1, const void* Ws2, const void* Ws3, void* y_host,
                                    void* ws, size_t ws_bytes, cudaStream_t st, bool wait) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (c.T == 0) return MOE_OK;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  const FwdLayout L = fwd_layout(c);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  void* x_dev = w + L.x_io;
  void* y_dev = w + L.y_io;
  const size_t bytes = (size_t)c.T * c.d * esize(c);
  MOE_CUDA(cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, st));
  const moe_status r = forward_impl(cfg, x_dev, W_g, logit_bias, sel_bias, W1, W2, W3, Ws1, Ws2, Ws3, y_dev, nullptr,
                                    nullptr, ws, ws_bytes, st, nullptr);
  if (r != MOE_OK) return r;
  MOE_CUDA(cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, st));
  return wait ? cuda_status(cudaStreamSynchronize(st)) : MOE_OK;
}

}  // extern "C"

extern "C" {

moe_status moe_forward_host(const moe_config* cfg, const void* x_host, const void* W_g, const float* logit_bias,
                            const float* sel_bias, const void* W1, const void* W2, const void* W3, const void* Ws1,
                            const void* Ws2, const void* Ws3, void* y_host, void* ws, size_t ws_bytes,
                            moe_stream_t stream) {
  return forward_host_impl(cfg, x_host, W_g, logit_bias, sel_bias, W1, W2, W3, Ws1, Ws2, Ws3, y_host, ws, ws_bytes,
                           (cudaStream_t)stream, true);
}

moe_status moe_forward_host_async(const moe_config* cfg, const void* x_host, const void* W_g, const float* logit_bias,
                                  const float* sel_bias, const void* W1, const void* W2, const void* W3,
                                  const void* Ws1, const void* Ws2, const void* Ws3, void* y_host, void* ws,
                                  size_t ws_bytes, moe_stream_t stream) {
  return forward_host_impl(cfg, x_host, W_g, logit_bias, sel_bias, W1, W2, W3, Ws1, Ws2, Ws3, y_host, ws, ws_bytes,
                           (cudaStream_t)stream, false);
}

moe_status moe_get_device_error(moe_stream_t stream, uint32_t* word) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_error_word, sizeof(w)) != cudaSuccess) return MOE_ERR_CUDA;
  if (word) *word = w;
  if (w != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_ERR_DEVICE;
  }
  return MOE_OK;
}

int32_t moe_last_launch_count(void) { return g_launches; }

moe_status moe_test_pipeline_fault(uint64_t wait_limit_ns) {
  if (wait_limit_ns == 0 || wait_limit_ns > kWaitLimitNs) return MOE_ERR_INVALID_ARG;
  arm_pipeline_fault((unsigned long long)wait_limit_ns);
  return MOE_OK;
}

const char* moe_status_string(moe_status status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE: return "device-side error flagged";
  }
  return "unknown status";
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// moe_dispatch_static: moe_dispatch with its scratch in a fixed device array owned by the
// library, for callers that cannot allocate device memory (see include/moe.h).

namespace moe {

constexpr size_t kStaticScratchInts = MOE_DISPATCH_STATIC_SCRATCH_BYTES / sizeof(int32_t);

// The scratch itself: chunk counts followed by chunk positions.  Each dispatch call fully
// rewrites the parts it reads (every chunk row of both tables), so nothing needs clearing.
static __device__ __align__(256) int32_t g_dispatch_scratch[kStaticScratchInts];

// Device address of g_dispatch_scratch, looked up once per device with that device current.
// In host code the array's name is only a host-side stand-in and must not reach a kernel.
static int32_t* dispatch_scratch_ptr() {
  static std::mutex mu;
  static int32_t* ptr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    int32_t* p = nullptr;
    if (cudaGetSymbolAddress((void**)&p, g_dispatch_scratch) != cudaSuccess) return nullptr;
    ptr[dev] = p;
  }
  return ptr[dev];
}

}  // namespace moe

extern "C" moe_status moe_dispatch_static(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                                          int32_t* counts, int32_t* offsets, int32_t* perm_tok, int32_t* inv_pos,
                                          void* x_perm, moe_stream_t stream) {
  g_launches = 0;
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (expert_choice(c)) return MOE_ERR_UNSUPPORTED;   // see moe_route_expert_choice
  if (c.T == 0) return MOE_OK;
  if (!topk_idx || !x || !counts || !offsets || !perm_tok || !inv_pos || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned4(topk_idx) || !aligned4(counts) || !aligned4(offsets) || !aligned4(perm_tok) || !aligned4(inv_pos) ||
      !aligned16(x) || !aligned16(x_perm))
    return MOE_ERR_INVALID_ARG;
  const size_t table_ints = (size_t)dispatch_num_chunks((long long)c.T * c.k) * (size_t)c.E;
  if (2 * table_ints > kStaticScratchInts) return MOE_ERR_UNSUPPORTED;
  int32_t* scratch = dispatch_scratch_ptr();
  if (!scratch) return MOE_ERR_CUDA;
  return stage_dispatch(c, topk_idx, x, counts, offsets, perm_tok, inv_pos, x_perm, scratch, scratch + table_ints,
                        (cudaStream_t)stream);
}
