// Grouped bf16 GEMM on the sm_103a tensor cores (tcgen05.mma, accumulators in TMEM, operands
// staged by TMA), for the expert matmuls of the MoE layer: one group per expert, each group a
// contiguous block of rows of the permuted activations (page "Mixture of Experts: What
// Actually Happens When a Token Hits the Router", Step 3: each expert processes its block as
// one dense matmul; page "8.6 - Mixture of Experts (MoE)", section 2: the SwiGLU expert).
//
// Two epilogues:
//   EPI_SWIGLU  h = (X W1) * SiLU(X W2), written as bf16.  An accumulator tile holds X W1 and
//               X W2 for the same output columns, so the pair is finished on chip.
//   EPI_F32     out (+)= X W, written as float32 (expert W3, shared W3, router logits).
//
// Three kernels, all persistent (one CTA per SM, or one CTA pair per two SMs), all reading the
// group sizes on the device from `offsets` (nothing is synchronised with the host):
//   grouped_gemm_kernel        1 CTA, 128 token rows x 256 MMA columns per tile, 4 x 48 KB
//                              stages.  For small expert blocks (decode, < 128 rows).
//   grouped_gemm_pair_kernel   a cluster of 2 CTAs shares one tcgen05.mma.cta_group::2 of
//                              256 token rows x 256 columns; each CTA loads its 128 rows and
//                              half of the weight columns; 6 x 32 KB stages.  W1/W2 + SwiGLU
//                              of one dense block of >= 512 rows (the shared experts).
//   grouped_gemm_tpair_kernel  the CTA pair with the roles swapped: weight features along the
//                              MMA's M (256), tokens along N in steps of 16 up to 256, so the
//                              last tile of a block carries at most 15 padding rows.  With
//                              "wide" tiles (an expert's last tile takes up to 32 more tokens)
//                              W1/W2 + SwiGLU for blocks averaging >= 128 rows and the
//                              float32-output GEMMs for 128..511; without them the float32
//                              GEMMs for blocks averaging >= 512 rows.
// Tiles are walked as (group, column tile, row tile), row tiles fastest, so the CTAs that run
// at the same time share one weight tile and the weights are streamed from HBM about once.
// Row tiles may run past the end of their group: the extra rows belong to the next group (or
// lie beyond the matrix and are zero-filled by TMA) and their results are not stored.
//
// Warp roles (256 threads): warp 0 lane 0 issues the TMA loads into the shared-memory ring;
// warp 1 lane 0 issues tcgen05.mma into one of two 256-column TMEM accumulators; warps 4-7
// drain the other accumulator (tcgen05.ld) and store; warp 2 owns the TMEM allocation; warp 3
// builds the group table.  Every wait is bounded (kWaitLimitNs, or a test hook's shorter
// limit) and on a timeout sets the device error word and unwinds.
#include <cudaTypedefs.h>
#include <atomic>
#include <mutex>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace tc {

constexpr int BM = 128;                   // rows per tile (MMA M)
constexpr int BN = 256;                   // MMA N (EPI_F32: output columns; SWIGLU: 128 + 128)
constexpr int BK = 64;                    // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int A_TILE = BM * BK * 2;       // 16 KB, K-major, 128B-swizzled
constexpr int B_SUB = BK * 64 * 2;        // 8 KB: 64 k-rows x 64 n-columns, MN-major, swizzled
constexpr int B_TILE = 4 * B_SUB;         // 32 KB
constexpr int STAGE = A_TILE + B_TILE;    // 48 KB
constexpr int MAX_GROUPS = 1024;
constexpr int TMEM_COLS = 512;            // two 256-column fp32 accumulators
constexpr int THREADS = 256;
constexpr uint32_t IDESC = idesc_bf16_f32_kmaj_a_mnmaj_b<BM, BN>();

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort;
  int tile_start[MAX_GROUPS + 1];
  int row_off[MAX_GROUPS + 1];
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE + sizeof(Ctrl);
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct Tile {
  int g, row0, row_end, n_tile;
  int tile_end;   // end of this tile's rows: row0 + TILE_M, or the group's end for its last tile
};

// Row tiles of a group of `rows` rows: tiles of TILE_M rows, except that the last one also takes
// up to WIDE extra rows (so a group of TILE_M + WIDE rows is one tile, not a full tile and a
// short one).
template <int TILE_M, int WIDE = 0>
__host__ __device__ __forceinline__ int row_tiles(int rows) {
  return rows <= TILE_M + WIDE ? 1 : (rows - WIDE + TILE_M - 1) / TILE_M;
}

template <int TILE_M = BM, int WIDE = 0, typename C>
__device__ __forceinline__ Tile decode_tile(const C& c, int G, int t) {
  int lo = 0, hi = G;  // largest g with tile_start[g] <= t (always a non-empty group)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (c.tile_start[mid] <= t) lo = mid; else hi = mid;
  }
  Tile r;
  r.g = lo;
  const int rows = c.row_off[lo + 1] - c.row_off[lo];
  const int mt = row_tiles<TILE_M, WIDE>(rows);
  const int local = t - c.tile_start[lo];
  r.n_tile = local / mt;
  const int m = local - r.n_tile * mt;
  r.row0 = c.row_off[lo] + m * TILE_M;
  r.row_end = c.row_off[lo + 1];
  r.tile_end = m == mt - 1 ? r.row_end : r.row0 + TILE_M;
  return r;
}

// Bounds-checking build: the rows a tile stores lie inside the output ([0, rows_cap]); the group
// table clamps the offsets it reads, so this only fails if that clamp is broken.
__device__ __forceinline__ void debug_tile_rows(const Tile& tl, const GemmArgs& a) {
  debug_bounds(tl.row0 >= 0 && tl.row0 <= tl.row_end && tl.row_end <= a.rows_cap, a.err);
}

// Warp-wide: the group table of a persistent grouped GEMM.  row_off[g] = offsets[g] clamped
// to the output's rows (a violation is flagged), tile_start[g] = first tile of group g, with
// row_tiles(rows) row tiles times n_tiles column tiles per non-empty group.
template <int TILE_M, int WIDE = 0, typename C>
__device__ __forceinline__ void build_group_table(C& c, const GemmArgs& a, int G, int lane) {
  bool bad = false;
  for (int base = 0; base <= G; base += 32) {
    const int g = base + lane;
    if (g <= G) {
      int off = a.offsets ? __ldg(a.offsets + g) : (g == 0 ? 0 : a.M);
      if (off < 0 || off > a.rows_cap) { bad = true; off = off < 0 ? 0 : a.rows_cap; }
      c.row_off[g] = off;
    }
  }
  __syncwarp();
  int carry = 0;
  for (int base = 0; base < G; base += 32) {
    const int g = base + lane;
    int tiles = 0;
    if (g < G) {
      const int rows = c.row_off[g + 1] - c.row_off[g];
      if (rows < 0) bad = true;
      tiles = rows > 0 ? row_tiles<TILE_M, WIDE>(rows) * a.n_tiles : 0;
    }
    int v = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (g < G) c.tile_start[g] = carry + v - tiles;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) c.tile_start[G] = carry;
  if (__any_sync(0xffffffffu, bad) && lane == 0) flag_error(a.err, ERR_OFFSETS);
}

// Epilogue of one accumulator tile for the 32 rows of this warp's TMEM lane quarter: read the
// 256 fp32 columns at `taddr` (tcgen05.ld, warp-collective) and store row `row` when `valid`.
//   EPI_SWIGLU: columns 0-127 hold X W1, 128-255 the same columns of X W2; h = u * SiLU(v) in bf16.
//   EPI_F32:    256 output columns in float32, added to the existing values when accumulating.
template <int EPI>
__device__ __forceinline__ void drain_tile(const GemmArgs& a, uint32_t taddr, int row, bool valid, int n_tile) {
  if (EPI == EPI_SWIGLU) {
    uint16_t* out = reinterpret_cast<uint16_t*>(a.out);
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t u[32], v[32];
      tmem_ld_32cols(taddr + ch * 32, u);
      tmem_ld_32cols(taddr + 128 + ch * 32, v);
      tmem_ld_wait();
      const int col0 = n_tile * (BN / 2) + ch * 32;
      if (valid) {
        uint32_t hp[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
          const float v0 = __uint_as_float(v[2 * i]), v1 = __uint_as_float(v[2 * i + 1]);
          const float h0 = u0 * __fdividef(v0, 1.0f + __expf(-v0));
          const float h1 = u1 * __fdividef(v1, 1.0f + __expf(-v1));
          hp[i] = pack_bf16x2(h0, h1);
        }
        uint16_t* dst = out + (size_t)row * a.ldo + col0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (col0 + 8 * j + 8 <= a.N)
            *reinterpret_cast<uint4*>(dst + 8 * j) = make_uint4(hp[4 * j], hp[4 * j + 1], hp[4 * j + 2], hp[4 * j + 3]);
      }
    }
  } else {
    float* out = reinterpret_cast<float*>(a.out);
#pragma unroll 1
    for (int ch = 0; ch < 8; ++ch) {
      uint32_t r[32];
      tmem_ld_32cols(taddr + ch * 32, r);
      tmem_ld_wait();
      const int col0 = n_tile * BN + ch * 32;
      if (valid) {
        float* dst = out + (size_t)row * a.ldo + col0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (col0 + 4 * j + 4 <= a.N) {
            float4 v = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                   __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            if (a.accumulate) {
              const float4 o = *reinterpret_cast<const float4*>(dst + 4 * j);
              v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
            }
            *reinterpret_cast<float4*>(dst + 4 * j) = v;
          }
        }
      }
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  Ctrl& c = *reinterpret_cast<Ctrl*>(smem + (size_t)STAGES * STAGE);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.offsets ? a.G : 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c.tfull[b], 1);
      mbar_init(&c.tempty[b], 4);
    }
    mbar_init(&c.drain, 1);
    c.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB0);
    prefetch_tensormap(&tmB1);
  }
  if (warp == 2) {
    tmem_alloc(&c.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  pdl_wait();      // offsets, A and the outputs belong to earlier kernels of the stream
  pdl_trigger();
  if (warp == 3) build_group_table<BM>(c, a, G, lane);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem = c.tmem_base;
  const int total = c.tile_start[G];
  const int num_kb = (a.K + BK - 1) / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      int s = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      bool ok = !a.starve;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode_tile(c, G, t);
        const int z = a.offsets ? tl.g : a.b_z;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&c.empty[s], phase ^ 1, &c.abort, a.wait_limit_ns)) {
            flag_error(a.err, ERR_WAIT_PRODUCER);
            c.abort = 1;
            ok = false;
            break;
          }
          uint8_t* sa = stages + (size_t)s * STAGE;
          uint8_t* sb = sa + A_TILE;
          mbar_arrive_expect_tx(&c.full[s], STAGE);
          armed |= 1u << s;
          armed_parity = (armed_parity & ~(1u << s)) | (phase << s);
          const int k0 = kb * BK;
          tma_load_2d(sa, &tmA, &c.full[s], k0, tl.row0);
          if (EPI == EPI_SWIGLU) {
            const int n0 = tl.n_tile * (BN / 2);
            tma_load_3d(sb + 0 * B_SUB, &tmB0, &c.full[s], n0, k0, z);
            tma_load_3d(sb + 1 * B_SUB, &tmB0, &c.full[s], n0 + 64, k0, z);
            tma_load_3d(sb + 2 * B_SUB, &tmB1, &c.full[s], n0, k0, z);
            tma_load_3d(sb + 3 * B_SUB, &tmB1, &c.full[s], n0 + 64, k0, z);
          } else {
            const int n0 = tl.n_tile * BN;
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_3d(sb + j * B_SUB, &tmB0, &c.full[s], n0 + 64 * j, k0, z);
          }
          if (++s == STAGES) { s = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA's shared memory is released.
        volatile int never = 0;
        for (int i = 0; i < STAGES; ++i)
          if (armed & (1u << i)) mbar_wait(&c.full[i], (armed_parity >> i) & 1u, &never, a.wait_limit_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      int s = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      // Stage-0 descriptors; a stage or K step adds its byte offset / 16 to the address field
      // (shared addresses stay below 2^18, so the field never carries).
      const uint64_t ad_base = sdesc_sw128(smem_addr(stages), 16, 1024);
      const uint64_t bd_base = sdesc_sw128(smem_addr(stages) + A_TILE, B_SUB, 1024);
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait(&c.tempty[buf], (use & 1u) ^ 1u, &c.abort, a.wait_limit_ns)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&c.full[s], phase, &c.abort, a.wait_limit_ns)) { ok = false; break; }
          tc_fence_after_sync();
          const uint64_t soff = (uint64_t)(((uint32_t)s * (uint32_t)STAGE) >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A: K-major rows of 128 B; a K step of 16 elements moves 32 B inside the swizzle atom.
            // B: MN-major; 8-row k-groups 1024 B apart, 64-column n-blocks B_SUB apart;
            // a K step of 16 rows moves 2048 B.
            umma_bf16(d_tmem, ad_base + soff + (uint64_t)(kk * (32 >> 4)), bd_base + soff + (uint64_t)(kk * (2048 >> 4)),
                      IDESC, (kb | kk) != 0);
          }
          umma_commit(&c.empty[s]);
          if (++s == STAGES) { s = 0; phase ^= 1; }
        }
        if (!ok) break;
        umma_commit(&c.tfull[buf]);
      }
      if (!ok) {
        flag_error(a.err, ERR_WAIT_MMA);
        c.abort = 1;
        // Wait for the MMAs already issued before TMEM is released.
        umma_commit(&c.drain);
        volatile int never = 0;
        mbar_wait(&c.drain, 0, &never, a.wait_limit_ns);
      }
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const Tile tl = decode_tile(c, G, t);
      if (lane == 0) debug_tile_rows(tl, a);
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      // Warp-uniform decision: the TMEM loads below are .sync.aligned.
      const bool got = __all_sync(0xffffffffu, mbar_wait(&c.tfull[buf], use & 1u, &c.abort, a.wait_limit_ns));
      if (!got) {
        if (lane == 0) flag_error(a.err, ERR_WAIT_EPILOGUE);
        c.abort = 1;
        break;
      }
      tc_fence_after_sync();
      const int row = tl.row0 + q * 32 + lane;
      const bool valid = row < tl.row_end;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      drain_tile<EPI>(a, taddr, row, valid, tl.n_tile);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.tempty[buf]);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------- dynamic tile schedule
// The CTA-pair kernels take their tiles dynamically.  One thread of CTA 0 (the scheduler) takes
// tile ids in increasing order from a counter in global memory shared by all clusters of the
// launch and hands each to both CTAs of its pair through a ring of SCHED_RING slots; every role
// of the pair takes the same sequence from the ring.  The scheduler takes the next id only when
// the pair's TMA producer starts its current tile, so each pair holds one id ahead and the
// tiles running at any moment are a narrow window of consecutive ids: the row (token) tiles of
// one expert's column (feature) tile, which share a weight slice, start at about the same time
// and find it in L2, and so do the column tiles that share rows.  A static round-robin schedule
// lets clusters drift apart over many rounds (tiles differ in length: token tiles of 16..288
// rows, DRAM and power stalls), and each then streams the slice from HBM; handing out ids
// further ahead scatters the running tiles the same way.  A tile's result does not depend on
// which cluster computes it.
constexpr int SCHED_RING = 4;
// Roles that take every tile id from the ring: in CTA 0 the TMA producer, the MMA issuer and
// four epilogue warps; in CTA 1 the TMA producer and four epilogue warps.
constexpr int SCHED_CONSUMERS = 11;

struct Sched {
  uint64_t full[SCHED_RING];    // slot holds the next tile id (arrived by the scheduler)
  uint64_t empty[SCHED_RING];   // CTA 0 only: every consumer has read the slot
  uint64_t taken;               // CTA 0 only: its TMA producer has taken the next tile id
  int ring[SCHED_RING];
};

__device__ __forceinline__ void sched_init(Sched& s) {
  for (int i = 0; i < SCHED_RING; ++i) {
    mbar_init(&s.full[i], 1);
    mbar_init(&s.empty[i], SCHED_CONSUMERS);
  }
  mbar_init(&s.taken, 1);
}

// Consumer side: wait for ring slot i % SCHED_RING and return its tile id (-1: no more tiles,
// -2: the wait failed).  The caller releases the slot with sched_release once it has read it.
__device__ __forceinline__ int sched_peek(Sched& s, volatile int* abort, int i, unsigned long long limit) {
  const int slot = i % SCHED_RING;
  if (!mbar_wait_acq_cluster(&s.full[slot], (uint32_t)(i / SCHED_RING) & 1u, abort, limit)) return -2;
  return s.ring[slot];
}

__device__ __forceinline__ void sched_release(Sched& s, int i) {
  mbar_arrive_cluster(mapa_shared(smem_addr(&s.empty[i % SCHED_RING]), 0));
}

// Scheduler (one thread of CTA 0): hands out tile ids until they run out, then counts its
// cluster as finished; the last cluster to finish resets the counters for the next launch.
// Id i + 1 is taken once CTA 0's producer has taken id i (`taken`) and its ring slot is free.
__device__ __forceinline__ void sched_run(Sched& s, volatile int* abort, const GemmArgs& a, int total,
                                          int nclusters) {
  for (int i = 0;; ++i) {
    const int slot = i % SCHED_RING;
    if ((i >= 1 && !mbar_wait(&s.taken, (uint32_t)(i - 1) & 1u, abort, a.wait_limit_ns)) ||
        (i >= SCHED_RING && !mbar_wait(&s.empty[slot], (uint32_t)(i / SCHED_RING - 1) & 1u, abort, a.wait_limit_ns))) {
      flag_error(a.err, ERR_WAIT_PRODUCER);
      *abort = 1;
      break;
    }
    int t = atomicAdd(a.tile_ctr, 1);
    if (t >= total) t = -1;
    s.ring[slot] = t;
    st_shared_cluster(mapa_shared(smem_addr(&s.ring[slot]), 1), t);
    mbar_arrive(&s.full[slot]);
    mbar_arrive_cluster(mapa_shared(smem_addr(&s.full[slot]), 1));   // releases the store above
    if (t < 0) break;
  }
  if (atomicAdd(a.tile_ctr + 1, 1) == nclusters - 1) {
    atomicExch(a.tile_ctr, 0);
    atomicExch(a.tile_ctr + 1, 0);
  }
}

// ------------------------------------------------------------------------- CTA-pair kernel
// The same grouped GEMM with one tcgen05.mma.cta_group::2 per 256 x 256 x 16 step shared by the
// two CTAs of a cluster.  CTA r of the pair loads rows row0 + 128 r .. + 127 of A and MMA
// columns 128 r .. 128 r + 127 of B (for SWIGLU: CTA 0 the W1 slice, CTA 1 the same slice of
// W2; for EPI_F32: output columns n0 + 128 r ..) into its own shared memory, and receives its
// 128 accumulator rows x 256 columns in its own tensor memory.  Per CTA a k-block stage is
// 32 KB (A 16 KB + half of B 16 KB) instead of 48 KB, so six stages fit.
//
// Synchronisation: both CTAs' copies of a stage complete on full[s] in CTA 0, whose producer
// expects 2 x 32 KB; the MMA thread (CTA 0 only) releases a stage to both producers with a
// multicast commit on empty[s]; finished accumulators are signalled to both epilogues by a
// multicast commit on tfull[b]; the eight epilogue warps of the pair release a buffer by
// arriving on tempty[b] in CTA 0.
namespace pair {
constexpr int BM = 128;                   // rows per CTA
constexpr int PAIR_M = 256;               // rows per pair tile (MMA M)
constexpr int STAGES = 6;
constexpr int A_TILE = BM * BK * 2;       // 16 KB
constexpr int B_HALF = 2 * B_SUB;         // 16 KB: this CTA's 128 of the 256 MMA columns
constexpr int STAGE = A_TILE + B_HALF;    // 32 KB
constexpr uint32_t IDESC = idesc_bf16_f32_kmaj_a_mnmaj_b<PAIR_M, BN>();

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  Sched sched;
  uint32_t tmem_base;
  volatile int abort;
  int tile_start[MAX_GROUPS + 1];
  int row_off[MAX_GROUPS + 1];
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE + sizeof(Ctrl);
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
}  // namespace pair

// A bounded pause (used only after a timed-out wait, so that copies already issued can land
// before the CTA's shared memory is released).
__device__ __forceinline__ void settle_after_abort() {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < 200000ull) __nanosleep(1000);
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                         const __grid_constant__ CUtensorMap tmB1, const GemmArgs a) {
  using pair::STAGES;
  using pair::STAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  pair::Ctrl& c = *reinterpret_cast<pair::Ctrl*>(smem + (size_t)STAGES * STAGE);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.offsets ? a.G : 1;
  const uint32_t rank = cluster_ctarank();
  const int nclusters = (int)(gridDim.x >> 1);   // clusters are pairs of consecutive blocks

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c.tfull[b], 1);
      mbar_init(&c.tempty[b], 8);
    }
    sched_init(c.sched);
    mbar_init(&c.drain, 1);
    c.abort = 0;
    fence_barrier_init_cluster();
    fence_proxy_async_smem();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB0);
    prefetch_tensormap(&tmB1);
  }
  if (warp == 2) tmem_alloc_pair(&c.tmem_base, TMEM_COLS);
  pdl_wait();      // offsets, A and the outputs belong to earlier kernels of the stream
  pdl_trigger();
  if (warp == 3) build_group_table<pair::PAIR_M>(c, a, G, lane);
  tc_fence_before_sync();
  cluster_sync();   // the peer's barriers are initialised and both CTAs hold their TMEM columns
  tc_fence_after_sync();

  const uint32_t tmem = c.tmem_base;
  const int total = c.tile_start[G];
  const int num_kb = (a.K + BK - 1) / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer (both CTAs)
      int s = 0;
      uint32_t phase = 0;
      for (int i = 0;; ++i) {
        const int t = sched_peek(c.sched, &c.abort, i, a.wait_limit_ns);
        sched_release(c.sched, i);
        if (rank == 0) mbar_arrive(&c.sched.taken);   // the scheduler may take the next id
        if (t == -2) {
          flag_error(a.err, ERR_WAIT_PRODUCER);
          c.abort = 1;
          break;
        }
        if (t < 0) break;
        if (a.starve) continue;   // test hook: no copies, so the MMA and epilogue waits run out
        const Tile tl = decode_tile<pair::PAIR_M>(c, G, t);
        const int z = a.offsets ? tl.g : a.b_z;
        const int arow = tl.row0 + (int)rank * pair::BM;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&c.empty[s], phase ^ 1, &c.abort, a.wait_limit_ns)) {
            flag_error(a.err, ERR_WAIT_PRODUCER);
            c.abort = 1;
            ok = false;
            break;
          }
          uint8_t* sa = stages + (size_t)s * STAGE;
          uint8_t* sb = sa + pair::A_TILE;
          if (rank == 0) mbar_arrive_expect_tx(&c.full[s], 2 * STAGE);
          const uint32_t fb = mapa_shared(smem_addr(&c.full[s]), 0);
          const int k0 = kb * BK;
          tma_load_2d_pair(sa, &tmA, fb, k0, arow);
          if (EPI == EPI_SWIGLU) {
            const CUtensorMap* mb = rank == 0 ? &tmB0 : &tmB1;
            const int n0 = tl.n_tile * (BN / 2);
            tma_load_3d_pair(sb, mb, fb, n0, k0, z);
            tma_load_3d_pair(sb + B_SUB, mb, fb, n0 + 64, k0, z);
          } else {
            const int n0 = tl.n_tile * BN + (int)rank * (BN / 2);
            tma_load_3d_pair(sb, &tmB0, fb, n0, k0, z);
            tma_load_3d_pair(sb + B_SUB, &tmB0, fb, n0 + 64, k0, z);
          }
          if (++s == STAGES) { s = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------------- MMA issuer (CTA 0)
      int s = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      const uint64_t ad_base = sdesc_sw128(smem_addr(stages), 16, 1024);   // stage 0, as above
      const uint64_t bd_base = sdesc_sw128(smem_addr(stages) + pair::A_TILE, B_SUB, 1024);
      for (;; ++it) {
        const int t = sched_peek(c.sched, &c.abort, it, a.wait_limit_ns);
        sched_release(c.sched, it);
        if (t == -2) { ok = false; break; }
        if (t < 0) break;
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait(&c.tempty[buf], (use & 1u) ^ 1u, &c.abort, a.wait_limit_ns)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&c.full[s], phase, &c.abort, a.wait_limit_ns)) { ok = false; break; }
          tc_fence_after_sync();
          const uint64_t soff = (uint64_t)(((uint32_t)s * (uint32_t)STAGE) >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // Same layouts as the single-CTA kernel; each CTA supplies its 128 rows of A and
            // its two 64-column blocks of B at these shared-memory offsets.
            umma_bf16_pair(d_tmem, ad_base + soff + (uint64_t)(kk * (32 >> 4)),
                           bd_base + soff + (uint64_t)(kk * (2048 >> 4)), pair::IDESC, (kb | kk) != 0);
          }
          umma_commit_pair(&c.empty[s], 0x3);
          if (++s == STAGES) { s = 0; phase ^= 1; }
        }
        if (!ok) break;
        umma_commit_pair(&c.tfull[buf], 0x3);
      }
      if (!ok) {
        flag_error(a.err, ERR_WAIT_MMA);
        c.abort = 1;
        umma_commit_pair(&c.drain, 0x1);
        volatile int never = 0;
        mbar_wait(&c.drain, 0, &never, a.wait_limit_ns);
      }
    }
  } else if (warp == 3) {
    if (lane == 0 && rank == 0) sched_run(c.sched, &c.abort, a, total, nclusters);   // ---- tile scheduler (CTA 0)
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;
    const uint32_t tempty0 = mapa_shared(smem_addr(&c.tempty[0]), 0);
    const uint32_t tempty1 = mapa_shared(smem_addr(&c.tempty[1]), 0);
    for (int it = 0;; ++it) {
      const int t_lane = sched_peek(c.sched, &c.abort, it, a.wait_limit_ns);
      const bool fed = __all_sync(0xffffffffu, t_lane != -2);
      const int t = __shfl_sync(0xffffffffu, t_lane, 0);
      __syncwarp();
      if (lane == 0) sched_release(c.sched, it);
      if (!fed) {
        if (lane == 0) flag_error(a.err, ERR_WAIT_EPILOGUE);
        c.abort = 1;
        break;
      }
      if (t < 0) break;
      const Tile tl = decode_tile<pair::PAIR_M>(c, G, t);
      if (lane == 0) debug_tile_rows(tl, a);
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      const bool got = __all_sync(0xffffffffu, mbar_wait(&c.tfull[buf], use & 1u, &c.abort, a.wait_limit_ns));
      if (!got) {
        if (lane == 0) flag_error(a.err, ERR_WAIT_EPILOGUE);
        c.abort = 1;
        break;
      }
      tc_fence_after_sync();
      const int row = tl.row0 + (int)rank * pair::BM + q * 32 + lane;
      const bool valid = row < tl.row_end;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      drain_tile<EPI>(a, taddr, row, valid, tl.n_tile);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(buf ? tempty1 : tempty0);
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && c.abort) settle_after_abort();
  tc_fence_before_sync();
  cluster_sync();   // neither CTA leaves while the peer may still use its shared memory
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------- token-wide CTA-pair kernel
// The CTA-pair GEMM with the operands' roles swapped: the weights' output features run along the
// MMA's M (256 per pair, 128 per CTA) and the tokens along its N, in steps of 16, so an expert
// block pays at most 15 rows of MMA padding (with tokens along M the padding reaches 255 rows per
// expert, about a tenth of the work on the Mixtral-shaped layer).
//
// Tiles hold 256 tokens, except that an expert's last tile also takes up to WIDE = 32 more
// ("wide" tile): a block of 257..288 rows is one pass over its weight slice instead of a full
// tile plus a short one.  A short tail tile costs almost as much as a full one, because the
// weight slice is streamed again for a few tokens; with ~256 rows per expert (DeepSeek-V3
// shapes) half the experts would need one.  A wide tile issues a second MMA per k step (N = 16
// or 32) on the same weight stage.
//
//   A (MMA M, weights, MN-major): per CTA and stage two 64-feature x 64-k boxes.  SWIGLU: box 0
//     is W1 for features f0 + 64 r .. + 63 and box 1 is W2 for the same features, so a CTA's
//     TMEM lanes 0-63 hold X W1 and lanes 64-127 hold X W2 of the same 64 features; EPI_F32:
//     the two boxes are output features f0 + 128 r .. + 127.
//   B (MMA N, tokens, K-major): the MMA takes N / 2 rows from each CTA.  A tile of n16 <= 256
//     (tokens rounded up to 16) has CTA r load the 128-row box at row0 + r n16 / 2.  A wide tile
//     (n16 = 256 + t16) has CTA r hold rows row0 + r half .. + half - 1, half = 128 + t16 / 2:
//     a 128-row box (for the N = 256 MMA) and a 16-row box behind it (for the N = t16 MMA).
//     Accumulator column c of the main MMA is token c (c < 128) or half + c - 128; column c of
//     the tail MMA is token 128 + c (c < t16 / 2) or half + 128 + c - t16 / 2.
//   TMEM: two 256-column accumulators (tile i uses buffer i & 1); the tail accumulator of a
//     wide tile in buffer b borrows columns 0..31 of buffer 1 - b.  The epilogue drains a tile's
//     tail and its columns 0..31 first and then arrives on thead[b], so the next tile's MMAs
//     wait only for those two chunks (not the whole drain) before they overwrite them.
// The SwiGLU epilogue passes X W1 from the warps that hold it (lanes 0-63) to the warps that
// hold X W2 of the same features through a small shared-memory buffer, 32 tokens at a time.
// Synchronisation is otherwise that of the pair kernel above.
namespace tpair {
constexpr int TOK = 256;                           // tokens of a full tile (MMA N)
constexpr int WIDE_ROWS = 32;                      // extra tokens an expert's last tile may take
constexpr int STAGES = 6;
constexpr int A_BYTES = 2 * B_SUB;                 // 16 KB
constexpr int B_MAIN = BM * BK * 2;                // 16 KB: 128 token rows x 64 k
constexpr int B_TAIL_ROWS = WIDE_ROWS / 2;         // 16 rows per CTA for the tail MMA
constexpr int B_TAIL = B_TAIL_ROWS * BK * 2;       // 2 KB
constexpr int XCHG_FLOATS = 2 * 32 * 32;           // X W1 of 64 features x 32 tokens
constexpr uint32_t IDESC_BASE = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((uint32_t)(256 >> 4) << 24);

// Instruction descriptor: D f32, A and B bf16, A MN-major, B K-major, M = 256, N = n.
__host__ __device__ __forceinline__ uint32_t idesc(int n) { return IDESC_BASE | ((uint32_t)(n >> 3) << 17); }

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t thead[2];
  uint64_t drain;
  Sched sched;
  uint32_t tmem_base;
  volatile int abort;
  int ep_ok[4];
  int tile_start[MAX_GROUPS + 1];
  int row_off[MAX_GROUPS + 1];
};

// The kernel is compiled with and without wide tiles (W): without, it has no tail MMA, no tail
// rows in its stages and no early hand-back, and blocks of 257..288 rows take two tiles.
template <bool W>
struct Cfg {
  static constexpr int wide_rows = W ? WIDE_ROWS : 0;
  static constexpr int STAGE = A_BYTES + B_MAIN + (W ? B_TAIL : 0);   // 34 or 32 KB
  static constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE + XCHG_FLOATS * 4 + sizeof(Ctrl);
  static_assert(STAGE % 1024 == 0, "stage alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Token layout of one tile (see above).
struct Shape {
  int n;       // tokens
  int n16;     // tokens rounded up to 16
  int t16;     // tail MMA width (0: not a wide tile)
  int half;    // rows each CTA holds
  __device__ __forceinline__ Shape(int tokens, bool wide_tiles) {
    n = tokens;
    n16 = (tokens + 15) & ~15;
    t16 = wide_tiles && n16 > TOK ? n16 - TOK : 0;
    half = t16 ? 128 + t16 / 2 : n16 / 2;
  }
  // token of main-accumulator column c (c < 256) or tail-accumulator column c
  __device__ __forceinline__ int main_token(int c) const { return (t16 == 0 || c < 128) ? c : half + c - 128; }
  __device__ __forceinline__ int tail_token(int c) const {
    return c < t16 / 2 ? 128 + c : half + 128 + c - t16 / 2;
  }
};
}  // namespace tpair

__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Stores of one 32-column chunk: column j of the chunk is token base + j for j0 <= j < end (the
// caller splits the chunk into runs on which the token map is affine).  One add, compare and
// store per column, as few instructions as possible: these warps share issue slots with the
// TMA producer and the MMA issuer.  SWIGLU: `r` holds X W2 and `xu` X W1 of the same features.
template <int EPI>
__device__ __forceinline__ void tpair_store_run(const GemmArgs& a, const Tile& tl, const uint32_t (&r)[32],
                                                const float* xu, int lane, int f, int base, int j0, int end) {
  if (EPI == EPI_SWIGLU) {
    uint16_t* p = reinterpret_cast<uint16_t*>(a.out) + (size_t)(tl.row0 + base) * a.ldo + f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j >= j0 && j < end) {
        const float u = xu[j * 32 + lane];
        const float v = __uint_as_float(r[j]);
        const float h = u * __fdividef(v, 1.0f + __expf(-v));
        p[(size_t)j * a.ldo] = __bfloat16_as_ushort(__float2bfloat16_rn(h));
      }
    }
  } else {
    float* p = reinterpret_cast<float*>(a.out) + (size_t)(tl.row0 + base) * a.ldo + f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j >= j0 && j < end) {
        float* dst = p + (size_t)j * a.ldo;
        const float v = __uint_as_float(r[j]);
        *dst = a.accumulate ? *dst + v : v;
      }
    }
  }
}

// Epilogue of 32 accumulator columns of a token-wide tile for this warp's 32 TMEM lanes, already
// read from TMEM into `r`: store every column whose token is valid.  `tail` selects the
// column-to-token map: main columns col0 + j are tokens main_token(col0) + j (a chunk never
// straddles column 128), tail columns j are tokens 128 + j (j < t16 / 2) and half + 128 + j -
// t16 / 2.  SWIGLU: all four epilogue warps must call it together (named barrier).
template <int EPI>
__device__ __forceinline__ void tpair_store_chunk(const GemmArgs& a, const tpair::Shape& sh, const Tile& tl,
                                                  const uint32_t (&r)[32], int col0, bool tail, int q, int lane,
                                                  uint32_t rank, float* xchg) {
  int f;
  float* xu = nullptr;
  if (EPI == EPI_SWIGLU) {
    // Warps 4-5 (TMEM lanes 0-63, X W1) hand their values to warps 6-7 (lanes 64-127, X W2 of
    // the same features), which finish and store h: the TMA producer and the MMA issuer run on
    // the same SM sub-partitions as warps 4 and 5 (warp w issues on sub-partition w % 4), so
    // the SiLU and the stores go to the sub-partitions of the idle warps 2 and 3.
    f = tl.n_tile * 128 + 64 * (int)rank + 32 * (q & 1) + lane;
    xu = xchg + (q & 1) * 32 * 32;
    if (q < 2) {
#pragma unroll
      for (int j = 0; j < 32; ++j) xu[j * 32 + lane] = __uint_as_float(r[j]);
    }
    epilogue_bar();
  } else {
    f = tl.n_tile * 256 + 128 * (int)rank + 32 * q + lane;
  }
  if ((EPI != EPI_SWIGLU || q >= 2) && f < a.N) {
    if (!tail) {
      const int base = sh.main_token(col0);
      const int end = min(min(32, (sh.t16 ? tpair::TOK : sh.n16) - col0), sh.n - base);
      tpair_store_run<EPI>(a, tl, r, xu, lane, f, base, 0, end);
    } else {
      const int split = sh.t16 / 2;
      tpair_store_run<EPI>(a, tl, r, xu, lane, f, 128, 0, min(split, sh.n - 128));
      const int base_b = sh.half + 128 - split;
      tpair_store_run<EPI>(a, tl, r, xu, lane, f, base_b, split, min(sh.t16, sh.n - base_b));
    }
  }
  if (EPI == EPI_SWIGLU) epilogue_bar();
}

// The MMA issuer's K loop over one tile of the token-wide kernel: per stage, wait for its data,
// issue the BK / 16 MMAs (two per K step for a wide tile: the main N = 256 one and the tail one
// on the same weight stage), and release the stage when they complete.  Returns false if a wait
// timed out.
template <bool WIDE_TILE, int STAGE>
__device__ __forceinline__ bool tpair_mma_kloop(tpair::Ctrl& c, const GemmArgs& a, int num_kb, int& s,
                                                uint32_t& phase, uint64_t ad_base, uint64_t bd_base, uint32_t d_main,
                                                uint32_t d_tail, uint32_t idesc_main, uint32_t idesc_tail) {
  for (int kb = 0; kb < num_kb; ++kb) {
    if (!mbar_wait(&c.full[s], phase, &c.abort, a.wait_limit_ns)) return false;
    tc_fence_after_sync();
    const uint64_t soff = (uint64_t)(((uint32_t)s * (uint32_t)STAGE) >> 4);
    const uint64_t ad0 = ad_base + soff, bd0 = bd_base + soff;
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      const uint64_t ad = ad0 + (uint64_t)(kk * (2048 >> 4));
      const uint64_t bd = bd0 + (uint64_t)(kk * (32 >> 4));
      umma_bf16_pair(d_main, ad, bd, idesc_main, (kb | kk) != 0);
      if (WIDE_TILE) umma_bf16_pair(d_tail, ad, bd + (uint64_t)(tpair::B_MAIN >> 4), idesc_tail, (kb | kk) != 0);
    }
    umma_commit_pair(&c.empty[s], 0x3);
    if (++s == tpair::STAGES) { s = 0; phase ^= 1; }
  }
  return true;
}

template <int EPI, bool WIDE>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_tpair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXt,
                          const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                          const GemmArgs a) {
  using tpair::STAGES;
  constexpr int STAGE = tpair::Cfg<WIDE>::STAGE;
  constexpr int WR = tpair::Cfg<WIDE>::wide_rows;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  float* xchg = reinterpret_cast<float*>(smem + (size_t)STAGES * STAGE);
  tpair::Ctrl& c = *reinterpret_cast<tpair::Ctrl*>(smem + (size_t)STAGES * STAGE + tpair::XCHG_FLOATS * 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.offsets ? a.G : 1;
  const uint32_t rank = cluster_ctarank();
  const int nclusters = (int)(gridDim.x >> 1);
  const int feat_per_tile = EPI == EPI_SWIGLU ? 128 : 256;   // output features of one pair tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c.tfull[b], 1);
      mbar_init(&c.tempty[b], 8);
      mbar_init(&c.thead[b], 8);
    }
    sched_init(c.sched);
    mbar_init(&c.drain, 1);
    c.abort = 0;
    fence_barrier_init_cluster();
    fence_proxy_async_smem();
    prefetch_tensormap(&tmX);
    if (WIDE) prefetch_tensormap(&tmXt);
    prefetch_tensormap(&tmW0);
    prefetch_tensormap(&tmW1);
  }
  if (warp == 2) tmem_alloc_pair(&c.tmem_base, TMEM_COLS);
  pdl_wait();      // offsets, rows and the outputs belong to earlier kernels of the stream
  pdl_trigger();
  if (warp == 3) build_group_table<tpair::TOK, WR>(c, a, G, lane);
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();

  const uint32_t tmem = c.tmem_base;
  const int total = c.tile_start[G];
  const int num_kb = (a.K + BK - 1) / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer (both CTAs)
      int s = 0;
      uint32_t phase = 0;
      for (int i = 0;; ++i) {
        const int t = sched_peek(c.sched, &c.abort, i, a.wait_limit_ns);
        sched_release(c.sched, i);
        if (rank == 0) mbar_arrive(&c.sched.taken);   // the scheduler may take the next id
        if (t == -2) {
          flag_error(a.err, ERR_WAIT_PRODUCER);
          c.abort = 1;
          break;
        }
        if (t < 0) break;
        if (a.starve) continue;   // test hook: no copies, so the MMA and epilogue waits run out
        const Tile tl = decode_tile<tpair::TOK, WR>(c, G, t);
        const tpair::Shape sh(tl.tile_end - tl.row0, WIDE);
        const int z = a.offsets ? tl.g : a.b_z;
        const int trow = tl.row0 + (int)rank * sh.half;
        const int fa = tl.n_tile * feat_per_tile + (EPI == EPI_SWIGLU ? 64 : 128) * (int)rank;
        const uint32_t tx = 2u * (uint32_t)(tpair::A_BYTES + tpair::B_MAIN + (sh.t16 ? tpair::B_TAIL : 0));
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&c.empty[s], phase ^ 1, &c.abort, a.wait_limit_ns)) {
            flag_error(a.err, ERR_WAIT_PRODUCER);
            c.abort = 1;
            ok = false;
            break;
          }
          uint8_t* sa = stages + (size_t)s * STAGE;
          uint8_t* sb = sa + tpair::A_BYTES;
          if (rank == 0) mbar_arrive_expect_tx(&c.full[s], tx);
          const uint32_t fb = mapa_shared(smem_addr(&c.full[s]), 0);
          const int k0 = kb * BK;
          if (EPI == EPI_SWIGLU) {
            tma_load_3d_pair(sa, &tmW0, fb, fa, k0, z);
            tma_load_3d_pair(sa + B_SUB, &tmW1, fb, fa, k0, z);
          } else {
            tma_load_3d_pair(sa, &tmW0, fb, fa, k0, z);
            tma_load_3d_pair(sa + B_SUB, &tmW0, fb, fa + 64, k0, z);
          }
          tma_load_2d_pair(sb, &tmX, fb, k0, trow);
          if (WIDE && sh.t16) tma_load_2d_pair(sb + tpair::B_MAIN, &tmXt, fb, k0, trow + 128);
          if (++s == STAGES) { s = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------------- MMA issuer (CTA 0)
      int s = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      bool prev_wide = false;
      const uint64_t ad_base = sdesc_sw128(smem_addr(stages), B_SUB, 1024);
      const uint64_t bd_base = sdesc_sw128(smem_addr(stages) + tpair::A_BYTES, 16, 1024);
      for (;; ++it) {
        const int t = sched_peek(c.sched, &c.abort, it, a.wait_limit_ns);
        sched_release(c.sched, it);
        if (t == -2) { ok = false; break; }
        if (t < 0) break;
        const Tile tl = decode_tile<tpair::TOK, WR>(c, G, t);
        const tpair::Shape sh(tl.tile_end - tl.row0, WIDE);
        const bool wide = WIDE && sh.t16 != 0;
        const uint32_t idesc_main = tpair::idesc(wide ? tpair::TOK : sh.n16);
        const uint32_t idesc_tail = tpair::idesc(wide ? sh.t16 : 16);
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait(&c.tempty[buf], (use & 1u) ^ 1u, &c.abort, a.wait_limit_ns)) { ok = false; break; }
        // A wide tile writes columns 0..31 of the other buffer, whose previous tile may still be
        // draining them; after a wide tile, its tail sits in columns 0..31 of this buffer.
        if (WIDE && it > 0 && (wide || prev_wide) &&
            !mbar_wait(&c.thead[buf ^ 1], (uint32_t)((it - 1) >> 1) & 1u, &c.abort, a.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_main = tmem + (uint32_t)(buf * BN);
        const uint32_t d_tail = tmem + (uint32_t)((buf ^ 1) * BN);
        // A: MN-major, two 64-feature blocks B_SUB apart, 8-row k-groups 1024 B apart; a K step
        // of 16 rows moves 2048 B.  B: K-major token rows of 128 B; a K step moves 32 B.  The
        // descriptors are the stage-0 ones plus the byte offset / 16 in their address field
        // (shared addresses stay below 2^18, so the field never carries), and the wide test sits
        // outside the K loop (one loop per case): the issuing thread is on the critical path.
        if (WIDE && wide) {
          ok = tpair_mma_kloop<true, STAGE>(c, a, num_kb, s, phase, ad_base, bd_base, d_main, d_tail, idesc_main,
                                            idesc_tail);
        } else {
          ok = tpair_mma_kloop<false, STAGE>(c, a, num_kb, s, phase, ad_base, bd_base, d_main, d_tail, idesc_main,
                                             idesc_tail);
        }
        if (!ok) break;
        umma_commit_pair(&c.tfull[buf], 0x3);
        prev_wide = wide;
      }
      if (!ok) {
        flag_error(a.err, ERR_WAIT_MMA);
        c.abort = 1;
        umma_commit_pair(&c.drain, 0x1);
        volatile int never = 0;
        mbar_wait(&c.drain, 0, &never, a.wait_limit_ns);
      }
    }
  } else if (warp == 3) {
    if (lane == 0 && rank == 0) sched_run(c.sched, &c.abort, a, total, nclusters);   // ---- tile scheduler (CTA 0)
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;   // TMEM lanes 32 q .. 32 q + 31
    const uint32_t tempty0 = mapa_shared(smem_addr(&c.tempty[0]), 0);
    const uint32_t tempty1 = mapa_shared(smem_addr(&c.tempty[1]), 0);
    const uint32_t thead0 = mapa_shared(smem_addr(&c.thead[0]), 0);
    const uint32_t thead1 = mapa_shared(smem_addr(&c.thead[1]), 0);
    for (int it = 0;; ++it) {
      // The four warps take the same decision: they meet at unbounded named barriers below.
      const int t_lane = sched_peek(c.sched, &c.abort, it, a.wait_limit_ns);
      const bool mine_fed = __all_sync(0xffffffffu, t_lane != -2);
      const int t = __shfl_sync(0xffffffffu, t_lane, 0);
      __syncwarp();
      if (lane == 0) {
        sched_release(c.sched, it);
        c.ep_ok[q] = mine_fed ? 1 : 0;
      }
      epilogue_bar();
      const bool fed = c.ep_ok[0] && c.ep_ok[1] && c.ep_ok[2] && c.ep_ok[3];
      epilogue_bar();
      if (!fed) {
        if (lane == 0 && !mine_fed) flag_error(a.err, ERR_WAIT_EPILOGUE);
        c.abort = 1;
        break;
      }
      if (t < 0) break;
      const Tile tl = decode_tile<tpair::TOK, WR>(c, G, t);
      if (lane == 0) debug_tile_rows(tl, a);
      const tpair::Shape sh(tl.tile_end - tl.row0, WIDE);
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      // the four epilogue warps take the same decision (they meet at named barriers below)
      const bool mine = __all_sync(0xffffffffu, mbar_wait(&c.tfull[buf], use & 1u, &c.abort, a.wait_limit_ns));
      if (lane == 0) c.ep_ok[q] = mine ? 1 : 0;
      epilogue_bar();
      const bool got = c.ep_ok[0] && c.ep_ok[1] && c.ep_ok[2] && c.ep_ok[3];
      epilogue_bar();
      if (!got) {
        if (lane == 0 && !mine) flag_error(a.err, ERR_WAIT_EPILOGUE);
        c.abort = 1;
        break;
      }
      tc_fence_after_sync();
      const uint32_t lanes = (uint32_t)(q * 32) << 16;
      const uint32_t t_main = tmem + lanes + (uint32_t)(buf * BN);
      const uint32_t t_tail = tmem + lanes + (uint32_t)((buf ^ 1) * BN);
      // The tail and columns 0..31 are read first and handed back (thead) before anything is
      // stored: the next tile's MMAs wait for these two chunks only, and the arrive's release
      // has no new stores to wait for.
      if (WIDE) {
        uint32_t rt[32], rh[32];
        if (sh.t16) tmem_ld_32cols(t_tail, rt);
        tmem_ld_32cols(t_main, rh);
        tmem_ld_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(buf ? thead1 : thead0);
        if (sh.t16) tpair_store_chunk<EPI>(a, sh, tl, rt, 0, true, q, lane, rank, xchg);
        tpair_store_chunk<EPI>(a, sh, tl, rh, 0, false, q, lane, rank, xchg);
      }
      const int main_cols = sh.t16 ? tpair::TOK : sh.n16;
#pragma unroll 1
      for (int col0 = WIDE ? 32 : 0; col0 < main_cols; col0 += 32) {
        uint32_t r[32];
        tmem_ld_32cols(t_main + (uint32_t)col0, r);
        tmem_ld_wait();
        tpair_store_chunk<EPI>(a, sh, tl, r, col0, false, q, lane, rank, xchg);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(buf ? tempty1 : tempty0);
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && c.abort) settle_after_abort();
  tc_fence_before_sync();
  cluster_sync();
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A operand: rows x K bf16 row-major; box 64 (K) x box_rows (rows), 128B swizzle.
static bool make_map_a(CUtensorMap* m, const void* ptr, long long rows, long long K, int box_rows = BM) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B operand: Z matrices of K x N bf16 row-major (N contiguous); box 64 (N) x 64 (K) x 1.
static bool make_map_b(CUtensorMap* m, const void* ptr, long long Z, long long K, long long N) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)K, (cuuint64_t)(Z > 0 ? Z : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)N * 2, (cuuint64_t)K * N * 2};
  cuuint32_t box[3] = {64, BK, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

template <int EPI>
static cudaError_t launch(const CUtensorMap& ma, const CUtensorMap& mb0, const CUtensorMap& mb1, const GemmArgs& a,
                          cudaStream_t st) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  MOE_RETURN_ON_ERROR(launch_k(grouped_gemm_kernel<EPI>, num_sms(), THREADS, SMEM_BYTES, st, ma, mb0, mb1, a));
  ++g_launches;
  return cudaGetLastError();
}

// Counters of the CTA-pair kernels' tile scheduler: a pair of ints (next tile, clusters
// finished) per launch slot, zero when the library loads.  Each launch takes the next slot in
// turn, and the kernel sets its pair back to zero before it completes, so a slot is free again
// once its launch has finished; launches kTileCtrSlots apart would have to run at the same time
// to collide.  Part of the library's device image, like the error word: nothing is allocated.
constexpr int kTileCtrSlots = 256;
static __device__ int g_tile_ctr[2 * kTileCtrSlots];
static std::atomic<unsigned> g_tile_ticket{0};

// Device address of this launch's counter pair on the current device (the array's address is
// looked up once per device, with that device current, under a lock).
static int* tile_ctr_slot() {
  static std::mutex mu;
  static int* base[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!base[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_tile_ctr) != cudaSuccess) return nullptr;
      base[dev] = static_cast<int*>(p);
    }
  }
  return base[dev] + 2 * (g_tile_ticket.fetch_add(1) % kTileCtrSlots);
}

// Persistent grid of CTA pairs: as many clusters of 2 as can be resident at once (at most
// half the SMs).  `slot` caches the per-kernel configuration.
struct PairLaunchCache {
  int device = -1;
  int clusters = 0;
};

template <typename Kernel, typename... Args>
static cudaError_t launch_cluster_pair(Kernel kernel, size_t smem, PairLaunchCache& cache, cudaStream_t st,
                                       const Args&... args) {
  int dev = 0;
  cudaGetDevice(&dev);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;   // the occupancy query takes the cluster shape only
  if (cache.device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int n = 0;
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    cache.clusters = n < num_sms() / 2 ? n : num_sms() / 2;
    cache.device = dev;
  }
  cfg.gridDim = dim3(2 * cache.clusters, 1, 1);
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  ++g_launches;
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int EPI>
static cudaError_t launch_pair(const CUtensorMap& ma, const CUtensorMap& mb0, const CUtensorMap& mb1,
                               const GemmArgs& a_in, cudaStream_t st) {
  static PairLaunchCache cache;
  GemmArgs a = a_in;
  a.tile_ctr = tile_ctr_slot();
  if (!a.tile_ctr) return cudaErrorInvalidDevice;
  return launch_cluster_pair(grouped_gemm_pair_kernel<EPI>, pair::SMEM_BYTES, cache, st, ma, mb0, mb1, a);
}

// The token-wide kernel with wide tiles also takes the rows through a 16-row box (the tail of a
// wide tile); without, that map is the main one and is not used.
template <int EPI, bool WIDE>
static cudaError_t launch_tpair(const CUtensorMap& mx, const void* A, long long rows_cap, int K,
                                const CUtensorMap& mw0, const CUtensorMap& mw1, const GemmArgs& a_in, cudaStream_t st) {
  static PairLaunchCache cache;
  CUtensorMap mxt = mx;
  if (WIDE && !make_map_a(&mxt, A, rows_cap, K, tpair::B_TAIL_ROWS)) return cudaErrorInvalidValue;
  GemmArgs a = a_in;
  a.tile_ctr = tile_ctr_slot();
  if (!a.tile_ctr) return cudaErrorInvalidDevice;
  return launch_cluster_pair(grouped_gemm_tpair_kernel<EPI, WIDE>, tpair::Cfg<WIDE>::SMEM_BYTES, cache, st, mx, mxt,
                             mw0, mw1, a);
}

// Test hook: one starved launch with a short wait limit (moe_test_pipeline_fault).
static std::atomic<unsigned long long> g_fault_limit_ns{0};

static void apply_test_hook(GemmArgs& a) {
  a.wait_limit_ns = kWaitLimitNs;
  a.starve = 0;
  const unsigned long long lim = g_fault_limit_ns.exchange(0);
  if (lim) {
    a.wait_limit_ns = lim;
    a.starve = 1;
  }
}

// Kernel choice, from measurements on B300 (Mixtral-, Hunyuan- and DeepSeek-V3-shaped layers,
// both CTA-pair kernels on the dynamic tile schedule):
//   one dense block (the shared experts, M = T rows): W1/W2 + SwiGLU on the CTA-pair kernel
//     ("pair", 256 token rows per tile): with no ragged ends it pads nothing and keeps the
//     tensor pipe busiest (DeepSeek-V3-shaped shared expert 0.55-0.56 ms against 0.58 on the
//     token-wide kernel); float32 outputs on the token-wide kernel;
//   expert blocks averaging >= 128 rows: W1/W2 + SwiGLU on the token-wide CTA-pair kernel with
//     wide tiles ("tpairw", tokens along N in steps of 16; an expert's last tile may take up to
//     32 tokens beyond 256 through a second MMA on the same weight stage).  A k-block of a
//     separate 16..32-token tail tile costs as many cycles as a full one (~530: its weight
//     stream sets the pace), the second MMA of a wide tile about 250, so the wide build wins on
//     every block size: Mixtral-shaped W1/W2 1.220-1.224 against 1.241-1.242 ms without wide
//     tiles, Hunyuan-shaped 2.25-2.29 against 2.28-2.31 ms (one box, three runs each);
//   W3 (float32 out) on blocks averaging >= 512 rows: the token-wide kernel without wide tiles
//     ("tpair"; Mixtral-shaped 0.625-0.630 against 0.669-0.676 ms with them), with wide tiles
//     for 128..511 rows (DeepSeek-V3 shapes, ~256 rows per expert: a block of up to 288 rows is
//     one pass over its weight slice);
//   fewer rows (decode-sized batches): the single-CTA kernel, which streams each expert's
//     weights once with the fewest bytes per row.
// MOE_GEMM_KERNEL=single|pair|tpair|tpairw overrides the choice (the tests run every kernel on
// the same inputs).
enum Variant { V_SINGLE = 0, V_PAIR = 1, V_TPAIR = 2, V_TPAIR_WIDE = 3 };

static Variant choose_variant(int epi, long long rows, int groups, bool dense) {
  const char* v = getenv("MOE_GEMM_KERNEL");
  if (v && strcmp(v, "single") == 0) return V_SINGLE;
  if (v && strcmp(v, "pair") == 0) return V_PAIR;
  if (v && strcmp(v, "tpair") == 0) return V_TPAIR;
  if (v && strcmp(v, "tpairw") == 0) return V_TPAIR_WIDE;
  const long long g = groups > 0 ? groups : 1;
  if (rows >= 512LL * g) return epi == EPI_SWIGLU ? (dense ? V_PAIR : V_TPAIR_WIDE) : V_TPAIR;
  return rows >= 128LL * g ? V_TPAIR_WIDE : V_SINGLE;
}

}  // namespace tc

void arm_pipeline_fault(unsigned long long wait_limit_ns) {
  tc::g_fault_limit_ns.store(wait_limit_ns ? wait_limit_ns : 1);
}

// h[rows, N] (bf16) = (A W1) * SiLU(A W2), grouped.  A is [rows_cap, K] bf16; W1, W2 are
// [Z][K][N] bf16.  N must be a multiple of 8, K a multiple of 8.
cudaError_t tc_swiglu(const void* A, long long rows_cap, int K, const void* W1, const void* W2, int Z, int N,
                      const int* offsets, int G, int M_dense, int b_z, void* h, uint32_t* err, cudaStream_t st) {
  CUtensorMap ma, mb0, mb1;
  if (!tc::make_map_a(&ma, A, rows_cap, K) || !tc::make_map_b(&mb0, W1, Z, K, N) || !tc::make_map_b(&mb1, W2, Z, K, N))
    return cudaErrorInvalidValue;
  GemmArgs a{};
  a.offsets = offsets; a.G = G; a.M = M_dense; a.K = K; a.N = N;
  a.n_tiles = (N + tc::BN / 2 - 1) / (tc::BN / 2);   // 128 output columns per tile (all variants)
  a.b_z = b_z; a.out = h; a.ldo = N; a.accumulate = 0; a.rows_cap = (int)rows_cap; a.err = err;
  tc::apply_test_hook(a);
  switch (tc::choose_variant(EPI_SWIGLU, offsets ? rows_cap : M_dense, offsets ? G : 1, offsets == nullptr)) {
    case tc::V_TPAIR: return tc::launch_tpair<EPI_SWIGLU, false>(ma, A, rows_cap, K, mb0, mb1, a, st);
    case tc::V_TPAIR_WIDE: return tc::launch_tpair<EPI_SWIGLU, true>(ma, A, rows_cap, K, mb0, mb1, a, st);
    case tc::V_PAIR: return tc::launch_pair<EPI_SWIGLU>(ma, mb0, mb1, a, st);
    default: return tc::launch<EPI_SWIGLU>(ma, mb0, mb1, a, st);
  }
}

// out[rows, N] (f32) (+)= A W, grouped.  A is [rows_cap, K] bf16; W is [Z][K][N] bf16.
cudaError_t tc_matmul_f32(const void* A, long long rows_cap, int K, const void* W, int Z, int N, const int* offsets,
                          int G, int M_dense, int b_z, float* out, long long ldo, int accumulate, uint32_t* err,
                          cudaStream_t st) {
  CUtensorMap ma, mb;
  if (!tc::make_map_a(&ma, A, rows_cap, K) || !tc::make_map_b(&mb, W, Z, K, N)) return cudaErrorInvalidValue;
  GemmArgs a{};
  a.offsets = offsets; a.G = G; a.M = M_dense; a.K = K; a.N = N;
  a.n_tiles = (N + tc::BN - 1) / tc::BN;             // 256 output columns per tile (all variants)
  a.b_z = b_z; a.out = out; a.ldo = ldo; a.accumulate = accumulate; a.rows_cap = (int)rows_cap; a.err = err;
  tc::apply_test_hook(a);
  switch (tc::choose_variant(EPI_F32, offsets ? rows_cap : M_dense, offsets ? G : 1, offsets == nullptr)) {
    case tc::V_TPAIR: return tc::launch_tpair<EPI_F32, false>(ma, A, rows_cap, K, mb, mb, a, st);
    case tc::V_TPAIR_WIDE: return tc::launch_tpair<EPI_F32, true>(ma, A, rows_cap, K, mb, mb, a, st);
    case tc::V_PAIR: return tc::launch_pair<EPI_F32>(ma, mb, mb, a, st);
    default: return tc::launch<EPI_F32>(ma, mb, mb, a, st);
  }
}

}  // namespace moe
