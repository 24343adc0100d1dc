// rz_gemm.cuh -- the one tensor-core pipeline every contraction of the
// library runs on: a persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   warp 0      TMA producer: one elected lane streams A and B tiles
//               (128x64 and 256x64 bf16, 128-byte swizzle) into a 4-stage
//               shared-memory ring, completion tracked by mbarriers.
//   warp 1      TMEM owner + MMA issuer: allocates 512 TMEM columns (two
//               128x256 fp32 accumulators), one lane issues
//               tcgen05.mma (M=128, N=256, K=16) per 16-wide K slice and
//               commits to the ring's "empty" barriers and to the
//               accumulator's "full" barrier.
//   warps 2..5  epilogue: each warp owns 32 TMEM lanes (= 32 output rows);
//               thread i holds row i of its quadrant, so row-wise
//               reductions (log-sum-exp over the vocabulary) need no
//               shuffles.  Double buffering lets the epilogue of tile j run
//               under the MMAs of tile j+1.
//
// Work is a list of tasks (m-block, group of consecutive n-tiles), walked
// m-major and handed to CTAs round-robin.  The tile shape, the K order (K
// blocks 0,1,2,... each as four K=16 MMAs into the same accumulator) and the
// grouping of n-tiles never depend on the number of rows, which is what makes
// a row's result independent of the batch it sits in.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "rz_check.cuh"
#include "rz_ptx.cuh"

namespace rz {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kTileABytes = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kTileBBytes = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kErrTimeout = 4;                    // RZ_DEVERR_TIMEOUT

constexpr uint32_t kSmemRing = kStages * (kTileABytes + kTileBBytes);
constexpr uint32_t kEpiStageBytes = 32 * 128;  // per epilogue warp: 32 rows x 128 B
// ring | barriers (first 256 B of a 1 KB block) | 4 epilogue stages, each
// 1024-byte aligned (a TMA box with 128-byte swizzle)
constexpr uint32_t kSmemBytes =
    kSmemRing + 1024 /*align*/ + 1024 /*barriers*/ + 4 * kEpiStageBytes;

struct GemmSched {
  int m_blocks;         // number of 128-row blocks
  int n_tiles;          // number of 256-wide tiles along N
  int n_groups;         // tasks per m-block (consecutive n-tiles per task)
  int tiles_per_group;  // ceil(n_tiles / n_groups)
  int k_blocks;         // number of 64-deep K blocks
  int num_tasks;        // m_blocks * n_groups
  int m_group;          // raster: m-blocks per group; inside a group tasks run
                        // group-of-n-tiles major, m-block minor (1 = m-major)
  int a_m_off;          // added to the M coordinate of A loads
  int a_k_off;          // added to the K coordinate of MN-major A loads
  int b_k_off;          // added to the K coordinate of B loads
  int* err;             // device error word (nullable)
  uint32_t a_bytes;     // bytes one A load brings (0: a full 128-row box).  A
                        // K-major A box of fewer rows (a batch of < 128 rows:
                        // exactly its rows) fills the first rows of the
                        // stage; the kernel keeps the rest of its A stages zero
};

template <bool kAMN, bool kBMN>
struct Operands {
  // K-major A: one 64(K) x 128(M) box.  MN-major A: two 64(M) x 64(K) boxes.
  static __device__ __forceinline__ void load_a(uint8_t* dst, const CUtensorMap* tm,
                                                uint64_t* bar, int m0, int k0) {
    if constexpr (!kAMN) {
      tma_load_2d(dst, tm, bar, k0, m0);
    } else {
      tma_load_2d(dst, tm, bar, m0, k0);
      tma_load_2d(dst + 8192, tm, bar, m0 + 64, k0);
    }
  }
  // K-major B: one 64(K) x 256(N) box.  MN-major B: four 64(N) x 64(K) boxes.
  static __device__ __forceinline__ void load_b(uint8_t* dst, const CUtensorMap* tm,
                                                uint64_t* bar, int n0, int k0) {
    if constexpr (!kBMN) {
      tma_load_2d(dst, tm, bar, k0, n0);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) tma_load_2d(dst + 8192 * j, tm, bar, n0 + 64 * j, k0);
    }
  }
  // Descriptor of the k-th K=16 slice of a stage.
  //   K-major (rows of 128 B along K): slice start +32 B, SBO = 8 rows = 1024 B.
  //   MN-major (rows of 128 B along MN, one row per k): slice start +16 rows
  //   = 2048 B, LBO = next 64-wide MN block = 8192 B, SBO = 8 k-rows = 1024 B.
  static __device__ __forceinline__ uint64_t desc_a(uint32_t base, int k) {
    if constexpr (!kAMN) return sdesc_sw128(base + 32u * k, 16u, 1024u);
    else return sdesc_sw128(base + 2048u * k, 8192u, 1024u);
  }
  static __device__ __forceinline__ uint64_t desc_b(uint32_t base, int k) {
    if constexpr (!kBMN) return sdesc_sw128(base + 32u * k, 16u, 1024u);
    else return sdesc_sw128(base + 2048u * k, 8192u, 1024u);
  }
};

// Task -> (m-block, n-tile group).  Tasks come in groups of m_group m-blocks;
// inside a group all m-blocks of n-group 0 come first, then n-group 1, ...,
// so CTAs running at the same time share the same B tiles (the LM-head
// weight) through L2.  The order never changes what a task computes.
__device__ __forceinline__ void task_coords(const GemmSched& s, int task, int& m_blk, int& grp,
                                            int& n_begin, int& n_end) {
  const int G = s.m_group;
  const int per = G * s.n_groups;
  const int mg = task / per;
  const int rem = task - mg * per;
  const int full_groups = s.m_blocks / G;
  const int Gl = mg < full_groups ? G : s.m_blocks - full_groups * G;
  grp = rem / Gl;
  m_blk = mg * G + (rem - grp * Gl);
  n_begin = grp * s.tiles_per_group;
  n_end = n_begin + s.tiles_per_group;
  if (n_end > s.n_tiles) n_end = s.n_tiles;
}

__device__ __forceinline__ void raise_abort(volatile int* abort, int* err) {
  *abort = 1;
  if (err) atomicOr(err, kErrTimeout);
}

// Epi must provide:
//   struct Params;  struct State;
//   static void task_begin(const Params&, State&, int m_blk, int grp, int row);
//   static void tile(const Params&, State&, int m_blk, int n_tile, uint32_t taddr, int row,
//                    uint8_t* stage);
//   static void task_end(const Params&, State&, int m_blk, int grp, int row);
// `row` is the thread's row inside the 128-row block; `taddr` the TMEM
// address of (this warp's 32 lanes, column 0) of the tile's accumulator;
// `stage` a private 4 KB shared-memory buffer of the warp (128 B per row,
// 1024-byte aligned).  Params is a __grid_constant__ kernel parameter, so a
// tensor map inside it can serve TMA stores.
template <class Epi, bool kAMN, bool kBMN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmSched sched, const __grid_constant__ typename Epi::Params ep) {
  using Ops = Operands<kAMN, kBMN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kTileABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSmemRing);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* issued_ring = reinterpret_cast<int*>(tmem_slot + 2);  // [0] issued, [1] consumed
  uint8_t* epi_stage = smem + kSmemRing + 1024;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    *abort = 0;
    issued_ring[0] = 0;  // loads issued
    issued_ring[1] = 0;  // loads consumed
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (sched.a_bytes != 0 && sched.a_bytes < kTileABytes) {
    // rows past the A box stay zero for the whole kernel, as a full box
    // would have filled them past the last row
    uint4* a4 = reinterpret_cast<uint4*>(sA);
    for (uint32_t i = threadIdx.x; i < kStages * kTileABytes / 16; i += kThreads)
      a4[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // visible to the tensor cores' reads
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Set-up done: the next kernel may be scheduled, and this one waits for
  // the kernel ahead of it (when launched to overlap its tail) before its
  // first global access.
  grid_dep_launch();
  grid_dep_wait();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int task = blockIdx.x; ok && task < sched.num_tasks; task += gridDim.x) {
        int m_blk, grp, nb, ne;
        task_coords(sched, task, m_blk, grp, nb, ne);
        if (!RZ_DCHECK(m_blk >= 0 && m_blk < sched.m_blocks && nb >= 0 && nb < ne &&
                           ne <= sched.n_tiles && grp >= 0 && grp < sched.n_groups,
                       1))
          ne = nb;  // (debug build) a task outside the problem loads nothing
        const int m0 = m_blk * kBM + sched.a_m_off;
        for (int n = nb; ok && n < ne; ++n) {
          for (int kb = 0; kb < sched.k_blocks; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort, kWaitLimitNs)) {
              raise_abort(abort, sched.err);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage],
                                  (sched.a_bytes != 0 ? sched.a_bytes : kTileABytes) + kTileBBytes);
            const int k0 = kb * kBK;
            Ops::load_a(sA + stage * kTileABytes, &tmA, &full[stage], m0, k0 + sched.a_k_off);
            Ops::load_b(sB + stage * kTileBBytes, &tmB, &full[stage], n * kBN,
                        k0 + sched.b_k_off);
            ++issued;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      issued_ring[0] = issued;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, kAMN, kBMN);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t it = 0;
      int consumed = 0;
      bool ok = true;
      for (int task = blockIdx.x; ok && task < sched.num_tasks; task += gridDim.x) {
        int m_blk, grp, nb, ne;
        task_coords(sched, task, m_blk, grp, nb, ne);
        for (int n = nb; ok && n < ne; ++n, ++it) {
          const uint32_t buf = it & 1u;
          const uint32_t use = it >> 1;
          if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort, kWaitLimitNs)) {
            raise_abort(abort, sched.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * kBN;
          for (int kb = 0; kb < sched.k_blocks; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort, kWaitLimitNs)) {
              raise_abort(abort, sched.err);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(sA + stage * kTileABytes);
            const uint32_t b_base = smem_u32(sB + stage * kTileBBytes);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              umma_bf16(d_tmem, Ops::desc_a(a_base, k), Ops::desc_b(b_base, k), idesc,
                        (kb > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit(&empty[stage]);
            ++consumed;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) umma_commit(&tfull[buf]);
        }
      }
      // Make sure every MMA this thread issued has finished before the CTA
      // can release TMEM (matters only on the abort path).
      umma_commit(drain);
      if (!mbar_wait(drain, 0, abort, kWaitLimitNs) && !*abort) raise_abort(abort, sched.err);
      issued_ring[1] = consumed;
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    typename Epi::State st;
    uint32_t it = 0;
    bool ok = true;
    for (int task = blockIdx.x; ok && task < sched.num_tasks; task += gridDim.x) {
      int m_blk, grp, nb, ne;
      task_coords(sched, task, m_blk, grp, nb, ne);
      Epi::task_begin(ep, st, m_blk, grp, row);
      for (int n = nb; n < ne; ++n, ++it) {
        const uint32_t buf = it & 1u;
        const uint32_t use = it >> 1;
        // One lane waits; the verdict is shared so the warp stays converged
        // for the .sync.aligned TMEM loads that follow.
        int got = 1;
        if (lane == 0) got = mbar_wait<true>(&tfull[buf], use & 1u, abort, kWaitLimitNs) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          if (lane == 0) raise_abort(abort, sched.err);
          ok = false;
          break;
        }
        tc_fence_after();
        Epi::tile(ep, st, m_blk, n, lane_addr + buf * kBN, row,
                  epi_stage + (warp - 2) * kEpiStageBytes);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
      if (ok) Epi::task_end(ep, st, m_blk, grp, row);
    }
    // bulk stores an epilogue issued from its stage have completed
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (*abort && threadIdx.x == 0) {
    // Wait (bounded) for tensor copies that were issued but never consumed,
    // so no copy lands in shared memory after the CTA has exited.
    const int issued = issued_ring[0];
    const int consumed = issued_ring[1];
    for (int i = consumed; i < issued; ++i) {
      const int s = i % kStages;
      const uint32_t ph = static_cast<uint32_t>((i / kStages) & 1);
      const uint32_t a = smem_u32(&full[s]);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(a, ph)) {
        if (globaltimer_ns() - t0 > 100000000ull) break;
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace rz
