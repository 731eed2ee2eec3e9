// engine.cuh — persistent, warp-specialised tcgen05 GEMM pipeline shared by every
// contraction of the head (forward logits, backward logit recompute, dh and dW).
//
// One CTA per SM.  Warp 0 issues TMA loads into a STAGES-deep shared-memory ring,
// warp 1 issues tcgen05.mma (one thread) into a double-buffered TMEM accumulator
// (2 x 256 fp32 columns = all 512 columns), warps 2..5 run the epilogue that the
// kernel supplies.  Each accumulator tile is BM x BN = 128 x 256, built from BK = 64
// wide k-blocks (128-byte swizzle rows) of bf16 operands.
//
// Operand staging in shared memory (per stage: A 16 KiB, B 32 KiB):
//   K-major operand  [rows, K] with K contiguous: one TMA box {64 (K), rows};
//                    rows at 128 B pitch, 8-row swizzle atoms 1024 B apart (SBO).
//   MN-major operand [K, rows] with rows contiguous: rows/64 TMA boxes {64, 64},
//                    each 64 k-rows x 128 B = 8 KiB (or one 3-D box over all of them);
//                    LBO = 8 KiB between 64-wide column blocks, SBO = 1 KiB between
//                    8-k-row groups.
// Options a kernel picks: a paired mode (2-CTA clusters that multicast halves of the
// B tile to each other, run_cta<true>), sparse K (a bitmap of k-block groups per tile,
// KWalk), a static or a dynamic unit feed, and an L2-aware unit order (chunk_decode).
// Every wait is bounded: a wait that exceeds kWaitLimitNs sets ORPO_STATUS_TIMEOUT,
// flags the CTA as aborted and every role drains its own in-flight work and returns.
#pragma once

#include "../../include/orpo_head.h"
#include "bounds.cuh"
#include "ptx.cuh"

namespace orpo {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int UMMA_K = 16;
constexpr int EPI_WARPS = 4;
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int TMEM_COLS = 512;

constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KiB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KiB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t BOX_BYTES = 4096;                 // one 32-row x 128-byte epilogue staging box
constexpr uint32_t STAGING_PER_WARP = 2 * BOX_BYTES;  // double-buffered
constexpr uint32_t SMEM_STAGING_OFF = STAGES * STAGE_BYTES;
constexpr uint32_t SMEM_CTL_OFF = SMEM_STAGING_OFF + EPI_WARPS * STAGING_PER_WARP;
constexpr uint32_t SMEM_CTL_BYTES = 256;
constexpr uint32_t SMEM_TOTAL = SMEM_CTL_OFF + SMEM_CTL_BYTES + 1024;  // + slack to align the base to 1 KiB

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far above any legitimate wait

constexpr int RING = 4;                     // unit indices in flight between the roles (dynamic feed)

struct SmemCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint64_t unit_full[RING];
  uint64_t unit_empty[RING];
  volatile int unit_ring[RING];
  uint32_t tmem_base;
  volatile int abort_flag;
};

// Source of work units.  Static: CTA b takes units b, b + G, b + 2G, ...
// Dynamic (counter != nullptr): the producer thread claims the next unit with
// an atomic add on a zeroed global counter and hands its index to the MMA and
// epilogue warps through a RING-deep shared-memory ring; index -1 ends the
// stream.  Every unit is still computed by exactly one CTA.
struct Feed {
  int* counter;
  int nu;
  int first = -1;  // static feed: first unit and stride (default: blockIdx.x, gridDim.x)
  int stride = 0;
};

__device__ __forceinline__ int static_unit(const Feed& f, uint32_t i) {
  const long long first = f.first >= 0 ? f.first : blockIdx.x;
  const long long stride = f.stride > 0 ? f.stride : gridDim.x;
  const long long u = first + (long long)i * stride;
  return u < f.nu ? (int)u : -1;
}

__device__ __forceinline__ bool wait_phase(SmemCtl* ctl, uint64_t* bar, uint32_t parity, int32_t* status,
                                           uint64_t limit_ns = kWaitLimitNs);

// Producer side: returns the next unit, -1 when done, -2 on abort.
__device__ __forceinline__ int feed_produce(const Feed& f, SmemCtl* ctl, uint32_t i, int32_t* status) {
  if (f.counter == nullptr) return static_unit(f, i);
  const uint32_t r = i % RING, ph = (i / RING) & 1u;
  if (!wait_phase(ctl, &ctl->unit_empty[r], ph ^ 1u, status)) return -2;
  int u = atomicAdd(f.counter, 1);
  if (u >= f.nu) u = -1;
  ctl->unit_ring[r] = u;
  mbar_arrive(&ctl->unit_full[r]);
  return u;
}

// Consumer side (the MMA thread, or a whole epilogue warp): same sequence as the producer's.
__device__ __forceinline__ int feed_consume(const Feed& f, SmemCtl* ctl, uint32_t i, int32_t* status,
                                            bool whole_warp) {
  if (f.counter == nullptr) return static_unit(f, i);
  const uint32_t r = i % RING, ph = (i / RING) & 1u;
  if (!wait_phase(ctl, &ctl->unit_full[r], ph, status)) return -2;
  const int u = ctl->unit_ring[r];
  if (whole_warp) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl->unit_empty[r]);
  } else {
    mbar_arrive(&ctl->unit_empty[r]);
  }
  return u;
}
static_assert(sizeof(SmemCtl) <= SMEM_CTL_BYTES, "control block too large");

// How one operand tile is fetched for one k-block.
struct Operand {
  const CUtensorMap* map;
  int mn_major;  // 0: K-major (K contiguous); 1: MN-major, one 2-D box {64, 64} per 64-wide column block;
                 // 2: MN-major, all column blocks in one 3-D box {64, 64, rows/64} (map dims
                 //    {64, K, MN/64}, strides {pitch, 128 B}; needs MN % 64 == 0)
  int mn0;       // first row of the tile (coordinate along the MN dimension of the tensor)
  int k0;        // first K coordinate of k-block 0
};

// kblocks k-blocks of BK, in order.  Dense (kbits == nullptr): k-block i is i.  Sparse: kbits is a
// bitmap (kwords 32-bit words) of groups of 2^kg_shift consecutive k-blocks; the tile walks the set
// groups in ascending order, and kblocks (the count of set groups x 2^kg_shift, less what lies past
// the operands' K extent in the last group) ends the walk.  A tile with kblocks == 0 issues no loads
// and no MMAs and takes no accumulator; the kernel's epilogue handles it without waiting on one.
struct TileOps {
  Operand a, b;
  int kblocks;
  const uint32_t* kbits = nullptr;
  int kwords = 0;
  int kg_shift = 0;
};

// Walks the k-blocks of a tile; a sparse bitmap is read one word ahead, so the TMA issue of a group
// seldom waits on the load of its own word.
struct KWalk {
  const uint32_t* bits;
  int words, shift, w, group;
  uint32_t cur, nxt;
  __device__ __forceinline__ explicit KWalk(const TileOps& t)
      : bits(t.kbits), words(t.kwords), shift(t.kg_shift), w(0), group(0), cur(0), nxt(0) {
    if (bits != nullptr && words > 0) {
      cur = __ldg(bits);
      nxt = words > 1 ? __ldg(bits + 1) : 0u;
    }
  }
  __device__ __forceinline__ int kblock(int i) {
    if (bits == nullptr) return i;
    const int off = i & ((1 << shift) - 1);
    if (off == 0) {
      while (cur == 0u && w + 1 < words) {  // next word with a set group (bounded by the bitmap)
        ++w;
        cur = nxt;
        nxt = w + 1 < words ? __ldg(bits + w + 1) : 0u;
      }
      group = 32 * w + __ffs((int)cur) - 1;
      cur &= cur - 1u;
    }
    return (group << shift) + off;
  }
};

__device__ __forceinline__ uint8_t* smem_base_aligned() {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uintptr_t p = reinterpret_cast<uintptr_t>(smem_raw);
  p = (p + 1023) & ~uintptr_t(1023);
  return reinterpret_cast<uint8_t*>(p);
}

// L2-aware unit order over an (m, n) grid of units: m in chunks of `chunk`, and within a chunk
// n-major (all m of the chunk for n = 0, then n = 1, ...).  Units that run at the same time then
// share a few n (the same W tiles) and at most `chunk` m (the same rows of h), so both stay in L2.
// chunk >= n_m gives the plain n-major order.
__device__ __forceinline__ void chunk_decode(int u, int n_m, int n_n, int chunk, int& m, int& n) {
  if (chunk >= n_m) {  // one chunk: plain n-major order
    n = u / n_m;
    m = u - n * n_m;
    return;
  }
  const int per = chunk * n_n;
  const int c = u / per;
  const int local = u - c * per;
  const int rc = min(chunk, n_m - c * chunk);
  n = local / rc;
  m = c * chunk + (local - n * rc);
}

// Bounded wait on an mbarrier phase.  Returns false on abort / timeout.
__device__ __forceinline__ bool wait_phase(SmemCtl* ctl, uint64_t* bar, uint32_t parity, int32_t* status,
                                           uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (ctl->abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicOr(status, ORPO_STATUS_TIMEOUT);
        ctl->abort_flag = 1;
        return false;
      }
    }
  }
}

// Wait used while draining after an abort: short limit, ignores the abort flag.
__device__ __forceinline__ void drain_phase(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

__device__ __forceinline__ void load_operand(const Operand& op, uint64_t* bar, uint8_t* dst, int rows, int kb) {
  if (op.mn_major == 0) {
    tma_load_2d(op.map, bar, dst, op.k0 + kb * BK, op.mn0);
  } else if (op.mn_major == 2) {
    tma_load_3d(op.map, bar, dst, 0, op.k0 + kb * BK, op.mn0 / 64);
  } else {
    const int kk = op.k0 + kb * BK;
#pragma unroll 1
    for (int c = 0; c < rows / 64; ++c) tma_load_2d(op.map, bar, dst + c * (BK * 128), op.mn0 + 64 * c, kk);
  }
}

// Paired mode: this CTA fetches its half of the B tile (rows [rank * BN/2, (rank + 1) * BN/2) of a
// K-major tile, through a map whose box is {64, BN/2}) and multicasts it to both CTAs of the cluster.
__device__ __forceinline__ void load_b_half(const Operand& op, uint64_t* bar, uint8_t* b_dst, int kb, uint32_t rank) {
  tma_load_2d_mc(op.map, bar, b_dst + rank * (B_BYTES / 2), op.k0 + kb * BK, op.mn0 + (int)rank * (BN / 2), 0x3);
}

__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int mn_major, int kk) {
  // K-major: advance 16 elements (32 B) inside the swizzle row; MN-major: advance 16 k-rows (2 KiB)
  return mn_major ? smem_desc_sw128(base + kk * (UMMA_K * 128), BK * 128, 1024)
                  : smem_desc_sw128(base + kk * (UMMA_K * 2), 16, 1024);
}

// ---------------------------------------------------------------- producer (one thread)
template <bool kPair, class Sched>
__device__ void producer_role(const Sched& sched, const Feed& feed, uint8_t* smem, SmemCtl* ctl, int32_t* status) {
  const uint32_t rank = kPair ? cluster_ctarank() : 0;
  uint32_t it = 0;
  bool ok = true;
  for (uint32_t i = 0; ok; ++i) {
    const int u = feed_produce(feed, ctl, i, status);
    if (u < 0) {
      ok = (u == -1);
      break;
    }
    const int len = sched.unit_len(u);
    for (int j = 0; ok && j < len; ++j) {
      const TileOps t = sched.tile(u, j);
      KWalk walk(t);
      for (int i = 0; i < t.kblocks; ++i, ++it) {
        const int kb = walk.kblock(i);
        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
        if (!wait_phase(ctl, &ctl->empty[s], ph ^ 1u, status)) {
          ok = false;
          break;
        }
        uint8_t* a_dst = smem + s * STAGE_BYTES;
        uint8_t* b_dst = a_dst + A_BYTES;
        mbar_arrive_expect_tx(&ctl->full[s], STAGE_BYTES);  // paired: half of B comes from the peer
        load_operand(t.a, &ctl->full[s], a_dst, BM, kb);
        if constexpr (kPair)
          load_b_half(t.b, &ctl->full[s], b_dst, kb, rank);
        else
          load_operand(t.b, &ctl->full[s], b_dst, BN, kb);
      }
    }
  }
  if (!ok) {
    // let the loads already issued land before the CTA can exit
    const uint32_t first = it > STAGES ? it - STAGES : 0;
    for (uint32_t k = first; k < it; ++k) drain_phase(&ctl->full[k % STAGES], (k / STAGES) & 1u);
  }
}

// ---------------------------------------------------------------- MMA issuer (one thread)
template <bool kPair, class Sched>
__device__ void mma_role(const Sched& sched, const Feed& feed, uint8_t* smem, SmemCtl* ctl, uint32_t tmem_base,
                         int32_t* status) {
  uint32_t it = 0, tcount = 0;
  bool ok = true;
  const uint32_t smem0 = smem_u32(smem);
  for (uint32_t i = 0; ok; ++i) {
    const int u = feed_consume(feed, ctl, i, status, false);
    if (u < 0) break;
    const int len = sched.unit_len(u);
    for (int j = 0; ok && j < len; ++j) {
      const TileOps t = sched.tile(u, j);
      if (t.kblocks == 0) continue;  // empty tile: no accumulator (the epilogue knows)
      const uint32_t buf = tcount & 1u, aph = (tcount >> 1) & 1u;
      ++tcount;
      if (!wait_phase(ctl, &ctl->acc_empty[buf], aph ^ 1u, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      const uint32_t idesc = make_idesc_bf16(BM, BN, t.a.mn_major != 0, t.b.mn_major != 0);
      for (int kb = 0; kb < t.kblocks; ++kb, ++it) {
        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
        if (!wait_phase(ctl, &ctl->full[s], ph, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem0 + s * STAGE_BYTES;
        const uint32_t b_base = a_base + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
          umma_bf16(d_tmem, operand_desc(a_base, t.a.mn_major != 0, kk), operand_desc(b_base, t.b.mn_major != 0, kk), idesc,
                    (kb | kk) != 0 ? 1u : 0u);
        }
        // frees the stage once these MMAs have read it (paired: in both CTAs, whose producers
        // write halves of B into each other's stage)
        if constexpr (kPair)
          umma_commit_mc(&ctl->empty[s], 0x3);
        else
          umma_commit(&ctl->empty[s]);
      }
      if (!ok) break;
      umma_commit(&ctl->acc_full[buf]);  // accumulator ready for the epilogue
    }
  }
  // make sure every issued MMA has finished before TMEM is released
  umma_commit(&ctl->drain);
  drain_phase(&ctl->drain, 0);
}

// ---------------------------------------------------------------- epilogue helpers

// Waits until accumulator tile `tcount` is ready; returns its TMEM address for
// this warp's 32 lanes (column 0 of the tile).
__device__ __forceinline__ bool epi_acquire(SmemCtl* ctl, uint32_t tmem_base, uint32_t tcount, int warp,
                                            int32_t* status, uint32_t* taddr) {
  const uint32_t buf = tcount & 1u, aph = (tcount >> 1) & 1u;
  if (!wait_phase(ctl, &ctl->acc_full[buf], aph, status)) return false;
  tc_fence_after();
  *taddr = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + buf * BN;
  return true;
}

__device__ __forceinline__ void epi_release(SmemCtl* ctl, uint32_t tcount) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl->acc_empty[tcount & 1u]);
}

// 32 fp32 values of one row -> 128-byte swizzled row `lane` of a 32 x 128 B staging box
__device__ __forceinline__ void stage_row_f32(uint32_t box, int lane, const uint32_t (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t addr = box + lane * 128 + ((uint32_t)(j ^ (lane & 7)) << 4);
    st_shared_v4(addr, v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
}

// 64 bf16 values (32 packed words) of one row -> swizzled row `lane` of a staging box
__device__ __forceinline__ void stage_row_bf16(uint32_t box, int lane, const uint32_t (&w)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t addr = box + lane * 128 + ((uint32_t)(j ^ (lane & 7)) << 4);
    st_shared_v4(addr, w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

// ---------------------------------------------------------------- CTA driver

// Runs the three roles; `epilogue(smem, ctl, tmem_base, warp, lane)` is the kernel's epilogue loop,
// which walks the units with feed_consume(feed, ctl, i, status, true).
template <bool kPair = false, class Sched, class EpiFn>
__device__ __forceinline__ void run_cta(const Sched& sched, const Feed& feed, int32_t* status, EpiFn&& epilogue) {
  uint8_t* smem = smem_base_aligned();
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + SMEM_CTL_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], kPair ? 2 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->acc_full[b], 1);
      mbar_init(&ctl->acc_empty[b], EPI_WARPS);
    }
    mbar_init(&ctl->drain, 1);
    for (int r = 0; r < RING; ++r) {
      mbar_init(&ctl->unit_full[r], 1);
      mbar_init(&ctl->unit_empty[r], 1 + EPI_WARPS);
    }
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();  // the peer's barriers exist before any multicast reaches them
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) producer_role<kPair>(sched, feed, smem, ctl, status);
  } else if (warp == 1) {
    if (lane == 0) mma_role<kPair>(sched, feed, smem, ctl, tmem_base, status);
  } else {
    epilogue(smem, ctl, tmem_base, warp, lane);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();  // no CTA leaves while its peer may still write into it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace orpo
