// engine.cuh — persistent, warp-specialised tcgen05 GEMM pipeline shared by every
// contraction of the head (forward logits, backward logit recompute, dh and dW).
//
// One CTA per SM.  Warp 0 issues TMA loads into a shared-memory ring of stages,
// warp 1 issues tcgen05.mma (one thread) into a double-buffered TMEM accumulator
// (2 x 256 fp32 columns = all 512 columns), warps 2..5 run the epilogue that the
// kernel supplies, and warps 6..8 run an optional side job of the kernel's (the
// quantised head dequantises its next vocabulary block there) or leave at once.
// Each CTA's accumulator tile is BM x BN = 128 x 256, built from BK = 64 wide
// k-blocks (128-byte swizzle rows) of bf16 operands.
//
// Two forms, chosen by the template argument CG (the tcgen05 CTA group):
//   CG = 1  one CTA per tile.  A stage holds one k-block of A (128 x 64) and B (256 x 64):
//           48 KiB, 4 stages.
//   CG = 2  a 2-CTA cluster computes a 256 x 256 tile with tcgen05.mma.cta_group::2, issued by
//           the even CTA.  Each CTA fetches its own 128 rows of A and its own half (128 rows)
//           of B into its own shared memory with plain (non-multicast) TMA loads, whose bytes
//           are counted on the even CTA's `full` barrier; each CTA's tensor memory receives its
//           128 rows of the accumulator.  A k-block is 32 KiB per CTA, and a stage holds two
//           (64 KiB, 3 stages): one wait and one pair of commits per 128 of K.  With one k-block
//           per stage (six 32 KiB stages) the tensor pipe spent ~9% of its cycles on other
//           work and the forward ran slower than on single CTAs; with two it is active ~90% of
//           cycles.  Every B tile crosses from L2 once per 256 rows instead of once per 128.  The
//           even CTA's commits free the stages and publish the accumulators in both CTAs (two
//           unicast commits, one per CTA); the odd CTA's epilogue warps release accumulators
//           and unit slots by remote arrivals on the even CTA's barriers.
//
// Operand staging in shared memory (per k-block: A 16 KiB, B 32 KiB / CG):
//   K-major operand  [rows, K] with K contiguous: one TMA box {64 (K), rows};
//                    rows at 128 B pitch, 8-row swizzle atoms 1024 B apart (SBO).
//   MN-major operand [K, rows] with rows contiguous: rows/64 TMA boxes {64, 64},
//                    each 64 k-rows x 128 B = 8 KiB (or one 3-D box over all of them);
//                    LBO = 8 KiB between 64-wide column blocks, SBO = 1 KiB between
//                    8-k-row groups.
// Options a kernel picks: sparse K (a bitmap of k-block groups per tile, KWalk; CG = 1 only), a
// static or a dynamic unit feed, and an L2-aware unit order (chunk_decode).
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
constexpr int MAX_STAGES = 6;
constexpr int UMMA_K = 16;
constexpr int EPI_WARPS = 4;
constexpr int SIDE_WARP = 2 + EPI_WARPS;  // the first spare warp
constexpr int SIDE_WARPS = 3;             // one spare warp took ~0.7 ms to dequantise an e4b block; three take
                                          // about as long as the block's contraction
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS + 32 * SIDE_WARPS;
constexpr int TMEM_COLS = 512;

constexpr uint32_t A_BYTES = BM * BK * 2;            // 16 KiB
constexpr uint32_t BOX_BYTES = 4096;                 // one 32-row x 128-byte epilogue staging box
constexpr uint32_t STAGING_PER_WARP = 2 * BOX_BYTES;  // double-buffered
constexpr uint32_t SMEM_CTL_BYTES = 256;

// Shared-memory geometry of one CTA for CTA group CG.
// A stage holds SUBS consecutive k-blocks, each laid out as a one-k-block stage would be: A
// sub-blocks first, then B sub-blocks.  The 2-CTA form takes two per stage (one wait and one commit
// pair per 128 of K), the single-CTA form one.
// W (wide, 2-CTA only): the pair's tile is 256 x 512, two 256-column halves that share the A tile.
// Each CTA fetches 128 rows of each half of B (32 KiB per k-block, one k-block per stage, four
// stages), and the single accumulator takes all 512 TMEM columns: the epilogue no longer overlaps
// the next tile's MMAs, but each k-block moves a quarter fewer operand bytes per flop.
template <int CG, bool W = false>
struct Geo {
  static_assert(CG == 1 || CG == 2, "CTA group 1 or 2");
  static_assert(!W || CG == 2, "wide tiles run on 2-CTA clusters");
  static constexpr int SUBS = W ? 1 : (CG == 2 ? 2 : 1);  // k-blocks per stage
  static constexpr int STAGES = W ? 4 : (CG == 2 ? 3 : 4);
  static constexpr int B_ROWS = (W ? 2 : 1) * BN / CG;    // rows of B this CTA fetches per k-block
  static constexpr int TN = W ? 2 * BN : BN;              // output columns of a tile
  static constexpr int NACC = W ? 1 : 2;                  // accumulators in TMEM
  static constexpr uint32_t B_BYTES = B_ROWS * BK * 2;    // one k-block of B: 32 KiB / CG (wide: 32 KiB)
  static constexpr uint32_t SUB_BYTES = A_BYTES + B_BYTES;  // one k-block of A and B
  static constexpr uint32_t STAGE_BYTES = SUBS * SUB_BYTES;
  static constexpr uint32_t STAGING_OFF = STAGES * STAGE_BYTES;
  static constexpr uint32_t CTL_OFF = STAGING_OFF + EPI_WARPS * STAGING_PER_WARP;
  static constexpr uint32_t SMEM = CTL_OFF + SMEM_CTL_BYTES + 1024;  // + slack to align the base to 1 KiB
  static_assert(STAGES <= MAX_STAGES, "control block holds MAX_STAGES stages");
  static_assert(SMEM <= 232448, "dynamic shared memory per CTA");
};

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far above any legitimate wait

constexpr int RING = 4;                     // unit indices in flight between the roles (dynamic feed)

struct SmemCtl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint64_t unit_full[RING];
  uint64_t unit_empty[RING];
  volatile int unit_ring[RING];
  uint32_t tmem_base;
  volatile int abort_flag;
  volatile int split_last;  // split-K epilogue: this CTA counted a tile's last part
  uint64_t split_in;        // split-K epilogue: the epilogue warps' partial rows are written
  uint64_t split_out;       //                   split_last is set
};
static_assert(sizeof(SmemCtl) <= SMEM_CTL_BYTES, "control block too large");

// Source of work units.  Static: CTA (or 2-CTA cluster) b takes units b, b + G, b + 2G, ...
// Dynamic (counter != nullptr): the producer thread (the even CTA's, in a pair) claims the next unit
// with an atomic add on a zeroed global counter and hands its index to the MMA and epilogue warps
// (and, in a pair, to the odd CTA's producer and epilogue warps) through a RING-deep shared-memory
// ring; index -1 ends the stream.  Every unit is still computed by exactly one CTA or pair.
struct Feed {
  int* counter;
  int nu;
};

template <int CG>
__device__ __forceinline__ int static_unit(const Feed& f, uint32_t i) {
  const long long first = CG == 2 ? (long long)cluster_id_x() : (long long)blockIdx.x;
  const long long stride = CG == 2 ? (long long)num_clusters_x() : (long long)gridDim.x;
  const long long u = first + (long long)i * stride;
  return u < f.nu ? (int)u : -1;
}

template <int CG>
__device__ __forceinline__ bool wait_phase(SmemCtl* ctl, uint64_t* bar, uint32_t parity, int32_t* status,
                                           uint64_t limit_ns = kWaitLimitNs);

// rank of this CTA in its pair (0 for CG = 1)
template <int CG>
__device__ __forceinline__ uint32_t pair_rank() {
  if constexpr (CG == 2)
    return cluster_ctarank() & 1u;
  else
    return 0u;
}

// An arrival on barrier `bar` of the even CTA: local for the even CTA (and CG = 1), remote for the odd.
template <int CG>
__device__ __forceinline__ void arrive_leader(uint64_t* bar, uint32_t rank) {
  if (CG == 2 && rank != 0)
    mbar_arrive_cluster(mapa_u32(smem_u32(bar), 0));
  else
    mbar_arrive(bar);
}

// Producer side: returns the next unit, -1 when done, -2 on abort.  In a pair the odd CTA's producer
// receives the even one's claims like the other consumers.
template <int CG>
__device__ __forceinline__ int feed_consume(const Feed& f, SmemCtl* ctl, uint32_t i, int32_t* status,
                                            bool whole_warp, uint32_t rank);
template <int CG>
__device__ __forceinline__ int feed_produce(const Feed& f, SmemCtl* ctl, uint32_t i, int32_t* status, uint32_t rank) {
  if (f.counter == nullptr) return static_unit<CG>(f, i);
  if (CG == 2 && rank != 0) return feed_consume<CG>(f, ctl, i, status, false, rank);
  const uint32_t r = i % RING, ph = (i / RING) & 1u;
  if (!wait_phase<CG>(ctl, &ctl->unit_empty[r], ph ^ 1u, status)) return -2;
  int u = atomicAdd(f.counter, 1);
  if (u >= f.nu) u = -1;
  ctl->unit_ring[r] = u;
  if constexpr (CG == 2) {  // the odd CTA's copy of the slot, then its notice
    st_shared_cluster_u32(mapa_u32(smem_u32((const void*)&ctl->unit_ring[r]), 1), (uint32_t)u);
    mbar_arrive_cluster(mapa_u32(smem_u32(&ctl->unit_full[r]), 1));
  }
  mbar_arrive(&ctl->unit_full[r]);
  return u;
}

// Consumer side (the MMA thread, a whole epilogue warp, or the odd CTA's producer): same sequence as
// the producer's.
template <int CG>
__device__ __forceinline__ int feed_consume(const Feed& f, SmemCtl* ctl, uint32_t i, int32_t* status,
                                            bool whole_warp, uint32_t rank) {
  if (f.counter == nullptr) return static_unit<CG>(f, i);
  const uint32_t r = i % RING, ph = (i / RING) & 1u;
  if (!wait_phase<CG>(ctl, &ctl->unit_full[r], ph, status)) return -2;
  const int u = ctl->unit_ring[r];
  if (whole_warp) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) arrive_leader<CG>(&ctl->unit_empty[r], rank);
  } else {
    arrive_leader<CG>(&ctl->unit_empty[r], rank);
  }
  return u;
}

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
// In a pair (CG = 2) a tile is this CTA's part of the pair's tile: its own 128 rows of A and its own
// half of B; both CTAs' parts agree on kblocks and on the operand layouts.
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

// Bounded wait on an mbarrier phase.  Returns false on abort / timeout.  In a pair every barrier may
// receive arrivals from the other CTA, so the wait acquires at cluster scope.
template <int CG>
__device__ __forceinline__ bool try_wait_cg(uint64_t* bar, uint32_t parity) {
  if constexpr (CG == 2)
    return mbar_try_wait_cluster(bar, parity);
  else
    return mbar_try_wait(bar, parity);
}

template <int CG>
__device__ __forceinline__ bool wait_phase(SmemCtl* ctl, uint64_t* bar, uint32_t parity, int32_t* status,
                                           uint64_t limit_ns) {
  if (try_wait_cg<CG>(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (try_wait_cg<CG>(bar, parity)) return true;
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
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

// One operand tile of one k-block into `dst`; its bytes are counted on the barrier at shared::cluster
// address `bar` (this CTA's own barrier for CG = 1, the even CTA's for CG = 2).
template <int CG>
__device__ __forceinline__ void load_operand(const Operand& op, uint32_t bar, uint8_t* dst, int rows, int kb) {
  const int kk = op.k0 + kb * BK;
  if constexpr (CG == 2) {
    if (op.mn_major == 0) {
      tma_load_2d_cg2(op.map, bar, dst, kk, op.mn0);
    } else if (op.mn_major == 2) {
      tma_load_3d_cg2(op.map, bar, dst, 0, kk, op.mn0 / 64);
    } else {
#pragma unroll 1
      for (int c = 0; c < rows / 64; ++c) tma_load_2d_cg2(op.map, bar, dst + c * (BK * 128), op.mn0 + 64 * c, kk);
    }
  } else {
    if (op.mn_major == 0) {
      tma_load_2d(op.map, bar, dst, kk, op.mn0);
    } else if (op.mn_major == 2) {
      tma_load_3d(op.map, bar, dst, 0, kk, op.mn0 / 64);
    } else {
#pragma unroll 1
      for (int c = 0; c < rows / 64; ++c) tma_load_2d(op.map, bar, dst + c * (BK * 128), op.mn0 + 64 * c, kk);
    }
  }
}

__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int mn_major, int kk) {
  // K-major: advance 16 elements (32 B) inside the swizzle row; MN-major: advance 16 k-rows (2 KiB)
  return mn_major ? smem_desc_sw128(base + kk * (UMMA_K * 128), BK * 128, 1024)
                  : smem_desc_sw128(base + kk * (UMMA_K * 2), 16, 1024);
}

// ---------------------------------------------------------------- producer (one thread per CTA)
template <int CG, bool W, class Sched>
__device__ void producer_role(const Sched& sched, const Feed& feed, uint8_t* smem, SmemCtl* ctl, int32_t* status,
                              uint32_t rank) {
  using G = Geo<CG, W>;
  uint32_t it = 0;
  bool ok = true;
  for (uint32_t i = 0; ok; ++i) {
    const int u = feed_produce<CG>(feed, ctl, i, status, rank);
    if (u < 0) {
      ok = (u == -1);
      break;
    }
    const int len = sched.unit_len(u);
    for (int j = 0; ok && j < len; ++j) {
      const TileOps t = sched.tile(u, j);
      KWalk walk(t);
      for (int i = 0; i < t.kblocks; ++i, ++it) {  // one stage per pass: i advances by SUBS
        const int kb = walk.kblock(i);
        const uint32_t s = it % G::STAGES, ph = (it / G::STAGES) & 1u;
        if (!wait_phase<CG>(ctl, &ctl->empty[s], ph ^ 1u, status)) {
          ok = false;
          break;
        }
        uint8_t* a_dst = smem + s * G::STAGE_BYTES;
        uint8_t* b_dst = a_dst + G::SUBS * A_BYTES;
        const int nv = min(G::SUBS, t.kblocks - i);  // k-blocks in this stage
        // the even CTA's full barrier counts both CTAs' bytes; only the even CTA arrives on it
        if (rank == 0) mbar_arrive_expect_tx(&ctl->full[s], (uint32_t)(nv * CG) * G::SUB_BYTES);
        const uint32_t bar = CG == 2 ? mapa_u32(smem_u32(&ctl->full[s]), 0) : smem_u32(&ctl->full[s]);
        for (int j = 0; j < nv; ++j) {
          const int kbj = j == 0 ? kb : walk.kblock(i + j);
          load_operand<CG>(t.a, bar, a_dst + j * A_BYTES, BM, kbj);
          if constexpr (W) {  // the two halves of the wide tile: B rows mn0 and mn0 + BN
            Operand b2 = t.b;
            b2.mn0 += BN;
            load_operand<CG>(t.b, bar, b_dst + j * G::B_BYTES, BN / CG, kbj);
            load_operand<CG>(b2, bar, b_dst + j * G::B_BYTES + G::B_BYTES / 2, BN / CG, kbj);
          } else {
            load_operand<CG>(t.b, bar, b_dst + j * G::B_BYTES, G::B_ROWS, kbj);
          }
        }
        i += nv - 1;
      }
    }
  }
  if (!ok && rank == 0) {
    // let the loads already issued land before the CTA can exit (in a pair the even CTA's barrier
    // also counts the odd CTA's loads)
    const uint32_t first = it > G::STAGES ? it - G::STAGES : 0;
    for (uint32_t k = first; k < it; ++k) drain_phase(&ctl->full[k % G::STAGES], (k / G::STAGES) & 1u);
  }
}

// ---------------------------------------------------------------- MMA issuer (one thread; the even CTA's in a pair)
template <int CG>
__device__ __forceinline__ void commit_both(uint64_t* bar) {
  if constexpr (CG == 2) {
    umma_commit_cg2(smem_u32(bar));
    umma_commit_cg2(mapa_u32(smem_u32(bar), 1));
  } else {
    umma_commit(bar);
  }
}

template <int CG, bool W, class Sched>
__device__ void mma_role(const Sched& sched, const Feed& feed, uint8_t* smem, SmemCtl* ctl, uint32_t tmem_base,
                         int32_t* status) {
  using G = Geo<CG, W>;
  uint32_t it = 0, tcount = 0;
  bool ok = true;
  const uint32_t smem0 = smem_u32(smem);
  for (uint32_t i = 0; ok; ++i) {
    const int u = feed_consume<CG>(feed, ctl, i, status, false, 0);
    if (u < 0) break;
    const int len = sched.unit_len(u);
    for (int j = 0; ok && j < len; ++j) {
      const TileOps t = sched.tile(u, j);
      if (t.kblocks == 0) continue;  // empty tile: no accumulator (the epilogue knows)
      const uint32_t buf = G::NACC == 2 ? tcount & 1u : 0u, aph = G::NACC == 2 ? (tcount >> 1) & 1u : tcount & 1u;
      ++tcount;
      if (!wait_phase<CG>(ctl, &ctl->acc_empty[buf], aph ^ 1u, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      const uint32_t idesc = make_idesc_bf16(BM * CG, BN, t.a.mn_major != 0, t.b.mn_major != 0);
      for (int kb = 0; kb < t.kblocks; kb += G::SUBS, ++it) {
        const uint32_t s = it % G::STAGES, ph = (it / G::STAGES) & 1u;
        if (!wait_phase<CG>(ctl, &ctl->full[s], ph, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int nv = min(G::SUBS, t.kblocks - kb);
#pragma unroll
        for (int j = 0; j < G::SUBS; ++j) {
          if (j < nv) {
            const uint32_t a_base = smem0 + s * G::STAGE_BYTES + j * A_BYTES;
            const uint32_t b_base = smem0 + s * G::STAGE_BYTES + G::SUBS * A_BYTES + j * G::B_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              const uint64_t ad = operand_desc(a_base, t.a.mn_major != 0, kk);
              const uint64_t bd = operand_desc(b_base, t.b.mn_major != 0, kk);
              if constexpr (CG == 2)
                umma_bf16_cg2(d_tmem, ad, bd, idesc, (kb | j | kk) != 0 ? 1u : 0u);
              else
                umma_bf16(d_tmem, ad, bd, idesc, (kb | j | kk) != 0 ? 1u : 0u);
              if constexpr (W)  // the second half: B rows BN on, accumulator columns BN on
                umma_bf16_cg2(d_tmem + BN, ad, operand_desc(b_base + G::B_BYTES / 2, t.b.mn_major != 0, kk), idesc,
                              (kb | j | kk) != 0 ? 1u : 0u);
            }
          }
        }
        commit_both<CG>(&ctl->empty[s]);  // frees the stage (in both CTAs) once these MMAs have read it
      }
      if (!ok) break;
      commit_both<CG>(&ctl->acc_full[buf]);  // accumulator ready for the epilogue warps (of both CTAs)
    }
  }
  // make sure every issued MMA has finished before TMEM is released
  if constexpr (CG == 2)
    umma_commit_cg2(smem_u32(&ctl->drain));
  else
    umma_commit(&ctl->drain);
  drain_phase(&ctl->drain, 0);
}

// ---------------------------------------------------------------- epilogue helpers

// Waits until accumulator tile `tcount` is ready; returns its TMEM address for
// this warp's 32 lanes (column 0 of the tile).
template <int CG = 1, bool W = false>
__device__ __forceinline__ bool epi_acquire(SmemCtl* ctl, uint32_t tmem_base, uint32_t tcount, int warp,
                                            int32_t* status, uint32_t* taddr) {
  const uint32_t buf = W ? 0u : tcount & 1u, aph = W ? tcount & 1u : (tcount >> 1) & 1u;
  if (!wait_phase<CG>(ctl, &ctl->acc_full[buf], aph, status)) return false;
  tc_fence_after();
  *taddr = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + buf * BN;
  return true;
}

// The accumulator's counter lives in the even CTA: the odd CTA's warps arrive on it remotely.
template <int CG = 1, bool W = false>
__device__ __forceinline__ void epi_release(SmemCtl* ctl, uint32_t tcount, uint32_t rank = 0) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) arrive_leader<CG>(&ctl->acc_empty[W ? 0u : tcount & 1u], rank);
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

// Runs the roles; `epilogue(staging, ctl, tmem_base, warp, lane, rank)` is the kernel's epilogue loop
// (`staging` is the base of the epilogue warps' staging boxes, STAGING_PER_WARP bytes per warp),
// which walks the units with feed_consume<CG>(feed, ctl, i, status, true, rank); `side()` is the
// spare warps' job, independent of the pipeline (it touches no barrier, TMEM or staging box).
// CG = 2 must run in 2-CTA clusters.
template <int CG, bool W = false, class Sched, class EpiFn, class SideFn>
__device__ __forceinline__ void run_cta(const Sched& sched, const Feed& feed, int32_t* status, EpiFn&& epilogue,
                                        SideFn&& side) {
  using G = Geo<CG, W>;
  uint8_t* smem = smem_base_aligned();
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + G::CTL_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = pair_rank<CG>();
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->acc_full[b], 1);
      mbar_init(&ctl->acc_empty[b], CG * EPI_WARPS);  // pair: both CTAs' epilogue warps
    }
    mbar_init(&ctl->drain, 1);
    mbar_init(&ctl->split_in, EPI_WARPS);
    mbar_init(&ctl->split_out, 1);
    for (int r = 0; r < RING; ++r) {
      mbar_init(&ctl->unit_full[r], 1);
      // MMA thread + epilogue warps; pair: + the odd CTA's producer and epilogue warps
      mbar_init(&ctl->unit_empty[r], CG == 2 ? 2 + 2 * EPI_WARPS : 1 + EPI_WARPS);
    }
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(&ctl->tmem_base, TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the other CTA's barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) producer_role<CG, W>(sched, feed, smem, ctl, status, rank);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) mma_role<CG, W>(sched, feed, smem, ctl, tmem_base, status);
  } else if (warp < SIDE_WARP) {
    epilogue(smem + G::STAGING_OFF, ctl, tmem_base, warp, lane, rank);
  } else {
    side();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // pair: the even CTA's MMAs read the odd CTA's shared memory and write its tensor memory, so neither
  // leaves (or frees its columns) before both are done
  if constexpr (CG == 2) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host: launches

// Launches an engine kernel of CTA group `cg`: CG = 2 kernels run as 2-CTA clusters, `grid` counting
// CTAs (even).
template <class... Params, class... Args>
inline cudaError_t launch_engine(void (*kernel)(Params...), int cg, int grid, uint32_t smem, cudaStream_t st,
                                 Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cg;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cg == 2 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Number of 2-CTA clusters of `kernel` (one CTA per SM) that fit on the current device at once; 0 when
// none can run.
template <class Kernel>
inline int max_pair_clusters(Kernel kernel, uint32_t smem) {
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
  cudaGetLastError();
  return n;
}

}  // namespace orpo
