// head_bwd.cu — backward of the flash-CCE head and the generic fp32-output GEMM.
//
// Fused-head spec, backward bullet: recompute the vocabulary tiles, rebuild the
// softmax from the saved lse, form g * (onehot - softmax) * sech^2 and contract
// it into dh (and, here, dW).  The "Steel flash-CCE — handoff" page accumulated
// dh with float atomics across vocabulary blocks; here the bf16 logit gradient
// of one (row block, vocabulary block) is streamed through a bounded workspace
// block S and contracted with two large-K GEMMs per block:
//   recompute kernel : S = bf16(dZ[m0:m0+Mc, v0:v0+Vc])             (K = d)
//   gemm kernel      : dh[m0 rows]  (+)= S   W[v0 rows]             (K = Vc)
//                      dW[v0 rows]  (+)= S^T h[m0 rows]             (K = Mc)
// Each output tile is written by exactly one CTA per launch (TMA store, or TMA
// reduce-add after the first block), so results are bitwise reproducible.
#include "engine.cuh"
#include "internal.h"

namespace orpo {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ================================================================ recompute -> S
// Unit = (M unit, vocabulary tile): an M unit is one row tile (CG = 1) or a pair's two row tiles
// (CG = 2, CTA rank r taking tile 2m + r; the pair shares the W tile, half fetched by each CTA).
template <int CG>
struct RecSched {
  const CUtensorMap* mh;
  const CUtensorMap* mw;
  int m0, v0, n_mt, n_vt, kblocks;
  int w_row0;        // row of the W map that holds vocabulary column v0
  const int* list;   // backward skips (CG = 1): the tiles to compute (vt * n_mt + mt, in unit order), or nullptr
  const int* count;  // number of entries of list
  int chunk;         // M units per L2 chunk (chunk_decode)
  int32_t* status = nullptr;
  int rank = 0;      // this CTA's rank in its pair (0 for CG = 1)
  __device__ int n_mu() const { return (n_mt + CG - 1) / CG; }
  __device__ int num_units() const { return list ? __ldg(count) : n_mu() * n_vt; }
  // unit u -> x = vt * n_mu + mu
  __device__ int tile_index(int u) const {
    int x;
    if (list) {
      x = in_bounds(status, u, kMaxTiles) ? __ldg(list + u) : 0;
    } else {
      int mu, vt;
      chunk_decode(u, n_mu(), n_vt, chunk, mu, vt);
      x = vt * n_mu() + mu;
    }
    return in_bounds(status, x, n_mu() * n_vt) ? x : 0;
  }
  __device__ int unit_len(int) const { return 1; }
  __device__ TileOps tile(int u, int) const {
    const int x = tile_index(u);
    const int vt = x / n_mu(), mt = (x - vt * n_mu()) * CG + rank;
    TileOps t;
    t.a = Operand{mh, 0, m0 + mt * BM, 0};
    t.b = Operand{mw, 0, w_row0 + vt * BN + rank * (BN / CG), 0};
    t.kblocks = kblocks;
    return t;
  }
};

struct RecArgs {
  const int32_t* targets;
  const uint8_t* mask;
  const float* lse;
  const float* g;
  int M, V;
  float softcap;
  int32_t* status;
  float eps;           // coefficient filter threshold (filter instances only)
  uint32_t* rowbits;   // filter instances: kept tiles by row tile, [n_mt][ld_row] bitmap over vt
  uint32_t* colbits;   //                   and by vocabulary tile, [n_vt][ld_col] bitmap over mt
  int ld_row, ld_col;
  DequantJob side;     // spare warps: dequantise the next vocabulary block (quantised head), or nothing
};

// dZ for 32 accumulator values of one row starting at vocabulary column col0;
// writes 16 packed bf16 pairs into w[0..15].
//   softcap on : t = tanh(z / c) = 1 - 2q, q = 1 / (1 + e^{2z/c}), z~ = c t,
//                sech^2(z/c) = 4q(1 - q); for caps above kCapExpMax, |z / c| < 1/8 uses the
//                Taylor form of t and 1 - t^2 (the forward's hybrid form)
//   dZ = g sech^2 (onehot - 2^(x - lse2)),  x = z~ log2(e)
constexpr int kCapOff = 0, kCapExp = 1, kCapHybrid = 2;  // softcap forms, as in the forward
constexpr float kCapExpMax = 64.f;

template <int cap, bool kFilter>
__device__ __forceinline__ void dz_chunk(const uint32_t (&r)[32], int col0, int V, int y, float gval, float lse2,
                                         float inv_c, float cl2, uint32_t* w, float& amax) {
  float dz[32], sl[32];
  if constexpr (cap == kCapExp) {
    const float K = 2.f * kLog2e * inv_c, A = cl2 - lse2, B2 = 2.f * cl2;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float q = rcp_approx(1.f + ex2_approx(__uint_as_float(r[i]) * K));
      sl[i] = 4.f * q * (1.f - q);
      dz[i] = -(gval * sl[i]) * ex2_approx(fmaf(-B2, q, A));  // 2^(x - lse2), x = A' - 2A' q
    }
  } else if constexpr (cap == kCapHybrid) {
    bool big = false;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      dz[i] = __uint_as_float(r[i]) * inv_c;  // u = z / c
      big |= fabsf(dz[i]) >= kTanhSmall;
    }
    if (__any_sync(0xffffffffu, big)) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float u = dz[i];
        float q = 0.5f, t;
        if (fabsf(u) < kTanhSmall) {
          t = tanh_small(u);
          sl[i] = fmaf(-t, t, 1.f);
        } else {
          t = tanh_exp(u, &q);
          sl[i] = 4.f * q * (1.f - q);
        }
        dz[i] = t * cl2;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float t = tanh_small(dz[i]);
        sl[i] = fmaf(-t, t, 1.f);
        dz[i] = t * cl2;
      }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) dz[i] = -(gval * sl[i]) * ex2_approx(dz[i] - lse2);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      sl[i] = 1.f;
      dz[i] = -gval * ex2_approx(__uint_as_float(r[i]) * kLog2e - lse2);
    }
  }
  if ((unsigned)(y - col0) < 32u) {  // the target column lies in this chunk: add g * sech^2 there
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i == y - col0) dz[i] += gval * sl[i];
  }
  if (col0 + 32 > V) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i >= V) dz[i] = 0.f;
  }
  if constexpr (kFilter) {
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(dz[i]));
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(dz[2 * i], dz[2 * i + 1]);
}

// kFilter: the coefficient filter of the backward skips ("Steel flash-CCE — handoff" §E).  A tile
// is kept (its bits set in rowbits and colbits) when some row with g != 0 has |dZ| >= eps |g|,
// i.e. an entry of (onehot - p) sech^2 reaches eps; the dh / dW GEMMs read only kept tiles.
template <int cap, bool kFilter, int CG>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    rec_kernel(const __grid_constant__ CUtensorMap mh, const __grid_constant__ CUtensorMap mw,
               const __grid_constant__ CUtensorMap ms, RecSched<CG> sched, RecArgs p) {
  static_assert(!(kFilter && CG == 2), "the backward skips run on single-CTA tiles");
  sched.mh = &mh;
  sched.mw = &mw;
  sched.status = p.status;
  sched.rank = (int)pair_rank<CG>();
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&mh);
    tma_prefetch_desc(&mw);
    tma_prefetch_desc(&ms);
  }
  const Feed feed{nullptr, sched.num_units()};
  run_cta<CG>(sched, feed, p.status, [&](uint8_t* stg, SmemCtl* ctl, uint32_t tmem_base, int warp, int lane,
                                         uint32_t rank) {
    const int q = warp & 3;
    uint8_t* stage_ptr = stg + (warp - 2) * STAGING_PER_WARP;
    const uint32_t staging = smem_u32(stage_ptr);
    const float inv_c = cap != kCapOff ? 1.f / p.softcap : 0.f;
    const float cl2 = p.softcap * kLog2e;
    uint32_t tcount = 0, nstore = 0;
    for (uint32_t i = 0;; ++i, ++tcount) {
      const int u = feed_consume<CG>(feed, ctl, i, p.status, true, rank);
      if (u < 0) break;
      const int x = sched.tile_index(u);
      const int vt = x / sched.n_mu(), mt = (x - vt * sched.n_mu()) * CG + (int)rank;
      uint32_t taddr;
      if (mt >= sched.n_mt) {  // the empty half of a pair whose row-tile count is odd: nothing to store
        if (!epi_acquire<CG>(ctl, tmem_base, tcount, warp, p.status, &taddr)) break;
        epi_release<CG>(ctl, tcount, rank);
        continue;
      }
      const int srow = mt * BM + 32 * q;  // first scratch row of this warp
      const int row = sched.m0 + srow + lane;
      float gval = 0.f, lse2 = 0.f;
      int y = -1;
      if (row < p.M && p.mask[row] != 0) {
        gval = p.g[row];
        y = p.targets[row];
        if (y < 0 || y >= p.V) {
          atomicOr(p.status, ORPO_STATUS_TARGET);
          y = -1;
        }
        lse2 = p.lse[row] * kLog2e;
      }
      const bool warp_zero = __all_sync(0xffffffffu, gval == 0.f);
      if (!epi_acquire<CG>(ctl, tmem_base, tcount, warp, p.status, &taddr)) break;
      const int vcol0 = sched.v0 + vt * BN;  // global vocabulary column of the tile
      float amax = 0.f;                       // largest |dZ| of this row in the tile (filter)
      uint32_t ra[32], rb[32];
      if (!warp_zero) tmem_ld32(taddr, ra);
#pragma unroll 1
      for (int gi = 0; gi < BN / 64; ++gi) {
        uint32_t w[32];
        if (warp_zero) {
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = 0u;
        } else {
          tmem_ld_wait(ra);
          tmem_ld32(taddr + gi * 64 + 32, rb);
          dz_chunk<cap, kFilter>(ra, vcol0 + gi * 64, p.V, y, gval, lse2, inv_c, cl2, w, amax);
          tmem_ld_wait(rb);
          if (gi + 1 < BN / 64) tmem_ld32(taddr + gi * 64 + 64, ra);
          dz_chunk<cap, kFilter>(rb, vcol0 + gi * 64 + 32, p.V, y, gval, lse2, inv_c, cl2, w + 16, amax);
        }
        const uint32_t box = staging + (nstore & 1u) * BOX_BYTES;
        if (lane == 0) bulk_wait_group_read<1>();  // the store that used this buffer has read it
        __syncwarp();
        stage_row_bf16(box, lane, w);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&ms, stage_ptr + (nstore & 1u) * BOX_BYTES, vt * BN + gi * 64, srow);
          bulk_commit_group();
        }
        ++nstore;
      }
      epi_release<CG>(ctl, tcount, rank);
      if constexpr (kFilter) {
        const bool keep = gval != 0.f && amax >= p.eps * fabsf(gval);
        if (__any_sync(0xffffffffu, keep) && lane == 0) {
          if (in_bounds(p.status, mt, sched.n_mt) && in_bounds(p.status, vt >> 5, p.ld_row))
            atomicOr(p.rowbits + mt * p.ld_row + (vt >> 5), 1u << (vt & 31));
          if (in_bounds(p.status, vt, sched.n_vt) && in_bounds(p.status, mt >> 5, p.ld_col))
            atomicOr(p.colbits + vt * p.ld_col + (mt >> 5), 1u << (mt & 31));
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }, [&] { side_dequant(p.side, p.status); });
}

// ================================================================ fp32-output GEMM (dh, dW, diagnostic)
struct GemmClass {
  int a_map, a_mn, a_mn_base, a_k_base;
  int b_map, b_mn, b_mn_base, b_k_base;
  int out_map, out_row_base, out_col_base, reduce;
  int out_rows, out_cols;
  int n_mt, n_nt, kblocks;
  int mt_major;
  // sparse K (backward skips): bitmap (mt >> list_shift) of kept groups of 2^kg_shift k-blocks,
  // kwords words each; ngroups groups in all, the last holding clip k-blocks fewer than the others
  // (past the operands' K extent).  kbits == nullptr: dense, kblocks.
  const uint32_t* kbits;
  int kwords, list_shift, kg_shift, ngroups, clip;
  int kbits_rows;  // bitmaps at kbits
  // split K (dense classes only): each output tile's K range in ksplit parts, each part a unit that
  // writes its fp32 partial tile to part[tile][part]; the tile's last part to finish (counted in
  // cnt[tile], which it resets to 0) sums the parts in part order and writes the tile.
  int ksplit;
  float* part;
  int* cnt;
};

// Unit = (class, M unit, N tile); an M unit is one 128-row output tile (CG = 1) or a pair's two
// (CG = 2: CTA rank r takes output tile 2m + r and fetches half of the B tile).
template <int CG, bool W = false>
struct GemmSched {
  static constexpr int TN = Geo<CG, W>::TN;  // output columns of a tile (512 for the wide form)
  const CUtensorMap* maps[6];
  GemmClass cls[2];
  int32_t* status;
  int rank = 0;  // this CTA's rank in its pair (0 for CG = 1)
  // constant-index selection keeps the pointer table in registers (no local-memory copy)
  __device__ __forceinline__ const CUtensorMap* map(int i) const {
    switch (i) {
      case 0: return maps[0];
      case 1: return maps[1];
      case 2: return maps[2];
      case 3: return maps[3];
      case 4: return maps[4];
      default: return maps[5];
    }
  }
  // class k by value, read through constant indices (no dynamically indexed copy of the table)
  __device__ __forceinline__ GemmClass pick(int k) const {
    GemmClass c;
    if (k == 0)
      c = cls[0];
    else
      c = cls[1];
    return c;
  }
  __device__ static int n_mu(const GemmClass& c) { return (c.n_mt + CG - 1) / CG; }
  __device__ int n0() const { return n_mu(cls[0]) * cls[0].n_nt * cls[0].ksplit; }
  __device__ int num_units() const { return n0() + n_mu(cls[1]) * cls[1].n_nt * cls[1].ksplit; }
  __device__ int unit_len(int) const { return 1; }
  // mt: this CTA's output row tile (c.n_mt or more: the empty half of a pair whose tile count is odd);
  // ks: the part of the tile's K range (0 without split K).  The parts of a tile are consecutive units.
  __device__ void decode(int u, int& k, int& mt, int& nt, int& ks) const {
    k = u < n0() ? 0 : 1;
    const GemmClass c = pick(k);
    const int w = k == 0 ? u : u - n0();
    const int v = w / c.ksplit;
    ks = w - v * c.ksplit;
    int mu;
    if (c.mt_major) {
      mu = v / c.n_nt;
      nt = v - mu * c.n_nt;
    } else {
      nt = v / n_mu(c);
      mu = v - nt * n_mu(c);
    }
    mt = mu * CG + rank;
  }
  // k-blocks [kb_first(c, ks), kb_first(c, ks + 1)) form part ks
  __device__ static int kb_first(const GemmClass& c, int ks) {
    return (int)(((long long)ks * c.kblocks) / c.ksplit);
  }
  __device__ TileOps tile(int u, int) const {
    int k, mt, nt, ks;
    decode(u, k, mt, nt, ks);
    const GemmClass c = pick(k);
    const int kb0 = kb_first(c, ks);
    TileOps t;
    t.a = Operand{map(c.a_map), c.a_mn, c.a_mn_base + mt * BM, c.a_k_base + kb0 * BK};
    t.b = Operand{map(c.b_map), c.b_mn, c.b_mn_base + nt * TN + rank * (BN / CG), c.b_k_base + kb0 * BK};
    t.kblocks = kb_first(c, ks + 1) - kb0;
    if (CG == 1 && c.kbits != nullptr) {
      const int br = in_bounds(status, mt >> c.list_shift, c.kbits_rows) ? mt >> c.list_shift : 0;
      const uint32_t* bits = c.kbits + (size_t)br * c.kwords;
      int n = 0;
      for (int w = 0; w < c.kwords; ++w) n += __popc(__ldg(bits + w));
      const int lg = c.ngroups - 1;
      const bool last = (__ldg(bits + (lg >> 5)) >> (lg & 31)) & 1u;
      t.kbits = bits;
      t.kwords = c.kwords;
      t.kg_shift = c.kg_shift;
      t.kblocks = (n << c.kg_shift) - (last ? c.clip : 0);
    }
    return t;
  }
};

// One part of a split-K tile (`c.ksplit` > 1), run by the four epilogue warps: this CTA's fp32
// accumulator goes to the part's slot (float4 index (col / 4) * BM + row: a warp's stores of one
// column group are contiguous); after a fence, one thread counts the part in.  The part counted last
// (whichever CTA runs it) reads every part's slot in part order (ld.global.cg: from L2, written by
// other SMs), adds them in that order, writes the tile as the unsplit epilogue would (store or
// reduce-add) and resets the counter for the next launch.  No CTA waits for another, and the sum
// is the same whichever part is last, so results stay bitwise reproducible.  The four warps meet on
// two mbarriers (split_in, split_out; phase = nsplit & 1, the CTA's split parts so far) through the
// engine's bounded wait, so a timeout elsewhere cannot leave a warp waiting.
constexpr int kSplitMaxParts = 8;  // parts per tile at most (the host's kSplitMax)

template <int CG>
__device__ __forceinline__ void split_part(const GemmClass& c, SmemCtl* ctl, uint32_t taddr, int mt, int nt, int ks,
                                           int q, int warp, int lane, int orow, int ocol0, const CUtensorMap* out,
                                           uint32_t staging, uint8_t* stage_ptr, uint32_t& nstore, uint32_t tcount,
                                           uint32_t rank, uint32_t& nsplit, int32_t* status) {
  constexpr int kSlot = BM * BN / 4;  // float4 per partial tile
  if (mt >= c.n_mt) {                 // the empty half of an odd pair: no tile, no count
    epi_release<CG>(ctl, tcount, rank);
    return;
  }
  const int tile = mt * c.n_nt + nt;
  if (!in_bounds(status, tile, (int64_t)c.n_mt * c.n_nt) || !in_bounds(status, ks, c.ksplit)) {
    epi_release<CG>(ctl, tcount, rank);
    return;
  }
  const int r = 32 * q + lane;  // this thread's row of the tile
  float4* slots = reinterpret_cast<float4*>(c.part) + (size_t)tile * c.ksplit * kSlot;
  float4* mine = slots + (size_t)ks * kSlot;
  uint32_t v[32];
#pragma unroll 1
  for (int ch = 0; ch < BN / 32; ++ch) {
    tmem_ld32(taddr + ch * 32, v);
    tmem_ld_wait(v);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      mine[(ch * 8 + j) * BM + r] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
  }
  epi_release<CG>(ctl, tcount, rank);
  __threadfence();
  __syncwarp();
  const uint32_t par = nsplit & 1u;
  ++nsplit;
  if (lane == 0) mbar_arrive(&ctl->split_in);
  if (warp == 2) {  // counts the part in once all four warps' rows are written
    const bool in = wait_phase<CG>(ctl, &ctl->split_in, par, status);
    if (lane == 0) {
      ctl->split_last = in && atomicAdd(c.cnt + tile, 1) == c.ksplit - 1 ? 1 : 0;
      mbar_arrive(&ctl->split_out);
    }
  }
  if (!wait_phase<CG>(ctl, &ctl->split_out, par, status) || !ctl->split_last) return;
  __threadfence();
  if (orow < c.out_rows) {
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
      const int col = ocol0 + ch * 32;
      if (col >= c.out_cols) break;
#pragma unroll
      for (int j = 0; j < 8; j += 2) {  // two float4 columns at a time: every part's loads in flight at once
        float4 x[2][kSplitMaxParts];
#pragma unroll
        for (int p = 0; p < kSplitMaxParts; ++p) {
          if (p < c.ksplit) {
            x[0][p] = __ldcg(slots + (size_t)p * kSlot + (ch * 8 + j) * BM + r);
            x[1][p] = __ldcg(slots + (size_t)p * kSlot + (ch * 8 + j + 1) * BM + r);
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float4 acc = x[e][0];
#pragma unroll
          for (int p = 1; p < kSplitMaxParts; ++p) {
            if (p < c.ksplit) {  // in part order
              acc.x += x[e][p].x;
              acc.y += x[e][p].y;
              acc.z += x[e][p].z;
              acc.w += x[e][p].w;
            }
          }
          v[4 * (j + e)] = __float_as_uint(acc.x);
          v[4 * (j + e) + 1] = __float_as_uint(acc.y);
          v[4 * (j + e) + 2] = __float_as_uint(acc.z);
          v[4 * (j + e) + 3] = __float_as_uint(acc.w);
        }
      }
      const uint32_t box = staging + (nstore & 1u) * BOX_BYTES;
      if (lane == 0) bulk_wait_group_read<1>();
      __syncwarp();
      stage_row_f32(box, lane, v);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const void* src = stage_ptr + (nstore & 1u) * BOX_BYTES;
        if (c.reduce)
          tma_reduce_add_2d(out, src, col, orow);
        else
          tma_store_2d(out, src, col, orow);
        bulk_commit_group();
      }
      ++nstore;
    }
  }
  if (warp == 2 && lane == 0) c.cnt[tile] = 0;
}

template <int CG, bool W>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap m0, const __grid_constant__ CUtensorMap m1,
                const __grid_constant__ CUtensorMap m2, const __grid_constant__ CUtensorMap m3,
                const __grid_constant__ CUtensorMap m4, const __grid_constant__ CUtensorMap m5,
                GemmSched<CG, W> sched, int* counter, int32_t* status) {
  constexpr int TN = GemmSched<CG, W>::TN;
  sched.maps[0] = &m0;
  sched.maps[1] = &m1;
  sched.maps[2] = &m2;
  sched.maps[3] = &m3;
  sched.maps[4] = &m4;
  sched.maps[5] = &m5;
  sched.status = status;
  sched.rank = (int)pair_rank<CG>();
  if (threadIdx.x == 0) {
    for (int i = 0; i < 6; ++i) tma_prefetch_desc(sched.maps[i]);
  }
  const Feed feed{counter, sched.num_units()};
  run_cta<CG, W>(sched, feed, status, [&](uint8_t* stg, SmemCtl* ctl, uint32_t tmem_base, int warp, int lane,
                                          uint32_t rank) {
    const int q = warp & 3;
    uint8_t* stage_ptr = stg + (warp - 2) * STAGING_PER_WARP;
    const uint32_t staging = smem_u32(stage_ptr);
    uint32_t tcount = 0, nstore = 0, nsplit = 0;
    for (uint32_t i = 0;; ++i) {
      const int u = feed_consume<CG>(feed, ctl, i, status, true, rank);
      if (u < 0) break;
      int k, mt, nt, ks;
      sched.decode(u, k, mt, nt, ks);
      const GemmClass c = sched.pick(k);
      const CUtensorMap* out = sched.map(c.out_map);
      const int orow = c.out_row_base + mt * BM + 32 * q;
      const int ocol0 = c.out_col_base + nt * TN;
      if (CG == 1 && sched.tile(u, 0).kblocks == 0) {
        // empty sparse tile: nothing to add; a first (store) write still owes the tile its zeros
        if (!c.reduce && orow < c.out_rows) {
#pragma unroll 1
          for (int ch = 0; ch < BN / 32; ++ch) {
            const int col = ocol0 + ch * 32;
            if (col >= c.out_cols) break;
            const uint32_t box = staging + (nstore & 1u) * BOX_BYTES;
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            const uint32_t zero[32] = {};
            stage_row_f32(box, lane, zero);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(out, stage_ptr + (nstore & 1u) * BOX_BYTES, col, orow);
              bulk_commit_group();
            }
            ++nstore;
          }
        }
        continue;
      }
      uint32_t taddr;
      if (!epi_acquire<CG, W>(ctl, tmem_base, tcount, warp, status, &taddr)) break;
      if constexpr (!W) {  // (the host never splits K with wide tiles)
        if (c.ksplit > 1) {
          split_part<CG>(c, ctl, taddr, mt, nt, ks, q, warp, lane, orow, ocol0, out, staging, stage_ptr, nstore,
                         tcount, rank, nsplit, status);
          ++tcount;
          continue;
        }
      }
      if (mt < c.n_mt && orow < c.out_rows) {  // (the empty half of an odd pair stores nothing)
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr, ra);
#pragma unroll 1
        for (int ch = 0; ch < TN / 32; ch += 2) {
          tmem_ld_wait(ra);
          tmem_ld32(taddr + (ch + 1) * 32, rb);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h == 1) {
              tmem_ld_wait(rb);
              if (ch + 2 < TN / 32) tmem_ld32(taddr + (ch + 2) * 32, ra);
            }
            const int col = ocol0 + (ch + h) * 32;
            if (col < c.out_cols) {
              const uint32_t box = staging + (nstore & 1u) * BOX_BYTES;
              if (lane == 0) bulk_wait_group_read<1>();
              __syncwarp();
              if (h == 0)
                stage_row_f32(box, lane, ra);
              else
                stage_row_f32(box, lane, rb);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                const void* src = stage_ptr + (nstore & 1u) * BOX_BYTES;
                if (c.reduce)
                  tma_reduce_add_2d(out, src, col, orow);
                else
                  tma_store_2d(out, src, col, orow);
                bulk_commit_group();
              }
              ++nstore;
            }
          }
        }
      }
      epi_release<CG, W>(ctl, tcount, rank);
      ++tcount;
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }, [] {});
}

}  // namespace

namespace {
template <int cap, bool kFilter, int CG>
cudaError_t launch_rec_kernel(const RecLaunch& L, cudaStream_t st) {
  static std::atomic<int> smem_set[64];
  if (cudaError_t e = opt_in_smem(rec_kernel<cap, kFilter, CG>, Geo<CG>::SMEM, smem_set)) return e;
  const int n_mu = (L.n_mt + CG - 1) / CG;
  const int chunk = L.chunk > 0 && L.chunk < n_mu ? L.chunk : n_mu;
  RecSched<CG> sched{nullptr, nullptr, L.m0, L.v0, L.n_mt, L.n_vt, L.kblocks, L.w_row0, L.list, L.count, chunk};
  RecArgs a{L.targets, L.mask, L.lse, L.g, L.M, L.V, L.softcap, L.status, L.eps, L.rowbits, L.colbits, L.ld_row,
            L.ld_col, L.side};
  prof_begin(K_REC, st);
  const cudaError_t e =
      launch_engine(rec_kernel<cap, kFilter, CG>, CG, L.grid, Geo<CG>::SMEM, st, L.mh, L.mw, L.ms_store, sched, a);
  prof_end(K_REC, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <bool kFilter, int CG>
cudaError_t launch_rec_cap(const RecLaunch& L, cudaStream_t st) {
  const int cap = L.softcap > 0.f ? (L.softcap <= kCapExpMax ? kCapExp : kCapHybrid) : kCapOff;
  return cap == kCapExp      ? launch_rec_kernel<kCapExp, kFilter, CG>(L, st)
         : cap == kCapHybrid ? launch_rec_kernel<kCapHybrid, kFilter, CG>(L, st)
                             : launch_rec_kernel<kCapOff, kFilter, CG>(L, st);
}

template <int CG, bool W>
cudaError_t launch_gemm_cg(const GemmLaunch& L, cudaStream_t st, int kind) {
  static std::atomic<int> smem_set[64];
  if (cudaError_t e = opt_in_smem(gemm_kernel<CG, W>, Geo<CG, W>::SMEM, smem_set)) return e;
  GemmSched<CG, W> sched;
  for (int i = 0; i < 6; ++i) sched.maps[i] = nullptr;
  sched.status = nullptr;
  for (int k = 0; k < 2; ++k) {
    const GemmClassH& h = L.cls[k];
    sched.cls[k] = GemmClass{h.a_map,     h.a_mn,      h.a_mn_base,  h.a_k_base,     h.b_map,        h.b_mn,
                             h.b_mn_base, h.b_k_base,  h.out_map,    h.out_row_base, h.out_col_base, h.reduce,
                             h.out_rows,  h.out_cols,  h.n_mt,       h.n_nt,         h.kblocks,      h.mt_major,
                             h.kbits,     h.kwords,    h.list_shift, h.kg_shift,     h.ngroups,      h.clip,
                             h.kbits_rows, h.ksplit,   h.part,       h.cnt};
  }
  prof_begin(kind, st);
  const cudaError_t e = launch_engine(gemm_kernel<CG, W>, CG, L.grid, Geo<CG, W>::SMEM, st, L.maps[0], L.maps[1],
                                      L.maps[2], L.maps[3], L.maps[4], L.maps[5], sched, L.counter, L.status);
  prof_end(kind, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}
}  // namespace

cudaError_t launch_recompute(const RecLaunch& L, cudaStream_t st) {
  if (L.rowbits) return launch_rec_cap<true, 1>(L, st);
  return L.cg == 2 ? launch_rec_cap<false, 2>(L, st) : launch_rec_cap<false, 1>(L, st);
}

cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t st, int kind) {
  if (L.cg == 2) return L.wide ? launch_gemm_cg<2, true>(L, st, kind) : launch_gemm_cg<2, false>(L, st, kind);
  return launch_gemm_cg<1, false>(L, st, kind);
}

}  // namespace orpo
