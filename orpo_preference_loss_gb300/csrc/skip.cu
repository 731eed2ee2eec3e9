// skip.cu — planning kernels of the backward skips.
//
// "Steel flash-CCE — handoff" §E and "Training — design" §5.1 (the Apple-CCE
// backward skips, eps 1e-5): the coefficient filter skips a block of the
// backward coefficient that lies wholly below eps, and the block skip uses the
// forward's block maxima to skip cold (token block, vocabulary block) work.
//
// Here a block is one 128 x 256 tile of dZ.  One plan launch serves a round of
// (row block, vocabulary block) pairs of the backward, one CTA per pair, before
// their recomputes.  Each CTA zeroes its pair's keep bitmaps (the recompute's
// filter sets the bits of the tiles it keeps; the dh / dW GEMMs walk them) and,
// when the forward's block maxima are given, lists the tiles to recompute.  A
// tile holds work unless it is provably cold: no row with g != 0 has its target
// in the tile, and for every 32-row group, (largest logit of the group in the
// tile) - (smallest lse of the group's rows with g != 0) lies below
// log2(eps) - kMargin in base-2 units, which bounds every p sech^2 of the tile
// below eps.  The filter would drop every cold tile anyway, so the block skip
// leaves the result unchanged.  The list follows the full recompute's unit
// order (row-tile chunks, vocabulary-tile-major within a chunk).
#include "engine.cuh"
#include "internal.h"

#include <cuda_runtime.h>

#include "../../include/orpo_head.h"

namespace orpo {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMargin = 1.f / 64.f;  // base-2 slack for the fp32 rounding of both sides of the bound
constexpr int kPlanThreads = 1024;
constexpr int kGroupsMax = kMcMax / 32;
constexpr int kPerThread = kMaxTiles / kPlanThreads;  // tiles each thread judges
static_assert(kMaxTiles == kPerThread * kPlanThreads, "tiles split evenly over the plan's threads");

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const SkipPlan P) {
  __shared__ uint8_t hot[kMaxTiles];        // [mt][vt]: a target of an active row lies in the tile
  __shared__ float minlse2[kGroupsMax];     // per 32-row group: min lse log2e over active rows (+inf: none)
  __shared__ int warp_sums[kPlanThreads / 32];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int b = P.first_block + (int)blockIdx.x;
  const int mb = b % P.n_mblocks, vb = b / P.n_mblocks;
  const int m0 = (int)(mb * P.Mc), v0 = (int)(vb * P.Vc);
  const int mc = (int)min((int64_t)P.M - m0, P.Mc), vc = (int)min((int64_t)P.V - v0, P.Vc);
  const int n_mt = (mc + 127) / 128, n_vt = (vc + 255) / 256;
  if (!in_bounds(P.status, (int64_t)(blockIdx.x + 1) * P.shape.slot_bytes - 1, P.area_bytes)) return;
  uint8_t* slot = P.area + (size_t)blockIdx.x * P.shape.slot_bytes;
  uint32_t* bits = reinterpret_cast<uint32_t*>(slot + P.shape.rowbits_off());  // rowbits, then colbits
  const int nwords = P.shape.n_mt * P.shape.ld_row + P.shape.n_vt * P.shape.ld_col;
  for (int i = tid; i < nwords; i += kPlanThreads) bits[i] = 0u;
  if (P.bmax == nullptr) return;  // filter alone: every tile is recomputed

  int* list = reinterpret_cast<int*>(slot + P.shape.list_off());
  int* count = reinterpret_cast<int*>(slot + P.shape.count_off());
  const int ntiles = n_mt * n_vt;
  const int ngroups = (mc + 31) / 32;
  // the shared tables hold a block of at most kMcMax rows and kMaxTiles tiles (uniform over the block)
  if (!in_bounds(P.status, ntiles - 1, kMaxTiles) || !in_bounds(P.status, ngroups - 1, kGroupsMax)) return;
  for (int i = tid; i < ntiles; i += kPlanThreads) hot[i] = 0;
  __syncthreads();
  // one row per thread: a warp covers one 32-row group per pass
  for (int r = tid; r < ngroups * 32; r += kPlanThreads) {
    const int t = m0 + r;
    const bool active = r < mc && t < P.M && P.mask[t] != 0 && P.g[t] != 0.f;
    float l2 = INFINITY;
    if (active) {
      l2 = P.lse[t] * kLog2e;
      const int y = P.targets[t];
      if (y < 0 || y >= P.V)
        atomicOr(P.status, ORPO_STATUS_TARGET);
      else if (y >= v0 && y < v0 + vc && in_bounds(P.status, (r / 128) * n_vt + (y - v0) / 256, kMaxTiles))
        hot[(r / 128) * n_vt + (y - v0) / 256] = 1;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l2 = fminf(l2, __shfl_xor_sync(0xffffffffu, l2, o));
    if (lane == 0 && in_bounds(P.status, r / 32, kGroupsMax)) minlse2[r / 32] = l2;
  }
  __syncthreads();
  // each thread judges kPerThread consecutive tiles in the recompute's unit order (chunk_decode),
  // then a block scan gives their places in the list, which holds tile ids vt * n_mt + mt
  const int chunk = l2_chunk(n_mt, P.chunk_bytes);
  int keep[kPerThread], c = 0;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int u = kPerThread * tid + k;
    keep[k] = 0;
    if (u >= ntiles) continue;
    int mt, vt;
    chunk_decode(u, n_mt, n_vt, chunk, mt, vt);
    int hit = in_bounds(P.status, mt * n_vt + vt, kMaxTiles) ? hot[mt * n_vt + vt] : 1;
    for (int gq = mt * 4; !hit && gq < min(ngroups, mt * 4 + 4); ++gq) {
      const float ml = minlse2[gq];
      if (ml == INFINITY) continue;
      if (!in_bounds(P.status, m0 / 32 + gq, ((int64_t)P.M + 31) / 32) ||
          !in_bounds(P.status, v0 / 256 + vt, P.bmax_ld)) {
        hit = 1;
        break;
      }
      const float bm = __ldg(P.bmax + (size_t)(m0 / 32 + gq) * P.bmax_ld + (v0 / 256 + vt));
      hit = bm - ml >= P.thr2 - kMargin;  // -inf block maxima (no supervised row) never hold work
    }
    keep[k] = hit;
    c += hit;
  }
  // exclusive scan of c over the block
  int x = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  int pos = x - c + (warp > 0 ? warp_sums[warp - 1] : 0);
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    if (!keep[k]) continue;
    int mt, vt;
    chunk_decode(kPerThread * tid + k, n_mt, n_vt, chunk, mt, vt);
    if (in_bounds(P.status, pos, (int64_t)P.shape.n_mt * P.shape.n_vt)) list[pos] = vt * n_mt + mt;
    ++pos;
  }
  if (tid == kPlanThreads - 1) *count = warp_sums[31];
}

}  // namespace

cudaError_t launch_skip_plan(const SkipPlan& P, cudaStream_t st) {
  prof_begin(K_SKIP, st);
  plan_kernel<<<P.nblocks, kPlanThreads, 0, st>>>(P);
  prof_end(K_SKIP, st);
  return cudaGetLastError();
}

}  // namespace orpo
