// skip.cu — planning kernels of the backward skips.
//
// "Steel flash-CCE — handoff" §E and "Training — design" §5.1 (the Apple-CCE
// backward skips, eps 1e-5): the coefficient filter skips a block of the
// backward coefficient that lies wholly below eps, and the block skip uses the
// forward's block maxima to skip cold (token block, vocabulary block) work.
//
// Here a block is one 128 x 256 tile of dZ.  Per (row block, vocabulary block)
// of the backward:
//   plan_kernel  : before the recompute.  A tile holds work unless it is
//                  provably cold: no row with g != 0 has its target in the
//                  tile, and for every 32-row group, (largest logit of the group
//                  in the tile) - (smallest lse of the group's rows with g != 0)
//                  lies below log2(eps) - kMargin in base-2 units, which bounds
//                  every p sech^2 of the tile below eps.  The remaining tiles
//                  are listed (vocabulary-tile-major, ascending) for the
//                  recompute; the filter would drop every cold tile anyway, so
//                  the block skip leaves the result unchanged.
//   index_kernel : after the recompute, whose filter marked the kept tiles.
//                  Builds, per row tile, the ascending list of kept vocabulary
//                  tiles (K of the dh GEMM) and, per vocabulary tile, the list
//                  of kept row tiles (K of the dW GEMM), with k-block counts.
#include "internal.h"

#include <cuda_runtime.h>

#include "../../include/orpo_head.h"

namespace orpo {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMargin = 1.f / 64.f;  // base-2 slack for the fp32 rounding of both sides of the bound
constexpr int kPlanThreads = 1024;
constexpr int kGroupsMax = kMcMax / 32;
static_assert(kMaxTiles == 4 * kPlanThreads, "the plan judges four tiles per thread");

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const float* __restrict__ g, const uint8_t* __restrict__ mask,
                                                            const int32_t* __restrict__ targets,
                                                            const float* __restrict__ lse,
                                                            const float* __restrict__ bmax, int bmax_ld, int m0, int mc,
                                                            int v0, int vc, int n_mt, int n_vt, int M, int V,
                                                            float thr2, int* __restrict__ list, int* __restrict__ count,
                                                            uint8_t* __restrict__ flags, int32_t* status) {
  __shared__ uint8_t hot[kMaxTiles];        // [mt][vt]: a target of an active row lies in the tile
  __shared__ float minlse2[kGroupsMax];     // per 32-row group: min lse log2e over active rows (+inf: none)
  __shared__ int warp_sums[kPlanThreads / 32];
  const int tid = threadIdx.x;
  const int ntiles = n_mt * n_vt;
  const int ngroups = (mc + 31) / 32;
  for (int i = tid; i < ntiles; i += kPlanThreads) {
    hot[i] = 0;
    flags[i] = 0;
  }
  __syncthreads();
  for (int qg = tid; qg < ngroups; qg += kPlanThreads) {
    float mn = INFINITY;
    for (int r = qg * 32; r < min(mc, qg * 32 + 32); ++r) {
      const int t = m0 + r;
      if (t >= M || mask[t] == 0 || g[t] == 0.f) continue;
      mn = fminf(mn, lse[t] * kLog2e);
      const int y = targets[t];
      if (y < 0 || y >= V) {
        atomicOr(status, ORPO_STATUS_TARGET);
        continue;
      }
      if (y >= v0 && y < v0 + vc) hot[(r / 128) * n_vt + (y - v0) / 256] = 1;
    }
    minlse2[qg] = mn;
  }
  __syncthreads();
  // each thread judges 4 consecutive tiles in list order (u = vt * n_mt + mt), then a block scan
  // gives their places in the list
  int keep[4], c = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int u = 4 * tid + k;
    keep[k] = 0;
    if (u >= ntiles) continue;
    const int vt = u / n_mt, mt = u - vt * n_mt;
    int hit = hot[mt * n_vt + vt];
    for (int gq = mt * 4; !hit && gq < min(ngroups, mt * 4 + 4); ++gq) {
      const float ml = minlse2[gq];
      if (ml == INFINITY) continue;
      const float bm = __ldg(bmax + (size_t)(m0 / 32 + gq) * bmax_ld + (v0 / 256 + vt));
      hit = bm - ml >= thr2 - kMargin;  // -inf block maxima (no supervised row) never hold work
    }
    keep[k] = hit;
    c += hit;
  }
  // exclusive scan of c over the block
  const int lane = tid & 31, warp = tid >> 5;
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
  for (int k = 0; k < 4; ++k)
    if (keep[k]) list[pos++] = 4 * tid + k;
  if (tid == kPlanThreads - 1) *count = warp_sums[31];
}

__global__ void __launch_bounds__(kPlanThreads) index_kernel(const uint8_t* __restrict__ flags, int n_mt, int n_vt,
                                                             int kbt_dh, int kbt_dw, int* __restrict__ rowlist,
                                                             int* __restrict__ rowcnt, int* __restrict__ collist,
                                                             int* __restrict__ colcnt) {
  for (int i = threadIdx.x; i < n_mt + n_vt; i += kPlanThreads) {
    if (i < n_mt) {  // row tile mt: kept vocabulary tiles, 4 k-blocks each (the last tile may hold fewer)
      const int mt = i;
      int c = 0, last = -1;
      for (int vt = 0; vt < n_vt; ++vt)
        if (flags[mt * n_vt + vt]) rowlist[mt * n_vt + c++] = last = vt;
      rowcnt[mt] = c * 4 - (last == n_vt - 1 ? n_vt * 4 - kbt_dh : 0);
    } else {  // vocabulary tile vt: kept row tiles, 2 k-blocks each (the last may hold fewer)
      const int vt = i - n_mt;
      int c = 0, last = -1;
      for (int mt = 0; mt < n_mt; ++mt)
        if (flags[mt * n_vt + vt]) collist[vt * n_mt + c++] = last = mt;
      colcnt[vt] = c * 2 - (last == n_mt - 1 ? n_mt * 2 - kbt_dw : 0);
    }
  }
}

}  // namespace

cudaError_t launch_skip_plan(const SkipPlan& P, cudaStream_t st) {
  prof_begin(K_SKIP, st);
  plan_kernel<<<1, kPlanThreads, 0, st>>>(P.g, P.mask, P.targets, P.lse, P.bmax, P.bmax_ld, P.m0, P.mc, P.v0, P.vc,
                                          P.n_mt, P.n_vt, P.M, P.V, P.thr2, P.list, P.count, P.flags, P.status);
  prof_end(K_SKIP, st);
  return cudaGetLastError();
}

cudaError_t launch_skip_index(const SkipPlan& P, cudaStream_t st) {
  prof_begin(K_SKIP, st);
  index_kernel<<<1, kPlanThreads, 0, st>>>(P.flags, P.n_mt, P.n_vt, (P.vc + 63) / 64, (P.mc + 63) / 64, P.rowlist,
                                           P.rowcnt, P.collist, P.colcnt);
  prof_end(K_SKIP, st);
  return cudaGetLastError();
}

}  // namespace orpo
