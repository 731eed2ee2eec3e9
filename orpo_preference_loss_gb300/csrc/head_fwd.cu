// head_fwd.cu — forward of the flash-CCE head.
//
// Design page "Training — design", §5.1 tier 4 (vocab-parallel grid with
// per-block partials merged per row) and the fused-head spec's forward bullet
// (online max / sum-exp over vocabulary tiles, softcap, target capture).
//
// Work unit = (row tile of 128, vocabulary split).  A CTA walks the 256-wide
// vocabulary tiles of its split; for each tile the tensor cores build the
// 128 x 256 fp32 logit block in TMEM, and the epilogue (one thread per row)
// applies the softcap, folds the block into the row's running (max, sum-exp)
// in base-2 units and captures the target logit.  At the end of the unit the
// row's partial (max, sum) is written to the workspace; a small merge kernel
// combines the splits into lse and logp.
#include <stdlib.h>

#include "engine.cuh"
#include "internal.h"

namespace orpo {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Unit = (M unit, split), where an M unit is one row tile (CG = 1) or the two row tiles of a 2-CTA
// pair (CG = 2; CTA rank r takes tile 2m + r, and the W tiles of the split are shared by the pair).
// Units are ordered split-major within L2 chunks of M units, so the CTAs running at the same time
// stream the same W split through L2.
template <int CG>
struct FwdSched {
  const CUtensorMap* mh;
  const CUtensorMap* mw;
  int n_mt, nsplit, n_vt, kblocks;
  int chunk;  // M units per L2 chunk (chunk_decode)
  int rank;   // this CTA's rank in its pair (0 for CG = 1)
  __device__ int n_mu() const { return (n_mt + CG - 1) / CG; }
  __device__ int num_units() const { return n_mu() * nsplit; }
  __device__ int split_of(int u) const {
    int m, s;
    chunk_decode(u, n_mu(), nsplit, chunk, m, s);
    return s;
  }
  __device__ int mt_of(int u) const {  // this CTA's row tile (n_mt itself: the empty half of an odd pair)
    int m, s;
    chunk_decode(u, n_mu(), nsplit, chunk, m, s);
    return m * CG + rank;
  }
  __device__ int vt_begin(int s) const { return (int)(((long long)s * n_vt) / nsplit); }
  __device__ int unit_len(int u) const {
    const int s = split_of(u);
    return vt_begin(s + 1) - vt_begin(s);
  }
  __device__ TileOps tile(int u, int j) const {
    const int s = split_of(u), mt = mt_of(u);
    const int vt = vt_begin(s) + j;
    TileOps t;
    t.a = Operand{mh, 0, mt * BM, 0};
    t.b = Operand{mw, 0, vt * BN + rank * (BN / CG), 0};  // a pair fetches one half of the W tile each
    t.kblocks = kblocks;
    return t;
  }
};

struct FwdArgs {
  const int32_t* targets;
  const uint8_t* mask;
  float* tgt;  // receives z~[t, y_t] (the logp buffer, finalised by the merge)
  float* part_m;
  float* part_s;
  int M, Mpad, V;
  float softcap;
  int32_t* status;
  int col0;    // vocabulary column of row 0 of the W map (0 unless W is a block of the vocabulary)
  int split0;  // index of this launch's first split in the partial arrays
  float* bmax;   // optional block maxima [ceil(M/32), bmax_ld]: max of x over a 32-row group's mask != 0
                 // rows and one 256-column vocabulary tile (-inf for a group with no such row)
  int bmax_ld;   // ceil(V / 256)
  int part_cap;  // splits the partial arrays hold (each Mpad floats)
  DequantJob side;  // spare warps: dequantise the next vocabulary block (quantised head), or nothing
};

// Per-row online softmax state of one epilogue thread, base-2 units.
struct RowState {
  float m, s;
};

// Softcap forms (chosen once per launch):
//   kCapExp    (c <= kCapExpMax): tanh u = 1 - 2 / (1 + e^{2u}); one ex2 + one rcp per logit,
//              absolute error ~ c * 2^-22 on z~ (<= 1.5e-5 at c = 64).
//   kCapHybrid (larger c): the same form loses ~c * 2^-23 to cancellation, so |u| < 1/8 uses the
//              Taylor series of tanh (tanh_small) and only larger |u| the exp form; the exp form
//              runs only when some lane of the warp needs it.
constexpr int kCapOff = 0, kCapExp = 1, kCapHybrid = 2;
constexpr float kCapExpMax = 64.f;

// Fold 32 logits (raw fp32 accumulator bits) starting at column col0 into the row state.
// x = z~ log2(e) (base-2 units), z~ = c tanh(z / c) with the softcap on, else z.
template <int cap>
__device__ __forceinline__ void fold_chunk(const uint32_t (&r)[32], int col0, int V, int y, float inv_c, float cl2,
                                           RowState& st, float* tgt_slot, float& tmax) {
  if (col0 >= V) return;
  float x[32];
  if constexpr (cap == kCapExp) {
    // x = c log2e (1 - 2 / (1 + 2^{z K})) = A - 2A / (1 + 2^{z K}),  A = c log2e, K = 2 log2e / c
    const float K = 2.f * kLog2e * inv_c, A = cl2, B2 = 2.f * cl2;
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = fmaf(-B2, rcp_approx(1.f + ex2_approx(__uint_as_float(r[i]) * K)), A);
  } else if constexpr (cap == kCapHybrid) {
    bool big = false;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      x[i] = __uint_as_float(r[i]) * inv_c;  // u = z / c
      big |= fabsf(x[i]) >= kTanhSmall;
    }
    if (__any_sync(0xffffffffu, big)) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float q;
        const float u = x[i];
        x[i] = (fabsf(u) < kTanhSmall ? tanh_small(u) : tanh_exp(u, &q)) * cl2;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = tanh_small(x[i]) * cl2;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]) * kLog2e;
  }
  if (col0 + 32 > V) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i >= V) x[i] = -INFINITY;
  }
  if ((unsigned)(y - col0) < 32u) {
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i == y - col0) v = x[i];
    *tgt_slot = v * kLn2;
  }
  float m0 = fmaxf(x[0], x[1]), m1 = fmaxf(x[2], x[3]), m2 = fmaxf(x[4], x[5]), m3 = fmaxf(x[6], x[7]);
#pragma unroll
  for (int i = 8; i < 32; i += 8) {
    m0 = fmaxf(m0, fmaxf(x[i], x[i + 1]));
    m1 = fmaxf(m1, fmaxf(x[i + 2], x[i + 3]));
    m2 = fmaxf(m2, fmaxf(x[i + 4], x[i + 5]));
    m3 = fmaxf(m3, fmaxf(x[i + 6], x[i + 7]));
  }
  const float cmax = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
  tmax = fmaxf(tmax, cmax);
  const float mnew = fmaxf(st.m, cmax);
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    a0 += ex2_approx(x[i] - mnew);
    a1 += ex2_approx(x[i + 1] - mnew);
    a2 += ex2_approx(x[i + 2] - mnew);
    a3 += ex2_approx(x[i + 3] - mnew);
  }
  st.s = fmaf(st.s, ex2_approx(st.m - mnew), (a0 + a1) + (a2 + a3));
  st.m = mnew;
}

template <int cap, int CG>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap mh, const __grid_constant__ CUtensorMap mw, FwdSched<CG> sched,
               FwdArgs p) {
  sched.mh = &mh;
  sched.mw = &mw;
  sched.rank = (int)pair_rank<CG>();
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&mh);
    tma_prefetch_desc(&mw);
  }
  const Feed feed{nullptr, sched.num_units()};
  run_cta<CG>(sched, feed, p.status, [&](uint8_t*, SmemCtl* ctl, uint32_t tmem_base, int warp, int lane,
                                         uint32_t rank) {
    const int q = warp & 3;
    const float inv_c = cap != kCapOff ? 1.f / p.softcap : 0.f;
    const float cl2 = p.softcap * kLog2e;
    uint32_t tcount = 0;
    for (uint32_t i = 0;; ++i) {
      const int u = feed_consume<CG>(feed, ctl, i, p.status, true, rank);
      if (u < 0) break;
      const int s = sched.split_of(u), mt = sched.mt_of(u);
      const int row = mt * BM + 32 * q + lane;
      const bool supervised = row < p.M && p.mask[row] != 0;
      const int grp = mt * (BM / 32) + q;  // this warp's 32-row group
      int y = -1;
      if (supervised) y = p.targets[row];
      float* tgt_slot = p.tgt + (row < p.M ? row : 0);
      RowState st{-INFINITY, 0.f};
      const int len = sched.unit_len(u);
      const int vt0 = sched.vt_begin(s);
      for (int j = 0; j < len; ++j, ++tcount) {
        uint32_t taddr;
        if (!epi_acquire<CG>(ctl, tmem_base, tcount, warp, p.status, &taddr)) return;
        const int col_base = p.col0 + (vt0 + j) * BN;
        uint32_t ra[32], rb[32];
        float tmax = -INFINITY;
        tmem_ld32(taddr, ra);
#pragma unroll 1
        for (int c = 0; c < BN / 32; c += 2) {
          tmem_ld_wait(ra);
          tmem_ld32(taddr + (c + 1) * 32, rb);
          fold_chunk<cap>(ra, col_base + c * 32, p.V, y, inv_c, cl2, st, tgt_slot, tmax);
          tmem_ld_wait(rb);
          if (c + 2 < BN / 32) tmem_ld32(taddr + (c + 2) * 32, ra);
          fold_chunk<cap>(rb, col_base + (c + 1) * 32, p.V, y, inv_c, cl2, st, tgt_slot, tmax);
        }
        epi_release<CG>(ctl, tcount, rank);
        if (p.bmax != nullptr) {
          float v = supervised ? tmax : -INFINITY;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
          if (lane == 0 && grp * 32 < p.M && in_bounds(p.status, col_base / BN, p.bmax_ld))
            p.bmax[(size_t)grp * p.bmax_ld + col_base / BN] = v;
        }
      }
      if (row < p.Mpad && in_bounds(p.status, p.split0 + s, p.part_cap)) {
        p.part_m[(size_t)(p.split0 + s) * p.Mpad + row] = st.m;
        p.part_s[(size_t)(p.split0 + s) * p.Mpad + row] = st.s;
      }
    }
  }, [&] { side_dequant(p.side, p.status); });
}

// lse[t] = ln2 * (gM + log2 sum_k s_k 2^(m_k - gM));  logp[t] = z~[t,y_t] - lse[t] on response rows.
// A CTA takes 32 consecutive rows; warp g of its kMergeGroups warps reads the splits k = g, g + 8, ...
// of those rows (one 128-byte line per split), so few rows still spread over many warps.  The
// partial sums are added in group order, the same order on every run.
constexpr int kMergeGroups = 8;
__global__ void __launch_bounds__(32 * kMergeGroups)
    merge_kernel(const float* __restrict__ part_m, const float* __restrict__ part_s, int nsplit, int Mpad, int M,
                 int V, const int32_t* __restrict__ targets, const uint8_t* __restrict__ mask,
                 float* __restrict__ logp, float* __restrict__ lse, int32_t* status) {
  __shared__ float red_m[kMergeGroups][32];
  __shared__ float red_s[kMergeGroups][32];
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const int t = blockIdx.x * 32 + lane;
  const bool live = t < M && in_bounds(status, t, Mpad);
  float gm = -INFINITY;
  if (live)
    for (int k = grp; k < nsplit; k += kMergeGroups) gm = fmaxf(gm, part_m[(size_t)k * Mpad + t]);
  red_m[grp][lane] = gm;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kMergeGroups; ++j) gm = fmaxf(gm, red_m[j][lane]);
  float S = 0.f;
  if (live)
    for (int k = grp; k < nsplit; k += kMergeGroups)
      S += part_s[(size_t)k * Mpad + t] * exp2f(part_m[(size_t)k * Mpad + t] - gm);
  red_s[grp][lane] = S;
  __syncthreads();
  if (grp != 0 || !live) return;
  S = 0.f;
#pragma unroll
  for (int j = 0; j < kMergeGroups; ++j) S += red_s[j][lane];
  const float l = (gm + log2f(S)) * kLn2;
  lse[t] = l;
  int32_t err = 0;
  if (!isfinite(l)) err |= ORPO_STATUS_NONFINITE;
  float out = 0.f;
  if (mask[t] != 0) {
    const int y = targets[t];
    if (y < 0 || y >= V)
      err |= ORPO_STATUS_TARGET;
    else
      out = logp[t] - l;
  }
  logp[t] = out;
  if (err) atomicOr(status, err);
}

template <int cap, int CG>
cudaError_t launch_fwd_kernel(const FwdLaunch& L, cudaStream_t st) {
  static std::atomic<int> smem_set[64];
  if (cudaError_t e = opt_in_smem(fwd_kernel<cap, CG>, Geo<CG>::SMEM, smem_set)) return e;
  const int n_mu = (L.n_mt + CG - 1) / CG;
  const int chunk = L.chunk > 0 && L.chunk < n_mu ? L.chunk : n_mu;
  FwdSched<CG> sched{nullptr, nullptr, L.n_mt, L.nsplit, L.n_vt, L.kblocks, chunk, 0};
  FwdArgs a{L.targets, L.mask, L.logp, L.part_m, L.part_s, L.M,      L.Mpad,       L.V,
            L.softcap, L.status, L.col0, L.split0, L.bmax, (L.V + BN - 1) / BN, L.part_cap, L.side};
  prof_begin(K_FWD, st);
  const cudaError_t e = launch_engine(fwd_kernel<cap, CG>, CG, L.grid, Geo<CG>::SMEM, st, L.mh, L.mw, sched, a);
  prof_end(K_FWD, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int CG>
cudaError_t launch_fwd_cg(const FwdLaunch& L, cudaStream_t st) {
  const int cap = L.softcap > 0.f ? (L.softcap <= kCapExpMax ? kCapExp : kCapHybrid) : kCapOff;
  return cap == kCapExp      ? launch_fwd_kernel<kCapExp, CG>(L, st)
         : cap == kCapHybrid ? launch_fwd_kernel<kCapHybrid, CG>(L, st)
                             : launch_fwd_kernel<kCapOff, CG>(L, st);
}

}  // namespace

// Looked up once per device.
int engine_pair_clusters() {
  static std::atomic<int> cached[64];  // 0 unknown, -1 none, else the cluster count
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int c = cached[dev].load(std::memory_order_acquire);
  if (c != 0) return c > 0 ? c : 0;
  const int n = max_pair_clusters(fwd_kernel<kCapExp, 2>, Geo<2>::SMEM);
  cached[dev].store(n > 0 ? n : -1, std::memory_order_release);
  return n > 0 ? n : 0;
}

// Read once per process: ORPO_CTA_GROUP=1 runs every engine kernel on single-CTA tiles; otherwise
// (unset, or =2) they run on 2-CTA clusters wherever clusters fit.
int engine_cta_group_override() {
  static const int v = [] {
    const char* env = getenv("ORPO_CTA_GROUP");
    if (env != nullptr && (env[0] == '1' || env[0] == '2') && env[1] == 0) return env[0] - '0';
    return 0;
  }();
  return v;
}

cudaError_t launch_forward_logits(const FwdLaunch& L, cudaStream_t st) {
  return L.cg == 2 ? launch_fwd_cg<2>(L, st) : launch_fwd_cg<1>(L, st);
}

cudaError_t launch_forward_merge(const FwdLaunch& L, int nsplit_total, cudaStream_t st) {
  prof_begin(K_MERGE, st);
  merge_kernel<<<(L.M + 31) / 32, 32 * kMergeGroups, 0, st>>>(L.part_m, L.part_s, nsplit_total, L.Mpad, L.M, L.V,
                                                              L.targets, L.mask, L.logp, L.lse, L.status);
  prof_end(K_MERGE, st);
  return cudaGetLastError();
}

cudaError_t launch_forward(const FwdLaunch& L, cudaStream_t st) {
  cudaError_t e = launch_forward_logits(L, st);
  if (e != cudaSuccess) return e;
  return launch_forward_merge(L, L.nsplit, st);
}

}  // namespace orpo
