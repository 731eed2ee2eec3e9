// orpo_loss.cu — the ORPO objective over per-token log-probs.
//
// Design page "Training — design", §1 "The objective": per sequence the mean
// response log-prob l_s, per pair the log-odds x = (l_w - l_r) - (log1mexp(l_w) -
// log1mexp(l_r)), loss = mean_p(-l_w + lambda * softplus(-x)), and the metrics
// loss / nll / or / accuracy / margin.  The gradient with respect to each
// token's logp is written in closed form (d x / d l_w = 1 / (1 - e^{l_w}), the
// "1/(1-P)" factor of §4), divided by the sequence's response-token count.
//
// One CTA of 1024 threads.  Rows are split into 1024 contiguous chunks; each
// thread sums the runs of equal sequence id inside its chunk in two-float
// arithmetic (ff, about 48 significant bits).  A run strictly inside a chunk is
// a whole sequence (ids are non-decreasing); the first and last runs of each
// chunk are partial and are combined per sequence by one warp in a fixed
// lane/butterfly order, so the result is bitwise reproducible.  Per-sequence
// means, per-pair differences and the metric sums stay two-float, the per-pair
// transcendentals and gradients are fp32 (see log1mexp_f); outputs are fp32.
// No fp64 arithmetic is left: it issues at a small fraction of the fp32 rate on
// this GPU and made the single-CTA reduction latency-bound.
//
// The same kernel evaluates the sibling objectives that share the logp engine
// ("Training — design" §8.3 SimPO; the xtrain post-training page's DPO with a
// summed sequence log-prob and cached reference log-probs; IPO and a hinge on
// the same reference log-ratio): only the per-pair term and its derivative
// change, and whether a sequence is summarised by its mean or its sum.
#include <math.h>

#include "../../include/orpo_head.h"
#include "bounds.cuh"
#include "internal.h"

namespace orpo {

namespace {

constexpr int T = 1024;
constexpr int kKindOrpo = 0, kKindSimpo = 1, kKindDpo = 2, kKindIpo = 3, kKindHinge = 4, kKindOrpoFull = 5;
static_assert(kKindOrpo == ORPO_PREF_ORPO && kKindSimpo == ORPO_PREF_SIMPO && kKindDpo == ORPO_PREF_DPO &&
                  kKindIpo == ORPO_PREF_IPO && kKindHinge == ORPO_PREF_HINGE && kKindOrpoFull == ORPO_PREF_ORPO_FULL,
              "kernel kinds are the ABI's ORPO_PREF_* values");
constexpr uint8_t kPromptRow = 2;  // mask value: prompt row, supervised only by the full-scope NLL
constexpr int32_t kSeqErr = ORPO_STATUS_SEQID, kEmptyErr = ORPO_STATUS_EMPTY_SEQ,
                  kNonfiniteErr = ORPO_STATUS_NONFINITE;

struct LossSmem {
  int head_sid[T], tail_sid[T], first_sid[T], last_sid[T];
  int head_cnt[T], tail_cnt[T];          // response rows of the partial runs
  int head_fcnt[T], tail_fcnt[T];        // response + prompt rows (full-scope NLL)
  float2 head_sum[T], tail_sum[T];       // two-float sums (ff)
  float2 head_fsum[T], tail_fsum[T];
  float2 red[5][T / 32];
  int err;
};
// followed by the per-sequence tables (SeqTables)

// Two-float ("double-single") arithmetic for the row sums and reductions: a value is hi + lo with
// |lo| <= ulp(hi) / 2, about 48 significant bits.  Additions use Knuth's two-sum for the high parts
// (exact error term) and fold the low parts in, all on the fp32 pipes: double-precision adds issue
// at a small fraction of the fp32 rate on this GPU, and a per-row fp64 add made the whole reduction
// latency-bound.  The order of every addition is fixed, so results are bitwise reproducible.
struct ff {
  float hi, lo;
};
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const float s = a.hi + b.hi;
  const float bp = s - a.hi;
  const float e = (a.hi - (s - bp)) + (b.hi - bp) + (a.lo + b.lo);
  const float hi = s + e;
  return ff{hi, e - (hi - s)};
}
__device__ __forceinline__ ff ff_of(float2 v) { return ff{v.x, v.y}; }
__device__ __forceinline__ float2 ff_pack(ff a) { return make_float2(a.hi, a.lo); }
__device__ __forceinline__ ff ff_neg(ff a) { return ff{-a.hi, -a.lo}; }
__device__ __forceinline__ float ff_f(ff a) { return a.hi + a.lo; }
__device__ __forceinline__ bool ff_gt(ff a, ff b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
// a / n for a count 0 < n < 2^24: the fp32 quotient, then the quotient of its exact remainder
__device__ __forceinline__ ff ff_div_n(ff a, int n) {
  const float fn = (float)n;
  const float q = a.hi / fn;
  const float r = fmaf(-q, fn, a.hi) + a.lo;
  const float q2 = r / fn;
  const float hi = q + q2;
  return ff{hi, q2 - (hi - q)};
}
__device__ __forceinline__ ff ff_shfl_xor(ff a, int o) {
  return ff{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}

// Per-pair transcendentals run in fp32 (the library's accurate logf / expm1f / log1pf / expf, a few
// ulp).  Their arguments (means, sums, log-ratio differences) are formed in two-float arithmetic
// first, so no cancellation happens in fp32.
__device__ __forceinline__ float log1mexp_f(float x) {
  // log(1 - e^x), x <= 0; two branches at -ln 2 (Maechler 2012)
  return x > -0.6931471805599453f ? logf(-expm1f(x)) : log1pf(-expf(x));
}

__device__ __forceinline__ float softplus_f(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }

__device__ __forceinline__ float sigmoid_f(float x) {
  const float e = expf(-fabsf(x));
  return x >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
}

// 1 / (1 - e^l) = -1 / expm1(l), l <= 0
__device__ __forceinline__ float inv_one_minus_exp(float l) { return -1.f / expm1f(l); }

// Per-sequence tables after LossSmem: two-float sums first (8-byte entries), then 4-byte ones.
struct SeqTables {
  size_t sum, fsum, cnt, fcnt, G, coef, coef_full, end;
};
__host__ __device__ inline SeqTables seq_tables(size_t S) {
  SeqTables t;
  size_t o = sizeof(LossSmem);
  t.sum = o, o += S * 8;   // float2 (ff): response-row sum, then the sequence statistic
  t.fsum = o, o += S * 8;  // float2 (ff): response + prompt rows
  t.cnt = o, o += S * 4;
  t.fcnt = o, o += S * 4;
  t.G = o, o += S * 4;     // float: d loss / d statistic
  t.coef = o, o += S * 4;
  t.coef_full = o, o += S * 4;
  t.end = o;
  return t;
}

__global__ void __launch_bounds__(T, 1)
    loss_kernel(int kind, const float* __restrict__ logp, const int32_t* __restrict__ seq_id,
                const uint8_t* __restrict__ mask, int M, int P, float lam_f, float gamma_f,
                const float* __restrict__ ref, float* __restrict__ out, float* __restrict__ ell,
                float* __restrict__ g, int32_t* status) {
  extern __shared__ __align__(16) uint8_t raw[];
  LossSmem& sm = *reinterpret_cast<LossSmem*>(raw);
  const int S = 2 * P;
  const SeqTables tb = seq_tables((size_t)S);
  float2* seq_sum = reinterpret_cast<float2*>(raw + tb.sum);
  float2* seq_fsum = reinterpret_cast<float2*>(raw + tb.fsum);
  int* seq_cnt = reinterpret_cast<int*>(raw + tb.cnt);
  int* seq_fcnt = reinterpret_cast<int*>(raw + tb.fcnt);
  float* G = reinterpret_cast<float*>(raw + tb.G);
  float* coef = reinterpret_cast<float*>(raw + tb.coef);
  float* coef_full = reinterpret_cast<float*>(raw + tb.coef_full);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float lam = lam_f;  // lambda for ORPO, beta for the other kinds
  const float gam = gamma_f;
  const bool orpo_kind = kind == kKindOrpo || kind == kKindOrpoFull;
  const bool mean_kind = orpo_kind || kind == kKindSimpo;
  const bool full_scope = kind == kKindOrpoFull;

  if (tid == 0) sm.err = 0;
  for (int s = tid; s < S; s += T) {
    seq_sum[s] = make_float2(0.f, 0.f);
    seq_cnt[s] = 0;
    seq_fsum[s] = make_float2(0.f, 0.f);
    seq_fcnt[s] = 0;
  }
  __syncthreads();

  // ---- phase 1: runs inside the contiguous chunk of this thread
  int err = 0;
  {
    const int chunk = (M + T - 1) / T;
    const int t0 = min(M, tid * chunk), t1 = min(M, t0 + chunk);
    int cur = -1, cnt = 0, fcnt = 0, nruns = 0, last = -1, first = -1;
    ff sum{0.f, 0.f}, fsum{0.f, 0.f};
    int hs = -1, hc = 0, hfc = 0, ts = -1, tc = 0, tfc = 0;
    ff hsum{0.f, 0.f}, hfsum{0.f, 0.f}, tsum{0.f, 0.f}, tfsum{0.f, 0.f};
    for (int t = t0; t < t1; ++t) {
      const int sid = seq_id[t];
      if (sid == -1) continue;
      if (sid < -1 || sid >= S) {
        err |= kSeqErr;
        continue;
      }
      if (sid < last) err |= kSeqErr;
      if (sid != cur) {
        if (cur >= 0) {
          if (nruns == 0) {
            hs = cur, hsum = sum, hc = cnt, hfsum = fsum, hfc = fcnt;
          } else if (in_bounds(status, cur, S)) {
            seq_sum[cur] = ff_pack(sum);  // a run strictly inside the chunk is the whole sequence
            seq_cnt[cur] = cnt;
            seq_fsum[cur] = ff_pack(fsum);
            seq_fcnt[cur] = fcnt;
          }
          ++nruns;
        }
        cur = sid;
        sum = fsum = ff{0.f, 0.f};
        cnt = fcnt = 0;
      }
      const uint8_t mk = mask[t];
      if (mk != 0) {
        const ff v{logp[t], 0.f};
        fsum = ff_add(fsum, v);
        ++fcnt;
        if (mk != kPromptRow) {
          sum = ff_add(sum, v);
          ++cnt;
        }
      }
      last = sid;
      if (first < 0) first = sid;
    }
    if (cur >= 0) {
      if (nruns == 0) {
        hs = cur, hsum = sum, hc = cnt, hfsum = fsum, hfc = fcnt;
      } else {
        ts = cur, tsum = sum, tc = cnt, tfsum = fsum, tfc = fcnt;
      }
    }
    sm.head_sid[tid] = hs;
    sm.head_sum[tid] = ff_pack(hsum);
    sm.head_cnt[tid] = hc;
    sm.head_fsum[tid] = ff_pack(hfsum);
    sm.head_fcnt[tid] = hfc;
    sm.tail_sid[tid] = ts;
    sm.tail_sum[tid] = ff_pack(tsum);
    sm.tail_cnt[tid] = tc;
    sm.tail_fsum[tid] = ff_pack(tfsum);
    sm.tail_fcnt[tid] = tfc;
    sm.first_sid[tid] = first;
    sm.last_sid[tid] = last;
  }
  __syncthreads();

  // ---- phase 1b: ids must not decrease across chunk boundaries
  if (sm.first_sid[tid] >= 0) {
    for (int j = tid - 1; j >= 0; --j) {
      if (sm.last_sid[j] >= 0) {
        if (sm.last_sid[j] > sm.first_sid[tid]) err |= kSeqErr;
        break;
      }
    }
  }

  // ---- phase 2: add the partial head / tail runs of every chunk to their sequence
  for (int s = warp; s < S; s += T / 32) {
    ff acc{0.f, 0.f}, facc{0.f, 0.f};
    int c = 0, fc = 0;
    for (int i = lane; i < T; i += 32) {
      if (sm.head_sid[i] == s) {
        acc = ff_add(acc, ff_of(sm.head_sum[i]));
        c += sm.head_cnt[i];
        facc = ff_add(facc, ff_of(sm.head_fsum[i]));
        fc += sm.head_fcnt[i];
      }
      if (sm.tail_sid[i] == s) {
        acc = ff_add(acc, ff_of(sm.tail_sum[i]));
        c += sm.tail_cnt[i];
        facc = ff_add(facc, ff_of(sm.tail_fsum[i]));
        fc += sm.tail_fcnt[i];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      acc = ff_add(acc, ff_shfl_xor(acc, o));
      c += __shfl_xor_sync(0xffffffffu, c, o);
      facc = ff_add(facc, ff_shfl_xor(facc, o));
      fc += __shfl_xor_sync(0xffffffffu, fc, o);
    }
    if (lane == 0) {
      seq_sum[s] = ff_pack(ff_add(ff_of(seq_sum[s]), acc));
      seq_cnt[s] += c;
      seq_fsum[s] = ff_pack(ff_add(ff_of(seq_fsum[s]), facc));
      seq_fcnt[s] += fc;
    }
  }
  __syncthreads();

  // ---- phase 3: per-sequence statistic: mean (ORPO, SimPO) or sum (DPO, IPO, hinge)
  for (int s = tid; s < S; s += T) {
    const int n = seq_cnt[s];
    ff l{NAN, 0.f};
    if (n == 0)
      err |= kEmptyErr;
    else
      l = mean_kind ? ff_div_n(ff_of(seq_sum[s]), n) : ff_of(seq_sum[s]);
    seq_sum[s] = ff_pack(l);
    ell[s] = ff_f(l);
  }
  __syncthreads();

  // ---- phase 4: per pair value, metrics and gradient (G = d loss / d statistic)
  const float inv_p = 1.f / (float)P;
  ff c_loss{0.f, 0.f}, c_nll{0.f, 0.f}, c_or{0.f, 0.f}, c_mar{0.f, 0.f};
  float c_acc = 0.f;
  for (int p = tid; p < P; p += T) {
    const ff lw = ff_of(seq_sum[2 * p]), lr = ff_of(seq_sum[2 * p + 1]);
    const ff dl = ff_add(lw, ff_neg(lr));
    float term = 0.f, dw = 0.f, Gw, Gr;
    ff loss_p, nll_p = ff_neg(lw), margin{0.f, 0.f};
    bool better;
    if (orpo_kind) {
      // x = (l_w - l_r) - (log1mexp(l_w) - log1mexp(l_r)); loss_p = NLL_p + lambda softplus(-x)
      const ff x = ff_add(dl, ff_add(ff{log1mexp_f(lr.hi), 0.f}, ff{-log1mexp_f(lw.hi), 0.f}));
      const float xf = ff_f(x);
      term = softplus_f(-xf);
      const float sg = sigmoid_f(-xf);
      const float inv_w = inv_one_minus_exp(lw.hi), inv_r = inv_one_minus_exp(lr.hi);
      // response scope folds the NLL gradient (-1/P on l_w) into G_w; full scope spreads
      // -1/(P N_w) over the chosen prompt + response rows in phase 5
      if (full_scope) nll_p = ff_neg(ff_div_n(ff_of(seq_fsum[2 * p]), max(seq_fcnt[2 * p], 1)));
      Gw = ((full_scope ? 0.f : -1.f) - lam * sg * inv_w) * inv_p;
      Gr = (lam * sg * inv_r) * inv_p;
      loss_p = ff_add(nll_p, ff{lam * term, 0.f});
      margin = x;
      better = ff_gt(lw, lr);
      if (lw.hi > 0.f || lr.hi > 0.f) err |= kNonfiniteErr;
    } else {
      float mf;
      if (kind == kKindSimpo) {
        mf = lam * (ff_f(dl) - gam);  // softplus(-beta((l_w - l_r) - gamma))
        term = softplus_f(-mf);
        dw = -lam * sigmoid_f(-mf);
        better = ff_gt(lw, lr);
      } else {
        const float D = ff_f(ff_add(dl, ff_add(ff{ref[2 * p + 1], 0.f}, ff{-ref[2 * p], 0.f})));
        better = D > 0.f;
        if (kind == kKindDpo) {  // -log sigmoid(beta D)
          mf = lam * D;
          term = softplus_f(-mf);
          dw = -lam * sigmoid_f(-mf);
        } else if (kind == kKindIpo) {  // (D - 1/(2 beta))^2
          const float c = D - 0.5f / lam;
          mf = D;
          term = c * c;
          dw = 2.f * c;
        } else {  // hinge: max(0, 1 - beta D)
          const float a = 1.f - lam * D;
          mf = lam * D;
          term = a > 0.f ? a : 0.f;
          dw = a > 0.f ? -lam : 0.f;
        }
      }
      Gw = dw * inv_p;
      Gr = -dw * inv_p;
      loss_p = ff{term, 0.f};
      margin = ff{mf, 0.f};
    }
    if (!isfinite(term) || !isfinite(Gw) || !isfinite(Gr) || !isfinite(lw.hi) || !isfinite(lr.hi) ||
        !isfinite(margin.hi))
      err |= kNonfiniteErr;
    G[2 * p] = Gw;
    G[2 * p + 1] = Gr;
    c_loss = ff_add(c_loss, loss_p);
    c_nll = ff_add(c_nll, nll_p);
    c_or = ff_add(c_or, ff{term, 0.f});
    c_acc += better ? 1.f : 0.f;
    c_mar = ff_add(c_mar, margin);
  }
  // fixed-order block reduction of the five sums (two-float)
  ff v[5] = {c_loss, c_nll, c_or, ff{c_acc, 0.f}, c_mar};
#pragma unroll
  for (int k = 0; k < 5; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] = ff_add(v[k], ff_shfl_xor(v[k], o));
    if (lane == 0) sm.red[k][warp] = ff_pack(v[k]);
  }
  if (err) atomicOr(&sm.err, err);
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      ff a = ff_of(sm.red[k][lane]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a = ff_add(a, ff_shfl_xor(a, o));
      if (lane == 0) out[k] = ff_f(ff_div_n(a, P));
    }
    if (lane == 0 && sm.err) atomicOr(status, sm.err);
  }

  // ---- phase 5: per-sequence coefficients, then the per-token gradient as a plain fp32 lookup:
  // g_t = coef[s] on response rows, plus coef_full[s] on every supervised row of a chosen sequence
  // under the full-scope NLL
  for (int s2 = tid; s2 < S; s2 += T) {
    const int n = seq_cnt[s2];
    coef[s2] = n > 0 ? (mean_kind ? G[s2] / (float)n : G[s2]) : 0.f;
    coef_full[s2] = (full_scope && (s2 & 1) == 0 && seq_fcnt[s2] > 0) ? -inv_p / (float)seq_fcnt[s2] : 0.f;
  }
  __syncthreads();
  for (int t = tid; t < M; t += T) {
    const int sid = seq_id[t];
    const uint8_t mk = mask[t];
    float gv = 0.f;
    if (sid >= 0 && sid < S && mk != 0) gv = (mk != kPromptRow ? coef[sid] : 0.f) + coef_full[sid];
    g[t] = gv;
  }
}

}  // namespace

size_t loss_smem_bytes(int P) { return seq_tables(2 * (size_t)P).end; }

cudaError_t launch_loss(int kind, const float* logp, const int32_t* seq_id, const uint8_t* mask, int M, int P,
                        float beta, float gamma, const float* ref, float* out, float* ell, float* g, int32_t* status,
                        cudaStream_t st) {
  const size_t smem = loss_smem_bytes(P);
  // one opt-in per device, at the size of the largest accepted batch (ORPO_MAX_PAIRS pairs)
  static std::atomic<int> smem_set[64];
  if (cudaError_t e = opt_in_smem(loss_kernel, (int)loss_smem_bytes(ORPO_MAX_PAIRS), smem_set)) return e;
  prof_begin(K_LOSS, st);
  loss_kernel<<<1, T, smem, st>>>(kind, logp, seq_id, mask, M, P, beta, gamma, ref, out, ell, g, status);
  prof_end(K_LOSS, st);
  return cudaGetLastError();
}

}  // namespace orpo
