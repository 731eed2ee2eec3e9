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
// thread sums the runs of equal sequence id inside its chunk in fp64.  A run
// strictly inside a chunk is a whole sequence (ids are non-decreasing); the
// first and last runs of each chunk are partial and are combined per sequence
// by one warp in a fixed lane/butterfly order, so the result is bitwise
// reproducible.  Sums and per-pair differences are fp64, the per-pair transcendentals fp32
// (see log1mexp_d); outputs are fp32.
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
  double head_sum[T], tail_sum[T];
  double head_fsum[T], tail_fsum[T];
  double red[5][T / 32];
  int err;
};
// followed by: double seq_sum[S]; int seq_cnt[S]; double G[S]; double seq_fsum[S]; int seq_fcnt[S];
//               float coef[S]; float coef_full[S]

// Per-pair transcendentals run in fp32 (the library's accurate logf / expm1f / log1pf / expf, a few
// ulp): double-precision transcendentals are very slow on this GPU and sit on a serial per-pair
// chain.  Their arguments (means, sums, log-ratio differences) are formed in fp64 first, so no
// cancellation happens in fp32; values return to fp64 for the reductions.
__device__ __forceinline__ double log1mexp_d(double x) {
  // log(1 - e^x), x <= 0; two branches at -ln 2 (Maechler 2012)
  const float xf = (float)x;
  return (double)(x > -0.6931471805599453 ? logf(-expm1f(xf)) : log1pf(-expf(xf)));
}

__device__ __forceinline__ double softplus_d(double x) {
  return fmax(x, 0.0) + (double)log1pf(expf(-(float)fabs(x)));
}

__device__ __forceinline__ double sigmoid_d(double x) {
  const float e = expf(-(float)fabs(x));
  return (double)(x >= 0 ? 1.f / (1.f + e) : e / (1.f + e));
}

// 1 / (1 - e^l) = -1 / expm1(l), l <= 0
__device__ __forceinline__ double inv_one_minus_exp(double l) { return (double)(-1.f / expm1f((float)l)); }

__global__ void __launch_bounds__(T, 1)
    loss_kernel(int kind, const float* __restrict__ logp, const int32_t* __restrict__ seq_id,
                const uint8_t* __restrict__ mask, int M, int P, float lam_f, float gamma_f,
                const float* __restrict__ ref, float* __restrict__ out, float* __restrict__ ell,
                float* __restrict__ g, int32_t* status) {
  extern __shared__ __align__(16) uint8_t raw[];
  LossSmem& sm = *reinterpret_cast<LossSmem*>(raw);
  const int S = 2 * P;
  double* seq_sum = reinterpret_cast<double*>(raw + sizeof(LossSmem));
  int* seq_cnt = reinterpret_cast<int*>(seq_sum + S);
  double* G = reinterpret_cast<double*>(raw + sizeof(LossSmem) + (size_t)S * 8 + (((size_t)S * 4 + 7) & ~size_t(7)));
  double* seq_fsum = G + S;
  int* seq_fcnt = reinterpret_cast<int*>(seq_fsum + S);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const double lam = (double)lam_f;  // lambda for ORPO, beta for the other kinds
  const double gam = (double)gamma_f;
  const bool orpo_kind = kind == kKindOrpo || kind == kKindOrpoFull;
  const bool mean_kind = orpo_kind || kind == kKindSimpo;
  const bool full_scope = kind == kKindOrpoFull;

  if (tid == 0) sm.err = 0;
  for (int s = tid; s < S; s += T) {
    seq_sum[s] = 0.0;
    seq_cnt[s] = 0;
    seq_fsum[s] = 0.0;
    seq_fcnt[s] = 0;
  }
  __syncthreads();

  // ---- phase 1: runs inside the contiguous chunk of this thread
  int err = 0;
  {
    const int chunk = (M + T - 1) / T;
    const int t0 = min(M, tid * chunk), t1 = min(M, t0 + chunk);
    int cur = -1, cnt = 0, fcnt = 0, nruns = 0, last = -1, first = -1;
    double sum = 0.0, fsum = 0.0;
    int hs = -1, hc = 0, hfc = 0, ts = -1, tc = 0, tfc = 0;
    double hsum = 0.0, hfsum = 0.0, tsum = 0.0, tfsum = 0.0;
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
            seq_sum[cur] = sum;  // a run strictly inside the chunk is the whole sequence
            seq_cnt[cur] = cnt;
            seq_fsum[cur] = fsum;
            seq_fcnt[cur] = fcnt;
          }
          ++nruns;
        }
        cur = sid;
        sum = fsum = 0.0;
        cnt = fcnt = 0;
      }
      const uint8_t mk = mask[t];
      if (mk != 0) {
        const double v = (double)logp[t];
        fsum += v;
        ++fcnt;
        if (mk != kPromptRow) {
          sum += v;
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
    sm.head_sum[tid] = hsum;
    sm.head_cnt[tid] = hc;
    sm.head_fsum[tid] = hfsum;
    sm.head_fcnt[tid] = hfc;
    sm.tail_sid[tid] = ts;
    sm.tail_sum[tid] = tsum;
    sm.tail_cnt[tid] = tc;
    sm.tail_fsum[tid] = tfsum;
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
    double acc = 0.0, facc = 0.0;
    int c = 0, fc = 0;
    for (int i = lane; i < T; i += 32) {
      if (sm.head_sid[i] == s) {
        acc += sm.head_sum[i];
        c += sm.head_cnt[i];
        facc += sm.head_fsum[i];
        fc += sm.head_fcnt[i];
      }
      if (sm.tail_sid[i] == s) {
        acc += sm.tail_sum[i];
        c += sm.tail_cnt[i];
        facc += sm.tail_fsum[i];
        fc += sm.tail_fcnt[i];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      acc += __shfl_xor_sync(0xffffffffu, acc, o);
      c += __shfl_xor_sync(0xffffffffu, c, o);
      facc += __shfl_xor_sync(0xffffffffu, facc, o);
      fc += __shfl_xor_sync(0xffffffffu, fc, o);
    }
    if (lane == 0) {
      seq_sum[s] += acc;
      seq_cnt[s] += c;
      seq_fsum[s] += facc;
      seq_fcnt[s] += fc;
    }
  }
  __syncthreads();

  // ---- phase 3: per-sequence statistic: mean (ORPO, SimPO) or sum (DPO, IPO, hinge)
  for (int s = tid; s < S; s += T) {
    const int n = seq_cnt[s];
    double l = NAN;
    if (n == 0)
      err |= kEmptyErr;
    else
      l = mean_kind ? seq_sum[s] / (double)n : seq_sum[s];
    seq_sum[s] = l;
    ell[s] = (float)l;
  }
  __syncthreads();

  // ---- phase 4: per pair value, metrics and gradient (G = d loss / d statistic)
  double c_loss = 0.0, c_nll = 0.0, c_or = 0.0, c_acc = 0.0, c_mar = 0.0;
  for (int p = tid; p < P; p += T) {
    const double lw = seq_sum[2 * p], lr = seq_sum[2 * p + 1];
    double term = 0.0, dw = 0.0, margin = 0.0, Gw, Gr, loss_p, nll_p = -lw;
    bool better;
    if (orpo_kind) {
      // x = (l_w - l_r) - (log1mexp(l_w) - log1mexp(l_r)); loss_p = NLL_p + lambda softplus(-x)
      const double x = (lw - lr) - (log1mexp_d(lw) - log1mexp_d(lr));
      term = softplus_d(-x);
      const double sg = sigmoid_d(-x);
      const double inv_w = inv_one_minus_exp(lw), inv_r = inv_one_minus_exp(lr);
      // response scope folds the NLL gradient (-1/P on l_w) into G_w; full scope spreads
      // -1/(P N_w) over the chosen prompt + response rows in phase 5
      if (full_scope) nll_p = -seq_fsum[2 * p] / (double)seq_fcnt[2 * p];
      Gw = ((full_scope ? 0.0 : -1.0) - lam * sg * inv_w) / (double)P;
      Gr = (lam * sg * inv_r) / (double)P;
      loss_p = nll_p + lam * term;
      margin = x;
      better = lw > lr;
      if (lw > 0.0 || lr > 0.0) err |= kNonfiniteErr;
    } else {
      if (kind == kKindSimpo) {
        margin = lam * ((lw - lr) - gam);  // softplus(-beta((l_w - l_r) - gamma))
        term = softplus_d(-margin);
        dw = -lam * sigmoid_d(-margin);
        better = lw > lr;
      } else {
        const double D = (lw - (double)ref[2 * p]) - (lr - (double)ref[2 * p + 1]);
        better = D > 0.0;
        if (kind == kKindDpo) {  // -log sigmoid(beta D)
          margin = lam * D;
          term = softplus_d(-margin);
          dw = -lam * sigmoid_d(-margin);
        } else if (kind == kKindIpo) {  // (D - 1/(2 beta))^2
          const double c = D - 1.0 / (2.0 * lam);
          margin = D;
          term = c * c;
          dw = 2.0 * c;
        } else {  // hinge: max(0, 1 - beta D)
          const double a = 1.0 - lam * D;
          margin = lam * D;
          term = a > 0.0 ? a : 0.0;
          dw = a > 0.0 ? -lam : 0.0;
        }
      }
      Gw = dw / (double)P;
      Gr = -dw / (double)P;
      loss_p = term;
    }
    if (!isfinite(term) || !isfinite(Gw) || !isfinite(Gr) || !isfinite(lw) || !isfinite(lr) || !isfinite(margin))
      err |= kNonfiniteErr;
    G[2 * p] = Gw;
    G[2 * p + 1] = Gr;
    c_loss += loss_p;
    c_nll += nll_p;
    c_or += term;
    c_acc += better ? 1.0 : 0.0;
    c_mar += margin;
  }
  // fixed-order block reduction of the five sums
  double v[5] = {c_loss, c_nll, c_or, c_acc, c_mar};
#pragma unroll
  for (int k = 0; k < 5; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
    if (lane == 0) sm.red[k][warp] = v[k];
  }
  if (err) atomicOr(&sm.err, err);
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      double a = sm.red[k][lane];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if (lane == 0) out[k] = (float)(a / (double)P);
    }
    if (lane == 0 && sm.err) atomicOr(status, sm.err);
  }

  // ---- phase 5: per-sequence coefficients (fp64 once per sequence), then the per-token gradient
  // as a plain fp32 lookup: g_t = coef[s] on response rows, plus coef_full[s] on every supervised
  // row of a chosen sequence under the full-scope NLL
  float* coef = reinterpret_cast<float*>(seq_fcnt + S);
  float* coef_full = coef + S;
  for (int s2 = tid; s2 < S; s2 += T) {
    const int n = seq_cnt[s2];
    coef[s2] = n > 0 ? (float)(mean_kind ? G[s2] / (double)n : G[s2]) : 0.f;
    coef_full[s2] = (full_scope && (s2 & 1) == 0 && seq_fcnt[s2] > 0)
                        ? (float)(-1.0 / ((double)P * seq_fcnt[s2]))
                        : 0.f;
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

size_t loss_smem_bytes(int P) {
  const size_t S = 2 * (size_t)P;
  return sizeof(LossSmem) + S * 8 + ((S * 4 + 7) & ~size_t(7)) + S * 8 + S * 8 + S * 4 + 2 * S * 4;
}

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
