// profile.cu — optional timing of the library's own kernel launches.
//
// While enabled, every launch is bracketed by a pair of CUDA events recorded on
// the launching stream; orpo_profile_stop waits for them and reports the total
// device time and launch count per kernel kind.  Events are host-side objects
// kept in a pool that is reused across sessions; no device memory is touched.
#include <mutex>
#include <vector>

#include "../../include/orpo_head.h"
#include "internal.h"

namespace orpo {
namespace {

struct Rec {
  int kind;
  cudaEvent_t e0, e1;
};

std::mutex g_mu;
bool g_on = false;
std::vector<cudaEvent_t> g_pool;
std::vector<Rec> g_recs;
size_t g_used = 0;

cudaEvent_t take_event() {
  if (g_used < g_pool.size()) return g_pool[g_used++];
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  g_pool.push_back(e);
  ++g_used;
  return e;
}

const char* kNames[K_NKINDS] = {"fwd_logits",    "fwd_merge",  "orpo_loss", "bwd_recompute",
                                "bwd_grad_gemm", "debug_gemm", "dequant",   "bwd_skip_plan"};

}  // namespace

void prof_begin(int kind, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on) return;
  Rec r{kind, take_event(), take_event()};
  if (!r.e0 || !r.e1) return;
  cudaEventRecord(r.e0, st);
  g_recs.push_back(r);
}

void prof_end(int kind, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || g_recs.empty() || g_recs.back().kind != kind) return;
  cudaEventRecord(g_recs.back().e1, st);
}

}  // namespace orpo

using namespace orpo;

extern "C" {

int orpo_profile_start(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_recs.clear();
  g_used = 0;
  g_on = true;
  return ORPO_OK;
}

int orpo_profile_stop(double* ms, int64_t* count, int nkinds) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = false;
  if (!ms || !count || nkinds < 1) return ORPO_ERR_NULL;
  for (int k = 0; k < nkinds; ++k) {
    ms[k] = 0.0;
    count[k] = 0;
  }
  int rc = ORPO_OK;
  for (const Rec& r : g_recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.e1) != cudaSuccess || cudaEventElapsedTime(&t, r.e0, r.e1) != cudaSuccess) {
      rc = ORPO_ERR_CUDA;
      continue;
    }
    if (r.kind < nkinds) {
      ms[r.kind] += t;
      count[r.kind] += 1;
    }
  }
  g_recs.clear();
  g_used = 0;
  return rc;
}

const char* orpo_profile_kind_name(int kind) {
  return (kind >= 0 && kind < K_NKINDS) ? kNames[kind] : "unknown";
}

}  // extern "C"
