// api.cu — the C ABI of liborpo_head: argument checks, workspace layout, tensor
// maps, blocking choices and the launch sequence of each entry point.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "../../include/orpo_head.h"
#include "internal.h"

namespace orpo {

size_t loss_smem_bytes(int P);

namespace {

// Largest M, V (and debug-GEMM extent): row and column indices, tile counts rounded up to whole tiles,
// and per-thread row chunks of the loss stay inside int32 with room to spare.
constexpr int64_t kMaxRows = (1ll << 31) - (1ll << 16);

// ---------------------------------------------------------------- driver entry point
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// ---------------------------------------------------------------- device facts
struct DevInfo {
  int ok = -1;  // -1 unknown, 0 unsupported, 1 ok
  int sms = 0;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

int device_check(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ORPO_ERR_CUDA;
  if (dev < 0 || dev >= 64) return ORPO_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& di = g_dev[dev];
  if (di.ok < 0) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ORPO_ERR_CUDA;
    di.ok = (major == 10 && minor == 3) ? 1 : 0;
    di.sms = n;
  }
  if (!di.ok) return ORPO_ERR_UNSUPPORTED;
  *sms = di.sms;
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return ORPO_ERR_CUDA;
  return ORPO_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- blocking
struct BwdBlocks {
  int64_t Mc, Vc;  // rows / columns of the scratch block (multiples of 128 / 256)
};

// quantised head: the bf16 copy of W is made one vocabulary block at a time, within this many bytes
// in all.  From kSideMinRows rows on, every block after the first is dequantised by the contraction
// kernels' spare warps while the previous one is multiplied, so the bytes form two buffers of half
// the size; below, where a block's contraction is shorter than that dequantisation (about 0.35 ms
// for a 16384 x 2560 block), each block is dequantised by a launch of its own into one buffer.
constexpr int64_t kWBudget = 256ll << 20;
constexpr int64_t kSideMinRows = 8192;

inline bool q_side(int64_t M) { return M >= kSideMinRows; }

// qd > 0: the quantised head of hidden size qd, whose vocabulary block must also fit one bf16 W
// buffer (with few rows the dZ budget alone would allow the whole vocabulary, and the dequantised
// copy would be all of W)
BwdBlocks bwd_blocks(int64_t M, int64_t V, int64_t qd = 0) {
  const int64_t Mpad = std::max<int64_t>(kBM, cdiv(M, kBM) * kBM);
  // row blocks of equal height (a multiple of a 2-CTA pair's 256 rows) rather than full blocks and
  // a short last one, whose launches would leave most SMs idle
  const int64_t nmb = cdiv(Mpad, kMcMax);
  const int64_t Mc = nmb == 1 ? Mpad : std::min(kMcMax, cdiv(cdiv(Mpad, nmb), 2 * kBM) * 2 * kBM);
  const int64_t Vpad = cdiv(V, kBN) * kBN;
  int64_t vc = (kScratchBudget / (2 * Mc)) / kBN * kBN;
  const int64_t wbuf = q_side(M) ? kWBudget / 2 : kWBudget;
  if (qd > 0) vc = std::min<int64_t>(vc, (wbuf / (2 * qd)) / kBN * kBN);
  vc = std::max<int64_t>(kBN, vc);
  // vocabulary blocks of equal width too (multiples of 256 columns, never wider than the budget's)
  const int64_t nvb = cdiv(Vpad, vc);
  vc = cdiv(cdiv(Vpad, nvb), kBN) * kBN;
  return BwdBlocks{Mc, std::min(Vpad, vc)};
}

// forward partials: (max, sum-exp) per row and vocabulary split
size_t partial_bytes(int64_t M, int nsplit_max) {
  const int64_t Mpad = std::max<int64_t>(kBM, cdiv(M, kBM) * kBM);
  return (size_t)2 * nsplit_max * Mpad * sizeof(float);
}

// quantised head: most splits over all dequantised blocks (at least one per block; see QLayout)
constexpr int kNsplitMaxQ = 256;

void* align_ws(void* ws) {
  uintptr_t p = reinterpret_cast<uintptr_t>(ws);
  return reinterpret_cast<void*>((p + 1023) & ~uintptr_t(1023));
}

// Row pitch of the dZ block in elements: 64 past the width, so that rows of the
// block (Vc is a power of two for the common vocabularies) do not all start on the
// same power-of-two address offsets.
inline int64_t scratch_pitch(const BwdBlocks& b) { return b.Vc + 64; }

size_t scratch_bytes(int64_t M, int64_t V, int64_t qd = 0) {
  const BwdBlocks b = bwd_blocks(M, V, qd);
  return (size_t)b.Mc * scratch_pitch(b) * 2;
}

// Unit counters of the dh/dW GEMM launches (dynamic scheduling): a fixed ring of
// kCounters slots; launch k uses slot k % kCounters and the ring is zeroed
// (stream-ordered) before every kCounters-th launch.
constexpr int kCounters = 4096;
constexpr size_t kCounterBytes = kCounters * sizeof(int);

// Backward-skip area after the counters: one slot per (row block, vocabulary block) of a plan round
// (tile list, count and keep bitmaps; SkipShape).  A slot is at most ~34 KiB, so a round covers
// 120 or more blocks.
constexpr size_t kSkipBytes = 4 << 20;

// Split K of the dh GEMM.  With few rows the dh class has few output tiles, each with K = the block's
// vocabulary columns (at M 512, d 2560: 20 units of 4096 k-blocks on 76 clusters), so most SMs idle.
// Each tile's K range is then cut into parts (see split_part in head_bwd.cu); the area after the skip
// area holds the parts' fp32 tiles and one counter per tile.
constexpr int kSplitSlotsMax = 320;  // partial tiles (128 x 256 fp32, 128 KiB each) the area holds
constexpr int kSplitMax = 8;         // parts per tile (the kernel's kSplitMaxParts)
constexpr int kSplitMinKb = 8;       // k-blocks per part at least
constexpr int kSplitFinalKb = 96;    // the last part's read-and-sum of every part, in k-block times
constexpr int64_t kSlotBytes = (int64_t)kBM * kBN * 4;

int64_t dh_tiles(int64_t M, int64_t d, int64_t qd = 0) {  // CTA tiles of the dh class of a full row block
  return cdiv(bwd_blocks(M, 1, qd).Mc, kBM) * cdiv(d, kBN);
}

size_t split_part_bytes(int64_t M, int64_t d, int64_t qd = 0) {
  const int64_t t = dh_tiles(M, d, qd);
  if (t > kSplitSlotsMax / 2) return 0;  // not even two parts fit: never split
  return (size_t)std::min<int64_t>(kSplitSlotsMax, t * kSplitMax) * kSlotBytes;
}

size_t split_bytes(int64_t M, int64_t d, int64_t qd = 0) {
  const size_t pb = split_part_bytes(M, d, qd);
  return pb ? pb + (((size_t)dh_tiles(M, d, qd) * 4 + 1023) & ~size_t(1023)) : 0;
}

// Parts per dh tile.  The launch takes at least (all its k-blocks) / slots, the dh units' own waves
// (waves of parts) x (k-blocks per part + 2 for writing the partial tile) + the last part's sum of all
// parts (a fixed cost: its loads are all in flight at once).  Minimise the larger of the two; ties
// to fewer parts.  A short K (the tiny config's 64 k-blocks) is not split, nor a launch whose other
// class (`other_kb` k-blocks of dW units) already fills the slots.
// Wide (256 x 512) GEMM tiles: a quarter fewer operand bytes per flop, but the accumulator takes all of
// TMEM, so a tile's epilogue no longer overlaps the next tile's MMAs, and twice-as-long tiles make the
// last wave coarser.  Measured 6-10% faster per tile on wave-aligned shapes.  Taken on 2-CTA clusters
// without split K when padding the output width to 512 columns adds at most an eighth (d 3840 pads to
// 4096 and still gains 2%) and there are at least three waves of wide tiles.  ORPO_GEMM_WIDE=0 never
// takes them, =1 wherever they are legal.
int gemm_wide_override() {
  static const int v = [] {
    const char* e = getenv("ORPO_GEMM_WIDE");
    return e != nullptr && (e[0] == '0' || e[0] == '1') ? e[0] - '0' : -1;
  }();
  return v;
}

bool use_wide(int cg, int ksplit, int64_t out_cols, int64_t wide_units, int slots) {
  if (cg != 2 || ksplit > 1) return false;
  const int o = gemm_wide_override();
  if (o >= 0) return o == 1;
  return cdiv(out_cols, 2 * kBN) * 2 * kBN * 8 <= out_cols * 9 && wide_units >= 3 * (int64_t)slots;
}

int choose_ksplit(int64_t units, int64_t kblocks, int64_t tiles, int slots, size_t part_bytes, int64_t other_kb) {
  if (part_bytes == 0) return 1;
  const int64_t smax = std::min<int64_t>({(int64_t)kSplitMax, (int64_t)(part_bytes / kSlotBytes) / tiles,
                                          kblocks / kSplitMinKb});
  const int64_t floor_kb = cdiv(units * kblocks + other_kb, slots);
  int best = 1;
  int64_t best_cost = std::max(floor_kb, cdiv(units, slots) * kblocks);
  for (int64_t k = 2; k <= smax; ++k) {
    const int64_t cost = std::max(floor_kb, cdiv(units * k, slots) * (cdiv(kblocks, k) + 2) + kSplitFinalKb);
    if (cost < best_cost) {
      best_cost = cost;
      best = (int)k;
    }
  }
  return best;
}

SkipShape skip_shape(const BwdBlocks& b) {
  SkipShape s{};
  s.n_mt = (int)(b.Mc / kBM);
  s.n_vt = (int)(b.Vc / kBN);
  s.ld_row = (s.n_vt + 31) / 32;
  s.ld_col = (s.n_mt + 31) / 32;
  s.slot_bytes = (s.end() + 255) & ~size_t(255);
  return s;
}

// Number of vocabulary splits: minimise (waves of units) x (tiles per unit);
// ties go to fewer splits (fewer partials to merge).
int choose_nsplit(int64_t n_mt, int64_t n_vt, int sms) {
  int best = 1;
  int64_t best_cost = INT64_MAX;
  const int64_t lim = std::min<int64_t>(n_vt, kNsplitMax);
  for (int64_t ns = 1; ns <= lim; ++ns) {
    const int64_t waves = cdiv(n_mt * ns, sms);
    const int64_t cost = waves * cdiv(n_vt, ns);
    if (cost < best_cost) {
      best_cost = cost;
      best = (int)ns;
    }
  }
  return best;
}

// Engine placement on the current device: 2-CTA clusters (slots = clusters) or single CTAs (slots =
// SMs).  Every contraction takes clusters where they fit (measured faster for each of them);
// ORPO_CTA_GROUP=1 forces single CTAs; `allow_pair` false forces them too (the backward skips'
// per-tile bitmaps and lists).
struct Placement {
  int cg;
  int slots;
};

Placement placement(int sms, bool allow_pair = true) {
  const bool want = allow_pair && engine_cta_group_override() != 1;
  const int clusters = want ? engine_pair_clusters() : 0;
  return clusters > 0 ? Placement{2, clusters} : Placement{1, sms};
}

}  // namespace

bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_map_mn3d(CUtensorMap* map, const void* base, uint64_t mn, uint64_t k, uint64_t row_bytes,
                     uint32_t chunks) {
  if (!g_encode || mn % 64 != 0) return false;
  const cuuint64_t dims[3] = {64, k, mn / 64};
  const cuuint64_t strides[2] = {row_bytes, 128};
  const cuuint32_t box[3] = {64, 64, chunks};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace orpo

using namespace orpo;

// ---------------------------------------------------------------- forward / backward implementations

// Source of an affine group-quantised head (nullptr: W is bf16).
struct QuantW {
  const uint8_t* wq;
  const void* scales;
  const void* biases;
  int bits, group;
};

int check_quant(const QuantW* q, int64_t d) {
  if (!q) return ORPO_OK;
  if (!q->wq || !q->scales || !q->biases) return ORPO_ERR_NULL;
  if ((q->bits != 4 && q->bits != 8) || q->group < 8 || q->group % 8 != 0 || d % q->group != 0)
    return ORPO_ERR_ARG;
  const uintptr_t a = reinterpret_cast<uintptr_t>(q->wq);
  if ((q->bits == 4 && (a & 3u)) || (q->bits == 8 && (a & 7u)) || (reinterpret_cast<uintptr_t>(q->scales) & 1u) ||
      (reinterpret_cast<uintptr_t>(q->biases) & 1u))
    return ORPO_ERR_ALIGN;
  return ORPO_OK;
}

// Quantised head: the forward and the backward walk W in the same vocabulary blocks (the backward's
// Vc), dequantised alternately into two bf16 buffers (one buffer below kSideMinRows rows).
// Workspace: [partials | S + counters + skip area], then the buffers.  The forward keeps at least
// one split per block, so the partials hold max(kNsplitMaxQ, blocks) splits.
struct QLayout {
  int64_t rows;     // vocabulary rows per block (= per buffer)
  int64_t nblocks;  // blocks covering V
  int nsplit_cap;   // forward splits the partial arrays hold
  size_t buf_off[2], total;  // one buffer: both offsets equal
};

QLayout q_layout(int64_t M, int64_t V, int64_t d) {
  QLayout L{};
  L.rows = bwd_blocks(M, V, d).Vc;
  L.nblocks = cdiv(V, L.rows);
  L.nsplit_cap = (int)std::max<int64_t>(kNsplitMaxQ, L.nblocks);
  const size_t head =
      std::max(partial_bytes(M, L.nsplit_cap), scratch_bytes(M, V, d) + kCounterBytes + kSkipBytes + split_bytes(M, d, d));
  const size_t buf = ((size_t)L.rows * d * 2 + 1023) & ~size_t(1023);
  L.buf_off[0] = (head + 1023) & ~size_t(1023);
  L.buf_off[1] = L.buf_off[0] + (q_side(M) ? buf : 0);
  L.total = L.buf_off[1] + buf + 1024;  // + slack for aligning the workspace base
  return L;
}

void* qbuf_ptr(void* workspace, const QLayout& L, int64_t block) {
  return static_cast<uint8_t*>(align_ws(workspace)) + L.buf_off[block & 1];
}

int head_fwd_impl(const void* h, const void* W, const QuantW* q, const int32_t* targets, const uint8_t* mask,
                  int64_t M, int64_t V, int64_t d, float softcap, float* logp, float* lse, float* bmax,
                  void* workspace, size_t ws_bytes, int32_t* status, void* stream) {
  if (M < 0 || M > kMaxRows || V < 1 || V > kMaxRows || d < 8 || d >= (1 << 20)) return ORPO_ERR_SHAPE;
  if (M == 0) return ORPO_OK;
  if (!h || (!W && !q) || !targets || !mask || !logp || !lse || !workspace || !status) return ORPO_ERR_NULL;
  if (d % 8 != 0 || !aligned16(h) || (W && !aligned16(W)) || !aligned16(workspace)) return ORPO_ERR_ALIGN;
  if (int e = check_quant(q, d)) return e;
  if (!isfinite(softcap)) return ORPO_ERR_ARG;
  if (ws_bytes < (q ? orpo_head_q_workspace_bytes(M, V, d) : orpo_head_workspace_bytes(M, V, d)))
    return ORPO_ERR_WORKSPACE;
  int sms = 0;
  if (int e = device_check(&sms)) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  FwdLaunch L;
  const int64_t n_mt = cdiv(M, kBM);
  const int64_t Mpad = n_mt * kBM;
  const QLayout ql = q ? q_layout(M, V, d) : QLayout{};
  const int nsplit_max = q ? ql.nsplit_cap : kNsplitMax;
  float* base = reinterpret_cast<float*>(align_ws(workspace));
  if (!encode_map_2d(&L.mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, d, M, d * 2, 64, kBM)) return ORPO_ERR_CUDA;
  L.n_mt = (int)n_mt;
  L.kblocks = (int)cdiv(d, 64);
  L.targets = targets;
  L.mask = mask;
  L.logp = logp;
  L.lse = lse;
  L.part_m = base;
  L.part_s = base + (size_t)nsplit_max * Mpad;
  L.part_cap = nsplit_max;
  L.M = (int)M;
  L.Mpad = (int)Mpad;
  L.V = (int)V;
  L.softcap = softcap > 0.f ? softcap : 0.f;
  L.status = status;
  L.bmax = bmax;
  // vocabulary blocks: the whole vocabulary for bf16 W; bounded dequantised blocks otherwise.  At
  // large M block k + 1 is dequantised by the spare warps of block k's launch (only block 0 by a
  // launch of its own); at small M every block by a launch of its own.
  const int64_t vb = q ? ql.rows : V;
  const int64_t nblocks = cdiv(V, vb);
  const int per_block = std::max<int>(1, nsplit_max / (int)nblocks);
  const bool side = q && q_side(M);
  const Placement pl = placement(sms);
  const int64_t n_mu = cdiv(n_mt, pl.cg);  // M units: row tiles, or pairs of them
  L.cg = pl.cg;
  L.chunk = l2_chunk((int)n_mu, (int64_t)pl.cg * kBM * d * 2);
  const uint32_t w_box = kBN / pl.cg;
  int split0 = 0;
  for (int64_t v0 = 0, blk = 0; v0 < V; v0 += vb, ++blk) {
    const int64_t vc = std::min(vb, V - v0);
    const int64_t n_vt = cdiv(vc, kBN);
    if (q) {
      if ((blk == 0 || !side) && launch_dequant(q->wq, q->scales, q->biases, q->bits, q->group, v0, vc, d, V,
                                                qbuf_ptr(workspace, ql, blk), status, st) != cudaSuccess)
        return ORPO_ERR_CUDA;
      if (!encode_map_2d(&L.mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qbuf_ptr(workspace, ql, blk), d, vc, d * 2, 64, w_box))
        return ORPO_ERR_CUDA;
      const int64_t n0 = v0 + vb;  // the next block, into the other buffer
      L.side = side && n0 < V ? dequant_job(q->wq, q->scales, q->biases, q->bits, q->group, n0, std::min(vb, V - n0),
                                            d, V, qbuf_ptr(workspace, ql, blk + 1))
                              : DequantJob{};
    } else if (!encode_map_2d(&L.mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, d, V, d * 2, 64, w_box)) {
      return ORPO_ERR_CUDA;
    }
    L.n_vt = (int)n_vt;
    L.nsplit = std::min<int>(choose_nsplit(n_mu, n_vt, pl.slots), per_block);
    L.col0 = (int)v0;
    L.split0 = split0;
    L.grid = (int)std::min<int64_t>(n_mu * L.nsplit, pl.slots) * pl.cg;
    if (launch_forward_logits(L, st) != cudaSuccess) return ORPO_ERR_CUDA;
    split0 += L.nsplit;
  }
  return launch_forward_merge(L, split0, st) == cudaSuccess ? ORPO_OK : ORPO_ERR_CUDA;
}

// The two GEMM classes of one backward block (gemm maps: 0 S K-major rows, 1 W MN-major, 2 S MN-major,
// 3 h MN-major, 4 dh, 5 dW).  With keep bitmaps (backward skips) K runs over the kept tiles only.

// dW[v0 + ..] (+)= S^T h[m0 + ..]: 128-column tiles of S against h, K = the block's rows
GemmClassH dw_class(int64_t v0, int64_t vc, int64_t m0, int64_t mc, int64_t V, int64_t d, int accumulate,
                    const uint32_t* colbits, int ld_col) {
  GemmClassH c{};
  c.a_map = 2, c.a_mn = 2, c.a_mn_base = 0, c.a_k_base = 0;
  c.b_map = 3, c.b_mn = d % 64 == 0 ? 2 : 1, c.b_mn_base = 0, c.b_k_base = (int)m0;
  c.out_map = 5, c.out_row_base = (int)v0, c.out_col_base = 0;
  c.reduce = (m0 > 0 || accumulate) ? 1 : 0;  // the first row block stores, later ones add
  c.out_rows = (int)V, c.out_cols = (int)d;
  c.n_mt = (int)cdiv(vc, kBM), c.n_nt = (int)cdiv(d, kBN), c.kblocks = (int)cdiv(mc, 64);
  c.mt_major = 1;  // CTAs running together share one column slab of S; h stays in L2
  if (colbits) {   // K: the kept row tiles of this 128-column tile's vocabulary tile, 2 k-blocks each
    const int n_mt = (int)cdiv(mc, kBM);
    c.kbits = colbits, c.kwords = ld_col, c.list_shift = 1, c.kg_shift = 1;
    c.ngroups = n_mt, c.clip = n_mt * 2 - c.kblocks;
    c.kbits_rows = (int)cdiv(vc, kBN);
  }
  return c;
}

// dh[m0 + ..] (+)= S W[v0 + ..]: row tiles of S against W, K = the block's vocabulary columns
GemmClassH dh_class(int64_t vc, int64_t m0, int64_t mc, int64_t M, int64_t d, bool reduce, int64_t w_k_base,
                    const uint32_t* rowbits, int ld_row) {
  GemmClassH c{};
  c.a_map = 0, c.a_mn = 0, c.a_mn_base = 0, c.a_k_base = 0;
  c.b_map = 1, c.b_mn = d % 64 == 0 ? 2 : 1, c.b_mn_base = 0, c.b_k_base = (int)w_k_base;
  c.out_map = 4, c.out_row_base = (int)m0, c.out_col_base = 0;
  c.reduce = reduce ? 1 : 0;  // the first vocabulary block stores, later ones add
  c.out_rows = (int)M, c.out_cols = (int)d;
  c.n_mt = (int)cdiv(mc, kBM), c.n_nt = (int)cdiv(d, kBN), c.kblocks = (int)cdiv(vc, 64);
  c.mt_major = 1;
  if (rowbits) {  // K: the kept vocabulary tiles of this row tile, 4 k-blocks each
    const int n_vt = (int)cdiv(vc, kBN);
    c.kbits = rowbits, c.kwords = ld_row, c.list_shift = 0, c.kg_shift = 2;
    c.ngroups = n_vt, c.clip = n_vt * 4 - c.kblocks;
    c.kbits_rows = (int)cdiv(mc, kBM);
  }
  return c;
}

int head_bwd_impl(const void* h, const void* W, const QuantW* q, const int32_t* targets, const uint8_t* mask,
                  const float* lse, const float* g, const float* bmax, float eps, int64_t M, int64_t V, int64_t d,
                  float softcap, float* dh, float* dW, int accumulate_dW, void* workspace, size_t ws_bytes,
                  int32_t* status, void* stream) {
  if (M < 0 || M > kMaxRows || V < 1 || V > kMaxRows || d < 8 || d >= (1 << 20)) return ORPO_ERR_SHAPE;
  if ((!W && !q) || !status) return ORPO_ERR_NULL;
  if (M > 0 && (!h || !targets || !mask || !lse || !g || !dh || !workspace)) return ORPO_ERR_NULL;
  if (d % 8 != 0 || (W && !aligned16(W)) || (dW && !aligned16(dW)) ||
      (M > 0 && (!aligned16(h) || !aligned16(dh) || !aligned16(workspace))))
    return ORPO_ERR_ALIGN;
  if (int e = check_quant(q, d)) return e;
  if (!isfinite(softcap) || !isfinite(eps) || eps < 0.f) return ORPO_ERR_ARG;
  if (M > 0 && ws_bytes < (q ? orpo_head_q_workspace_bytes(M, V, d) : orpo_head_workspace_bytes(M, V, d)))
    return ORPO_ERR_WORKSPACE;
  int sms = 0;
  if (int e = device_check(&sms)) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    if (!dW || accumulate_dW) return ORPO_OK;
    return cudaMemsetAsync(dW, 0, (size_t)V * d * sizeof(float), st) == cudaSuccess ? ORPO_OK : ORPO_ERR_CUDA;
  }

  const BwdBlocks B = bwd_blocks(M, V, q ? d : 0);
  void* S = align_ws(workspace);
  int* counters = reinterpret_cast<int*>(static_cast<uint8_t*>(S) + scratch_bytes(M, V, q ? d : 0));
  // backward skips: plan rounds over the blocks, slots in the area after the counters
  const bool skip = eps > 0.f;
  SkipPlan P{};
  const int64_t n_mblocks = cdiv(M, B.Mc), nblocks_all = n_mblocks * cdiv(V, B.Vc);
  int round_slots = 1;
  if (skip) {
    P.g = g, P.mask = mask, P.targets = targets, P.lse = lse, P.bmax = bmax;
    P.bmax_ld = (int)cdiv(V, kBN);
    P.M = (int)M, P.V = (int)V, P.status = status;
    P.Mc = B.Mc, P.Vc = B.Vc, P.n_mblocks = (int)n_mblocks;
    P.shape = skip_shape(B);
    P.area = reinterpret_cast<uint8_t*>(counters + kCounters);
    P.area_bytes = kSkipBytes;
    P.thr2 = log2f(eps);
    P.chunk_bytes = (int64_t)kBM * d * 2;
    if ((int64_t)P.shape.n_mt * P.shape.n_vt > kMaxTiles) return ORPO_ERR_SHAPE;  // cannot happen: Mc Vc bounded
    round_slots = (int)std::min<int64_t>(nblocks_all, (int64_t)(kSkipBytes / P.shape.slot_bytes));
  }
  const QLayout ql = q ? q_layout(M, V, d) : QLayout{};
  int64_t launch = 0;
  // split-K area after the skip area: partial tiles, then one counter per dh tile (zeroed once per call)
  const size_t split_parts = skip ? 0 : split_part_bytes(M, d, q ? d : 0);
  float* split_part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(counters + kCounters) + kSkipBytes);
  int* split_cnt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(split_part) + split_parts);
  bool split_zeroed = false;
  const int64_t sp = scratch_pitch(B);
  // the skips' bitmaps and tile lists are per 128-row tile
  const Placement pl = placement(sms, !skip);  // recompute and dh / dW GEMM
  const uint32_t b_rows = kBN / pl.cg;                // rows or columns of the GEMMs' B per CTA
  const bool d64 = d % 64 == 0;  // MN-major h / W fetched with one 3-D box per stage
  RecLaunch R;
  GemmLaunch G;
  bool ok = encode_map_2d(&R.mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, d, M, d * 2, 64, kBM) &&
            encode_map_2d(&R.ms_store, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, S, B.Vc, B.Mc, sp * 2, 64, 32) &&
            // gemm maps: 0 S K-major rows, 1 W MN-major, 2 S MN-major, 3 h MN-major, 4 dh, 5 dW
            encode_map_2d(&G.maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, S, B.Vc, B.Mc, sp * 2, 64, kBM) &&
            encode_map_mn3d(&G.maps[2], S, B.Vc, B.Mc, sp * 2, kBM / 64) &&
            (d64 ? encode_map_mn3d(&G.maps[3], h, d, M, d * 2, b_rows / 64)
                 : encode_map_2d(&G.maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, d, M, d * 2, 64, 64)) &&
            encode_map_2d(&G.maps[4], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dh, d, M, d * 4, 32, 32) &&
            (!dW || encode_map_2d(&G.maps[5], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dW, d, V, d * 4, 32, 32));
  if (!ok) return ORPO_ERR_CUDA;
  if (!dW) G.maps[5] = G.maps[4];
  // W maps over the whole bf16 head (encoded once), or per block over the dequantised copy
  auto encode_w = [&](const void* base, int64_t rows) {
    return encode_map_2d(&R.mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, d, rows, d * 2, 64, kBN / pl.cg) &&
           (d64 ? encode_map_mn3d(&G.maps[1], base, d, rows, d * 2, b_rows / 64)
                : encode_map_2d(&G.maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, d, rows, d * 2, 64, 64));
  };
  if (!q && !encode_w(W, V)) return ORPO_ERR_CUDA;
  G.status = status;
  G.cg = pl.cg;
  R.cg = pl.cg;
  R.targets = targets;
  R.mask = mask;
  R.lse = lse;
  R.g = g;
  R.M = (int)M;
  R.V = (int)V;
  R.softcap = softcap > 0.f ? softcap : 0.f;
  R.status = status;
  R.kblocks = (int)cdiv(d, 64);

  // quantised head: vocabulary block 0 is dequantised by a launch of its own; at large M block v + 1
  // by the spare warps of block v's first recompute (into the other buffer; the block's last GEMM,
  // which read that buffer's previous block, precedes it on the stream), at small M by a launch of its
  // own before the block
  const bool side = q && q_side(M);
  int64_t block = 0;  // v-block major, m-block minor
  for (int64_t v0 = 0, vblock = 0; v0 < V; v0 += B.Vc, ++vblock) {
    const int64_t vc = std::min(B.Vc, V - v0);
    if (q && (vblock == 0 || !side) &&
        launch_dequant(q->wq, q->scales, q->biases, q->bits, q->group, v0, vc, d, V, qbuf_ptr(workspace, ql, vblock),
                       status, st) != cudaSuccess)
      return ORPO_ERR_CUDA;
    if (q && !encode_w(qbuf_ptr(workspace, ql, vblock), vc)) return ORPO_ERR_CUDA;
    for (int64_t m0 = 0; m0 < M; m0 += B.Mc) {
      const int64_t mc = std::min(B.Mc, M - m0);
      const int n_mt = (int)cdiv(mc, kBM);
      const int n_vt = (int)cdiv(vc, kBN);
      R.m0 = (int)m0;
      R.v0 = (int)v0;
      R.w_row0 = q ? 0 : (int)v0;
      R.n_mt = n_mt;
      R.n_vt = n_vt;
      const int64_t n_mu = cdiv(n_mt, pl.cg);
      R.chunk = l2_chunk((int)n_mu, (int64_t)pl.cg * kBM * d * 2);
      R.grid = (int)std::min<int64_t>(n_mu * n_vt, pl.slots) * pl.cg;
      uint32_t *rowbits = nullptr, *colbits = nullptr;
      if (skip) {
        const int64_t slot = block % round_slots;
        if (slot == 0) {  // plan the next round of blocks (zeroed bitmaps; tile lists with block maxima)
          P.first_block = (int)block;
          P.nblocks = (int)std::min<int64_t>(round_slots, nblocks_all - block);
          if (launch_skip_plan(P, st) != cudaSuccess) return ORPO_ERR_CUDA;
        }
        uint8_t* base = P.area + (size_t)slot * P.shape.slot_bytes;
        rowbits = reinterpret_cast<uint32_t*>(base + P.shape.rowbits_off());
        colbits = reinterpret_cast<uint32_t*>(base + P.shape.colbits_off());
        if (bmax) {
          R.list = reinterpret_cast<const int*>(base + P.shape.list_off());
          R.count = reinterpret_cast<const int*>(base + P.shape.count_off());
        }
        R.rowbits = rowbits, R.colbits = colbits, R.ld_row = P.shape.ld_row, R.ld_col = P.shape.ld_col;
        R.eps = eps;
      }
      ++block;
      const int64_t n0 = v0 + B.Vc;
      R.side = side && m0 == 0 && n0 < V ? dequant_job(q->wq, q->scales, q->biases, q->bits, q->group, n0,
                                                    std::min(B.Vc, V - n0), d, V, qbuf_ptr(workspace, ql, vblock + 1))
                                      : DequantJob{};
      if (launch_recompute(R, st) != cudaSuccess) return ORPO_ERR_CUDA;

      GemmClassH cdw =
          dW ? dw_class(v0, vc, m0, mc, V, d, accumulate_dW, skip ? colbits : nullptr, P.shape.ld_col) : GemmClassH{};
      GemmClassH cdh = dh_class(vc, m0, mc, M, d, vblock > 0, q ? 0 : v0, skip ? rowbits : nullptr, P.shape.ld_row);
      const int64_t dw_kb = dW ? cdiv(cdw.n_mt, pl.cg) * cdw.n_nt * cdw.kblocks : 0;
      cdh.ksplit = choose_ksplit(cdiv(cdh.n_mt, pl.cg) * cdh.n_nt, cdh.kblocks, (int64_t)cdh.n_mt * cdh.n_nt, pl.slots,
                                 split_parts, dw_kb);
      if (cdh.ksplit > 1) {
        cdh.part = split_part;
        cdh.cnt = split_cnt;
        if (!split_zeroed && cudaMemsetAsync(split_cnt, 0, (size_t)dh_tiles(M, d, q ? d : 0) * 4, st) != cudaSuccess)
          return ORPO_ERR_CUDA;
        split_zeroed = true;
      }
      const int64_t wn = cdiv(d, 2 * kBN);
      const int64_t wide_units = (dW ? cdiv(cdw.n_mt, 2) * wn : 0) + cdiv(cdh.n_mt, 2) * wn;
      const bool wide = use_wide(pl.cg, cdh.ksplit, d, wide_units, pl.slots);
      if (wide) {  // classes count 512-column tiles
        cdh.n_nt = (int)wn;
        if (dW) cdw.n_nt = (int)wn;
      }
      G.wide = wide ? 1 : 0;
      // longer units first
      if (dW && cdw.kblocks >= cdiv(cdh.kblocks, cdh.ksplit)) {
        G.cls[0] = cdw;
        G.cls[1] = cdh;
      } else {
        G.cls[0] = cdh;
        G.cls[1] = cdw;
      }
      const int64_t units = cdiv(cdw.n_mt, pl.cg) * cdw.n_nt + cdiv(cdh.n_mt, pl.cg) * cdh.n_nt * cdh.ksplit;
      G.grid = (int)std::min<int64_t>(units, pl.slots) * pl.cg;
      if (launch % kCounters == 0 && cudaMemsetAsync(counters, 0, kCounterBytes, st) != cudaSuccess)
        return ORPO_ERR_CUDA;
      G.counter = counters + (launch++ % kCounters);
      if (launch_gemm(G, st, K_GEMM) != cudaSuccess) return ORPO_ERR_CUDA;
    }
  }
  return ORPO_OK;
}

extern "C" {

size_t orpo_head_workspace_bytes(int64_t M, int64_t V, int64_t d) {
  if (M < 0 || M > kMaxRows || V < 1 || V > kMaxRows || d < 8 || d >= (1 << 20)) return 0;
  return std::max(partial_bytes(M, kNsplitMax), scratch_bytes(M, V) + kCounterBytes + kSkipBytes + split_bytes(M, d)) +
         1024;
}

size_t orpo_head_q_workspace_bytes(int64_t M, int64_t V, int64_t d) {
  if (M < 0 || M > kMaxRows || V < 1 || V > kMaxRows || d < 8 || d >= (1 << 20)) return 0;
  return q_layout(M, V, d).total;
}

int orpo_head_fwd(const void* h, const void* W, const int32_t* targets, const uint8_t* mask, int64_t M, int64_t V,
                  int64_t d, float softcap, float* logp, float* lse, void* workspace, size_t ws_bytes,
                  int32_t* status, void* stream) {
  return head_fwd_impl(h, W, nullptr, targets, mask, M, V, d, softcap, logp, lse, nullptr, workspace, ws_bytes,
                       status, stream);
}

int orpo_head_fwd_q(const void* h, const uint8_t* wq, const void* scales, const void* biases, int bits, int group,
                    const int32_t* targets, const uint8_t* mask, int64_t M, int64_t V, int64_t d, float softcap,
                    float* logp, float* lse, void* workspace, size_t ws_bytes, int32_t* status, void* stream) {
  const QuantW q{wq, scales, biases, bits, group};
  return head_fwd_impl(h, nullptr, &q, targets, mask, M, V, d, softcap, logp, lse, nullptr, workspace, ws_bytes,
                       status, stream);
}

int orpo_loss(const float* logp, const int32_t* seq_id, const uint8_t* mask, int64_t M, int32_t n_pairs,
              float lambda, float* out, float* ell, float* g, int32_t* status, void* stream) {
  if (M < 0 || M > kMaxRows || n_pairs < 1 || n_pairs > ORPO_MAX_PAIRS) return ORPO_ERR_SHAPE;
  if (!out || !ell || !status || (M > 0 && (!logp || !seq_id || !mask || !g))) return ORPO_ERR_NULL;
  if (!isfinite(lambda) || lambda < 0.f) return ORPO_ERR_ARG;
  int sms = 0;
  if (int e = device_check(&sms)) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launch_loss(ORPO_PREF_ORPO, logp, seq_id, mask, (int)M, n_pairs, lambda, 0.f, nullptr, out, ell, g, status,
                     st) == cudaSuccess
             ? ORPO_OK
             : ORPO_ERR_CUDA;
}

int orpo_pref_loss(int kind, const float* logp, const int32_t* seq_id, const uint8_t* mask, int64_t M,
                   int32_t n_pairs, float beta, float gamma, const float* ref_logp, float* out, float* ell, float* g,
                   int32_t* status, void* stream) {
  if (kind < ORPO_PREF_ORPO || kind > ORPO_PREF_ORPO_FULL) return ORPO_ERR_ARG;
  if (M < 0 || M > kMaxRows || n_pairs < 1 || n_pairs > ORPO_MAX_PAIRS) return ORPO_ERR_SHAPE;
  const bool needs_ref = kind == ORPO_PREF_DPO || kind == ORPO_PREF_IPO || kind == ORPO_PREF_HINGE;
  if (!out || !ell || !status || (M > 0 && (!logp || !seq_id || !mask || !g)) || (needs_ref && !ref_logp))
    return ORPO_ERR_NULL;
  if (!isfinite(beta) || beta < 0.f || !isfinite(gamma) || (kind == ORPO_PREF_IPO && !(beta > 0.f)))
    return ORPO_ERR_ARG;
  int sms = 0;
  if (int e = device_check(&sms)) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launch_loss(kind, logp, seq_id, mask, (int)M, n_pairs, beta, gamma, needs_ref ? ref_logp : nullptr, out,
                     ell, g, status, st) == cudaSuccess
             ? ORPO_OK
             : ORPO_ERR_CUDA;
}

int orpo_head_bwd(const void* h, const void* W, const int32_t* targets, const uint8_t* mask, const float* lse,
                  const float* g, int64_t M, int64_t V, int64_t d, float softcap, float* dh, float* dW,
                  int accumulate_dW, void* workspace, size_t ws_bytes, int32_t* status, void* stream) {
  return head_bwd_impl(h, W, nullptr, targets, mask, lse, g, nullptr, 0.f, M, V, d, softcap, dh, dW, accumulate_dW,
                       workspace, ws_bytes, status, stream);
}

int orpo_head_bwd_q(const void* h, const uint8_t* wq, const void* scales, const void* biases, int bits, int group,
                    const int32_t* targets, const uint8_t* mask, const float* lse, const float* g, int64_t M,
                    int64_t V, int64_t d, float softcap, float* dh, float* dW, int accumulate_dW, void* workspace,
                    size_t ws_bytes, int32_t* status, void* stream) {
  const QuantW q{wq, scales, biases, bits, group};
  return head_bwd_impl(h, nullptr, &q, targets, mask, lse, g, nullptr, 0.f, M, V, d, softcap, dh, dW,
                       accumulate_dW, workspace, ws_bytes, status, stream);
}

size_t orpo_head_block_max_elems(int64_t M, int64_t V) {
  if (M < 0 || M > kMaxRows || V < 1 || V > kMaxRows) return 0;
  return (size_t)cdiv(M, 32) * (size_t)cdiv(V, kBN);
}

int orpo_head_fwd_bmax(const void* h, const void* W, const int32_t* targets, const uint8_t* mask, int64_t M,
                       int64_t V, int64_t d, float softcap, float* logp, float* lse, float* block_max, void* workspace,
                       size_t ws_bytes, int32_t* status, void* stream) {
  if (M > 0 && !block_max) return ORPO_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(block_max) & 3u) return ORPO_ERR_ALIGN;
  return head_fwd_impl(h, W, nullptr, targets, mask, M, V, d, softcap, logp, lse, block_max, workspace, ws_bytes,
                       status, stream);
}

int orpo_head_bwd_skip(const void* h, const void* W, const int32_t* targets, const uint8_t* mask, const float* lse,
                       const float* g, const float* block_max, float eps, int64_t M, int64_t V, int64_t d,
                       float softcap, float* dh, float* dW, int accumulate_dW, void* workspace, size_t ws_bytes,
                       int32_t* status, void* stream) {
  if (reinterpret_cast<uintptr_t>(block_max) & 3u) return ORPO_ERR_ALIGN;
  return head_bwd_impl(h, W, nullptr, targets, mask, lse, g, block_max, eps, M, V, d, softcap, dh, dW,
                       accumulate_dW, workspace, ws_bytes, status, stream);
}

int orpo_head_fwd_q_bmax(const void* h, const uint8_t* wq, const void* scales, const void* biases, int bits,
                         int group, const int32_t* targets, const uint8_t* mask, int64_t M, int64_t V, int64_t d,
                         float softcap, float* logp, float* lse, float* block_max, void* workspace, size_t ws_bytes,
                         int32_t* status, void* stream) {
  if (M > 0 && !block_max) return ORPO_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(block_max) & 3u) return ORPO_ERR_ALIGN;
  const QuantW q{wq, scales, biases, bits, group};
  return head_fwd_impl(h, nullptr, &q, targets, mask, M, V, d, softcap, logp, lse, block_max, workspace, ws_bytes,
                       status, stream);
}

int orpo_head_bwd_q_skip(const void* h, const uint8_t* wq, const void* scales, const void* biases, int bits,
                         int group, const int32_t* targets, const uint8_t* mask, const float* lse, const float* g,
                         const float* block_max, float eps, int64_t M, int64_t V, int64_t d, float softcap, float* dh,
                         float* dW, int accumulate_dW, void* workspace, size_t ws_bytes, int32_t* status,
                         void* stream) {
  if (reinterpret_cast<uintptr_t>(block_max) & 3u) return ORPO_ERR_ALIGN;
  const QuantW q{wq, scales, biases, bits, group};
  return head_bwd_impl(h, nullptr, &q, targets, mask, lse, g, block_max, eps, M, V, d, softcap, dh, dW,
                       accumulate_dW, workspace, ws_bytes, status, stream);
}

int orpo_debug_gemm(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int a_mn_major,
                    int b_mn_major, int32_t* status, void* stream) {
  if (M < 1 || N < 1 || K < 1 || M > kMaxRows || N > kMaxRows || K > kMaxRows) return ORPO_ERR_SHAPE;
  if (!A || !B || !C || !status) return ORPO_ERR_NULL;
  const int64_t a_inner = a_mn_major ? M : K, b_inner = b_mn_major ? N : K;
  if (a_inner % 8 || b_inner % 8 || N % 4 || !aligned16(A) || !aligned16(B) || !aligned16(C))
    return ORPO_ERR_ALIGN;
  int sms = 0;
  if (int e = device_check(&sms)) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  GemmLaunch G;
  const Placement pl = placement(sms);
  const uint32_t b_rows = kBN / pl.cg;
  // MN-major operands whose contiguous extent is a multiple of 64 use the one-box 3-D fetch
  const int a_mode = a_mn_major ? (M % 64 == 0 ? 2 : 1) : 0;
  const int b_mode = b_mn_major ? (N % 64 == 0 ? 2 : 1) : 0;
  bool ok = a_mode == 2   ? encode_map_mn3d(&G.maps[0], A, M, K, M * 2, kBM / 64)
            : a_mode == 1 ? encode_map_2d(&G.maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, M, K, M * 2, 64, 64)
                          : encode_map_2d(&G.maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, K * 2, 64, kBM);
  ok = ok && (b_mode == 2   ? encode_map_mn3d(&G.maps[1], B, N, K, N * 2, b_rows / 64)
              : b_mode == 1 ? encode_map_2d(&G.maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, N, K, N * 2, 64, 64)
                            : encode_map_2d(&G.maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, K * 2, 64, b_rows));
  ok = ok && encode_map_2d(&G.maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, N, M, N * 4, 32, 32);
  if (!ok) return ORPO_ERR_CUDA;
  G.maps[3] = G.maps[4] = G.maps[5] = G.maps[0];
  GemmClassH c{};
  c.a_map = 0, c.a_mn = a_mode;
  c.b_map = 1, c.b_mn = b_mode;
  c.out_map = 2, c.reduce = 0, c.out_rows = (int)M, c.out_cols = (int)N;
  c.n_mt = (int)cdiv(M, kBM), c.n_nt = (int)cdiv(N, kBN), c.kblocks = (int)cdiv(K, 64), c.mt_major = 1;
  const int64_t wn = cdiv(N, 2 * kBN);
  G.wide = use_wide(pl.cg, 1, N, cdiv(c.n_mt, 2) * wn, pl.slots) ? 1 : 0;
  if (G.wide) c.n_nt = (int)wn;
  G.cls[0] = c;
  G.cls[1] = GemmClassH{};
  G.counter = nullptr;
  G.status = status;
  G.cg = pl.cg;
  G.grid = (int)std::min<int64_t>(cdiv(c.n_mt, pl.cg) * c.n_nt, pl.slots) * pl.cg;
  return launch_gemm(G, st, K_DEBUG) == cudaSuccess ? ORPO_OK : ORPO_ERR_CUDA;
}

const char* orpo_status_string(int code) {
  switch (code) {
    case ORPO_OK: return "ok";
    case ORPO_ERR_NULL: return "a required pointer is NULL";
    case ORPO_ERR_SHAPE: return "M, V, d or n_pairs out of range";
    case ORPO_ERR_ALIGN: return "pointer not 16-byte aligned or d not a multiple of 8";
    case ORPO_ERR_ARG: return "softcap or lambda not finite, or lambda < 0";
    case ORPO_ERR_WORKSPACE: return "workspace smaller than orpo_head_workspace_bytes()";
    case ORPO_ERR_CUDA: return "CUDA runtime error";
    case ORPO_ERR_UNSUPPORTED: return "current device is not compute capability 10.3";
    case ORPO_ERR_TOO_LARGE: return "M exceeds ORPO_FWD_STATIC_MAX_ROWS for orpo_head_fwd_static";
    default: break;
  }
  static thread_local char buf[160];
  if (code < 16) return "unknown code";
  buf[0] = 0;
  const struct {
    int bit;
    const char* text;
  } bits[] = {{ORPO_STATUS_TARGET, "target out of range"},
              {ORPO_STATUS_SEQID, "bad sequence id"},
              {ORPO_STATUS_EMPTY_SEQ, "empty sequence"},
              {ORPO_STATUS_NONFINITE, "non-finite value"},
              {ORPO_STATUS_TIMEOUT, "on-chip wait timed out"},
              {ORPO_STATUS_BOUNDS, "index out of bounds (bounds-checked build)"}};
  for (const auto& b : bits) {
    if (code & b.bit) {
      if (buf[0]) strncat(buf, "; ", sizeof(buf) - strlen(buf) - 1);
      strncat(buf, b.text, sizeof(buf) - strlen(buf) - 1);
    }
  }
  return buf[0] ? buf : "unknown status";
}

}  // extern "C"

// ---------------------------------------------------------------- forward without a caller workspace
//
// For callers that may not allocate: the forward's per-split (max, sum-exp)
// partials live in this fixed device array instead of a workspace.  Capacity
// 2^20 floats (4 MiB): 2 * nsplit * Mpad floats, with nsplit capped so that the
// largest accepted M (65536 rows, Mpad 65536) still has 8 splits.
namespace orpo {
namespace {

constexpr int64_t kStaticFloats = 1 << 20;
static __device__ __align__(256) float g_fwd_static_partials[kStaticFloats];

struct StaticAddr {
  float* ptr = nullptr;
};
StaticAddr g_static_addr[64];
std::mutex g_static_mu;

// Device address of the array for the current device (looked up once per device).
int static_partials(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ORPO_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_addr[dev].ptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_static_partials) != cudaSuccess || !p) return ORPO_ERR_CUDA;
    g_static_addr[dev].ptr = static_cast<float*>(p);
  }
  *out = g_static_addr[dev].ptr;
  return ORPO_OK;
}

}  // namespace
}  // namespace orpo

extern "C" int orpo_head_fwd_static(const void* h, const void* W, const int32_t* targets, const uint8_t* mask,
                                    int64_t M, int64_t V, int64_t d, float softcap, float* logp, float* lse,
                                    int32_t* status, void* stream) {
  if (M < 0 || V < 1 || V > kMaxRows || d < 8 || d >= (1 << 20)) return ORPO_ERR_SHAPE;
  if (M > ORPO_FWD_STATIC_MAX_ROWS) return ORPO_ERR_TOO_LARGE;
  if (M == 0) return ORPO_OK;
  if (!h || !W || !targets || !mask || !logp || !lse || !status) return ORPO_ERR_NULL;
  if (d % 8 != 0 || !aligned16(h) || !aligned16(W)) return ORPO_ERR_ALIGN;
  if (!isfinite(softcap)) return ORPO_ERR_ARG;
  int sms = 0;
  if (int e = device_check(&sms)) return e;
  float* part = nullptr;
  if (int e = static_partials(&part)) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  FwdLaunch L;
  const int64_t n_mt = cdiv(M, kBM), n_vt = cdiv(V, kBN);
  const int64_t Mpad = n_mt * kBM;
  const Placement pl = placement(sms);
  const int64_t n_mu = cdiv(n_mt, pl.cg);
  if (!encode_map_2d(&L.mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, d, M, d * 2, 64, kBM) ||
      !encode_map_2d(&L.mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, d, V, d * 2, 64, kBN / pl.cg))
    return ORPO_ERR_CUDA;
  const int cap = (int)std::max<int64_t>(1, kStaticFloats / (2 * Mpad));
  L.cg = pl.cg;
  L.chunk = l2_chunk((int)n_mu, (int64_t)pl.cg * kBM * d * 2);
  L.n_mt = (int)n_mt;
  L.n_vt = (int)n_vt;
  L.nsplit = std::min(choose_nsplit(n_mu, n_vt, pl.slots), cap);
  L.kblocks = (int)cdiv(d, 64);
  L.targets = targets;
  L.mask = mask;
  L.logp = logp;
  L.lse = lse;
  L.part_m = part;
  L.part_s = part + (size_t)L.nsplit * Mpad;
  L.part_cap = L.nsplit;
  L.M = (int)M;
  L.Mpad = (int)Mpad;
  L.V = (int)V;
  L.softcap = softcap > 0.f ? softcap : 0.f;
  L.status = status;
  L.grid = (int)std::min<int64_t>(n_mu * L.nsplit, pl.slots) * pl.cg;
  return launch_forward(L, st) == cudaSuccess ? ORPO_OK : ORPO_ERR_CUDA;
}
