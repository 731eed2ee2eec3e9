// internal.h — host-side declarations shared by the translation units of liborpo_head.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "quant.cuh"

namespace orpo {

// ---- kernels using more than 48 KiB of dynamic shared memory opt in once per device
// (`done` is the caller's per-kernel table of devices already set; host threads may race to set
// it, which only repeats an idempotent attribute call)
template <class Kernel>
inline cudaError_t opt_in_smem(Kernel kernel, int bytes, std::atomic<int> (&done)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (dev < 0 || dev >= 64 || done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
  return e;
}

// ---- launch timing (profile.cu); no-ops unless orpo_profile_start() was called
enum KernelKind { K_FWD = 0, K_MERGE, K_LOSS, K_REC, K_GEMM, K_DEBUG, K_DEQUANT, K_SKIP, K_NKINDS };
void prof_begin(int kind, cudaStream_t st);
void prof_end(int kind, cudaStream_t st);

// ---- tiling / blocking constants visible to the host
constexpr int kBM = 128;          // rows per accumulator tile
constexpr int kBN = 256;          // columns per accumulator tile
constexpr int kNsplitMax = 64;    // most vocabulary splits of the forward
constexpr int64_t kMcMax = 16384; // rows per backward block
constexpr int64_t kScratchBudget = 256ll << 20;  // bytes of the bf16 dZ block
constexpr int kMaxTiles = (int)(kScratchBudget / 2 / (kBM * kBN));  // 128 x 256 tiles in one dZ block

// ---- L2-aware unit order (chunk_decode in engine.cuh): units along M per chunk.  The rows of h
// that concurrently running units re-read (one 128-row tile per M unit) are kept within
// kL2ChunkBytes; the chunks are then made about equal.
constexpr int64_t kL2ChunkBytes = 48ll << 20;
__host__ __device__ inline int l2_chunk(int n_m, int64_t bytes_per_m) {
  const int64_t rmax = bytes_per_m > 0 ? (kL2ChunkBytes / bytes_per_m > 1 ? kL2ChunkBytes / bytes_per_m : 1) : n_m;
  if (rmax >= n_m) return n_m > 0 ? n_m : 1;
  const int64_t nc = (n_m + rmax - 1) / rmax;
  return (int)((n_m + nc - 1) / nc);
}

// ---- tensor-core CTA group of the engine kernels (engine.cuh): 2 = 2-CTA clusters sharing each
// tcgen05.mma, 1 = single-CTA tiles.  The host encodes the B operand's tensor map with boxes of
// kBN / cg rows (each CTA of a pair fetches half of B).  Every contraction runs on clusters where
// they fit; ORPO_CTA_GROUP=1 forces single CTAs everywhere.
int engine_pair_clusters();       // co-resident 2-CTA clusters on the current device (0: none)
int engine_cta_group_override();  // 0 (default policy), 1 or 2 (ORPO_CTA_GROUP)

// ---- forward
struct FwdLaunch {
  CUtensorMap mh, mw;  // h K-major box {64,128}; W K-major box {64,256 / cg}
  int n_mt, nsplit, n_vt, kblocks;
  const int32_t* targets;
  const uint8_t* mask;
  float* logp;
  float* lse;
  float* part_m;
  float* part_s;
  int M, Mpad, V;
  float softcap;
  int32_t* status;
  int grid;
  int col0 = 0;    // vocabulary column of row 0 of mw
  int split0 = 0;  // first split index this launch writes
  int part_cap = 0;  // splits part_m / part_s hold (Mpad floats each)
  float* bmax = nullptr;  // optional block maxima [ceil(M/32), ceil(V/256)] (base-2 softcapped logits)
  int chunk = 0;          // M units (row tiles, or pairs of them) per L2 chunk (l2_chunk); 0: all of them
  int cg = 1;             // CTA group; grid = cg x (CTAs or clusters)
  DequantJob side{};      // quantised head: the next block's dequantisation, done by the spare warps
};
cudaError_t launch_forward(const FwdLaunch& L, cudaStream_t st);  // logits kernel + merge of L.nsplit splits
cudaError_t launch_forward_logits(const FwdLaunch& L, cudaStream_t st);
cudaError_t launch_forward_merge(const FwdLaunch& L, int nsplit_total, cudaStream_t st);

// ---- backward: recompute dZ for one (row block, vocab block) into the scratch
struct RecLaunch {
  CUtensorMap mh, mw, ms_store;  // h, W as in the forward (W box {64, 256 / cg}); S store box {64,32}
  int m0, v0, n_mt, n_vt, kblocks;
  const int32_t* targets;
  const uint8_t* mask;
  const float* lse;
  const float* g;
  int M, V;
  float softcap;
  int32_t* status;
  int grid;
  int w_row0;  // row of mw holding vocabulary column m0's block start v0 (v0 itself unless W is a block copy)
  // backward skips
  const int* list = nullptr;   // tiles to compute (vt * n_mt + mt, ascending) and their count, or all tiles
  const int* count = nullptr;
  uint32_t* rowbits = nullptr;  // coefficient filter: zeroed keep bitmaps [n_mt][ld_row] and [n_vt][ld_col],
  uint32_t* colbits = nullptr;  // or nullptr for no filter
  int ld_row = 0, ld_col = 0;
  float eps = 0.f;
  int chunk = 0;                // M units per L2 chunk (l2_chunk); 0: all of them
  int cg = 1;                   // CTA group (1 whenever the skip bitmaps or lists are used)
  DequantJob side{};            // quantised head: the next block's dequantisation, done by the spare warps
};
cudaError_t launch_recompute(const RecLaunch& L, cudaStream_t st);

// ---- backward skips (skip.cu): per (row block, vocabulary block), tiles of 128 x 256
// One plan launch covers a round of consecutive blocks (v-block major, m-block minor, as the backward
// walks them), one CTA per block, each with its own slot in the skip area:
//   ints  list[n_mt * n_vt]  tiles to recompute (vt * n_mt + mt, ascending), then count
//   words rowbits[n_mt][ld_row], colbits[n_vt][ld_col]  the filter's keep bitmaps (zeroed by the plan)
struct SkipShape {
  int n_mt, n_vt, ld_row, ld_col;
  size_t slot_bytes;
  __host__ __device__ size_t list_off() const { return 0; }
  __host__ __device__ size_t count_off() const { return (size_t)n_mt * n_vt * 4; }
  __host__ __device__ size_t rowbits_off() const { return count_off() + 16; }
  __host__ __device__ size_t colbits_off() const { return rowbits_off() + (size_t)n_mt * ld_row * 4; }
  __host__ __device__ size_t end() const { return colbits_off() + (size_t)n_vt * ld_col * 4; }
};
struct SkipPlan {
  const float* g;
  const uint8_t* mask;
  const int32_t* targets;
  const float* lse;
  const float* bmax;  // forward block maxima [ceil(M/32)][bmax_ld], base 2; nullptr: filter only (no lists)
  int bmax_ld;
  int M, V;
  int64_t Mc, Vc;     // block sizes; blocks are numbered b = vblock * n_mblocks + mblock
  int n_mblocks;
  int first_block, nblocks;  // this round: blocks first_block .. first_block + nblocks - 1, slot b - first_block
  SkipShape shape;    // of a full block (edge blocks use a prefix of it)
  uint8_t* area;      // slot s at area + s * shape.slot_bytes
  size_t area_bytes;
  float thr2;         // log2(eps)
  int32_t* status;
  int64_t chunk_bytes;  // h bytes per row tile: the list follows the recompute's l2_chunk order
};
cudaError_t launch_skip_plan(const SkipPlan& P, cudaStream_t st);  // lists and zeroed bitmaps for a round

// ---- quantised head: affine group dequantisation of W rows [v0, v0 + rows) into bf16 [rows, d]
cudaError_t launch_dequant(const uint8_t* wq, const void* scales, const void* biases, int bits, int group,
                           int64_t v0, int64_t rows, int64_t d, int64_t V, void* out_bf16, int32_t* status,
                           cudaStream_t st);
DequantJob dequant_job(const uint8_t* wq, const void* scales, const void* biases, int bits, int group, int64_t v0,
                       int64_t rows, int64_t d, int64_t V, void* out_bf16);

// ---- generic two-class GEMM with an fp32 store / reduce-add epilogue
struct GemmClassH {
  int a_map, a_mn, a_mn_base, a_k_base;
  int b_map, b_mn, b_mn_base, b_k_base;
  int out_map, out_row_base, out_col_base, reduce;
  int out_rows, out_cols;  // valid extent of the output tensor
  int n_mt, n_nt, kblocks;
  int mt_major;
  // sparse K (backward skips): bitmap (mt >> list_shift) of kept groups of 2^kg_shift k-blocks at
  // kbits + index * kwords; ngroups groups, the last clip k-blocks short; nullptr: dense
  const uint32_t* kbits = nullptr;
  int kwords = 0, list_shift = 0, kg_shift = 0, ngroups = 0, clip = 0;
  int kbits_rows = 0;  // bitmaps at kbits (bounds-checked build)
  // split K (dense only): K in ksplit parts; part holds n_mt * n_nt * ksplit fp32 tiles of 128 x 256,
  // cnt n_mt * n_nt zeroed counters (reset by the kernel after use)
  int ksplit = 1;
  float* part = nullptr;
  int* cnt = nullptr;
};
struct GemmLaunch {
  CUtensorMap maps[6];   // B operands' boxes cover kBN / cg rows or columns
  GemmClassH cls[2];     // n_mt counts 128-row output tiles; a pair takes two
  int* counter;  // zeroed unit counter (dynamic scheduling), or nullptr for static round-robin
  int32_t* status;
  int grid;
  int cg = 1;    // CTA group (1 whenever a class has sparse K)
  int wide = 0;  // 2-CTA only, no split K: 256 x 512 tiles (classes' n_nt count 512-column tiles)
};
cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t st, int kind);

// ---- loss
// kind: 0 ORPO (beta = lambda), 1 SimPO, 2 DPO, 3 IPO, 4 hinge; ref = per-sequence reference sums or nullptr
cudaError_t launch_loss(int kind, const float* logp, const int32_t* seq_id, const uint8_t* mask, int M, int P,
                        float beta, float gamma, const float* ref, float* out, float* ell, float* g, int32_t* status,
                        cudaStream_t st);

// ---- tensor maps (driver entry point fetched through the runtime)
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// MN-major bf16 operand [K, MN] (MN contiguous, MN % 64 == 0) viewed as {64, K, MN/64}: one TMA box
// {64, 64, chunks} fetches `chunks` 64-wide column blocks of 64 k-rows, laid out block after block.
bool encode_map_mn3d(CUtensorMap* map, const void* base, uint64_t mn, uint64_t k, uint64_t row_bytes,
                     uint32_t chunks);

}  // namespace orpo
