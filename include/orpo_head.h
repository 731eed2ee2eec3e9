/*
 * orpo_head.h — C ABI of the flash-CCE ORPO head for one GB300 GPU (sm_103a).
 *
 * The head computes, for M response rows of hidden state h and a vocabulary
 * head W, the per-token log-probability of the target token, the ORPO loss
 * over chosen / rejected pairs, and the gradients of that loss with respect to
 * h and W, without ever holding the [M, V] logits in memory.
 *
 * Where each operation is defined (mlx-bun documentation pages):
 *   - "Training — design (ORPO, flash-CCE head, prefix sharing, segmented
 *     backward)", §1 "The objective" (ORPO loss, log1mexp log-odds, mean
 *     response log-prob), §5.1 "The head: from token-chunking to the flash-CCE
 *     kernel" (tier 4: vocab-parallel online softmax, per-block partials and
 *     their merge, recompute backward), and the fused linear-CE implementation
 *     spec (forward / backward bullets, Gemma softcap and its sech^2 slope);
 *   - "Steel flash-CCE — handoff", "The architecture (what's proven)"
 *     (forward partials per vocab block, backward coefficient
 *     g * (onehot - softmax(logit - lse)) * sech^2 and its contraction into dh).
 * The weight gradient dW = dZ^T h is the head-LoRA follow-on that the design
 * page leaves open; it is computed here with the same dZ.
 *
 * Conventions shared by every entry point
 *   - Layouts are row-major and contiguous: h [M, d] bf16, W [V, d] bf16,
 *     dh [M, d] fp32, dW [V, d] fp32; per-row vectors have M entries.
 *   - bf16 data is passed as raw 16-bit words (uint16 bit patterns).
 *   - Every pointer argument is a DEVICE pointer except the stream handle.
 *     The caller allocates every buffer, including the workspace, and keeps
 *     them alive until the work on `stream` has finished.  The library never
 *     allocates, frees or caches device memory and keeps no pointer after it
 *     returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous and stream-ordered.
 *   - Return value: ORPO_OK or a host-detected error code (< 16).  On an error
 *     nothing is launched and no output is touched.
 *   - `status` (device int32, 1 word): data errors found on the GPU are OR-ed
 *     into it as ORPO_STATUS_* bits.  The caller zeroes it before the first
 *     call and reads it after synchronising.  Device code never traps.
 *   - Alignment: h, W, dh, dW and the workspace must be 16-byte aligned
 *     (cudaMalloc'd memory is 256-byte aligned); d must be a multiple of 8.
 *   - Requires a compute-capability 10.3 device (GB300); other devices get
 *     ORPO_ERR_UNSUPPORTED.
 */
#ifndef ORPO_HEAD_H
#define ORPO_HEAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* host-detected return codes */
enum {
  ORPO_OK = 0,
  ORPO_ERR_NULL = 1,        /* a required pointer is NULL */
  ORPO_ERR_SHAPE = 2,       /* M, V, d or n_pairs out of the supported range */
  ORPO_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned or d % 8 != 0 */
  ORPO_ERR_ARG = 4,         /* softcap / lambda not finite, or lambda < 0 */
  ORPO_ERR_WORKSPACE = 5,   /* ws_bytes < orpo_head_workspace_bytes(M, V, d) */
  ORPO_ERR_CUDA = 6,        /* a CUDA runtime call or a launch failed */
  ORPO_ERR_UNSUPPORTED = 7, /* the current device is not compute capability 10.3 */
  ORPO_ERR_TOO_LARGE = 8     /* M exceeds ORPO_FWD_STATIC_MAX_ROWS (orpo_head_fwd_static only) */
};

/* device-detected status bits (OR-ed into *status) */
enum {
  ORPO_STATUS_TARGET = 1 << 4,     /* a mask = 1 row has a target outside [0, V) */
  ORPO_STATUS_SEQID = 1 << 5,      /* seq_id outside [-1, 2P) or ids not non-decreasing */
  ORPO_STATUS_EMPTY_SEQ = 1 << 6,  /* a sequence has no mask = 1 row (its mean is undefined) */
  ORPO_STATUS_NONFINITE = 1 << 7,  /* a non-finite lse, loss, log-odds or gradient */
  ORPO_STATUS_TIMEOUT = 1 << 8,    /* a bounded on-chip wait gave up (the kernel returned early) */
  ORPO_STATUS_BOUNDS = 1 << 9      /* bounds-checked build only (ORPO_DEBUG_BOUNDS): a computed index fell
                                      outside its buffer; the access was skipped */
};

/* Largest number of pairs orpo_loss accepts. */
#define ORPO_MAX_PAIRS 2048

/*
 * Bytes of scratch that orpo_head_fwd and orpo_head_bwd need for these sizes
 * (one workspace serves both).  It holds the per-vocab-split partials of the
 * forward (O(M)) and the bounded bf16 block of logit gradients that the
 * backward streams through (at most 256 MiB whatever M and V are), and, for
 * batches whose dh GEMM has few output tiles (at most 160 tiles of 128 x 256,
 * e.g. M <= 2048 at d = 2560), up to 40 MiB of fp32 partial tiles with which
 * that GEMM splits its K range over more SMs.  The extra memory never grows
 * like M * V.  Returns 0 for invalid sizes.
 */
size_t orpo_head_workspace_bytes(int64_t M, int64_t V, int64_t d);

/*
 * Forward of the head (design page §5.1 tier 4; fused-head spec, forward).
 *   z = h W^T (fp32 accumulation of bf16 products);
 *   z~ = softcap * tanh(z / softcap) if softcap > 0, else z;
 *   lse[t]  = log sum_v exp(z~[t, v])              for every row t;
 *   logp[t] = z~[t, targets[t]] - lse[t]           for mask[t] = 1 rows,
 *   logp[t] = 0                                    for mask[t] = 0 rows
 *             (their targets are never read).
 * The vocabulary is processed in splits with an online (max, sum-exp) state
 * per row and merged per row at the end; no [M, V] buffer exists.
 * targets: int32 [M]; mask: uint8 [M] (nonzero = response row).
 * Device errors: ORPO_STATUS_TARGET (logp[t] is then 0),
 * ORPO_STATUS_NONFINITE (an lse that is not finite).
 * M = 0 is a no-op.  Limits: 1 <= V <= 2^31 - 2^16, 8 <= d < 2^20, M <= 2^31 - 2^16.
 */
int orpo_head_fwd(const void* h_bf16, const void* W_bf16, const int32_t* targets,
                  const uint8_t* mask, int64_t M, int64_t V, int64_t d, float softcap,
                  float* logp, float* lse, void* workspace, size_t ws_bytes,
                  int32_t* status, void* stream);

/*
 * ORPO loss and its gradient with respect to every logp (design page §1;
 * the length-normalised mean and the 1/(1 - P) gradient factor of §4).
 * Sequence 2p is the chosen response of pair p, sequence 2p+1 the rejected one.
 *   seq_id: int32 [M], -1 = padding row, else in [0, 2P); the ids that are not
 *           -1 must be non-decreasing in row order (padding may sit anywhere).
 *   mask: 0 = not supervised, 2 = prompt row (ignored here: see ORPO_PREF_ORPO_FULL),
 *         any other nonzero value = response row
 *   l_s  = mean of logp over the response rows of sequence s     -> ell[2P]
 *   x_p  = (l_w - l_r) - (log1mexp(l_w) - log1mexp(l_r)), log1mexp(x) = log(1 - e^x)
 *   loss = (1/P) sum_p [ -l_w + lambda * softplus(-x_p) ]  (NLL over the chosen response)
 *   out[0..4] = loss, nll = mean(-l_w), or = mean(softplus(-x)),
 *               accuracy = mean(l_w > l_r), margin = mean(x_p)
 *   g[t] = dloss/dlogp[t] = mask[t] * G_{s(t)} / n_{s(t)}, with
 *          G_w = (-1 - lambda * sigmoid(-x) / (1 - e^{l_w})) / P,
 *          G_r = ( lambda * sigmoid(-x) / (1 - e^{l_r})) / P;  g = 0 on pad rows.
 * Sums, means and per-pair differences are taken in two-float arithmetic (pairs
 * of fp32 values, about 48 significant bits) in a fixed order (bitwise
 * reproducible); the per-pair transcendentals and gradients are fp32.
 * Device errors: ORPO_STATUS_SEQID, ORPO_STATUS_EMPTY_SEQ, ORPO_STATUS_NONFINITE
 * (e.g. l = 0 makes log1mexp -inf; it is reported, not clamped).
 * Limits: 1 <= n_pairs <= ORPO_MAX_PAIRS, 0 <= M <= 2^31 - 2^16, lambda >= 0.
 */
int orpo_loss(const float* logp, const int32_t* seq_id, const uint8_t* mask, int64_t M,
              int32_t n_pairs, float lambda, float* out, float* ell, float* g,
              int32_t* status, void* stream);

/*
 * Sibling preference objectives on the same per-token logp (design page §8.3
 * "Objective variants": SimPO, IPO, hinge/SLiC; the xtrain post-training page,
 * Stage P1, for DPO with cached reference log-probs).  Same layouts, status
 * bits, determinism and limits as orpo_loss; only the per-pair term differs.
 * Per sequence the statistic is the mean of logp over its response rows
 * (ORPO, SimPO) or the sum (DPO, IPO, hinge), written to ell[2P].  With
 * D = (s_w - ref_logp[2p]) - (s_r - ref_logp[2p+1]) (ref_logp: device fp32
 * [2P], per-sequence reference sums; required for DPO, IPO, hinge):
 *   ORPO_PREF_ORPO  : exactly orpo_loss with lambda = beta (gamma unused)
 *   ORPO_PREF_SIMPO : softplus(-beta((l_w - l_r) - gamma))
 *   ORPO_PREF_DPO   : -log sigmoid(beta D)
 *   ORPO_PREF_IPO   : (D - 1/(2 beta))^2            (beta > 0)
 *   ORPO_PREF_HINGE : max(0, 1 - beta D)
 *   ORPO_PREF_ORPO_FULL : ORPO with sft_scope = full (design page §1,
 *                     combineFullNll): the NLL is the token mean of -logp over
 *                     the chosen sequence's prompt rows (mask = 2) and response
 *                     rows, -((P-1) pm + M l_w) / ((P-1) + M); the log-odds keep
 *                     response-only means; beta = lambda
 * Mask values for every kind: 0 = row not supervised; 2 = prompt row, read by the
 * head like a response row but seen only by the full-scope NLL (it gets g = 0
 * otherwise); any other nonzero value = response row.
 * loss = mean over pairs; out[0..4] = loss, mean(-statistic_w), mean preference
 * term, accuracy (chosen statistic beats rejected: l_w > l_r, or D > 0), margin
 * (mean of the argument of the term: x, beta((l_w-l_r)-gamma), beta D, D, beta D).
 * g[t] = d loss / d logp[t]: G_s / n_s for the mean kinds, G_s for the sum kinds.
 */
enum {
  ORPO_PREF_ORPO = 0,
  ORPO_PREF_SIMPO = 1,
  ORPO_PREF_DPO = 2,
  ORPO_PREF_IPO = 3,
  ORPO_PREF_HINGE = 4,
  ORPO_PREF_ORPO_FULL = 5
};
int orpo_pref_loss(int kind, const float* logp, const int32_t* seq_id, const uint8_t* mask, int64_t M,
                   int32_t n_pairs, float beta, float gamma, const float* ref_logp, float* out, float* ell,
                   float* g, int32_t* status, void* stream);

/*
 * Backward of the head (fused-head spec, backward bullet; steel handoff,
 * backward structure).  With p = exp(z~ - lse) rebuilt from the saved lse and
 * the logits recomputed tile by tile:
 *   dZ[t, v] = g[t] * (onehot(v == targets[t]) - p[t, v]) * sech^2(z[t, v] / softcap)
 *              (sech^2 factor only when softcap > 0; dZ = 0 on mask = 0 rows),
 *   dh  = dZ W     (fp32 [M, d], overwritten),
 *   dW  = dZ^T h   (fp32 [V, d]; overwritten, or added to when accumulate_dW != 0;
 *                  dW = NULL skips it: a frozen head needs dh only, and the
 *                  backward then does two thirds of the work).
 * g is dloss/dlogp (what orpo_loss returns).  dZ is rounded to bf16 once, in a
 * bounded workspace block, before the two contractions; accumulation is fp32
 * and the result does not depend on run-to-run scheduling (no float atomics).
 * Device errors: ORPO_STATUS_TARGET.
 */
int orpo_head_bwd(const void* h_bf16, const void* W_bf16, const int32_t* targets,
                  const uint8_t* mask, const float* lse, const float* g, int64_t M,
                  int64_t V, int64_t d, float softcap, float* dh, float* dW,
                  int accumulate_dW, void* workspace, size_t ws_bytes, int32_t* status,
                  void* stream);

/*
 * Quantised head (design page §5.1 tier 4: the pages' head is a 4/8-bit affine
 * group-quantised weight with per-group scales and biases).  Same contract as
 * orpo_head_fwd / orpo_head_bwd with W replaced by:
 *   wq      uint8 [V, d * bits / 8]: 4-bit values two per byte (even column in the
 *           low nibble), or one 8-bit value per byte; 4-byte (4-bit) or 8-byte
 *           (8-bit) aligned;
 *   scales, biases  bf16 bit patterns [V, d / group];
 *   bits    4 or 8;  group  a multiple of 8 that divides d.
 * The head's weight is W[v, j] = bf16(scales[v, j/group] * q[v, j] + biases[v, j/group])
 * (fp32 arithmetic, one nearest-even rounding).  Each call walks W in vocabulary
 * blocks dequantised into bf16 buffers of the workspace.  From M = 8192 rows on
 * there are two buffers of at most 128 MiB: the first block is dequantised by a
 * launch of its own, every later one by spare warps of the tensor-core kernels
 * while the previous block is multiplied.  Below 8192 rows (where a block's
 * contraction is too short to hide that work) there is one buffer of at most
 * 256 MiB and a dequantisation launch per block.  (A single 256-row block can
 * exceed these sizes when d is very large.)  The bf16 tensor-core path runs on
 * the dequantised blocks; nothing grows like V * d beyond the quantised weights.  dW, when given, is the gradient with respect to
 * the dequantised weight.  The workspace must hold orpo_head_q_workspace_bytes.
 * Host errors: ORPO_ERR_ARG for bits / group, ORPO_ERR_ALIGN for wq alignment.
 */
size_t orpo_head_q_workspace_bytes(int64_t M, int64_t V, int64_t d);
int orpo_head_fwd_q(const void* h_bf16, const uint8_t* wq, const void* scales_bf16,
                    const void* biases_bf16, int bits, int group, const int32_t* targets,
                    const uint8_t* mask, int64_t M, int64_t V, int64_t d, float softcap,
                    float* logp, float* lse, void* workspace, size_t ws_bytes,
                    int32_t* status, void* stream);
int orpo_head_bwd_q(const void* h_bf16, const uint8_t* wq, const void* scales_bf16,
                    const void* biases_bf16, int bits, int group, const int32_t* targets,
                    const uint8_t* mask, const float* lse, const float* g, int64_t M,
                    int64_t V, int64_t d, float softcap, float* dh, float* dW,
                    int accumulate_dW, void* workspace, size_t ws_bytes, int32_t* status,
                    void* stream);

/*
 * Backward skips ("Steel flash-CCE — handoff" §E, coefficient filter and
 * blockMax vocabulary-block skip; "Training — design" §5.1, the Apple-CCE skips
 * with eps 1e-5 by default).  An approximation that drops the parts of the
 * logit gradient that lie wholly below eps.  Its unit is one tile of 128 rows x
 * 256 vocabulary columns of dZ, aligned to row 0 and column 0.
 *
 * Coefficient filter: a tile is dropped when no row t with g[t] != 0 has an
 * entry with |(onehot - p) sech^2| >= eps in it; dropped tiles contribute
 * nothing to dh or dW, kept tiles contribute exactly what orpo_head_bwd would.
 * Block skip: the forward's block maxima (orpo_head_fwd_bmax) bound p from
 * above; a tile that holds no target of a row with g != 0 and whose bound lies
 * below eps is not recomputed at all.  The filter would drop every such tile,
 * so the block skip changes no result bit; it only saves the recompute.
 *
 * orpo_head_block_max_elems(M, V) = ceil(M / 32) * ceil(V / 256): floats of the
 *   block-max array.
 * orpo_head_fwd_bmax: orpo_head_fwd, and it also writes block_max (fp32,
 *   [ceil(M/32)][ceil(V/256)], row-major, 4-byte aligned; caller-owned): entry
 *   [q][j] = max of z~[t, v] * log2(e) over the rows t of group q (rows 32q ..
 *   32q+31) with mask != 0 and the columns v of tile j (256j .. 256j+255);
 *   -inf when the group has no such row.
 * orpo_head_bwd_skip: orpo_head_bwd with the coefficient filter at threshold
 *   eps (0 <= eps, finite; eps = 0 is exactly orpo_head_bwd).  block_max, when
 *   not NULL, must be what orpo_head_fwd_bmax wrote for the same h, W, mask and
 *   softcap; it enables the block skip.  NULL runs the filter alone.
 * orpo_head_fwd_q_bmax / orpo_head_bwd_q_skip: the same two calls for the
 *   quantised head (arguments as orpo_head_fwd_q / orpo_head_bwd_q, workspace
 *   orpo_head_q_workspace_bytes); the skips then act on the dequantised weight.
 *   The pages run their head this way: quantised, with the skips on.
 * Host errors: ORPO_ERR_ARG for a negative or non-finite eps; otherwise those
 * of orpo_head_fwd / orpo_head_bwd (or their quantised forms).  The workspace
 * is orpo_head_workspace_bytes (orpo_head_q_workspace_bytes when quantised).
 */
size_t orpo_head_block_max_elems(int64_t M, int64_t V);
int orpo_head_fwd_bmax(const void* h_bf16, const void* W_bf16, const int32_t* targets,
                       const uint8_t* mask, int64_t M, int64_t V, int64_t d, float softcap,
                       float* logp, float* lse, float* block_max, void* workspace, size_t ws_bytes,
                       int32_t* status, void* stream);
int orpo_head_bwd_skip(const void* h_bf16, const void* W_bf16, const int32_t* targets,
                       const uint8_t* mask, const float* lse, const float* g, const float* block_max,
                       float eps, int64_t M, int64_t V, int64_t d, float softcap, float* dh,
                       float* dW, int accumulate_dW, void* workspace, size_t ws_bytes,
                       int32_t* status, void* stream);
int orpo_head_fwd_q_bmax(const void* h_bf16, const uint8_t* wq, const void* scales_bf16,
                         const void* biases_bf16, int bits, int group, const int32_t* targets,
                         const uint8_t* mask, int64_t M, int64_t V, int64_t d, float softcap,
                         float* logp, float* lse, float* block_max, void* workspace,
                         size_t ws_bytes, int32_t* status, void* stream);
int orpo_head_bwd_q_skip(const void* h_bf16, const uint8_t* wq, const void* scales_bf16,
                         const void* biases_bf16, int bits, int group, const int32_t* targets,
                         const uint8_t* mask, const float* lse, const float* g,
                         const float* block_max, float eps, int64_t M, int64_t V, int64_t d,
                         float softcap, float* dh, float* dW, int accumulate_dW, void* workspace,
                         size_t ws_bytes, int32_t* status, void* stream);

/* Text of a return code or of a set of ORPO_STATUS_* bits (static storage). */
const char* orpo_status_string(int code);

/*
 * Diagnostic: C = A * B on the same tensor-core engine as the head, for
 * checking the engine in isolation (a plain matrix product; it has no
 * counterpart on the pages).  A is [M, K] bf16 row-major (a_mn_major = 0) or
 * stored transposed as [K, M] (a_mn_major = 1); B is [N, K] (b_mn_major = 0)
 * or stored as [K, N] (b_mn_major = 1); C is fp32 [M, N] row-major and is
 * overwritten.  M, N, K >= 1; the contiguous extent of every operand must be a
 * multiple of 8 elements and of C a multiple of 4.  It takes the engine's tile
 * forms by the same rules as the head's dh / dW contraction (2-CTA clusters where
 * they fit, 256 x 512 pair tiles for wide outputs with several waves of tiles),
 * including the ORPO_CTA_GROUP and ORPO_GEMM_WIDE overrides.
 */
int orpo_debug_gemm(const void* A_bf16, const void* B_bf16, float* C, int64_t M, int64_t N,
                    int64_t K, int a_mn_major, int b_mn_major, int32_t* status, void* stream);

/*
 * Forward for callers that cannot allocate device memory (no counterpart on
 * the pages; a packaging variant of orpo_head_fwd).  Some callers hold only
 * their inputs and outputs: a plugin or custom-call hook of another framework
 * whose enqueue step receives buffers but is not allowed to allocate, or a
 * service that fixes its device-memory budget at start-up and forbids
 * cudaMalloc afterwards.  This entry point computes exactly what orpo_head_fwd
 * computes, but keeps the per-split softmax partials in a fixed 4 MiB array
 * that lives inside the library (every GPU that loads the library holds it
 * until the process exits) instead of in a caller workspace.  It allocates
 * nothing and calls no allocating routine.
 *   - Limit: M <= ORPO_FWD_STATIC_MAX_ROWS; larger M returns ORPO_ERR_TOO_LARGE
 *     and launches nothing.  Large M may use fewer vocabulary splits than
 *     orpo_head_fwd (results agree to rounding).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current).  Under lazy module
 *     loading (the CUDA default since 12.2) that lookup is also what loads the
 *     library's host-side module on the device and reserves the 4 MiB, so it can
 *     fail with ORPO_ERR_CUDA if the device is already out of memory.  A caller
 *     with a fixed memory budget makes that first call (any M >= 1) at start-up,
 *     before it fixes the budget and before any stream capture.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents; nothing in it needs to start at zero (every entry read was
 *     written by the same call).  Calls whose GPU work overlaps in time (other
 *     streams, other host threads) race on it: order them on one stream.
 * Arguments, outputs and device status bits are those of orpo_head_fwd.
 */
#define ORPO_FWD_STATIC_MAX_ROWS 65536
int orpo_head_fwd_static(const void* h_bf16, const void* W_bf16, const int32_t* targets,
                         const uint8_t* mask, int64_t M, int64_t V, int64_t d, float softcap,
                         float* logp, float* lse, int32_t* status, void* stream);

/*
 * Diagnostic: failure detection without a fault (no counterpart on the pages).
 * Launches one thread that waits, through the same bounded wait every pipeline
 * role of the library uses, on a shared-memory barrier that nothing completes.
 * After limit_ns (1 us .. 2 s) the wait gives up, ORPO_STATUS_TIMEOUT is OR-ed
 * into *status (device word) and the kernel returns; the context stays usable.
 */
int orpo_debug_wait_timeout(int32_t* status, int64_t limit_ns, void* stream);

/*
 * Diagnostic: device time of the library's own launches (no counterpart on
 * the pages).  Between orpo_profile_start() and orpo_profile_stop(), every
 * kernel the library launches is bracketed by two CUDA events on its stream.
 * orpo_profile_stop() waits for those events and writes, for kernel kinds
 * 0 .. nkinds-1 (names from orpo_profile_kind_name: fwd_logits, fwd_merge,
 * orpo_loss, bwd_recompute, bwd_grad_gemm, debug_gemm), the summed milliseconds
 * into ms[] and the launch count into count[] (host arrays).  Events are
 * host-side objects pooled inside the library; no device memory is used.
 */
int orpo_profile_start(void);
int orpo_profile_stop(double* ms, int64_t* count, int nkinds);
const char* orpo_profile_kind_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* ORPO_HEAD_H */
