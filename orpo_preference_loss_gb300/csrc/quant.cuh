// quant.cuh — dequantisation of rows of an affine group-quantised head into bf16.
//
// Design page "Training — design", §5.1 tier 4: the pages' head is a 4/8-bit affine
// group-quantised weight (per-group scale and bias) dequantised inside the GEMM loader.  Here
// rows of it are dequantised into a bounded bf16 buffer that the bf16 tensor-core kernels read:
// W[v, j] = bf16(scale[v, j/group] * q[v, j] + bias[v, j/group]) (fp32 arithmetic, one
// nearest-even rounding); 4-bit q are packed two per byte, even column low.  The same loop runs in
// a standalone kernel and in the spare warps of the contraction kernels (at large M, every block
// after the first is dequantised there while the previous one is multiplied).
// Memory-bound: reads bits/8 + 4/group bytes and writes 2 bytes per weight.  4-bit rows are read as
// 32-bit words and 8-bit rows as 64-bit words: wq is 4- (4-bit) or 8-byte (8-bit) aligned and d is a
// multiple of 8 (checked by the host).
#pragma once

#include <stdint.h>

#include "bounds.cuh"

namespace orpo {

// Rows [v0, v0 + rows) of the quantised head into out (bf16 [rows, d], row-major).  rows == 0: no job.
struct DequantJob {
  const uint8_t* wq;
  const uint16_t* scales;
  const uint16_t* biases;
  uint4* out;
  int64_t v0, V;
  int rows, d, bits, group;
};

__device__ __forceinline__ uint32_t dq_pack2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

__device__ __forceinline__ float dq_bf16_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Slice = 8 consecutive weights of a row (one 16-byte bf16 store).  Thread `tid` of T handles slices
// tid, tid + T, ..., kUnroll of them per trip, so a warp's 32 stores of one round cover 512
// contiguous bytes and kUnroll independent loads are in flight per thread.  A block holds at most
// 2^31 slices (the host bounds it), so slice indices fit 32 bits.
template <int kBits, int kUnroll>
__device__ __forceinline__ void dequant_slices(const DequantJob& j, uint32_t tid, uint32_t T, int32_t* status) {
  const uint32_t per_row = (uint32_t)j.d / 8u;
  const uint32_t nslices = (uint32_t)j.rows * per_row;
  const uint32_t ngroups = (uint32_t)(j.d / j.group);
  for (uint32_t base = tid; base < nslices; base += kUnroll * T) {
    uint2 raw[kUnroll];
    float sc[kUnroll], bi[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const uint32_t idx = base + k * T;
      raw[k] = make_uint2(0u, 0u);
      sc[k] = bi[k] = 0.f;
      if (idx < nslices) {
        const uint32_t r = idx / per_row, c = idx - r * per_row;
        const int64_t v = j.v0 + r;
        if (!in_bounds(status, v, j.V)) continue;
        const uint8_t* row = j.wq + v * (int64_t)(j.d * kBits / 8);
        if constexpr (kBits == 4)
          raw[k].x = __ldg(reinterpret_cast<const uint32_t*>(row) + c);
        else
          raw[k] = __ldg(reinterpret_cast<const uint2*>(row) + c);
        const int64_t gi = v * ngroups + (8u * c) / (uint32_t)j.group;
        sc[k] = dq_bf16_to_float(__ldg(j.scales + gi));
        bi[k] = dq_bf16_to_float(__ldg(j.biases + gi));
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const uint32_t idx = base + k * T;
      if (idx >= nslices) break;
      float w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t q =
            kBits == 4 ? (raw[k].x >> (4 * e)) & 15u : ((e < 4 ? raw[k].x : raw[k].y) >> (8 * (e & 3))) & 255u;
        w[e] = fmaf(sc[k], (float)q, bi[k]);
      }
      uint4 o;
      o.x = dq_pack2(w[0], w[1]);
      o.y = dq_pack2(w[2], w[3]);
      o.z = dq_pack2(w[4], w[5]);
      o.w = dq_pack2(w[6], w[7]);
      j.out[idx] = o;  // slices are row-major over [rows, d]
    }
  }
}

// The contraction kernels' spare warps: the last SIDE threads of every CTA take the job, all CTAs of
// the grid sharing it.
__device__ __forceinline__ void side_dequant(const DequantJob& j, int32_t* status) {
  if (j.rows <= 0) return;
  constexpr uint32_t kSide = 96u;  // threads of the spare warps per CTA (the last three warps; engine.cuh)
  const uint32_t tid = blockIdx.x * kSide + (threadIdx.x - (blockDim.x - kSide));
  const uint32_t T = gridDim.x * kSide;
  if (j.bits == 4)
    dequant_slices<4, 8>(j, tid, T, status);
  else
    dequant_slices<8, 8>(j, tid, T, status);
}

}  // namespace orpo
