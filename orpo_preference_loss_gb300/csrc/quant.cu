// quant.cu — dequantisation of an affine group-quantised head into a bf16 block.
//
// Design page "Training — design", §5.1 tier 4: the pages' head is 4/8-bit affine
// group-quantised (per-group scale and bias) and dequantised inside the GEMM
// loader.  On sm_103a a per-tile dequantisation inside the contraction would cost
// most of the SM's ALU throughput (each W tile is consumed once per 128 rows), so
// the head is dequantised once per call, one vocabulary block at a time, into a
// bounded bf16 buffer that the bf16 tensor-core kernels then read.  The weight is
// W[v, j] = bf16(scale[v, j/group] * q[v, j] + bias[v, j/group]) (fp32 arithmetic,
// one nearest-even rounding); 4-bit q are packed two per byte, even column low.
// Memory-bound: reads bits/8 + 4/group bytes and writes 2 bytes per weight.  4-bit rows are read as
// 32-bit words and 8-bit rows as 64-bit words: wq is 4- (4-bit) or 8-byte (8-bit) aligned and d is a
// multiple of 8 (checked by the host).
#include <cuda_bf16.h>

#include <algorithm>

#include "bounds.cuh"
#include "internal.h"

namespace orpo {
namespace {

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// 8 weights (one 8-element slice of a row starting at column j0) -> one 16-byte bf16 store
__device__ __forceinline__ uint4 dequant8(const uint32_t (&q)[8], float s, float b) {
  uint4 o;
  o.x = pack2(fmaf(s, (float)q[0], b), fmaf(s, (float)q[1], b));
  o.y = pack2(fmaf(s, (float)q[2], b), fmaf(s, (float)q[3], b));
  o.z = pack2(fmaf(s, (float)q[4], b), fmaf(s, (float)q[5], b));
  o.w = pack2(fmaf(s, (float)q[6], b), fmaf(s, (float)q[7], b));
  return o;
}

// Slice = 8 consecutive weights of a row (one 16-byte bf16 store).  Thread t of T handles slices
// t, t + T, t + 2T, t + 3T per trip, so a warp's 32 stores of one round cover 512 contiguous bytes
// and four independent loads are in flight per thread.  A block holds at most kWBlockBudget bytes
// of bf16 (rows * d / 8 < 2^31 slices), so slice indices fit 32 bits.
constexpr int kUnroll = 4;

template <int kBits>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ wq,
                                                      const uint16_t* __restrict__ scales,
                                                      const uint16_t* __restrict__ biases, int group, int64_t v0,
                                                      int rows, int d, int64_t V, uint4* __restrict__ out,
                                                      int32_t* status) {
  const uint32_t per_row = (uint32_t)d / 8u;
  const uint32_t nslices = (uint32_t)rows * per_row;
  const uint32_t ngroups = (uint32_t)(d / group);
  const uint32_t T = gridDim.x * blockDim.x;
  for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < nslices; base += kUnroll * T) {
    uint2 raw[kUnroll];
    float sc[kUnroll], bi[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const uint32_t idx = base + k * T;
      raw[k] = make_uint2(0u, 0u);
      sc[k] = bi[k] = 0.f;
      if (idx < nslices) {
        const uint32_t r = idx / per_row, c = idx - r * per_row;
        const int64_t v = v0 + r;
        if (!in_bounds(status, v, V)) continue;
        const uint8_t* row = wq + v * (int64_t)(d * kBits / 8);
        if constexpr (kBits == 4)
          raw[k].x = __ldg(reinterpret_cast<const uint32_t*>(row) + c);
        else
          raw[k] = __ldg(reinterpret_cast<const uint2*>(row) + c);
        const int64_t gi = v * ngroups + (8u * c) / (uint32_t)group;
        sc[k] = bf16_bits_to_float(__ldg(scales + gi));
        bi[k] = bf16_bits_to_float(__ldg(biases + gi));
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const uint32_t idx = base + k * T;
      if (idx >= nslices) break;
      uint32_t q[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        q[e] = kBits == 4 ? (raw[k].x >> (4 * e)) & 15u : ((e < 4 ? raw[k].x : raw[k].y) >> (8 * (e & 3))) & 255u;
      out[idx] = dequant8(q, sc[k], bi[k]);  // slices are row-major over [rows, d]
    }
  }
}

}  // namespace

cudaError_t launch_dequant(const uint8_t* wq, const void* scales, const void* biases, int bits, int group,
                           int64_t v0, int64_t rows, int64_t d, int64_t V, void* out_bf16, int32_t* status,
                           cudaStream_t st) {
  const int64_t n = rows * (d / 8);
  if (n >= (1ll << 31)) return cudaErrorInvalidValue;  // cannot happen: a block is bounded by kWBlockBudget
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((n + threads * kUnroll - 1) / (threads * kUnroll), 152 * 16);
  const uint16_t* sc = static_cast<const uint16_t*>(scales);
  const uint16_t* bi = static_cast<const uint16_t*>(biases);
  uint4* o = static_cast<uint4*>(out_bf16);
  prof_begin(K_DEQUANT, st);
  if (bits == 4)
    dequant_kernel<4><<<(int)blocks, threads, 0, st>>>(wq, sc, bi, group, v0, (int)rows, (int)d, V, o, status);
  else
    dequant_kernel<8><<<(int)blocks, threads, 0, st>>>(wq, sc, bi, group, v0, (int)rows, (int)d, V, o, status);
  prof_end(K_DEQUANT, st);
  return cudaGetLastError();
}

}  // namespace orpo
