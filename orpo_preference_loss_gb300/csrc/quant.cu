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
// Memory-bound: reads bits/8 + 4/group bytes and writes 2 bytes per weight.
#include <cuda_bf16.h>

#include <algorithm>

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

// one thread: kSpan consecutive weights of one row (kSpan / 8 sixteen-byte stores); kSpan is 32
// when d % 32 == 0 (wider loads, more bytes in flight per thread), else 8
template <int kBits, int kSpan>
__global__ void dequant_kernel(const uint8_t* __restrict__ wq, const uint16_t* __restrict__ scales,
                               const uint16_t* __restrict__ biases, int group, int64_t v0, int64_t rows, int64_t d,
                               uint4* __restrict__ out) {
  const int64_t per_row = d / kSpan;
  const int64_t n = rows * per_row;
  const int64_t ngroups = d / group;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row, c = i - r * per_row;
    const int64_t v = v0 + r, j0 = c * kSpan;
    uint32_t words[kSpan * kBits / 32];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(wq + v * (d * kBits / 8) + j0 * kBits / 8);
    if constexpr (kSpan * kBits / 32 % 4 == 0) {
#pragma unroll
      for (int k = 0; k < kSpan * kBits / 128; ++k) {
        const uint4 x = reinterpret_cast<const uint4*>(src)[k];
        words[4 * k] = x.x, words[4 * k + 1] = x.y, words[4 * k + 2] = x.z, words[4 * k + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < kSpan * kBits / 32; ++k) words[k] = src[k];
    }
#pragma unroll
    for (int sub = 0; sub < kSpan / 8; ++sub) {
      const int64_t gi = v * ngroups + (j0 + 8 * sub) / group;
      const float s = bf16_bits_to_float(scales[gi]), b = bf16_bits_to_float(biases[gi]);
      uint32_t q[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int e = 8 * sub + k;  // element within the span
        q[k] = kBits == 4 ? (words[e / 8] >> (4 * (e % 8))) & 15u : (words[e / 4] >> (8 * (e % 4))) & 255u;
      }
      out[(r * d + j0) / 8 + sub] = dequant8(q, s, b);
    }
  }
}

}  // namespace

cudaError_t launch_dequant(const uint8_t* wq, const void* scales, const void* biases, int bits, int group,
                           int64_t v0, int64_t rows, int64_t d, void* out_bf16, cudaStream_t st) {
  // 32 weights per thread needs 16-byte loads: d % 32 == 0 keeps every row 16-byte aligned
  const bool wide = d % 32 == 0 && (reinterpret_cast<uintptr_t>(wq) & 15u) == 0;
  const int64_t n = rows * (d / (wide ? 32 : 8));
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((n + threads - 1) / threads, 152 * 16);
  const uint16_t* sc = static_cast<const uint16_t*>(scales);
  const uint16_t* bi = static_cast<const uint16_t*>(biases);
  uint4* o = static_cast<uint4*>(out_bf16);
  prof_begin(K_DEQUANT, st);
  if (bits == 4 && wide)
    dequant_kernel<4, 32><<<(int)blocks, threads, 0, st>>>(wq, sc, bi, group, v0, rows, d, o);
  else if (bits == 4)
    dequant_kernel<4, 8><<<(int)blocks, threads, 0, st>>>(wq, sc, bi, group, v0, rows, d, o);
  else if (wide)
    dequant_kernel<8, 32><<<(int)blocks, threads, 0, st>>>(wq, sc, bi, group, v0, rows, d, o);
  else
    dequant_kernel<8, 8><<<(int)blocks, threads, 0, st>>>(wq, sc, bi, group, v0, rows, d, o);
  prof_end(K_DEQUANT, st);
  return cudaGetLastError();
}

}  // namespace orpo
