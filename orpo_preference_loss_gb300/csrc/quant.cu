// quant.cu — the standalone dequantisation kernel of the quantised head (quant.cuh holds the loop).
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "quant.cuh"

namespace orpo {
namespace {

constexpr int kUnroll = 4;

template <int kBits>
__global__ void __launch_bounds__(256) dequant_kernel(DequantJob j, int32_t* status) {
  dequant_slices<kBits, kUnroll>(j, blockIdx.x * blockDim.x + threadIdx.x, gridDim.x * blockDim.x, status);
}

}  // namespace

cudaError_t launch_dequant(const uint8_t* wq, const void* scales, const void* biases, int bits, int group,
                           int64_t v0, int64_t rows, int64_t d, int64_t V, void* out_bf16, int32_t* status,
                           cudaStream_t st) {
  const int64_t n = rows * (d / 8);
  if (n >= (1ll << 31)) return cudaErrorInvalidValue;  // cannot happen: a block fits one W buffer (at most 128 MiB of bf16)
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((n + threads * kUnroll - 1) / (threads * kUnroll), 152 * 16);
  const DequantJob j = dequant_job(wq, scales, biases, bits, group, v0, rows, d, V, out_bf16);
  prof_begin(K_DEQUANT, st);
  if (bits == 4)
    dequant_kernel<4><<<(int)blocks, threads, 0, st>>>(j, status);
  else
    dequant_kernel<8><<<(int)blocks, threads, 0, st>>>(j, status);
  prof_end(K_DEQUANT, st);
  return cudaGetLastError();
}

DequantJob dequant_job(const uint8_t* wq, const void* scales, const void* biases, int bits, int group, int64_t v0,
                       int64_t rows, int64_t d, int64_t V, void* out_bf16) {
  return DequantJob{wq, static_cast<const uint16_t*>(scales), static_cast<const uint16_t*>(biases),
                    static_cast<uint4*>(out_bf16), v0, V, (int)rows, (int)d, bits, group};
}

}  // namespace orpo
