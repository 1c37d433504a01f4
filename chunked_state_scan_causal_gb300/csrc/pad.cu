// States of bf16 d = 64 problems that run on the d = 128 tensor-core kernels:
// [n][64][64] fp32 to and from the top-left block of [n][128][128] (zeros
// elsewhere).  The padded problem is the same problem: with the columns 64..127
// of q, k, v zero (the kernels' tiles load them as zeros), the state's rows and
// columns 64..127 stay zero.
#include <cuda_bf16.h>

#include "internal.h"

namespace linattn {
namespace {

constexpr int kPadThreads = 256;

// dst [n][128][128] <- src [n][64][64] in the top-left block, zeros elsewhere (fp32)
__global__ void __launch_bounds__(kPadThreads) pad_state_kernel(const float *src, float *dst, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * kPadThreads + threadIdx.x;
  if (i >= n * 128 * 128) return;
  const int64_t m = i >> 14;
  const int r = (int)((i >> 7) & 127), c = (int)(i & 127);
  dst[i] = (r < 64 && c < 64) ? src[m * 4096 + r * 64 + c] : 0.f;
}

// dst [n][64][64] <- the top-left block of src [n][128][128]
__global__ void __launch_bounds__(kPadThreads) unpad_state_kernel(const float *src, float *dst, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * kPadThreads + threadIdx.x;
  if (i >= n * 64 * 64) return;
  const int64_t m = i >> 12;
  const int r = (int)((i >> 6) & 63), c = (int)(i & 63);
  dst[i] = src[m * 16384 + r * 128 + c];
}

unsigned blocks_for(int64_t n) { return (unsigned)((n + kPadThreads - 1) / kPadThreads); }

}  // namespace

cudaError_t pad_state_d64(const float *src, float *dst, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  TimedLaunch t(K_PAD_D64, s);
  pad_state_kernel<<<blocks_for(n * 16384), kPadThreads, 0, s>>>(src, dst, n);
  return cudaGetLastError();
}

cudaError_t unpad_state_d64(const float *src, float *dst, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  TimedLaunch t(K_PAD_D64, s);
  unpad_state_kernel<<<blocks_for(n * 4096), kPadThreads, 0, s>>>(src, dst, n);
  return cudaGetLastError();
}

}  // namespace linattn
