// Zero padding of d = 64 bf16 problems to d = 128, so that they run on the
// tensor-core kernels: with the columns 64..127 of q, k and v zero, every q . k
// is unchanged, the rows and columns 64..127 of the state stay zero, and so do
// the padded columns of every output -- the padded problem is the same problem.
// Rows move in 16-byte pieces (8 bf16); states in fp32.
#include <cuda_bf16.h>

#include "internal.h"

namespace linattn {
namespace {

constexpr int kPadThreads = 256;

// dst [rows][128] contiguous <- src rows of 64 bf16 at the request's strides (zeros past 64)
__global__ void __launch_bounds__(kPadThreads) pad_rows_kernel(const __nv_bfloat16 *src, int H, int T, int64_t sb,
                                                               int64_t sh, int64_t st, __nv_bfloat16 *dst,
                                                               int64_t rows) {
  const int64_t i = (int64_t)blockIdx.x * kPadThreads + threadIdx.x;  // 16-byte piece of the padded rows
  if (i >= rows * 16) return;
  const int64_t r = i >> 4;
  const int c = (int)(i & 15);
  uint4 x = make_uint4(0u, 0u, 0u, 0u);
  if (c < 8) {
    const int64_t bh = r / T, t = r % T;
    const __nv_bfloat16 *row = src + (bh / H) * sb + (bh % H) * sh + t * st;
    x = *reinterpret_cast<const uint4 *>(row + 8 * c);
  }
  *reinterpret_cast<uint4 *>(dst + r * 128 + 8 * c) = x;
}

// dst rows of 64 bf16 at the request's strides <- columns 0..63 of src [rows][128]
__global__ void __launch_bounds__(kPadThreads) unpad_rows_kernel(const __nv_bfloat16 *src, int H, int T, int64_t sb,
                                                                 int64_t sh, int64_t st, __nv_bfloat16 *dst,
                                                                 int64_t rows) {
  const int64_t i = (int64_t)blockIdx.x * kPadThreads + threadIdx.x;
  if (i >= rows * 8) return;
  const int64_t r = i >> 3;
  const int c = (int)(i & 7);
  const int64_t bh = r / T, t = r % T;
  __nv_bfloat16 *row = dst + (bh / H) * sb + (bh % H) * sh + t * st;
  *reinterpret_cast<uint4 *>(row + 8 * c) = *reinterpret_cast<const uint4 *>(src + r * 128 + 8 * c);
}

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

cudaError_t pad_rows_d64(const Problem &p, const void *src, void *dst, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.H * p.T;
  if (rows == 0) return cudaSuccess;
  TimedLaunch t(K_PAD_D64, s);
  pad_rows_kernel<<<blocks_for(rows * 16), kPadThreads, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), p.H, p.T,
                                                                p.sb, p.sh, p.st, static_cast<__nv_bfloat16 *>(dst),
                                                                rows);
  return cudaGetLastError();
}

cudaError_t unpad_rows_d64(const Problem &p, const void *src, void *dst, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.H * p.T;
  if (rows == 0) return cudaSuccess;
  TimedLaunch t(K_PAD_D64, s);
  unpad_rows_kernel<<<blocks_for(rows * 8), kPadThreads, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), p.H, p.T,
                                                                 p.sb, p.sh, p.st, static_cast<__nv_bfloat16 *>(dst),
                                                                 rows);
  return cudaGetLastError();
}

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
