// Recurrent decode: the constant-memory inference form of the same attention
// ("LASP-2", abstract: linear attention gives constant-memory inference over
// the sequence length).  For a handful of new tokens per sequence,
//     S <- lambda S + k_t v_t^T,   o_t = S^T q_t,
// with the fp32 state read from and written back to caller memory.  The work
// is a rank-1 update and a matrix-vector product per token, bound by the state
// traffic (2 x d^2 x 4 bytes per sequence), so it runs on the CUDA cores: a CTA
// owns 32 state columns of one sequence, thread r owns state row r of them.
#include <cuda_bf16.h>

#include "internal.h"

namespace linattn {
namespace {

__device__ __forceinline__ float ld_val(const float *p) { return *p; }
__device__ __forceinline__ float ld_val(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_val(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_val(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

template <int D, typename TIn>
__global__ void __launch_bounds__(D) decode_kernel(Problem p, const TIn *q, const TIn *k, const TIn *v, TIn *o,
                                                   float *state) {
  constexpr int NW = D / 32;
  __shared__ float vcol[32];
  __shared__ float part[NW][32];
  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
  const int c0 = blockIdx.y * 32;
  const int r = threadIdx.x, lane = r & 31, warp = r >> 5;
  const int64_t off = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float lam = p.decay ? p.decay[h] : 1.f;
  float *srow = state + ((int64_t)bh * D + r) * D + c0;
  float s[32];
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const float4 x = *reinterpret_cast<const float4 *>(srow + j);
    s[j] = x.x; s[j + 1] = x.y; s[j + 2] = x.z; s[j + 3] = x.w;
  }
  for (int t = 0; t < p.T; ++t) {
    const int64_t row = off + (int64_t)t * p.st;
    if (r < 32) vcol[r] = ld_val(v + row + c0 + r);
    const float kr = ld_val(k + row + r), qr = ld_val(q + row + r);
    __syncthreads();
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      s[j] = fmaf(lam, s[j], kr * vcol[j]);
      acc[j] = s[j] * qr;
    }
    // column sums over the D state rows: warp shuffles, then across warps
#pragma unroll
    for (int j = 0; j < 32; ++j) {
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], m);
    }
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < 32; ++j) part[warp][j] = acc[j];
    }
    __syncthreads();
    if (r < 32) {
      float x = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) x += part[w][r];
      st_val(o + row + c0 + r, x);
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < 32; j += 4)
    *reinterpret_cast<float4 *>(srow + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
}

template <int D, typename TIn>
cudaError_t launch(const Problem &p, const void *q, const void *k, const void *v, void *o, float *state,
                   cudaStream_t s) {
  TimedLaunch t(K_DECODE, s);
  decode_kernel<D, TIn><<<dim3(p.B * p.H, D / 32), D, 0, s>>>(p, (const TIn *)q, (const TIn *)k,
                                                             (const TIn *)v, (TIn *)o, state);
  return cudaGetLastError();
}

}  // namespace

cudaError_t decode(const Problem &p, const void *q, const void *k, const void *v, void *o, float *state,
                   cudaStream_t s) {
  if (p.d == 64)
    return p.dtype == 1 ? launch<64, float>(p, q, k, v, o, state, s)
                        : launch<64, __nv_bfloat16>(p, q, k, v, o, state, s);
  return p.dtype == 1 ? launch<128, float>(p, q, k, v, o, state, s)
                      : launch<128, __nv_bfloat16>(p, q, k, v, o, state, s);
}

}  // namespace linattn
