// Recurrent decode: the constant-memory inference form of the same attention
// ("LASP-2", abstract: linear attention gives constant-memory inference over
// the sequence length).  For a handful of new tokens per sequence,
//     S <- lambda S + k_t v_t^T,   o_t = S^T q_t,
// with the fp32 state read from and written back to caller memory.  The work
// is a rank-1 update and a matrix-vector product per token, bound by the state
// traffic (2 x d^2 x 4 bytes per sequence), so it runs on the CUDA cores with
// the state in registers: CS CTAs of 8 warps per sequence, CTA y owning the
// column block [y D/CS, (y+1) D/CS) (its outputs depend on nothing else), lane
// l two consecutive columns of it in rows warp, warp + 8, ... -- every warp
// instruction of the state's load and store covers a contiguous row segment,
// and the output's column sums are reduced across the 8 warps in shared
// memory.  Splitting d = 128 over two CTAs halves the registers per thread so
// that more CTAs keep state loads in flight on every SM.
#include <cuda_bf16.h>

#include "internal.h"

namespace linattn {
namespace {

__device__ __forceinline__ float ld_val(const float *p) { return *p; }
__device__ __forceinline__ float ld_val(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_val(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_val(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

constexpr int kDecodeThreads = 256;

template <int D, int CS, typename TIn>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(Problem p, const TIn *q, const TIn *k, const TIn *v,
                                                                TIn *o, float *state) {
  constexpr int W = D / CS;    // columns of this CTA
  constexpr int NC = W / 32;   // columns per lane
  constexpr int NR = D / 8;    // rows per thread (8 warps)
  __shared__ float kk[D], qq[D];
  __shared__ __align__(16) float vv[W];
  __shared__ __align__(16) float part[8][W];
  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H, c0 = blockIdx.y * W;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int64_t off = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float lam = p.decay ? p.decay[h] : 1.f;
  float *base = state + (int64_t)bh * D * D + c0 + NC * lane;
  float s[NR][NC];
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const float *src = base + (warp + 8 * i) * D;
#pragma unroll
    for (int c = 0; c < NC; ++c) s[i][c] = src[c];
  }
  for (int t = 0; t < p.T; ++t) {
    const int64_t row = off + (int64_t)t * p.st;
    if (tid < D) {
      kk[tid] = ld_val(k + row + tid);
      qq[tid] = ld_val(q + row + tid);
    } else if (tid < D + W) {
      vv[tid - D] = ld_val(v + row + c0 + tid - D);
    }
    __syncthreads();
    float vc[NC], acc[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      vc[c] = vv[NC * lane + c];
      acc[c] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      const float kr = kk[warp + 8 * i], qr = qq[warp + 8 * i];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        s[i][c] = fmaf(lam, s[i][c], kr * vc[c]);
        acc[c] = fmaf(s[i][c], qr, acc[c]);
      }
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) part[warp][NC * lane + c] = acc[c];
    __syncthreads();
    if (tid < W) {
      float x = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) x += part[w][tid];
      st_val(o + row + c0 + tid, x);
    }
    __syncthreads();  // kk, qq, vv and part are rewritten by the next token
  }
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    float *dst = base + (warp + 8 * i) * D;
#pragma unroll
    for (int c = 0; c < NC; ++c) dst[c] = s[i][c];
  }
}

template <int D, typename TIn>
cudaError_t launch(const Problem &p, const void *q, const void *k, const void *v, void *o, float *state,
                   cudaStream_t s) {
  TimedLaunch t(K_DECODE, s);
  constexpr int CS = D == 128 ? 2 : 1;
  decode_kernel<D, CS, TIn><<<dim3(p.B * p.H, CS), kDecodeThreads, 0, s>>>(p, (const TIn *)q, (const TIn *)k,
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
