// CUDA-core kernels for per-dimension gates: one decay per token, head and key
// dimension (the vector form of the data-dependent gate; "Gated Linear
// Attention ..." on the LASP-2 page's related list),
//   S_t = diag(alpha_t) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t,   alpha_t = exp(log_gate_t).
// One CTA walks one (batch, head) sequence token by token with the fp32 state
// in shared memory (row stride d + 1: row walks and column walks are free of
// bank conflicts).  Row i of the state only ever sees key dimension i's gates.
//
// The backward walks the sequence forward once (dq_t = S_t dO_t, and the term
// q_t[i] dq_t[i] of every key dimension, kept in d_log_gate), then backward
// with R_t = diag(alpha_{t+1}) R_{t+1} + q_t dO_t^T (R_{T-1} starts from the
// gradient arriving at the final state): dk_t = R_t v_t, dv_t = R_t^T k_t,
// d_init = diag(alpha_0) R_0, and the gradient of every log-gate
//   d_log_gate[t][i] = sum_{u >= t} (q_u[i] dq_u[i] - k_u[i] dk_u[i]) + sum_j D[i][j] S_T[i][j]
// (d/dC_u[i] of the loss, C the cumulative log-gates: token u as a query gives
// q_u[i] dq_u[i], as a key -k_u[i] dk_u[i], and the final state the last sum;
// summed over u >= t).
#include <cuda_bf16.h>

#include "internal.h"

namespace linattn {
namespace {

constexpr int kVecThreads = 256;

__device__ __forceinline__ float ld_val(const float *p) { return *p; }
__device__ __forceinline__ float ld_val(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_val(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_val(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// shared memory: the state [D][D+1], five vectors of D, two partial-sum buffers of kVecThreads
template <int D>
constexpr size_t vec_smem() {
  return sizeof(float) * ((size_t)D * (D + 1) + 5 * D + 2 * kVecThreads);
}

template <int D, typename TIn>
__global__ void __launch_bounds__(kVecThreads) vec_fwd_kernel(Problem p, const TIn *q, const TIn *k, const TIn *v,
                                                             const float *lg, TIn *o, const float *init,
                                                             float *fin) {
  constexpr int kParts = kVecThreads / D, kSpan = D / kParts;  // row (or column) ranges per thread
  extern __shared__ float sm[];
  float *S = sm, *vq = S + D * (D + 1), *vk = vq + D, *va = vk + D, *vv = va + D, *part = vv + 2 * D;
  const int tid = threadIdx.x, bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
  const int64_t base = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float *g = lg + (int64_t)bh * p.T * D;
  for (int e = tid; e < D * D; e += kVecThreads)
    S[(e / D) * (D + 1) + e % D] = init ? init[(int64_t)bh * D * D + e] : 0.f;
  const int c = tid % D, r0 = (tid / D) * kSpan;  // output column, first row of this thread's range
  for (int t = 0; t < p.T; ++t) {
    const int64_t row = base + (int64_t)t * p.st;
    if (tid < D) {
      vq[tid] = ld_val(q + row + tid);
      vk[tid] = ld_val(k + row + tid);
      vv[tid] = ld_val(v + row + tid);
      va[tid] = expf(g[(int64_t)t * D + tid]);
    }
    __syncthreads();
    for (int e = tid; e < D * D; e += kVecThreads) {
      const int i = e / D, j = e % D;
      float &s = S[i * (D + 1) + j];
      s = fmaf(va[i], s, vk[i] * vv[j]);
    }
    __syncthreads();
    float acc = 0.f;
#pragma unroll 8
    for (int i = r0; i < r0 + kSpan; ++i) acc = fmaf(S[i * (D + 1) + c], vq[i], acc);
    part[tid] = acc;
    __syncthreads();
    if (tid < D) {
      float x = 0.f;
#pragma unroll
      for (int m = 0; m < kParts; ++m) x += part[m * D + tid];
      st_val(o + row + tid, x);
    }
  }
  if (fin) {
    __syncthreads();
    for (int e = tid; e < D * D; e += kVecThreads) fin[(int64_t)bh * D * D + e] = S[(e / D) * (D + 1) + e % D];
  }
}

template <int D, typename TIn>
__global__ void __launch_bounds__(kVecThreads) vec_bwd_kernel(Problem p, const TIn *q, const TIn *k, const TIn *v,
                                                             const TIn *dO, const float *lg, const float *init,
                                                             const float *dfin, TIn *dq, TIn *dk, TIn *dv,
                                                             float *dlg, float *dinit) {
  constexpr int kParts = kVecThreads / D, kSpan = D / kParts;
  extern __shared__ float sm[];
  float *S = sm, *vq = S + D * (D + 1), *vk = vq + D, *va = vk + D, *vv = va + D, *vg = vv + D;
  float *partA = vg + D, *partB = partA + kVecThreads;
  const int tid = threadIdx.x, bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
  const int64_t base = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float *g = lg + (int64_t)bh * p.T * D;
  float *dg = dlg + (int64_t)bh * p.T * D;
  const int c = tid % D, r0 = (tid / D) * kSpan;  // this thread's row / column and its range of the other index

  // forward sweep: S_t, dq_t = S_t dO_t, and q_t[i] dq_t[i] into d_log_gate
  for (int e = tid; e < D * D; e += kVecThreads)
    S[(e / D) * (D + 1) + e % D] = init ? init[(int64_t)bh * D * D + e] : 0.f;
  for (int t = 0; t < p.T; ++t) {
    const int64_t row = base + (int64_t)t * p.st;
    if (tid < D) {
      vq[tid] = ld_val(q + row + tid);
      vk[tid] = ld_val(k + row + tid);
      vv[tid] = ld_val(v + row + tid);
      vg[tid] = ld_val(dO + row + tid);
      va[tid] = expf(g[(int64_t)t * D + tid]);
    }
    __syncthreads();
    for (int e = tid; e < D * D; e += kVecThreads) {
      const int i = e / D, j = e % D;
      float &s = S[i * (D + 1) + j];
      s = fmaf(va[i], s, vk[i] * vv[j]);
    }
    __syncthreads();
    float acc = 0.f;  // row c of S against dO over this thread's column range
#pragma unroll 8
    for (int j = r0; j < r0 + kSpan; ++j) acc = fmaf(S[c * (D + 1) + j], vg[j], acc);
    partA[tid] = acc;
    __syncthreads();
    if (tid < D) {
      float x = 0.f;
#pragma unroll
      for (int m = 0; m < kParts; ++m) x += partA[m * D + tid];
      st_val(dq + row + tid, x);
      dg[(int64_t)t * D + tid] = vq[tid] * x;
    }
  }
  __syncthreads();
  // the final state's term of the log-gate gradient (row tid), then R from d_final
  float gacc = 0.f;
  if (tid < D && dfin) {
    const float *Dr = dfin + (int64_t)bh * D * D + (int64_t)tid * D;
    for (int j = 0; j < D; ++j) gacc = fmaf(Dr[j], S[tid * (D + 1) + j], gacc);
  }
  __syncthreads();
  for (int e = tid; e < D * D; e += kVecThreads)
    S[(e / D) * (D + 1) + e % D] = dfin ? dfin[(int64_t)bh * D * D + e] : 0.f;

  // reverse sweep
  for (int t = p.T - 1; t >= 0; --t) {
    const int64_t row = base + (int64_t)t * p.st;
    if (tid < D) {
      vq[tid] = ld_val(q + row + tid);
      vk[tid] = ld_val(k + row + tid);
      vv[tid] = ld_val(v + row + tid);
      vg[tid] = ld_val(dO + row + tid);
      va[tid] = t == p.T - 1 ? 1.f : expf(g[(int64_t)(t + 1) * D + tid]);  // the carry alpha_{t+1}
    }
    __syncthreads();
    for (int e = tid; e < D * D; e += kVecThreads) {
      const int i = e / D, j = e % D;
      float &s = S[i * (D + 1) + j];
      s = fmaf(va[i], s, vq[i] * vg[j]);
    }
    __syncthreads();
    float a = 0.f, bsum = 0.f;  // dk: row c against v; dv: column c against k
#pragma unroll 8
    for (int m = r0; m < r0 + kSpan; ++m) {
      a = fmaf(S[c * (D + 1) + m], vv[m], a);
      bsum = fmaf(S[m * (D + 1) + c], vk[m], bsum);
    }
    partA[tid] = a;
    partB[tid] = bsum;
    __syncthreads();
    if (tid < D) {
      float x = 0.f, y = 0.f;
#pragma unroll
      for (int m = 0; m < kParts; ++m) {
        x += partA[m * D + tid];
        y += partB[m * D + tid];
      }
      st_val(dk + row + tid, x);
      st_val(dv + row + tid, y);
      gacc += dg[(int64_t)t * D + tid] - vk[tid] * x;
      dg[(int64_t)t * D + tid] = gacc;
    }
  }
  if (dinit) {
    __syncthreads();
    for (int e = tid; e < D * D; e += kVecThreads) {
      const int i = e / D;
      const float a0 = p.T > 0 ? expf(g[i]) : 1.f;
      dinit[(int64_t)bh * D * D + e] = a0 * S[i * (D + 1) + e % D];
    }
  }
}

template <int D, typename TIn>
cudaError_t launch_vec_fwd(const Problem &p, const void *q, const void *k, const void *v, const float *lg, void *o,
                           const float *init, float *fin, cudaStream_t s) {
  auto kern = vec_fwd_kernel<D, TIn>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vec_smem<D>());
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_GATED_VEC_FWD, s);
  kern<<<p.B * p.H, kVecThreads, vec_smem<D>(), s>>>(p, (const TIn *)q, (const TIn *)k, (const TIn *)v, lg,
                                                     (TIn *)o, init, fin);
  return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_vec_bwd(const Problem &p, const void *q, const void *k, const void *v, const void *dO,
                           const float *lg, const float *init, const float *dfin, void *dq, void *dk, void *dv,
                           float *dlg, float *dinit, cudaStream_t s) {
  auto kern = vec_bwd_kernel<D, TIn>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vec_smem<D>());
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_GATED_VEC_BWD, s);
  kern<<<p.B * p.H, kVecThreads, vec_smem<D>(), s>>>(p, (const TIn *)q, (const TIn *)k, (const TIn *)v,
                                                     (const TIn *)dO, lg, init, dfin, (TIn *)dq, (TIn *)dk,
                                                     (TIn *)dv, dlg, dinit);
  return cudaGetLastError();
}

}  // namespace

cudaError_t gated_vec_fwd(const Problem &p, const void *q, const void *k, const void *v, const float *log_gate,
                          void *o, const float *init, float *final_state, cudaStream_t s) {
  if (p.d == 64)
    return p.dtype == 1 ? launch_vec_fwd<64, float>(p, q, k, v, log_gate, o, init, final_state, s)
                        : launch_vec_fwd<64, __nv_bfloat16>(p, q, k, v, log_gate, o, init, final_state, s);
  return p.dtype == 1 ? launch_vec_fwd<128, float>(p, q, k, v, log_gate, o, init, final_state, s)
                      : launch_vec_fwd<128, __nv_bfloat16>(p, q, k, v, log_gate, o, init, final_state, s);
}

cudaError_t gated_vec_bwd(const Problem &p, const void *q, const void *k, const void *v, const void *dO,
                          const float *log_gate, const float *init, const float *d_final, void *dq, void *dk,
                          void *dv, float *d_log_gate, float *d_init, cudaStream_t s) {
  if (p.d == 64)
    return p.dtype == 1 ? launch_vec_bwd<64, float>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv, d_log_gate,
                                                    d_init, s)
                        : launch_vec_bwd<64, __nv_bfloat16>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv,
                                                            d_log_gate, d_init, s);
  return p.dtype == 1 ? launch_vec_bwd<128, float>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv, d_log_gate,
                                                   d_init, s)
                      : launch_vec_bwd<128, __nv_bfloat16>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv,
                                                           d_log_gate, d_init, s);
}

}  // namespace linattn
