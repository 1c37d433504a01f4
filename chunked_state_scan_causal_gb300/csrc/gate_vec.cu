// CUDA-core kernels for per-dimension gates: one decay per token, head and key
// dimension (the vector form of the data-dependent gate; "Gated Linear
// Attention ..." on the LASP-2 page's related list),
//   S_t = diag(alpha_t) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t,   alpha_t = exp(log_gate_t).
// A CTA walks one chunk group of one (batch, head) sequence token by token with
// the fp32 state in shared memory (row stride d + 1: row walks and column walks
// are free of bank conflicts).  Row i of the state only ever sees key dimension
// i's gates, so the groups are joined by scans whose multipliers are per row:
//   forward:  S_{g+1} = diag(A_g) S_g + U_g,   A_g[i] = prod of group g's gates of dimension i,
//             U_g the group's state walked from zero;
//   backward: Dfin_{g-1} = W_g + diag(A_g) Dfin_g, Dfin_{G-1} = the gradient at the final state,
//             W_g = sum_{t in g} diag(alpha_start .. alpha_t) q_t dO_t^T (walked backward),
// Dfin_g being the gradient arriving at group g's last state from the groups after it.
//
// The backward of a group walks it forward once (dq_t = S_t dO_t, and the term
// q_t[i] dq_t[i] of every key dimension, kept in d_log_gate), then backward
// with R_t = diag(alpha_{t+1}) R_{t+1} + q_t dO_t^T (R at the group's last token
// starts from Dfin_g): dk_t = R_t v_t, dv_t = R_t^T k_t, d_init = diag(alpha_0) R_0
// (group 0), and the gradient of every log-gate of the group
//   d_log_gate[t][i] = sum_{u >= t in g} (q_u[i] dq_u[i] - k_u[i] dk_u[i]) + sum_j Dfin_g[i][j] S_end[i][j]
// (d/dC_u[i] of the loss, C the cumulative log-gates: token u as a query gives
// q_u[i] dq_u[i], as a key -k_u[i] dk_u[i]; every later token sees the gates of
// group g only through its last state S_end, whence the last sum).
#include <cuda_bf16.h>

#include <algorithm>

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

// Chunk groups of L tokens (the last one shorter): CTA (bh, g) walks tokens [g L, min(T, (g+1) L)).
struct VecGroups {
  int G, L;
  __device__ int start(int g) const { return g * L; }
  __device__ int end(int g, int T) const { return min(T, (g + 1) * L); }
};

// Forward walk of group g = blockIdx.y of sequence bh = blockIdx.x from its entering
// state (init [G][BH][D][D], or zero), with the outputs o (or none), the group's last
// state (fin [G][BH][D][D], or none) and the sums of its log-gates per key dimension
// (gsum [G][BH][D], or none).
template <int D, typename TIn>
__global__ void __launch_bounds__(kVecThreads) vec_fwd_kernel(Problem p, VecGroups gr, const TIn *q, const TIn *k,
                                                             const TIn *v, const float *lg, TIn *o,
                                                             const float *init, float *fin, float *gsum) {
  constexpr int kParts = kVecThreads / D, kSpan = D / kParts;  // row (or column) ranges per thread
  extern __shared__ float sm[];
  float *S = sm, *vq = S + D * (D + 1), *vk = vq + D, *va = vk + D, *vv = va + D, *part = vv + 2 * D;
  const int tid = threadIdx.x, bh = blockIdx.x, gi = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int64_t BH = (int64_t)p.B * p.H, slot = (int64_t)gi * BH + bh;
  const int64_t base = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float *g = lg + (int64_t)bh * p.T * D;
  const int t0 = gr.start(gi), t1 = gr.end(gi, p.T);
  for (int e = tid; e < D * D; e += kVecThreads)
    S[(e / D) * (D + 1) + e % D] = init ? init[slot * D * D + e] : 0.f;
  float gs = 0.f;  // this thread's key dimension: the group's sum of log-gates
  const int c = tid % D, r0 = (tid / D) * kSpan;  // output column, first row of this thread's range
  for (int t = t0; t < t1; ++t) {
    const int64_t row = base + (int64_t)t * p.st;
    if (tid < D) {
      if (o) vq[tid] = ld_val(q + row + tid);
      vk[tid] = ld_val(k + row + tid);
      vv[tid] = ld_val(v + row + tid);
      const float lgv = g[(int64_t)t * D + tid];
      gs += lgv;
      va[tid] = expf(lgv);
    }
    __syncthreads();
    for (int e = tid; e < D * D; e += kVecThreads) {
      const int i = e / D, j = e % D;
      float &s = S[i * (D + 1) + j];
      s = fmaf(va[i], s, vk[i] * vv[j]);
    }
    __syncthreads();
    if (o) {
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
  }
  if (fin) {
    __syncthreads();
    for (int e = tid; e < D * D; e += kVecThreads) fin[slot * D * D + e] = S[(e / D) * (D + 1) + e % D];
  }
  if (gsum && tid < D) gsum[slot * D + tid] = gs;
}

// The reverse aggregate of group g = blockIdx.y of sequence bh = blockIdx.x:
//   W_g = sum_{t in g} diag(alpha_start .. alpha_t) q_t dO_t^T,
// walked backward (A <- diag(alpha_t) (A + q_t dO_t^T)), into W [G][BH][D][D].
template <int D, typename TIn>
__global__ void __launch_bounds__(kVecThreads) vec_ragg_kernel(Problem p, VecGroups gr, const TIn *q,
                                                              const TIn *dO, const float *lg, float *W) {
  extern __shared__ float sm[];
  float *A = sm, *vq = A + D * (D + 1), *vg = vq + D, *va = vg + D;
  const int tid = threadIdx.x, bh = blockIdx.x, gi = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int64_t BH = (int64_t)p.B * p.H, slot = (int64_t)gi * BH + bh;
  const int64_t base = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float *g = lg + (int64_t)bh * p.T * D;
  const int t0 = gr.start(gi), t1 = gr.end(gi, p.T);
  for (int e = tid; e < D * D; e += kVecThreads) A[(e / D) * (D + 1) + e % D] = 0.f;
  for (int t = t1 - 1; t >= t0; --t) {
    const int64_t row = base + (int64_t)t * p.st;
    __syncthreads();  // the previous token's update has read the vectors
    if (tid < D) {
      vq[tid] = ld_val(q + row + tid);
      vg[tid] = ld_val(dO + row + tid);
      va[tid] = expf(g[(int64_t)t * D + tid]);
    }
    __syncthreads();
    for (int e = tid; e < D * D; e += kVecThreads) {
      const int i = e / D, j = e % D;
      float &a = A[i * (D + 1) + j];
      a = va[i] * fmaf(vq[i], vg[j], a);
    }
  }
  __syncthreads();
  for (int e = tid; e < D * D; e += kVecThreads) W[slot * D * D + e] = A[(e / D) * (D + 1) + e % D];
}

// The scans across groups, one thread per (sequence, state element (i, j)), with the
// per-row multipliers A_g[i] = exp(gsum[g][bh][i]):
//   forward: out[g] = S_g, S_0 = init (or 0), S_{g+1} = A_g S_g + X_g; total = S_G
//   reverse: out[g] = Dfin_g, Dfin_{G-1} = init (or 0), Dfin_{g-1} = X_g + A_g Dfin_g; total = Dfin_{-1}
__global__ void __launch_bounds__(256) vec_scan_kernel(int G, int64_t BH, int D, const float *X,
                                                       const float *gsum, const float *init, float *out,
                                                       float *total, int reverse) {
  const int64_t DD = (int64_t)D * D, n = BH * DD;
  const int64_t x = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (x >= n) return;
  const int64_t bh = x / DD, e = x % DD, i = e / D;
  float s = init ? init[x] : 0.f;
  for (int m = 0; m < G; ++m) {
    const int gi = reverse ? G - 1 - m : m;
    const int64_t slot = (int64_t)gi * BH + bh;
    out[slot * DD + e] = s;
    s = fmaf(expf(gsum[slot * D + i]), s, X[slot * DD + e]);
  }
  if (total) total[x] = s;
}

// Backward of group g = blockIdx.y of sequence bh = blockIdx.x from its entering state
// (init [G][BH][D][D], or zero) and the gradient arriving at its last state (dfin
// [G][BH][D][D], or zero); d_init from group 0.
template <int D, typename TIn>
__global__ void __launch_bounds__(kVecThreads) vec_bwd_kernel(Problem p, VecGroups gr, const TIn *q, const TIn *k,
                                                             const TIn *v, const TIn *dO, const float *lg,
                                                             const float *init, const float *dfin, TIn *dq,
                                                             TIn *dk, TIn *dv, float *dlg, float *dinit) {
  constexpr int kParts = kVecThreads / D, kSpan = D / kParts;
  extern __shared__ float sm[];
  float *S = sm, *vq = S + D * (D + 1), *vk = vq + D, *va = vk + D, *vv = va + D, *vg = vv + D;
  float *partA = vg + D, *partB = partA + kVecThreads;
  const int tid = threadIdx.x, bh = blockIdx.x, gi = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int64_t BH = (int64_t)p.B * p.H, slot = (int64_t)gi * BH + bh;
  const int64_t base = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float *g = lg + (int64_t)bh * p.T * D;
  float *dg = dlg + (int64_t)bh * p.T * D;
  const int t0 = gr.start(gi), t1 = gr.end(gi, p.T);
  const int c = tid % D, r0 = (tid / D) * kSpan;  // this thread's row / column and its range of the other index

  // forward sweep: S_t, dq_t = S_t dO_t, and q_t[i] dq_t[i] into d_log_gate
  for (int e = tid; e < D * D; e += kVecThreads)
    S[(e / D) * (D + 1) + e % D] = init ? init[slot * D * D + e] : 0.f;
  for (int t = t0; t < t1; ++t) {
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
  // the group's last state's term of the log-gate gradient (row tid), then R from dfin
  float gacc = 0.f;
  if (tid < D && dfin) {
    const float *Dr = dfin + slot * D * D + (int64_t)tid * D;
    for (int j = 0; j < D; ++j) gacc = fmaf(Dr[j], S[tid * (D + 1) + j], gacc);
  }
  __syncthreads();
  for (int e = tid; e < D * D; e += kVecThreads)
    S[(e / D) * (D + 1) + e % D] = dfin ? dfin[slot * D * D + e] : 0.f;

  // reverse sweep
  for (int t = t1 - 1; t >= t0; --t) {
    const int64_t row = base + (int64_t)t * p.st;
    if (tid < D) {
      vq[tid] = ld_val(q + row + tid);
      vk[tid] = ld_val(k + row + tid);
      vv[tid] = ld_val(v + row + tid);
      vg[tid] = ld_val(dO + row + tid);
      va[tid] = t == t1 - 1 ? 1.f : expf(g[(int64_t)(t + 1) * D + tid]);  // the carry alpha_{t+1}
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
  if (dinit && gi == 0) {
    __syncthreads();
    for (int e = tid; e < D * D; e += kVecThreads) {
      const int i = e / D;
      const float a0 = t1 > t0 ? expf(g[(int64_t)t0 * D + i]) : 1.f;
      dinit[(int64_t)bh * D * D + e] = a0 * S[i * (D + 1) + e % D];
    }
  }
}

template <int D, typename TIn>
cudaError_t launch_vec_fwd(const Problem &p, VecGroups gr, const void *q, const void *k, const void *v,
                           const float *lg, void *o, const float *init, float *fin, float *gsum, cudaStream_t s) {
  auto kern = vec_fwd_kernel<D, TIn>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vec_smem<D>());
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_GATED_VEC_FWD, s);
  kern<<<dim3(p.B * p.H, gr.G), kVecThreads, vec_smem<D>(), s>>>(p, gr, (const TIn *)q, (const TIn *)k,
                                                                 (const TIn *)v, lg, (TIn *)o, init, fin, gsum);
  return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_vec_ragg(const Problem &p, VecGroups gr, const void *q, const void *dO, const float *lg, float *W,
                            cudaStream_t s) {
  auto kern = vec_ragg_kernel<D, TIn>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vec_smem<D>());
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_GATED_VEC_BWD, s);
  kern<<<dim3(p.B * p.H, gr.G), kVecThreads, vec_smem<D>(), s>>>(p, gr, (const TIn *)q, (const TIn *)dO, lg, W);
  return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_vec_bwd(const Problem &p, VecGroups gr, const void *q, const void *k, const void *v,
                           const void *dO, const float *lg, const float *init, const float *dfin, void *dq, void *dk,
                           void *dv, float *dlg, float *dinit, cudaStream_t s) {
  auto kern = vec_bwd_kernel<D, TIn>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vec_smem<D>());
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_GATED_VEC_BWD, s);
  kern<<<dim3(p.B * p.H, gr.G), kVecThreads, vec_smem<D>(), s>>>(p, gr, (const TIn *)q, (const TIn *)k,
                                                                 (const TIn *)v, (const TIn *)dO, lg, init, dfin,
                                                                 (TIn *)dq, (TIn *)dk, (TIn *)dv, dlg, dinit);
  return cudaGetLastError();
}

cudaError_t launch_vec_scan(const Problem &p, VecGroups gr, const float *X, const float *gsum, const float *init,
                            float *out, float *total, bool reverse, cudaStream_t s) {
  const int64_t n = (int64_t)p.B * p.H * p.d * p.d;
  TimedLaunch t(reverse ? K_GATED_VEC_BWD : K_GATED_VEC_FWD, s);
  vec_scan_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(gr.G, (int64_t)p.B * p.H, p.d, X, gsum, init, out,
                                                              total, reverse ? 1 : 0);
  return cudaGetLastError();
}

// Groups: enough (group, sequence) CTAs for about two per SM, of at least 256 tokens.
VecGroups vec_groups(const Problem &p) {
  const int64_t BH = (int64_t)p.B * p.H, sms = p.num_sms > 0 ? p.num_sms : 1;
  int64_t G = (2 * sms + BH - 1) / BH;
  G = std::max<int64_t>(1, std::min<int64_t>(G, (p.T + 255) / 256));
  VecGroups gr;
  gr.L = (int)((p.T + G - 1) / G);
  gr.G = gr.L > 0 ? (int)((p.T + gr.L - 1) / gr.L) : 1;
  return gr;
}

struct VecLayout {
  size_t states = 0, agg = 0, gsum = 0, dfin = 0, total = 0;
};
VecLayout vec_layout(const Problem &p, bool bwd) {
  VecLayout w;
  const VecGroups gr = vec_groups(p);
  const size_t st = align256((size_t)gr.G * p.B * p.H * p.d * p.d * sizeof(float));
  w.states = 0;
  w.agg = st;
  w.gsum = 2 * st;
  w.dfin = w.gsum + align256((size_t)gr.G * p.B * p.H * p.d * sizeof(float));
  w.total = w.dfin + (bwd ? st : 0);
  return w;
}

template <int D, typename TIn>
cudaError_t vec_fwd_path(const Problem &p, const void *q, const void *k, const void *v, const float *lg, void *o,
                         const float *init, float *final_state, char *ws, cudaStream_t s) {
  const VecGroups gr = vec_groups(p);
  if (gr.G == 1) return launch_vec_fwd<D, TIn>(p, gr, q, k, v, lg, o, init, final_state, nullptr, s);
  const VecLayout w = vec_layout(p, false);
  float *states = reinterpret_cast<float *>(ws + w.states), *agg = reinterpret_cast<float *>(ws + w.agg);
  float *gsum = reinterpret_cast<float *>(ws + w.gsum);
  // the groups' own states from zero and their gate sums, the scan, the outputs
  cudaError_t e = launch_vec_fwd<D, TIn>(p, gr, q, k, v, lg, nullptr, nullptr, agg, gsum, s);
  if (e == cudaSuccess) e = launch_vec_scan(p, gr, agg, gsum, init, states, final_state, false, s);
  if (e == cudaSuccess) e = launch_vec_fwd<D, TIn>(p, gr, q, k, v, lg, o, states, nullptr, nullptr, s);
  return e;
}

template <int D, typename TIn>
cudaError_t vec_bwd_path(const Problem &p, const void *q, const void *k, const void *v, const void *dO,
                         const float *lg, const float *init, const float *d_final, void *dq, void *dk, void *dv,
                         float *dlg, float *dinit, char *ws, cudaStream_t s) {
  const VecGroups gr = vec_groups(p);
  if (gr.G == 1) return launch_vec_bwd<D, TIn>(p, gr, q, k, v, dO, lg, init, d_final, dq, dk, dv, dlg, dinit, s);
  const VecLayout w = vec_layout(p, true);
  float *states = reinterpret_cast<float *>(ws + w.states), *agg = reinterpret_cast<float *>(ws + w.agg);
  float *gsum = reinterpret_cast<float *>(ws + w.gsum), *dfin = reinterpret_cast<float *>(ws + w.dfin);
  // forward states entering every group; reverse aggregates and the gradients arriving
  // at every group's last state; then every group's backward
  cudaError_t e = launch_vec_fwd<D, TIn>(p, gr, q, k, v, lg, nullptr, nullptr, agg, gsum, s);
  if (e == cudaSuccess) e = launch_vec_scan(p, gr, agg, gsum, init, states, nullptr, false, s);
  if (e == cudaSuccess) e = launch_vec_ragg<D, TIn>(p, gr, q, dO, lg, agg, s);
  if (e == cudaSuccess) e = launch_vec_scan(p, gr, agg, gsum, d_final, dfin, nullptr, true, s);
  if (e == cudaSuccess) e = launch_vec_bwd<D, TIn>(p, gr, q, k, v, dO, lg, states, dfin, dq, dk, dv, dlg, dinit, s);
  return e;
}

}  // namespace

size_t gated_vec_ws_bytes(const Problem &p, bool bwd) {
  if (p.T == 0 || vec_groups(p).G == 1) return 0;
  return vec_layout(p, bwd).total;
}

cudaError_t gated_vec_fwd(const Problem &p, const void *q, const void *k, const void *v, const float *log_gate,
                          void *o, const float *init, float *final_state, void *ws, cudaStream_t s) {
  char *w = static_cast<char *>(ws);
  if (p.d == 64)
    return p.dtype == 1 ? vec_fwd_path<64, float>(p, q, k, v, log_gate, o, init, final_state, w, s)
                        : vec_fwd_path<64, __nv_bfloat16>(p, q, k, v, log_gate, o, init, final_state, w, s);
  return p.dtype == 1 ? vec_fwd_path<128, float>(p, q, k, v, log_gate, o, init, final_state, w, s)
                      : vec_fwd_path<128, __nv_bfloat16>(p, q, k, v, log_gate, o, init, final_state, w, s);
}

cudaError_t gated_vec_bwd(const Problem &p, const void *q, const void *k, const void *v, const void *dO,
                          const float *log_gate, const float *init, const float *d_final, void *dq, void *dk,
                          void *dv, float *d_log_gate, float *d_init, void *ws, cudaStream_t s) {
  char *w = static_cast<char *>(ws);
  if (p.d == 64)
    return p.dtype == 1 ? vec_bwd_path<64, float>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv, d_log_gate,
                                                  d_init, w, s)
                        : vec_bwd_path<64, __nv_bfloat16>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv,
                                                          d_log_gate, d_init, w, s);
  return p.dtype == 1 ? vec_bwd_path<128, float>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv, d_log_gate,
                                                 d_init, w, s)
                      : vec_bwd_path<128, __nv_bfloat16>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv,
                                                         d_log_gate, d_init, w, s);
}

}  // namespace linattn
