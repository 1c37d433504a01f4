// CUDA-core (SIMT) kernels in fp32 arithmetic: the path for fp32 inputs, for
// head dimension 64, and for requests of per-chunk states.  One CTA walks one
// (batch, head) sequence chunk by chunk (chunk = 64 tokens), in the order the
// chunked method states it: masked attention inside the chunk, query times the
// running state across chunks, then the state update ("Lightning Attention-2"
// entry and abstract of the LASP-2 page).  All tiles live in shared memory
// with a padded row stride (d + 1) so that column walks are bank-conflict free.
#include <cuda_bf16.h>

#include "internal.h"

namespace linattn {
namespace {

constexpr int kC = 64;          // chunk length
constexpr int kThreads = 256;

__device__ __forceinline__ float ld_elem(const float *p) { return *p; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_elem(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_elem(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// pw[k] = lambda^k for k = 0..kC, by repeated multiplication in double.
__device__ void fill_powers(float *pw, float lam) {
  if (threadIdx.x == 0) {
    double x = 1.0;
    for (int i = 0; i <= kC; ++i) {
      pw[i] = (float)x;
      x *= (double)lam;
    }
  }
}

// gc[i] = sum of the log-gates of tokens c0 .. c0+i (natural log), for i < n;
// rows past the end repeat the last sum (finite weights for zero rows).
__device__ void gate_sums(float *gc, const float *lg, int c0, int n) {
  if (threadIdx.x == 0) {
    float acc = 0.f;
    for (int i = 0; i < kC; ++i) {
      if (i < n) acc += lg[c0 + i];
      gc[i] = acc;
    }
  }
}

// Load rows [c0, c0+n) of one head into a [kC][D+1] fp32 tile; rows >= n are zero.
template <int D, typename TIn>
__device__ void load_tile(float *tile, const TIn *base, int64_t st, int c0, int n) {
  for (int e = threadIdx.x; e < kC * D; e += kThreads) {
    const int r = e / D, c = e % D;
    tile[r * (D + 1) + c] = r < n ? ld_elem(base + (int64_t)(c0 + r) * st + c) : 0.f;
  }
}

// ------------------------------------------------------------------ forward
template <int D, typename TIn>
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(Problem p, const TIn *q, const TIn *k,
                                                            const TIn *v, TIn *o, const float *init,
                                                            float *final_state, float *chunk_states,
                                                            const float *log_gate) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1;
  float *S = sm;                 // [D][LD]
  float *Q = S + D * LD;         // [kC][LD]
  float *K = Q + kC * LD;
  float *V = K + kC * LD;
  float *P = V + kC * LD;        // [kC][kC]
  float *pw = P + kC * kC;       // [kC + 1]
  float *gc = pw + kC + 1;       // [kC] gates: the chunk's cumulative log-gate sums

  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
  const int64_t off = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float lam = p.decay ? p.decay[h] : 1.f;
  const float *lg = log_gate ? log_gate + (int64_t)bh * p.T : nullptr;
  fill_powers(pw, lam);
  for (int e = threadIdx.x; e < D * D; e += kThreads)
    S[(e / D) * LD + e % D] = init ? init[(int64_t)bh * D * D + e] : 0.f;
  __syncthreads();

  const int nchunk = (p.T + kC - 1) / kC;
  for (int c = 0; c < nchunk; ++c) {
    const int c0 = c * kC, n = min(kC, p.T - c0);
    if (chunk_states) {
      float *cs = chunk_states + ((int64_t)bh * nchunk + c) * D * D;
      for (int e = threadIdx.x; e < D * D; e += kThreads) cs[e] = S[(e / D) * LD + e % D];
    }
    load_tile<D>(Q, q + off, p.st, c0, n);
    load_tile<D>(K, k + off, p.st, c0, n);
    load_tile<D>(V, v + off, p.st, c0, n);
    if (lg) gate_sums(gc, lg, c0, n);
    __syncthreads();
    // weights: lambda powers, or products of the gates between two tokens
    auto w_diff = [&](int i, int j) { return lg ? expf(gc[i] - gc[j]) : pw[i - j]; };
    auto w_inter = [&](int i) { return lg ? expf(gc[i]) : pw[i + 1]; };
    auto w_key = [&](int j) { return lg ? expf(gc[n - 1] - gc[j]) : pw[n - 1 - j]; };
    const float w_blk = lg ? expf(gc[n - 1]) : pw[n];
    // intra-chunk scores with the causal decay mask
    for (int e = threadIdx.x; e < kC * kC; e += kThreads) {
      const int i = e / kC, j = e % kC;
      float s = 0.f;
      if (j <= i) {
        for (int a = 0; a < D; ++a) s = fmaf(Q[i * LD + a], K[j * LD + a], s);
        s *= w_diff(i, j);
      }
      P[e] = s;
    }
    __syncthreads();
    // outputs: lambda^{i+1} S^T q_i + sum_j P_ij v_j
    for (int e = threadIdx.x; e < kC * D; e += kThreads) {
      const int i = e / D, bb = e % D;
      if (i >= n) continue;
      float inter = 0.f, intra = 0.f;
      for (int a = 0; a < D; ++a) inter = fmaf(Q[i * LD + a], S[a * LD + bb], inter);
      for (int j = 0; j <= i; ++j) intra = fmaf(P[i * kC + j], V[j * LD + bb], intra);
      st_elem(o + off + (int64_t)(c0 + i) * p.st + bb, fmaf(w_inter(i), inter, intra));
    }
    __syncthreads();
    // state update: S <- lambda^n S + sum_j lambda^{n-1-j} k_j v_j^T
    for (int e = threadIdx.x; e < D * D; e += kThreads) {
      const int a = e / D, bb = e % D;
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = fmaf(w_key(j) * K[j * LD + a], V[j * LD + bb], acc);
      S[a * LD + bb] = fmaf(w_blk, S[a * LD + bb], acc);
    }
    __syncthreads();
  }
  if (final_state)
    for (int e = threadIdx.x; e < D * D; e += kThreads)
      final_state[(int64_t)bh * D * D + e] = S[(e / D) * LD + e % D];
}

// ------------------------------------------------------------------ backward
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

// With gates (log_gate != NULL) every lambda power becomes the product of the
// gates between the two tokens, and the gradient of the log-gates is formed as
//     d_log_gate[t] = sum_{u >= t} (q_u . dq_u - k_u . dk_u) + <D, S_final>:
// the forward sweep stores q_t . dq_t in d_log_gate, and the reverse sweep, which
// meets the tokens from the end, subtracts k_t . dk_t and accumulates (in double).
// Both dot products are taken from the fp32 gradients before they are rounded.
template <int D, typename TIn>
__global__ void __launch_bounds__(kThreads) simt_bwd_kernel(Problem p, const TIn *q, const TIn *k,
                                                            const TIn *v, const TIn *dO,
                                                            const float *init, const float *dfin,
                                                            TIn *dq, TIn *dk, TIn *dv, float *dinit,
                                                            const float *log_gate, float *dlg) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1;
  constexpr int NW = D / 32;     // warps per row of a [kC][D] result
  float *S = sm;                 // forward state, then the reverse state
  float *Q = S + D * LD;
  float *K = Q + kC * LD;
  float *V = K + kC * LD;
  float *G = V + kC * LD;        // dO tile
  float *P = G + kC * LD;        // [kC][kC]
  float *dP = P + kC * kC;       // [kC][kC]
  float *pw = dP + kC * kC;      // [kC + 1]; with gates the cumulative log-gate sums instead
  float *gc = pw;
  float *part = pw + kC + 1;     // gates: [kC][NW] per-warp parts of the row dot products

  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
  const int64_t off = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float lam = p.decay ? p.decay[h] : 1.f;
  const float *lg = log_gate ? log_gate + (int64_t)bh * p.T : nullptr;
  float *dl = lg ? dlg + (int64_t)bh * p.T : nullptr;
  const int lane = threadIdx.x & 31;
  if (!lg) fill_powers(pw, lam);
  for (int e = threadIdx.x; e < D * D; e += kThreads)
    S[(e / D) * LD + e % D] = init ? init[(int64_t)bh * D * D + e] : 0.f;
  __syncthreads();
  const int nchunk = (p.T + kC - 1) / kC;

  // forward sweep: dq_i = sum_{j<=i} lambda^{i-j} (dO_i.v_j) k_j + lambda^{i+1} S_prev dO_i
  for (int c = 0; c < nchunk; ++c) {
    const int c0 = c * kC, n = min(kC, p.T - c0);
    load_tile<D>(K, k + off, p.st, c0, n);
    load_tile<D>(V, v + off, p.st, c0, n);
    load_tile<D>(G, dO + off, p.st, c0, n);
    if (lg) {
      load_tile<D>(Q, q + off, p.st, c0, n);
      gate_sums(gc, lg, c0, n);
    }
    __syncthreads();
    auto w_diff = [&](int i, int j) { return lg ? expf(gc[i] - gc[j]) : pw[i - j]; };
    auto w_inter = [&](int i) { return lg ? expf(gc[i]) : pw[i + 1]; };
    auto w_key = [&](int j) { return lg ? expf(gc[n - 1] - gc[j]) : pw[n - 1 - j]; };
    const float w_blk = lg ? expf(gc[n - 1]) : pw[n];
    for (int e = threadIdx.x; e < kC * kC; e += kThreads) {
      const int i = e / kC, j = e % kC;
      float s = 0.f;
      if (j <= i) {
        for (int a = 0; a < D; ++a) s = fmaf(G[i * LD + a], V[j * LD + a], s);
        s *= w_diff(i, j);
      }
      dP[e] = s;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kC * D; e += kThreads) {
      const int i = e / D, a = e % D;
      if (i >= n) continue;  // uniform across the warp: a warp covers 32 columns of one row
      float inter = 0.f, intra = 0.f;
      for (int bb = 0; bb < D; ++bb) inter = fmaf(S[a * LD + bb], G[i * LD + bb], inter);
      for (int j = 0; j <= i; ++j) intra = fmaf(dP[i * kC + j], K[j * LD + a], intra);
      const float x = fmaf(w_inter(i), inter, intra);
      st_elem(dq + off + (int64_t)(c0 + i) * p.st + a, x);
      if (lg) {
        const float r = warp_sum(Q[i * LD + a] * x);
        if (lane == 0) part[i * NW + a / 32] = r;
      }
    }
    __syncthreads();
    if (lg && (int)threadIdx.x < n) {
      float r = 0.f;
      for (int w = 0; w < NW; ++w) r += part[threadIdx.x * NW + w];
      dl[c0 + threadIdx.x] = r;  // q . dq, completed by the reverse sweep
    }
    for (int e = threadIdx.x; e < D * D; e += kThreads) {
      const int a = e / D, bb = e % D;
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = fmaf(w_key(j) * K[j * LD + a], V[j * LD + bb], acc);
      S[a * LD + bb] = fmaf(w_blk, S[a * LD + bb], acc);
    }
    __syncthreads();
  }

  // the gate gradient starts from <D, S_final> (S holds S_final here)
  double carry = 0.0;
  if (lg && dfin) {
    float r = 0.f;
    for (int e = threadIdx.x; e < D * D; e += kThreads)
      r = fmaf(dfin[(int64_t)bh * D * D + e], S[(e / D) * LD + e % D], r);
    r = warp_sum(r);
    if (lane == 0) part[threadIdx.x / 32] = r;
    __syncthreads();
    if (threadIdx.x == 0)
      for (int w = 0; w < kThreads / 32; ++w) carry += part[w];
  }

  // reverse sweep with Rbar = sum_{u > chunk end} lambda^{u-end} q_u dO_u^T
  // (+ lambda^{T-1-end} d_final: the gradient arriving at the final state)
  for (int e = threadIdx.x; e < D * D; e += kThreads)
    S[(e / D) * LD + e % D] = dfin ? dfin[(int64_t)bh * D * D + e] : 0.f;
  __syncthreads();
  for (int c = nchunk - 1; c >= 0; --c) {
    const int c0 = c * kC, n = min(kC, p.T - c0);
    load_tile<D>(Q, q + off, p.st, c0, n);
    load_tile<D>(K, k + off, p.st, c0, n);
    load_tile<D>(V, v + off, p.st, c0, n);
    load_tile<D>(G, dO + off, p.st, c0, n);
    if (lg) gate_sums(gc, lg, c0, n);
    __syncthreads();
    auto w_diff = [&](int i, int j) { return lg ? expf(gc[i] - gc[j]) : pw[i - j]; };
    auto w_inter = [&](int i) { return lg ? expf(gc[i]) : pw[i + 1]; };
    auto w_key = [&](int j) { return lg ? expf(gc[n - 1] - gc[j]) : pw[n - 1 - j]; };
    const float w_blk = lg ? expf(gc[n - 1]) : pw[n];
    for (int e = threadIdx.x; e < kC * kC; e += kThreads) {
      const int i = e / kC, j = e % kC;
      float s = 0.f, g = 0.f;
      if (j <= i) {
        for (int a = 0; a < D; ++a) {
          s = fmaf(Q[i * LD + a], K[j * LD + a], s);
          g = fmaf(G[i * LD + a], V[j * LD + a], g);
        }
        const float w = w_diff(i, j);
        s *= w;
        g *= w;
      }
      P[e] = s;
      dP[e] = g;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kC * D; e += kThreads) {
      const int j = e / D, a = e % D;
      if (j >= n) continue;  // warp-uniform, as above
      // dk_j[a] = sum_i dP_ij q_i[a] + lambda^{n-1-j} (Rbar v_j)[a]
      float intra = 0.f, inter = 0.f;
      for (int i = j; i < n; ++i) intra = fmaf(dP[i * kC + j], Q[i * LD + a], intra);
      for (int bb = 0; bb < D; ++bb) inter = fmaf(S[a * LD + bb], V[j * LD + bb], inter);
      const float wk = w_key(j);
      const float x = fmaf(wk, inter, intra);
      st_elem(dk + off + (int64_t)(c0 + j) * p.st + a, x);
      if (lg) {
        const float r = warp_sum(K[j * LD + a] * x);
        if (lane == 0) part[j * NW + a / 32] = r;
      }
      // dv_j[a] = sum_i P_ij dO_i[a] + lambda^{n-1-j} (Rbar^T k_j)[a]
      float intra2 = 0.f, inter2 = 0.f;
      for (int i = j; i < n; ++i) intra2 = fmaf(P[i * kC + j], G[i * LD + a], intra2);
      for (int aa = 0; aa < D; ++aa) inter2 = fmaf(S[aa * LD + a], K[j * LD + aa], inter2);
      st_elem(dv + off + (int64_t)(c0 + j) * p.st + a, fmaf(wk, inter2, intra2));
    }
    __syncthreads();
    if (lg && threadIdx.x == 0)
      for (int i = n - 1; i >= 0; --i) {
        float kdk = 0.f;
        for (int w = 0; w < NW; ++w) kdk += part[i * NW + w];
        carry += (double)dl[c0 + i] - (double)kdk;
        dl[c0 + i] = (float)carry;
      }
    for (int e = threadIdx.x; e < D * D; e += kThreads) {
      const int a = e / D, bb = e % D;
      float acc = 0.f;
      for (int i = 0; i < n; ++i) acc = fmaf(w_inter(i) * Q[i * LD + a], G[i * LD + bb], acc);
      S[a * LD + bb] = fmaf(w_blk, S[a * LD + bb], acc);
    }
    __syncthreads();
  }
  if (dinit)
    for (int e = threadIdx.x; e < D * D; e += kThreads)
      dinit[(int64_t)bh * D * D + e] = S[(e / D) * LD + e % D];
}

// ------------------------------------------------------------------ segment-local states
template <int D, typename TIn>
__global__ void __launch_bounds__(kThreads) simt_segment_kernel(Problem p, int seg_len, const TIn *k,
                                                                const TIn *v, bool reverse, float *out) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1;
  constexpr int PER = D * D / kThreads;
  float *K = sm;
  float *V = K + kC * LD;
  float *pw = V + kC * LD;
  const int g = blockIdx.y, bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
  const int64_t off = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float lam = p.decay ? p.decay[h] : 1.f;
  fill_powers(pw, lam);
  float acc[PER];
#pragma unroll
  for (int m = 0; m < PER; ++m) acc[m] = 0.f;
  // forward weights lambda^{end - s}: chunks in order, acc <- lambda^n acc + sum_j lambda^{n-1-j} k_j v_j^T;
  // reverse weights lambda^{s - start + 1}: chunks from the end, acc <- lambda^n acc + sum_j lambda^{j+1} ...
  const int s0 = g * seg_len, s1 = min(p.T, s0 + seg_len);
  const int nck = (s1 - s0 + kC - 1) / kC;
  for (int ci = 0; ci < nck; ++ci) {
    const int c0 = s0 + kC * (reverse ? nck - 1 - ci : ci);
    const int n = min(kC, s1 - c0);
    __syncthreads();
    load_tile<D>(K, k + off, p.st, c0, n);
    load_tile<D>(V, v + off, p.st, c0, n);
    __syncthreads();
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = threadIdx.x + m * kThreads, a = e / D, bb = e % D;
      float x = 0.f;
      for (int j = 0; j < n; ++j) x = fmaf(pw[reverse ? j + 1 : n - 1 - j] * K[j * LD + a], V[j * LD + bb], x);
      acc[m] = fmaf(pw[n], acc[m], x);
    }
  }
  float *U = out + ((int64_t)g * p.B * p.H + bh) * D * D;
#pragma unroll
  for (int m = 0; m < PER; ++m) U[threadIdx.x + m * kThreads] = acc[m];
}

template <int D>
size_t fwd_smem() { return sizeof(float) * (D * (D + 1) + 3 * kC * (D + 1) + kC * kC + 2 * kC + 1); }
template <int D>
size_t bwd_smem() { return sizeof(float) * (D * (D + 1) + 4 * kC * (D + 1) + 2 * kC * kC + kC + 1 + kC * (D / 32)); }
template <int D>
size_t seg_smem() { return sizeof(float) * (2 * kC * (D + 1) + kC + 1); }

template <int D, typename TIn>
cudaError_t launch_fwd(const Problem &p, const void *q, const void *k, const void *v, void *o,
                       const float *init, float *fin, float *cs, const float *lg, cudaStream_t s) {
  auto kern = simt_fwd_kernel<D, TIn>;
  const size_t sm = fwd_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_SIMT_FWD, s);
  kern<<<p.B * p.H, kThreads, sm, s>>>(p, (const TIn *)q, (const TIn *)k, (const TIn *)v, (TIn *)o,
                                        init, fin, cs, lg);
  return cudaGetLastError();
}
template <int D, typename TIn>
cudaError_t launch_bwd(const Problem &p, const void *q, const void *k, const void *v, const void *dO,
                       const float *init, const float *dfin, void *dq, void *dk, void *dv, float *dinit,
                       const float *lg, float *dlg, cudaStream_t s) {
  auto kern = simt_bwd_kernel<D, TIn>;
  const size_t sm = bwd_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_SIMT_BWD, s);
  kern<<<p.B * p.H, kThreads, sm, s>>>(p, (const TIn *)q, (const TIn *)k, (const TIn *)v,
                                        (const TIn *)dO, init, dfin, (TIn *)dq, (TIn *)dk, (TIn *)dv, dinit,
                                        lg, dlg);
  return cudaGetLastError();
}
template <int D, typename TIn>
cudaError_t launch_seg(const Problem &p, int seg_len, const void *k, const void *v, bool reverse, float *out,
                       cudaStream_t s) {
  auto kern = simt_segment_kernel<D, TIn>;
  const size_t sm = seg_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int G = (p.T + seg_len - 1) / seg_len;
  TimedLaunch t(K_SIMT_SEGMENT, s);
  kern<<<dim3(p.B * p.H, G), kThreads, sm, s>>>(p, seg_len, (const TIn *)k, (const TIn *)v, reverse, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t simt_fwd(const Problem &p, const void *q, const void *k, const void *v, void *o,
                     const float *init, float *final_state, float *chunk_states, cudaStream_t s,
                     const float *log_gate) {
  if (p.d == 64)
    return p.dtype == 1 ? launch_fwd<64, float>(p, q, k, v, o, init, final_state, chunk_states, log_gate, s)
                        : launch_fwd<64, __nv_bfloat16>(p, q, k, v, o, init, final_state, chunk_states, log_gate, s);
  return p.dtype == 1 ? launch_fwd<128, float>(p, q, k, v, o, init, final_state, chunk_states, log_gate, s)
                      : launch_fwd<128, __nv_bfloat16>(p, q, k, v, o, init, final_state, chunk_states, log_gate, s);
}

cudaError_t simt_bwd(const Problem &p, const void *q, const void *k, const void *v, const void *dO,
                     const float *init, const float *d_final, void *dq, void *dk, void *dv, float *dinit,
                     cudaStream_t s, const float *log_gate, float *d_log_gate) {
  const float *g = log_gate;
  float *dg = d_log_gate;
  if (p.d == 64)
    return p.dtype == 1 ? launch_bwd<64, float>(p, q, k, v, dO, init, d_final, dq, dk, dv, dinit, g, dg, s)
                        : launch_bwd<64, __nv_bfloat16>(p, q, k, v, dO, init, d_final, dq, dk, dv, dinit, g, dg, s);
  return p.dtype == 1 ? launch_bwd<128, float>(p, q, k, v, dO, init, d_final, dq, dk, dv, dinit, g, dg, s)
                      : launch_bwd<128, __nv_bfloat16>(p, q, k, v, dO, init, d_final, dq, dk, dv, dinit, g, dg, s);
}

cudaError_t simt_segment_states(const Problem &p, int seg_len, const void *x, const void *y, bool reverse,
                                float *out, cudaStream_t s) {
  if (p.d == 64)
    return p.dtype == 1 ? launch_seg<64, float>(p, seg_len, x, y, reverse, out, s)
                        : launch_seg<64, __nv_bfloat16>(p, seg_len, x, y, reverse, out, s);
  return p.dtype == 1 ? launch_seg<128, float>(p, seg_len, x, y, reverse, out, s)
                      : launch_seg<128, __nv_bfloat16>(p, seg_len, x, y, reverse, out, s);
}

}  // namespace linattn
