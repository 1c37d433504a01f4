// Data-dependent gates: a decay alpha_t = exp(g_t) per token per head
// (S_t = alpha_t S_{t-1} + k_t v_t^T), the gated variant the LASP-2 page names
// beside the plain one.  Every weight the chunked kernels need is a ratio of
// products of gates inside one chunk group, so they work from group-local
// cumulative sums of the gates in base 2,
//     C[t] = log2(e) * sum_{u = group start .. t} g_u,
// and a weight exp(sum_{u in (j, i]} g_u) is exp2(C[i] - C[j]).
//
// This file holds the small passes around the chunked kernels: the cumulative
// sums (and each group's total, the scan multiplier of the group), and the
// gradient of the gates, which follows from the other gradients:
//     dL/dG_t = q_t . dq_t - k_t . dk_t  (+ <D, S_final> at t = T-1),
//     dL/dg_u = sum_{t >= u} dL/dG_t      (G_t = sum_{u <= t} g_u),
// with dq, dk the gradients of the backward (dk includes the part that reaches
// the final state's gradient D).  The two dot products are taken by the dq
// and dk/dv passes from their fp32 results before these are rounded to the
// output dtype, and the sums run inside one chunk group, each anchored at the
// exact value at the next group's start (dgate_kernel).
#include <cuda_bf16.h>

#include "internal.h"

namespace linattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// One warp per (sequence, group): inclusive prefix sums in steps of 32 tokens,
// and the widest span (max - min) of the sums over any 128-token block of the
// group together with the sum before the block.
__global__ void __launch_bounds__(256) gate_prep_kernel(const float *lg, int T, GroupPlan gp, int BH, float *C,
                                                        float *tot, int *wflag) {
  const int G = gp.G;
  const int w = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32), lane = threadIdx.x & 31;
  if (w >= BH * G) return;  // warp-uniform
  const int bh = w / G, g = w % G;
  const int s0 = gp.start(g), s1 = min(T, gp.start(g + 1));
  const float *src = lg + (int64_t)bh * T;
  float *dst = C + (int64_t)bh * T;
  float carry = 0.f;
  float bmin = 0.f, bmax = 0.f, span = 0.f;  // the current block's range (from the sum before it)
  constexpr int kTiles = 8;                   // tiles of 32 tokens whose loads are in flight together
  for (int t0 = s0; t0 < s1; t0 += 32 * kTiles) {
    float xs[kTiles];
#pragma unroll
    for (int j = 0; j < kTiles; ++j) {
      const int tt = t0 + 32 * j + lane;
      xs[j] = tt < s1 ? src[tt] * kLog2e : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kTiles; ++j) {
      const int t = t0 + 32 * j, tt = t + lane;
      if (t >= s1) break;  // warp-uniform
      float x = xs[j];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
      }
      x += carry;
      if (tt < s1) dst[tt] = x;
      // lanes past the end hold the last sum, so all 32 lanes take part
      float mn = x, mx = x;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, d));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
      }
      bmin = fminf(bmin, mn);
      bmax = fmaxf(bmax, mx);
      carry = __shfl_sync(0xffffffffu, x, 31);
      if (((t - s0) & 127) == 96 || t + 32 >= s1) {  // a block ends (groups start on 128-token boundaries)
        span = fmaxf(span, bmax - bmin);
        bmin = bmax = carry;
      }
    }
  }
  if (lane == 0) {
    tot[(int64_t)g * BH + bh] = carry;
    if (wflag) wflag[(int64_t)g * BH + bh] = span <= kGateWeightedSpan ? 1 : 0;  // an infinite span fails
  }
}

// w[i] += exp2(tot[bh]) d[i] over n = BH * DD elements.
__global__ void fold_log2_kernel(float *w, const float *d, const float *tot, int DD, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    w[i] = fmaf(exp2f(tot[i / DD]), d[i], w[i]);
}

// One block of 256 threads per (sequence, group): the reverse inclusive sums of
// gx inside the group, walked from the end in tiles of 256 tokens, plus the
// exact value of the sum over everything after the group:
//     sum_{t > group end} dL/dG_t = dL/dg at the next group's first token
//       = alpha R at that token . S before it = <Rbar_g, S_{g+1}>,
// Rbar_g the reverse state at the group's end (what the dk/dv pass starts
// from) and S_{g+1} the forward state entering the next group (checkpoint);
// for the last group it is <D, S_final> (or 0).  Anchoring each group at an
// exact value keeps the sums short: a running sum over the whole sequence
// would accumulate the errors of every later token.
__global__ void __launch_bounds__(256) dgate_kernel(int T, GroupPlan gp, int BH, int DD, const float *gx,
                                                    const float *rbar, const float *states, const float *D,
                                                    const float *Sfin, float *dlg) {
  __shared__ float wsum[8];
  const int G = gp.G;
  const int bh = blockIdx.x / G, g = blockIdx.x % G;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  // the anchor: <Rbar_g, S_{g+1}> or <D, S_final>
  const float *a = nullptr, *b = nullptr;
  if (g + 1 < G) {
    a = rbar + ((int64_t)g * BH + bh) * DD;
    b = states + ((int64_t)(g + 1) * BH + bh) * DD;
  } else if (D) {
    a = D + (int64_t)bh * DD;
    b = Sfin + (int64_t)bh * DD;
  }
  float acc = 0.f;
  if (a)
    for (int i = threadIdx.x; i < DD; i += 256) acc = fmaf(a[i], b[i], acc);
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (lane == 0) wsum[warp] = acc;
  __syncthreads();
  float carry = 0.f;
  for (int w2 = 0; w2 < 8; ++w2) carry += wsum[w2];
  __syncthreads();
  const int s0 = gp.start(g), s1 = min(T, gp.start(g + 1));
  constexpr int kTiles = 4;  // tiles of 256 tokens whose loads are in flight together
  for (int tb = s1; tb > s0; tb -= 256 * kTiles) {
    float vs[kTiles];
#pragma unroll
    for (int j = 0; j < kTiles; ++j) {
      const int te = tb - 256 * j, ts = max(s0, te - 256);
      vs[j] = te > s0 && (int)threadIdx.x < te - ts ? gx[(int64_t)bh * T + ts + threadIdx.x] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kTiles; ++j) {
      const int te = tb - 256 * j, ts = max(s0, te - 256), n = te - ts;
      if (te <= s0) break;  // block-uniform
      float v = vs[j];
      // reverse inclusive scan: thread i owns token ts + i
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, v, d);
        if (lane + d < 32) v += y;
      }
      if (lane == 0) wsum[warp] = v;  // lane 0 holds its warp's total
      __syncthreads();
      float later = 0.f, tile = 0.f;  // sums of the later warps of the tile, of the whole tile
      for (int w2 = 0; w2 < 8; ++w2) {
        tile += wsum[w2];
        if (w2 > warp) later += wsum[w2];
      }
      if ((int)threadIdx.x < n) dlg[(int64_t)bh * T + ts + threadIdx.x] = v + later + carry;
      carry += tile;
      __syncthreads();  // wsum is rewritten by the next tile
    }
  }
}

}  // namespace

cudaError_t gate_prep(const Problem &p, const GroupPlan &gp, const float *log_gate, float *C, float *tot,
                      int *wflag, cudaStream_t s) {
  const int BH = p.B * p.H;
  const int64_t warps = (int64_t)BH * gp.G;
  TimedLaunch t(K_GATE, s);
  gate_prep_kernel<<<(int)((warps + 7) / 8), 256, 0, s>>>(log_gate, p.T, gp, BH, C, tot, wflag);
  return cudaGetLastError();
}

cudaError_t fold_state_log2(float *w, const float *d, const float *tot_last, int DD, int64_t n, cudaStream_t s) {
  const int64_t want = (n + 255) / 256;
  TimedLaunch t(K_SCAN, s);
  fold_log2_kernel<<<(int)(want < 1024 ? want : 1024), 256, 0, s>>>(w, d, tot_last, DD, n);
  return cudaGetLastError();
}

cudaError_t gate_grad(const Problem &p, const GroupPlan &gp, const float *gx, const float *rbar, const float *states,
                      const float *d_final, const float *final_state, float *dlg, cudaStream_t s) {
  const int BH = p.B * p.H;
  TimedLaunch t(K_GATE, s);
  dgate_kernel<<<BH * gp.G, 256, 0, s>>>(p.T, gp, BH, p.d * p.d, gx, rbar, states, d_final, final_state, dlg);
  return cudaGetLastError();
}

}  // namespace linattn
