// CUDA-core kernels for per-dimension gates: one decay per token, head and key
// dimension (the vector form of the data-dependent gate; "Gated Linear
// Attention ..." on the LASP-2 page's related list),
//   S_t = diag(alpha_t) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t,   alpha_t = exp(log_gate_t).
// A CTA walks one chunk group of one (batch, head) sequence with the fp32 state in
// registers (each of its 256 threads holds a tile of it), staging the tokens'
// vectors in shared memory eight at a time.  Row i of the state only ever sees key
// dimension i's gates, so the groups are joined by scans whose multipliers are per row:
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

constexpr int kVecThreads = 256, kVecWarps = kVecThreads / 32;
constexpr int kVecChunk = 8;  // tokens staged in shared memory per step of a walk

__device__ __forceinline__ void st_val(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_val(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// Two fp32 lanes per instruction (the packed f32x2 forms of sm_100 and later); each
// lane rounds exactly as the scalar instruction does.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 dup2(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 ld2(const float *p) { return *reinterpret_cast<const float2 *>(p); }
__device__ __forceinline__ void st2(float *p, float2 x) { *reinterpret_cast<float2 *>(p) = x; }

// Two consecutive input elements, held raw between their global load and their
// staging (the pointers and strides are 16-byte aligned and the index is even).
template <typename T>
struct PairOf;
template <>
struct PairOf<float> {
  using type = float2;
};
template <>
struct PairOf<__nv_bfloat16> {
  using type = __nv_bfloat162;
};
__device__ __forceinline__ void ld_raw(float2 &r, const float *p) { r = *reinterpret_cast<const float2 *>(p); }
__device__ __forceinline__ void ld_raw(__nv_bfloat162 &r, const __nv_bfloat16 *p) {
  r = *reinterpret_cast<const __nv_bfloat162 *>(p);
}
__device__ __forceinline__ void zero_raw(float2 &r) { r = make_float2(0.f, 0.f); }
__device__ __forceinline__ void zero_raw(__nv_bfloat162 &r) { r = __floats2bfloat162_rn(0.f, 0.f); }
__device__ __forceinline__ float2 to_f2(float2 x) { return x; }
__device__ __forceinline__ float2 to_f2(__nv_bfloat162 x) { return __bfloat1622float2(x); }

// The sum of x[c] over the 32 lanes of a warp, scattered over the lanes: lane l returns
// the total of value l >> (5 - log2 N), the lanes with equal high bits holding the same
// total.  Each halving step sends half of the values still held to the partner lane.
template <int N>
__device__ __forceinline__ float lanes_reduce_scatter(float (&x)[N], int lane) {
  static_assert(N >= 2 && N <= 32 && (N & (N - 1)) == 0, "a power of two up to 32 values");
#pragma unroll
  for (int half = N / 2, off = 16; half >= 1; half /= 2, off /= 2) {
    const bool up = lane & off;
#pragma unroll
    for (int m = 0; m < half; ++m) {
      const float send = up ? x[m] : x[m + half], keep = up ? x[m + half] : x[m];
      x[m] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  constexpr int kLog = N == 2 ? 1 : N == 4 ? 2 : N == 8 ? 3 : N == 16 ? 4 : 5;
#pragma unroll
  for (int off = 16 >> kLog; off >= 1; off /= 2) x[0] += __shfl_xor_sync(0xffffffffu, x[0], off);
  return x[0];
}

// lanes_reduce_scatter for values held in a lane-dependent order of 4-value blocks:
// slot block b of lane l holds column block b ^ ((l >> (5 - log2 NB)) & (NB - 1)), NB = N / 4.
// In that order the half a lane keeps in each of the first log2 NB halving steps is
// always its first half (the partner, whose block mask differs in that step's bit,
// holds the same columns in its second half), so those steps need no selects; the
// last two steps split a block as lanes_reduce_scatter does.  Same result, same
// column per lane: l >> (5 - log2 N).
template <int N>
__device__ __forceinline__ float lanes_reduce_scatter_blocked(float (&x)[N], int lane) {
  static_assert(N == 8 || N == 16, "two or four blocks of four values");
  constexpr int kBlockSteps = N == 16 ? 2 : 1;
#pragma unroll
  for (int st = 0, half = N / 2, off = 16; st < kBlockSteps; ++st, half /= 2, off /= 2) {
#pragma unroll
    for (int m = 0; m < half; ++m) x[m] += __shfl_xor_sync(0xffffffffu, x[m + half], off);
  }
  constexpr int kOff = 16 >> kBlockSteps;  // then 4 values left, as in the plain form
#pragma unroll
  for (int half = 2, off = kOff; half >= 1; half /= 2, off /= 2) {
    const bool up = lane & off;
#pragma unroll
    for (int m = 0; m < half; ++m) {
      const float send = up ? x[m] : x[m + half], keep = up ? x[m + half] : x[m];
      x[m] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
#pragma unroll
  for (int off = kOff / 4; off >= 1; off /= 2) x[0] += __shfl_xor_sync(0xffffffffu, x[0], off);
  return x[0];
}

// shared memory of a walk: `vectors` staged vectors of kVecChunk x D, the per-warp
// partial sums [kVecChunk][kVecWarps][D] (when it reduces across warps) and kVecThreads pairs
template <int D>
constexpr size_t vec_smem(int vectors, bool partial) {
  return sizeof(float) * ((size_t)vectors * kVecChunk * D + (partial ? (size_t)kVecChunk * kVecWarps * D : 0) +
                          2 * kVecThreads);
}

// Chunk groups of L tokens (the last one shorter): CTA (bh, g) walks tokens [g L, min(T, (g+1) L)).
struct VecGroups {
  int G, L;
  __device__ int start(int g) const { return g * L; }
  __device__ int end(int g, int T) const { return min(T, (g + 1) * L); }
};

// The staged inputs of a walk.  Every kVecChunk tokens the CTA writes the pairs its
// threads fetched into shared memory as fp32 (the gates as alpha = exp(log_gate)),
// then fetches the next kVecChunk tokens' pairs into registers while it walks these.
// Thread tid holds pairs 2 (tid + kVecThreads m) of the chunk's kVecChunk x D
// elements, always the same two key dimensions 2 tid mod D.
template <int D, typename TIn, int NV>
struct VecStage {
  using Raw = typename PairOf<TIn>::type;
  static constexpr int kPairs = kVecChunk * D / (2 * kVecThreads);
  Raw x[NV][kPairs];
  float2 lg[kPairs];
  // the first NV of src; token tt of the chunk is time t = tb + dir * tt; its gate is
  // the log-gate at time t + gshift (0 at or past t1); tokens outside [t0, t1) are zero
  __device__ void fetch(const TIn *const *src, int64_t base, int64_t st, const float *g, int tb, int dir,
                        int gshift, int t0, int t1) {
#pragma unroll
    for (int m = 0; m < kPairs; ++m) {
      const int e = 2 * (threadIdx.x + kVecThreads * m), t = tb + dir * (e / D), i = e % D;
      if (t >= t0 && t < t1) {
        const int64_t row = base + (int64_t)t * st + i;
#pragma unroll
        for (int n = 0; n < NV; ++n) ld_raw(x[n][m], src[n] + row);
        const int tg = t + gshift;
        lg[m] = tg < t1 ? ld2(g + (int64_t)tg * D + i) : make_float2(0.f, 0.f);
      } else {
#pragma unroll
        for (int n = 0; n < NV; ++n) zero_raw(x[n][m]);
        lg[m] = make_float2(0.f, 0.f);
      }
    }
  }
  // the vectors to dst[n], alpha to alpha; returns this thread's sum of the log-gates
  __device__ float2 store(float *const *dst, float *alpha) const {
    float2 sum = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kPairs; ++m) {
      const int e = 2 * (threadIdx.x + kVecThreads * m);
#pragma unroll
      for (int n = 0; n < NV; ++n) st2(dst[n] + e, to_f2(x[n][m]));
      st2(alpha + e, make_float2(expf(lg[m].x), expf(lg[m].y)));
      sum.x += lg[m].x;
      sum.y += lg[m].y;
    }
    return sum;
  }
};

// Forward walk of group g = blockIdx.y of sequence bh = blockIdx.x from its entering
// state (init [G][BH][D][D], or zero), with the outputs o and the group's last state
// (fin [G][BH][D][D], or none).  The fp32 state lives in registers: warp w holds rows
// [w D/8, (w+1) D/8), lane l columns [l D/32, (l+1) D/32), as pairs of adjacent rows;
// o_t = S_t^T q_t sums each thread's rows and then the warps' partial sums.
template <int D, typename TIn>
__global__ void __launch_bounds__(kVecThreads, 2)
    vec_fwd_kernel(Problem p, VecGroups gr, const TIn *q, const TIn *k, const TIn *v, const float *lg, TIn *o,
                   const float *init, float *fin) {
  constexpr int RW = D / kVecWarps, CL = D / 32, ND = kVecChunk * D, NV = 3;
  extern __shared__ float sm[];
  float *sk = sm, *sv = sk + ND, *sq = sv + ND, *sa = sm + NV * ND, *part = sa + ND;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, bh = blockIdx.x, gi = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int64_t BH = (int64_t)p.B * p.H, slot = (int64_t)gi * BH + bh;
  const int64_t base = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float *g = lg + (int64_t)bh * p.T * D;
  const int t0 = gr.start(gi), t1 = gr.end(gi, p.T), r0 = w * RW, c0 = lane * CL;

  float2 s[RW / 2][CL];  // s[m][c] = (S[r0 + 2m][c0 + c], S[r0 + 2m + 1][c0 + c])
#pragma unroll
  for (int m = 0; m < RW / 2; ++m)
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      const float *src = init + slot * D * D + (int64_t)(r0 + 2 * m) * D + c0 + c;
      s[m][c] = init ? make_float2(src[0], src[D]) : make_float2(0.f, 0.f);
    }

  VecStage<D, TIn, NV> stage;
  const TIn *const srcs[3] = {k, v, q};
  float *const dsts[3] = {sk, sv, sq};
  stage.fetch(srcs, base, p.st, g, t0, 1, 0, t0, t1);
  for (int tc = t0; tc < t1; tc += kVecChunk) {
    const int nt = min(kVecChunk, t1 - tc);
    __syncthreads();  // the previous step is done with the staged vectors and the partial sums
    stage.store(dsts, sa);
    if (tc + kVecChunk < t1) stage.fetch(srcs, base, p.st, g, tc + kVecChunk, 1, 0, t0, t1);
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      const float *ra = sa + tt * D + r0, *rk = sk + tt * D + r0, *rq = sq + tt * D + r0;
      float2 vv[CL], acc[CL];
#pragma unroll
      for (int c = 0; c < CL; ++c) {
        vv[c] = dup2(sv[tt * D + c0 + c]);
        acc[c] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int m = 0; m < RW / 2; ++m) {
        const float2 a = ld2(ra + 2 * m), kk = ld2(rk + 2 * m);
#pragma unroll
        for (int c = 0; c < CL; ++c) s[m][c] = fma2(a, s[m][c], mul2(kk, vv[c]));
        const float2 qq = ld2(rq + 2 * m);
#pragma unroll
        for (int c = 0; c < CL; ++c) acc[c] = fma2(qq, s[m][c], acc[c]);
      }
#pragma unroll
      for (int c = 0; c < CL; ++c) part[(tt * kVecWarps + w) * D + c0 + c] = acc[c].x + acc[c].y;
    }
    __syncthreads();
    for (int e = tid; e < nt * D; e += kVecThreads) {
      const int tt = e / D, j = e % D;
      float x = 0.f;
#pragma unroll
      for (int u = 0; u < kVecWarps; ++u) x += part[(tt * kVecWarps + u) * D + j];
      st_val(o + base + (int64_t)(tc + tt) * p.st + j, x);
    }
  }
  if (fin) {
#pragma unroll
    for (int m = 0; m < RW / 2; ++m)
#pragma unroll
      for (int c = 0; c < CL; ++c) {
        float *dst = fin + slot * D * D + (int64_t)(r0 + 2 * m) * D + c0 + c;
        dst[0] = s[m][c].x;
        dst[D] = s[m][c].y;
      }
  }
}

// The state a group builds from zero, group g = blockIdx.y of sequence bh = blockIdx.x:
//   forward (REV = false): S <- diag(alpha_t) S + k_t v_t^T over the group's tokens in
//     order, i.e. U_g into out [G][BH][D][D], and the group's log-gate sums per key
//     dimension into gsum [G][BH][D] (or none);
//   reverse (REV = true): A <- diag(alpha_t) (A + q_t dO_t^T) from the group's last token
//     back, i.e. W_g = sum_{t in g} diag(alpha_start .. alpha_t) q_t dO_t^T into out.
// Both are S <- diag(a) S + x y^T (x = k, or alpha q), and two tokens u then w of the
// walk fold into one update, S <- diag(a_u a_w) S + (a_w x_u) y_u^T + x_w y_w^T: three
// packed operations per pair of state elements for two tokens instead of four.  Every
// step walks all kVecChunk staged tokens; those outside the group are staged as x = y
// = 0 and alpha = 1, which leave S exactly as it is.  The state lives in registers:
// warp w holds columns [w D/8, (w+1) D/8), lane l rows [l D/32, (l+1) D/32), as pairs
// of adjacent columns, so a row's products serve 16 (or 8) columns.
template <int D, typename TIn, bool REV>
__global__ void __launch_bounds__(kVecThreads, 2)
    vec_agg_kernel(Problem p, VecGroups gr, const TIn *x, const TIn *y, const float *lg, float *out, float *gsum) {
  static_assert(kVecChunk % 2 == 0, "tokens are folded in pairs");
  constexpr int CW = D / kVecWarps, RL = D / 32, ND = kVecChunk * D;
  extern __shared__ float sm[];
  float *sx = sm, *sy = sx + ND, *sa = sy + ND, *red = sa + ND;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, bh = blockIdx.x, gi = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int64_t BH = (int64_t)p.B * p.H, slot = (int64_t)gi * BH + bh;
  const int64_t base = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float *g = lg + (int64_t)bh * p.T * D;
  const int t0 = gr.start(gi), t1 = gr.end(gi, p.T), r0 = lane * RL, c0 = w * CW;

  float2 s[RL][CW / 2];  // s[r][n] = (S[r0 + r][c0 + 2n], S[r0 + r][c0 + 2n + 1])
#pragma unroll
  for (int r = 0; r < RL; ++r)
#pragma unroll
    for (int n = 0; n < CW / 2; ++n) s[r][n] = make_float2(0.f, 0.f);

  VecStage<D, TIn, 2> stage;
  const TIn *const srcs[2] = {x, y};
  float *const dsts[2] = {sx, sy};
  float2 gs = make_float2(0.f, 0.f);  // this thread's two key dimensions' log-gate sums
  // token tt of a step is time tb + tt (forward) or hi - 1 - tt (reverse)
  const int nsteps = (t1 - t0 + kVecChunk - 1) / kVecChunk;
  stage.fetch(srcs, base, p.st, g, REV ? t1 - 1 : t0, REV ? -1 : 1, 0, t0, t1);
  for (int k = 0; k < nsteps; ++k) {
    __syncthreads();  // the previous step is done with the staged vectors
    const float2 add = stage.store(dsts, sa);
    gs.x += add.x;
    gs.y += add.y;
    if (k + 1 < nsteps)
      stage.fetch(srcs, base, p.st, g, REV ? t1 - 1 - (k + 1) * kVecChunk : t0 + (k + 1) * kVecChunk, REV ? -1 : 1, 0,
                  t0, t1);
    __syncthreads();
#pragma unroll 1
    for (int tt = 0; tt < kVecChunk; tt += 2) {
      const float *au = sa + tt * D + r0, *aw = au + D, *xu = sx + tt * D + r0, *xw = xu + D;
      float2 A[RL], Xu[RL], Xw[RL];
#pragma unroll
      for (int r = 0; r < RL; ++r) {
        const float a1 = au[r], a2 = aw[r];
        const float x1 = REV ? a1 * xu[r] : xu[r], x2 = REV ? a2 * xw[r] : xw[r];
        A[r] = dup2(a1 * a2);
        Xu[r] = dup2(a2 * x1);
        Xw[r] = dup2(x2);
      }
#pragma unroll
      for (int n = 0; n < CW / 2; ++n) {
        const float2 yu = ld2(sy + tt * D + c0 + 2 * n), yw = ld2(sy + (tt + 1) * D + c0 + 2 * n);
#pragma unroll
        for (int r = 0; r < RL; ++r) s[r][n] = fma2(A[r], s[r][n], fma2(Xu[r], yu, mul2(Xw[r], yw)));
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RL; ++r)
#pragma unroll
    for (int n = 0; n < CW / 2; ++n) st2(out + slot * D * D + (int64_t)(r0 + r) * D + c0 + 2 * n, s[r][n]);
  if (gsum) {
    // threads tid = u D/2 + n (u < 2 kVecThreads / D) hold key dimensions 2n and 2n + 1
    reinterpret_cast<float2 *>(red)[tid] = gs;
    __syncthreads();
    if (tid < D / 2) {
      float2 z = make_float2(0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 2 * kVecThreads / D; ++u) {
        const float2 v = reinterpret_cast<const float2 *>(red)[tid + u * D / 2];
        z.x += v.x;
        z.y += v.y;
      }
      st2(gsum + slot * D + 2 * tid, z);
    }
  }
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
// [G][BH][D][D], or zero); d_init from group 0.  S and then R live in registers as in
// the reverse aggregate (warp: columns, lane: rows).  dq_t = S_t dO_t and dk_t = R_t v_t
// sum each thread's columns and then the warps' partial sums; dv_t = R_t^T k_t sums
// each thread's rows and then the warp's lanes.
template <int D, typename TIn>
__global__ void __launch_bounds__(kVecThreads, 2)
    vec_bwd_kernel(Problem p, VecGroups gr, const TIn *q, const TIn *k, const TIn *v, const TIn *dO,
                   const float *lg, const float *init, const float *dfin, TIn *dq, TIn *dk, TIn *dv, float *dlg,
                   float *dinit) {
  constexpr int CW = D / kVecWarps, RL = D / 32, ND = kVecChunk * D;
  extern __shared__ float sm[];
  float *sq = sm, *sk = sq + ND, *sv = sk + ND, *sg = sv + ND, *sa = sg + ND, *part = sa + ND;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, bh = blockIdx.x, gi = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int64_t BH = (int64_t)p.B * p.H, slot = (int64_t)gi * BH + bh;
  const int64_t base = (int64_t)b * p.sb + (int64_t)h * p.sh;
  const float *g = lg + (int64_t)bh * p.T * D;
  float *dg = dlg + (int64_t)bh * p.T * D;
  const int t0 = gr.start(gi), t1 = gr.end(gi, p.T), r0 = lane * RL, c0 = w * CW;
  // this lane's order of its columns: pair n of the slots is column pair pc(n), the
  // 4-column blocks permuted by the lane's bits the dv reduction splits first
  constexpr int NB = CW / 4, kLogNB = NB == 4 ? 2 : 1;
  const int mb = (lane >> (5 - kLogNB)) & (NB - 1);
  auto pc = [&](int n) { return 2 * ((n >> 1) ^ mb) + (n & 1); };

  float2 s[RL][CW / 2];  // s[r][n] = (S[r0 + r][c0 + 2 pc(n)], S[r0 + r][c0 + 2 pc(n) + 1])
#pragma unroll
  for (int r = 0; r < RL; ++r)
#pragma unroll
    for (int n = 0; n < CW / 2; ++n)
      s[r][n] = init ? ld2(init + slot * D * D + (int64_t)(r0 + r) * D + c0 + 2 * pc(n)) : make_float2(0.f, 0.f);

  VecStage<D, TIn, 4> stage;
  const TIn *const srcs[4] = {q, k, v, dO};
  float *const dsts[4] = {sq, sk, sv, sg};

  // forward sweep: S_t, dq_t = S_t dO_t, and q_t[i] dq_t[i] into d_log_gate
  stage.fetch(srcs, base, p.st, g, t0, 1, 0, t0, t1);
  for (int tc = t0; tc < t1; tc += kVecChunk) {
    const int nt = min(kVecChunk, t1 - tc);
    __syncthreads();
    stage.store(dsts, sa);
    if (tc + kVecChunk < t1) stage.fetch(srcs, base, p.st, g, tc + kVecChunk, 1, 0, t0, t1);
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      float2 ad[RL], kd[RL], acc[RL];
#pragma unroll
      for (int r = 0; r < RL; ++r) {
        ad[r] = dup2(sa[tt * D + r0 + r]);
        kd[r] = dup2(sk[tt * D + r0 + r]);
        acc[r] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int n = 0; n < CW / 2; ++n) {
        const float2 vp = ld2(sv + tt * D + c0 + 2 * pc(n)), dp = ld2(sg + tt * D + c0 + 2 * pc(n));
#pragma unroll
        for (int r = 0; r < RL; ++r) {
          s[r][n] = fma2(ad[r], s[r][n], mul2(kd[r], vp));
          acc[r] = fma2(s[r][n], dp, acc[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < RL; ++r) part[(tt * kVecWarps + w) * D + r0 + r] = acc[r].x + acc[r].y;
    }
    __syncthreads();
    for (int e = tid; e < nt * D; e += kVecThreads) {
      const int tt = e / D, i = e % D;
      float x = 0.f;
#pragma unroll
      for (int u = 0; u < kVecWarps; ++u) x += part[(tt * kVecWarps + u) * D + i];
      st_val(dq + base + (int64_t)(tc + tt) * p.st + i, x);
      dg[(int64_t)(tc + tt) * D + i] = sq[tt * D + i] * x;
    }
  }

  // the group's last state's term of the log-gate gradient (row i: sum_j Dfin[i][j]
  // S_end[i][j]), then R from Dfin
  {
    float2 acc[RL];
#pragma unroll
    for (int r = 0; r < RL; ++r) {
      acc[r] = make_float2(0.f, 0.f);
#pragma unroll
      for (int n = 0; n < CW / 2; ++n) {
        const float2 df =
            dfin ? ld2(dfin + slot * D * D + (int64_t)(r0 + r) * D + c0 + 2 * pc(n)) : make_float2(0.f, 0.f);
        acc[r] = fma2(df, s[r][n], acc[r]);
        s[r][n] = df;
      }
    }
    __syncthreads();  // the last step's sums are read
#pragma unroll
    for (int r = 0; r < RL; ++r) part[w * D + r0 + r] = acc[r].x + acc[r].y;
    __syncthreads();
  }
  float gacc = 0.f;  // key dimension tid's running log-gate gradient
  if (tid < D) {
#pragma unroll
    for (int u = 0; u < kVecWarps; ++u) gacc += part[u * D + tid];
  }

  // reverse sweep, R_t = diag(alpha_{t+1}) R_{t+1} + q_t dO_t^T; token tt of a step is time hi - 1 - tt
  constexpr int kLowBits = 5 - (CW == 8 ? 3 : 4);  // lanes sharing one column total of dv
  stage.fetch(srcs, base, p.st, g, t1 - 1, -1, 1, t0, t1);
  for (int hi = t1; hi > t0; hi -= kVecChunk) {
    const int nt = min(kVecChunk, hi - t0);
    __syncthreads();
    stage.store(dsts, sa);
    if (hi - kVecChunk > t0) stage.fetch(srcs, base, p.st, g, hi - kVecChunk - 1, -1, 1, t0, t1);
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      const int t = hi - 1 - tt;
      float2 ad[RL], qd[RL], kd[RL], dka[RL];
#pragma unroll
      for (int r = 0; r < RL; ++r) {
        ad[r] = dup2(sa[tt * D + r0 + r]);
        qd[r] = dup2(sq[tt * D + r0 + r]);
        kd[r] = dup2(sk[tt * D + r0 + r]);
        dka[r] = make_float2(0.f, 0.f);
      }
      float dva[CW];
#pragma unroll
      for (int n = 0; n < CW / 2; ++n) {
        const float2 vp = ld2(sv + tt * D + c0 + 2 * pc(n)), dp = ld2(sg + tt * D + c0 + 2 * pc(n));
        float2 col = make_float2(0.f, 0.f);
#pragma unroll
        for (int r = 0; r < RL; ++r) {
          s[r][n] = fma2(ad[r], s[r][n], mul2(qd[r], dp));
          dka[r] = fma2(s[r][n], vp, dka[r]);
          col = fma2(s[r][n], kd[r], col);
        }
        dva[2 * n] = col.x;
        dva[2 * n + 1] = col.y;
      }
#pragma unroll
      for (int r = 0; r < RL; ++r) part[(tt * kVecWarps + w) * D + r0 + r] = dka[r].x + dka[r].y;
      const float x = lanes_reduce_scatter_blocked<CW>(dva, lane);
      if ((lane & ((1 << kLowBits) - 1)) == 0)
        st_val(dv + base + (int64_t)t * p.st + c0 + (lane >> kLowBits), x);
    }
    __syncthreads();
    // dk, and each token's own log-gate term q_t[i] dq_t[i] - k_t[i] dk_t[i] (into the
    // staged gates' place, free until the next step) ...
    constexpr int kPer = kVecChunk * D / kVecThreads;
    float own[kPer];  // q_t[i] dq_t[i] from the forward sweep, all loads in flight at once
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int e = tid + m * kVecThreads, tt = e / D;
      own[m] = tt < nt ? dg[(int64_t)(hi - 1 - tt) * D + e % D] : 0.f;
    }
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int e = tid + m * kVecThreads, tt = e / D, i = e % D;
      if (tt < nt) {
        float x = 0.f;
#pragma unroll
        for (int u = 0; u < kVecWarps; ++u) x += part[(tt * kVecWarps + u) * D + i];
        st_val(dk + base + (int64_t)(hi - 1 - tt) * p.st + i, x);
        sa[tt * D + i] = own[m] - sk[tt * D + i] * x;
      }
    }
    __syncthreads();
    // ... then their running sums down the step's tokens
    if (tid < D) {
      for (int tt = 0; tt < nt; ++tt) {
        gacc += sa[tt * D + tid];
        dg[(int64_t)(hi - 1 - tt) * D + tid] = gacc;
      }
    }
  }
  if (dinit && gi == 0) {
#pragma unroll
    for (int r = 0; r < RL; ++r) {
      const float a0 = t1 > t0 ? expf(g[(int64_t)t0 * D + r0 + r]) : 1.f;
#pragma unroll
      for (int n = 0; n < CW / 2; ++n)
        st2(dinit + (int64_t)bh * D * D + (int64_t)(r0 + r) * D + c0 + 2 * pc(n), mul2(dup2(a0), s[r][n]));
    }
  }
}

template <int D, typename TIn>
cudaError_t launch_vec_fwd(const Problem &p, VecGroups gr, const void *q, const void *k, const void *v,
                           const float *lg, void *o, const float *init, float *fin, cudaStream_t s) {
  auto kern = vec_fwd_kernel<D, TIn>;
  const size_t smem = vec_smem<D>(4, true);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_GATED_VEC_FWD, s);
  kern<<<dim3(p.B * p.H, gr.G), kVecThreads, smem, s>>>(p, gr, (const TIn *)q, (const TIn *)k, (const TIn *)v, lg,
                                                        (TIn *)o, init, fin);
  return cudaGetLastError();
}

// The groups' own states from zero (forward: x = k, y = v, with the log-gate sums) or
// their reverse aggregates (x = q, y = dO).
template <int D, typename TIn, bool REV>
cudaError_t launch_vec_agg(const Problem &p, VecGroups gr, const void *x, const void *y, const float *lg, float *out,
                           float *gsum, cudaStream_t s) {
  auto kern = vec_agg_kernel<D, TIn, REV>;
  const size_t smem = vec_smem<D>(3, false);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  TimedLaunch t(REV ? K_GATED_VEC_BWD : K_GATED_VEC_FWD, s);
  kern<<<dim3(p.B * p.H, gr.G), kVecThreads, smem, s>>>(p, gr, (const TIn *)x, (const TIn *)y, lg, out, gsum);
  return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_vec_bwd(const Problem &p, VecGroups gr, const void *q, const void *k, const void *v,
                           const void *dO, const float *lg, const float *init, const float *dfin, void *dq, void *dk,
                           void *dv, float *dlg, float *dinit, cudaStream_t s) {
  auto kern = vec_bwd_kernel<D, TIn>;
  const size_t smem = vec_smem<D>(5, true);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_GATED_VEC_BWD, s);
  kern<<<dim3(p.B * p.H, gr.G), kVecThreads, smem, s>>>(p, gr, (const TIn *)q, (const TIn *)k, (const TIn *)v,
                                                        (const TIn *)dO, lg, init, dfin, (TIn *)dq, (TIn *)dk,
                                                        (TIn *)dv, dlg, dinit);
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

// Groups: the count that minimises waves x (group length + a fixed cost of about 128
// tokens per group: its state in and out, its share of the scans) x the walks a token
// takes, with two CTAs per SM and groups of at least 256 tokens; the fewest groups
// among equals.  One group per sequence walks each token 10 state-updates' worth
// (forward 3, backward 7 in FMA-pipe operations per state element); a split adds
// the forward's pass for the groups' own states and the backward's reverse
// aggregates (14 with the checkpoint).
VecGroups vec_groups(const Problem &p) {
  const int64_t BH = (int64_t)p.B * p.H, slots = 2 * (int64_t)(p.num_sms > 0 ? p.num_sms : 1);
  const int64_t gmax = std::max<int64_t>(1, std::min<int64_t>(p.T / 256, 8 * slots / BH + 1));
  int64_t best = 1, best_cost = -1;
  for (int64_t G = 1; G <= gmax; ++G) {
    const int64_t L = (p.T + G - 1) / G, waves = (G * BH + slots - 1) / slots;
    const int64_t cost = waves * (L + 128) * (G > 1 ? 14 : 10);
    if (best_cost < 0 || cost < best_cost) {
      best = G;
      best_cost = cost;
    }
  }
  VecGroups gr;
  gr.L = (int)((p.T + best - 1) / best);
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

// The checkpoint of a chunk-group split: every group's entering state [G][BH][D][D]
// and its log-gate sums [G][BH][D].
struct VecCkpt {
  size_t states = 0, gsum = 0, total = 0;
};
VecCkpt vec_ckpt_layout(const Problem &p) {
  VecCkpt c;
  const VecGroups gr = vec_groups(p);
  c.gsum = align256((size_t)gr.G * p.B * p.H * p.d * p.d * sizeof(float));
  c.total = c.gsum + align256((size_t)gr.G * p.B * p.H * p.d * sizeof(float));
  return c;
}

template <int D, typename TIn>
cudaError_t vec_fwd_path(const Problem &p, const void *q, const void *k, const void *v, const float *lg, void *o,
                         const float *init, float *final_state, char *ws, char *ckpt, cudaStream_t s) {
  const VecGroups gr = vec_groups(p);
  if (gr.G == 1) return launch_vec_fwd<D, TIn>(p, gr, q, k, v, lg, o, init, final_state, s);
  const VecLayout w = vec_layout(p, false);
  const VecCkpt c = vec_ckpt_layout(p);
  float *agg = reinterpret_cast<float *>(ws + w.agg);
  float *states = reinterpret_cast<float *>(ckpt ? ckpt + c.states : ws + w.states);
  float *gsum = reinterpret_cast<float *>(ckpt ? ckpt + c.gsum : ws + w.gsum);
  // the groups' own states from zero and their gate sums, the scan, the outputs
  cudaError_t e = launch_vec_agg<D, TIn, false>(p, gr, k, v, lg, agg, gsum, s);
  if (e == cudaSuccess) e = launch_vec_scan(p, gr, agg, gsum, init, states, final_state, false, s);
  if (e == cudaSuccess) e = launch_vec_fwd<D, TIn>(p, gr, q, k, v, lg, o, states, nullptr, s);
  return e;
}

template <int D, typename TIn>
cudaError_t vec_bwd_path(const Problem &p, const void *q, const void *k, const void *v, const void *dO,
                         const float *lg, const float *init, const float *d_final, void *dq, void *dk, void *dv,
                         float *dlg, float *dinit, char *ws, const char *ckpt, cudaStream_t s) {
  const VecGroups gr = vec_groups(p);
  if (gr.G == 1) return launch_vec_bwd<D, TIn>(p, gr, q, k, v, dO, lg, init, d_final, dq, dk, dv, dlg, dinit, s);
  const VecLayout w = vec_layout(p, true);
  const VecCkpt c = vec_ckpt_layout(p);
  float *agg = reinterpret_cast<float *>(ws + w.agg), *dfin = reinterpret_cast<float *>(ws + w.dfin);
  cudaError_t e = cudaSuccess;
  const float *states, *gsum;
  if (ckpt) {
    // the forward states entering every group, kept by the forward
    states = reinterpret_cast<const float *>(ckpt + c.states);
    gsum = reinterpret_cast<const float *>(ckpt + c.gsum);
  } else {
    float *st = reinterpret_cast<float *>(ws + w.states), *gs = reinterpret_cast<float *>(ws + w.gsum);
    e = launch_vec_agg<D, TIn, false>(p, gr, k, v, lg, agg, gs, s);
    if (e == cudaSuccess) e = launch_vec_scan(p, gr, agg, gs, init, st, nullptr, false, s);
    states = st;
    gsum = gs;
  }
  // reverse aggregates and the gradients arriving at every group's last state; then
  // every group's backward
  if (e == cudaSuccess) e = launch_vec_agg<D, TIn, true>(p, gr, q, dO, lg, agg, nullptr, s);
  if (e == cudaSuccess) e = launch_vec_scan(p, gr, agg, gsum, d_final, dfin, nullptr, true, s);
  if (e == cudaSuccess) e = launch_vec_bwd<D, TIn>(p, gr, q, k, v, dO, lg, states, dfin, dq, dk, dv, dlg, dinit, s);
  return e;
}

}  // namespace

size_t gated_vec_ws_bytes(const Problem &p, bool bwd) {
  if (p.T == 0 || vec_groups(p).G == 1) return 0;
  return vec_layout(p, bwd).total;
}

size_t gated_vec_ckpt_bytes(const Problem &p) {
  if (p.T == 0 || vec_groups(p).G == 1) return 0;
  return vec_ckpt_layout(p).total;
}

cudaError_t gated_vec_fwd(const Problem &p, const void *q, const void *k, const void *v, const float *log_gate,
                          void *o, const float *init, float *final_state, void *ws, void *ckpt, cudaStream_t s) {
  char *w = static_cast<char *>(ws), *c = static_cast<char *>(ckpt);
  if (p.d == 64)
    return p.dtype == 1 ? vec_fwd_path<64, float>(p, q, k, v, log_gate, o, init, final_state, w, c, s)
                        : vec_fwd_path<64, __nv_bfloat16>(p, q, k, v, log_gate, o, init, final_state, w, c, s);
  return p.dtype == 1 ? vec_fwd_path<128, float>(p, q, k, v, log_gate, o, init, final_state, w, c, s)
                      : vec_fwd_path<128, __nv_bfloat16>(p, q, k, v, log_gate, o, init, final_state, w, c, s);
}

cudaError_t gated_vec_bwd(const Problem &p, const void *q, const void *k, const void *v, const void *dO,
                          const float *log_gate, const float *init, const float *d_final, void *dq, void *dk,
                          void *dv, float *d_log_gate, float *d_init, void *ws, const void *ckpt, cudaStream_t s) {
  char *w = static_cast<char *>(ws);
  const char *c = static_cast<const char *>(ckpt);
  if (p.d == 64)
    return p.dtype == 1 ? vec_bwd_path<64, float>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv, d_log_gate,
                                                  d_init, w, c, s)
                        : vec_bwd_path<64, __nv_bfloat16>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv,
                                                          d_log_gate, d_init, w, c, s);
  return p.dtype == 1 ? vec_bwd_path<128, float>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv, d_log_gate,
                                                 d_init, w, c, s)
                      : vec_bwd_path<128, __nv_bfloat16>(p, q, k, v, dO, log_gate, init, d_final, dq, dk, dv,
                                                         d_log_gate, d_init, w, c, s);
}

}  // namespace linattn
