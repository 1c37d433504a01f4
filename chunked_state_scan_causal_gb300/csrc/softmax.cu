// Causal softmax attention of a query segment over its gathered key/value
// prefix, on the tensor cores (tcgen05 + TMEM + TMA), bf16 with d = 128.
//
// The hybrid variant on the LASP-2 page ("LASP-2: Rethinking Sequence
// Parallelism for Linear Attention and Its Hybrid", abstract: LASP-2H carries
// the one-gather exchange over to the softmax attention layers of hybrid
// models) gives each sequence-parallel rank, by one gather, the keys and values of every
// position up to the end of its own segment; the rank's queries then attend
// causally over that prefix.  Here the queries are the last Tq positions of
// a prefix of Tk tokens (offset = Tk - Tq):
//
//   o_i   = sum_{j <= offset + i} softmax_j(scale q_i . k_j) v_j,
//   lse_i = log sum_{j <= offset + i} exp(scale q_i . k_j)      (optional output)
//
// computed blockwise with a running maximum and sum per query row (the
// softmax of the whole row is never formed): per 128-query tile, for every
// 128-key tile up to the diagonal,
//   S = Q K^T (TMEM, fp32)  ->  p = exp2(scale log2(e) S - m)  (bf16, back into TMEM)
//   O += P V                (TMEM accumulator, P read from TMEM as the A operand)
// The reference maximum m of a row moves only when a tile raises the row's
// maximum by more than 8 (in log2 units): p then stays below 2^8, and O and
// the row sum are rescaled only on those rare tiles.
//
// Persistent CTAs draw (query tile, sequence) items at run time, longest
// (most key tiles) first.  Warp roles:
//   warp 0      TMA producer (one thread): the item's Q tile, then K and V tiles
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 4..7  softmax (one thread per query row)
//   warps 8..11 output: O / rowsum to bf16, log-sum-exp
// Two score buffers let the product of the next key tile run while the
// softmax of the current one is formed; two output regions let an item's
// output be written while the next item accumulates.  Every wait is bounded.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace linattn {
namespace {

constexpr int kSmThreads = 384;
constexpr int kKvStages = 3;                               // stages of (K tile, V tile)
constexpr uint32_t kSmOffKv = kTileBytes;                  // after the Q tile
constexpr uint32_t kSmOffBar = kSmOffKv + kKvStages * 2 * kTileBytes;
constexpr uint32_t kSmOffStats = kSmOffBar + 256;          // [128] row maxima, [128] row sums
constexpr size_t kSmSmem = kSmOffStats + 1024 + 1024;      // (+ 1024: alignment of the tiles)
static_assert(kSmSmem + 128 <= 232448, "tiles, barriers, row statistics and static shared memory fit 227 KB");

enum { S_QFULL = 0, S_QEMPTY, S_KFULL, S_KEMPTY = S_KFULL + kKvStages, S_SFULL = S_KEMPTY + kKvStages,
       S_PREADY = S_SFULL + 2, S_PVC = S_PREADY + 2, S_OFULL, S_OEMPTY = S_OFULL + 2, S_LFULL = S_OEMPTY + 2,
       S_LEMPTY, S_COUNT };
static_assert(S_COUNT * 8 + 4 <= 256, "softmax kernel barriers and the TMEM slot fit their 256 bytes");

constexpr int kRingS = 4;

struct SoftmaxParams {
  int B, H, Tq, Tk, off, nqt, nitems;
  float scale_log2;            // softmax scale times log2(e)
  __nv_bfloat16 *o;            // [B,H,Tq,d]
  int64_t osb, osh, ost;       // element strides of o
  float *lse;                  // [B,H,Tq] fp32, or null
  int wide;                    // every row of o starts on a 32-byte boundary
  int *status;
  int *counter;                // [2] item counter and finished CTAs (zero at launch)
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// 2^x with the PTX ex2.approx instruction (flush-to-zero; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// item -> (query tile, sequence): the query tiles with the most key tiles first
__device__ __forceinline__ void sm_item(const SoftmaxParams &P, int item, int &qt, int &bh, int &nt) {
  const int BH = P.B * P.H;
  qt = P.nqt - 1 - item / BH;
  bh = item % BH;
  const int kend = min(P.Tk, P.off + 128 * qt + 128);  // keys up to the tile's last query
  nt = (kend + 127) / 128;
}

// 32 fp32 values -> 64 contiguous bytes of bf16 in global memory, streaming stores
// (two 32-byte stores when dst is 32-byte aligned, else four 16-byte ones).
__device__ __forceinline__ void st_row_chunk(__nv_bfloat16 *dst, const float (&x)[32], bool wide) {
  if (wide) {
#pragma unroll
    for (int q = 0; q < 2; ++q)
      asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 16 * q),
                   "r"(pack_bf16(x[16 * q + 0], x[16 * q + 1])), "r"(pack_bf16(x[16 * q + 2], x[16 * q + 3])),
                   "r"(pack_bf16(x[16 * q + 4], x[16 * q + 5])), "r"(pack_bf16(x[16 * q + 6], x[16 * q + 7])),
                   "r"(pack_bf16(x[16 * q + 8], x[16 * q + 9])), "r"(pack_bf16(x[16 * q + 10], x[16 * q + 11])),
                   "r"(pack_bf16(x[16 * q + 12], x[16 * q + 13])), "r"(pack_bf16(x[16 * q + 14], x[16 * q + 15]))
                   : "memory");
    return;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 8 * q),
                 "r"(pack_bf16(x[8 * q + 0], x[8 * q + 1])), "r"(pack_bf16(x[8 * q + 2], x[8 * q + 3])),
                 "r"(pack_bf16(x[8 * q + 4], x[8 * q + 5])), "r"(pack_bf16(x[8 * q + 6], x[8 * q + 7]))
                 : "memory");
}

__global__ void __launch_bounds__(kSmThreads, 1)
    softmax_segment_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                           const __grid_constant__ CUtensorMap mv, SoftmaxParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kSmOffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + S_COUNT);
  float *stat_m = reinterpret_cast<float *>(smem + kSmOffStats);  // [128]
  float *stat_l = stat_m + 128;                                  // [128]
  __shared__ int abort_flag;
  __shared__ int ring_item[kRingS];
  __shared__ uint64_t ring_bar[2 * kRingS];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int BH = P.B * P.H;
  int *const detail = P.status ? P.status + 1 + warp : nullptr;
  uint64_t *ring_full = ring_bar, *ring_empty = ring_bar + kRingS;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar[S_QFULL], 1);
    mbar_init(&bar[S_QEMPTY], 1);
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(&bar[S_KFULL + s], 1);
      mbar_init(&bar[S_KEMPTY + s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[S_SFULL + i], 1);
      mbar_init(&bar[S_PREADY + i], 128);
      mbar_init(&bar[S_OFULL + i], 1);
      mbar_init(&bar[S_OEMPTY + i], 128);
    }
    mbar_init(&bar[S_LFULL], 128);
    mbar_init(&bar[S_LEMPTY], 128);
    mbar_init(&bar[S_PVC], 1);
    for (int i = 0; i < kRingS; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1 + 128 + 128);  // readers: MMA thread, softmax and output groups
    }
    fence_mbar_init();
    prefetch_tensormap(&mq);
    prefetch_tensormap(&mk);
    prefetch_tensormap(&mv);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  auto tS = [&](int u) { return tmem + (uint32_t)(u & 1) * 128u; };          // score buffer of tile u
  auto tOut = [&](int it) { return tmem + 256u + (uint32_t)(it & 1) * 128u; };  // output region of item it
  const uint32_t sQ = smem_u32(smem);
  auto kv_addr = [&](int kt) { return smem_u32(smem + kSmOffKv) + (uint32_t)(kt % kKvStages) * 2u * kTileBytes; };
  auto wait = [&](int idx, int parity) { return mbar_wait(&bar[idx], parity & 1, &abort_flag, P.status, detail); };
  // the shared item ring: the producer draws, every other role reads in the same order
  auto take = [&](int k, int &item) {
    const int s = k % kRingS;
    if (!mbar_wait(&ring_full[s], (k / kRingS) & 1, &abort_flag, P.status, detail)) return false;
    item = *reinterpret_cast<volatile int *>(&ring_item[s]);
    mbar_arrive(&ring_empty[s]);
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int kt = 0, nq = 0;  // K/V tiles and Q tiles loaded
      bool ok = true;
      for (int k = 0;; ++k) {
        const int s = k % kRingS;
        if (k >= kRingS && !(ok = mbar_wait(&ring_empty[s], (k / kRingS - 1) & 1, &abort_flag, P.status, detail)))
          break;
        const int x = atomicAdd(P.counter, 1), item = x < P.nitems ? x : -1;
        *reinterpret_cast<volatile int *>(&ring_item[s]) = item;
        mbar_arrive(&ring_full[s]);
        if (item < 0) break;
        int qt, bh, nt;
        sm_item(P, item, qt, bh, nt);
        const int b = bh / P.H, h = bh % P.H;
        if (k > 0 && !(ok = wait(S_QEMPTY, k - 1))) break;  // the previous item's products read Q
        mbar_arrive_expect_tx(&bar[S_QFULL], kTileBytes);
        tma_load_4d(&mq, &bar[S_QFULL], smem, 0, 128 * qt, h, b, kPolicyEvictFirst);
        tma_load_4d(&mq, &bar[S_QFULL], smem + kTileHalfBytes, 64, 128 * qt, h, b, kPolicyEvictFirst);
        ++nq;
        for (int t = 0; t < nt && ok; ++t, ++kt) {
          const int st = kt % kKvStages, u = kt / kKvStages;
          if (u > 0 && !(ok = wait(S_KEMPTY + st, u - 1))) break;
          uint8_t *dst = smem + kSmOffKv + st * 2 * kTileBytes;
          mbar_arrive_expect_tx(&bar[S_KFULL + st], 2 * kTileBytes);
          tma_load_4d(&mk, &bar[S_KFULL + st], dst, 0, 128 * t, h, b, kPolicyEvictLast);
          tma_load_4d(&mk, &bar[S_KFULL + st], dst + kTileHalfBytes, 64, 128 * t, h, b, kPolicyEvictLast);
          tma_load_4d(&mv, &bar[S_KFULL + st], dst + kTileBytes, 0, 128 * t, h, b, kPolicyEvictLast);
          tma_load_4d(&mv, &bar[S_KFULL + st], dst + kTileBytes + kTileHalfBytes, 64, 128 * t, h, b,
                      kPolicyEvictLast);
        }
        if (!ok) break;
      }
      // time-bounded drain of the loads in flight (also after an abort)
      volatile int no_abort = 0;
      if (nq > 0) mbar_wait(&bar[S_QFULL], (nq - 1) & 1, &no_abort, P.status);
      for (int st = 0; st < kKvStages; ++st) {
        const int uses = kt > st ? (kt - 1 - st) / kKvStages + 1 : 0;
        if (uses > 0) mbar_wait(&bar[S_KFULL + st], (uses - 1) & 1, &no_abort, P.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16(128, 128, false, false);  // Q K^T
      const uint32_t id_pv = idesc_bf16(128, 128, false, true);   // P V (P from TMEM)
      int kt = 0, u = 0;
      bool ok = true;
      for (int k = 0, item; ok; ++k) {
        if (!(ok = take(k, item)) || item < 0) break;
        int qt, bh, nt;
        sm_item(P, item, qt, bh, nt);
        const uint32_t tO = tOut(k);
        // O += P V for the tile at counters (u0, kt0), the item's t0-th
        auto pv = [&](int u0, int kt0, int t0) {
          if (!(ok = wait(S_PREADY + (u0 & 1), u0 >> 1))) return;
          if (t0 == 0 && k >= 2 && !(ok = wait(S_OEMPTY + (k & 1), (k >> 1) - 1))) return;
          tc_fence_after();
          const uint32_t V = kv_addr(kt0) + kTileBytes;
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks)
            mma_ts(tO, tS(u0) + ks * 8, desc_mnmajor(V, ks), id_pv, (t0 > 0 || ks > 0) ? 1u : 0u);
          mma_commit(&bar[S_KEMPTY + kt0 % kKvStages]);
          mma_commit(&bar[S_PVC]);
        };
        if (!(ok = wait(S_QFULL, k))) break;
        for (int t = 0; t < nt && ok; ++t, ++kt, ++u) {
          if (!(ok = wait(S_KFULL + kt % kKvStages, kt / kKvStages))) break;
          tc_fence_after();
          const uint32_t K = kv_addr(kt);
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) mma_ss(tS(u), desc_kmajor(sQ, ks), desc_kmajor(K, ks), id_qk, ks > 0);
          mma_commit(&bar[S_SFULL + (u & 1)]);
          if (t + 1 == nt) mma_commit(&bar[S_QEMPTY]);
          if (t > 0) pv(u - 1, kt - 1, t - 1);  // the previous tile's softmax overlapped this product
        }
        if (!ok) break;
        pv(u - 1, kt - 1, nt - 1);
        if (!ok) break;
        mma_commit(&bar[S_OFULL + (k & 1)]);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax: one query row per thread
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    int u = 0;
    bool ok = true;
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, take(k, item))) || item < 0) break;
      int qt, bh, nt;
      sm_item(P, item, qt, bh, nt);
      const int qabs = P.off + 128 * qt + (int)row;  // this row's query position in the prefix
      const uint32_t tO = tOut(k);
      float m_ref = -INFINITY, l = 0.f;
      for (int t = 0; t < nt; ++t, ++u) {
        if (!(ok = __all_sync(0xffffffffu, wait(S_SFULL + (u & 1), u >> 1)))) break;
        tc_fence_after();
        // the tile's scaled, masked row maximum (all four loads in flight at once; the
        // scores are read again below)
        float mt = -INFINITY;
        const int kmax = qabs - 128 * t;  // the last key column this row may see
        {
          uint32_t r[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS(u) + lb + c * 32, r[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (32 * c + j <= kmax) mt = fmaxf(mt, __uint_as_float(r[c][j]));
        }
        mt *= P.scale_log2;
        // move the reference maximum only when this tile raises the row's maximum by more than 8
        const bool move = t == 0 || mt > m_ref + 8.f;
        if (t > 0 && __any_sync(0xffffffffu, move)) {
          // rescale this warp's rows of O (the previous tile's product must be done)
          if (!(ok = __all_sync(0xffffffffu, wait(S_PVC, u - 1)))) break;
          tc_fence_after();
          const float f = move ? ex2(m_ref - mt) : 1.f;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld32(tO + lb + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
            tmem_st32(tO + lb + c * 32, r);
          }
          tmem_st_wait();
          l *= f;
        }
        if (move) m_ref = mt;
        // p = exp2(scale log2(e) s - m_ref), 0 past the diagonal, as bf16 pairs: chunk c goes to
        // columns 16c..16c+15, which hold scores this pass has already read
#pragma unroll 1
        for (int c2 = 0; c2 < 4; c2 += 2) {
          uint32_t r[2][32];
          tmem_ld32(tS(u) + lb + c2 * 32, r[0]);
          tmem_ld32(tS(u) + lb + c2 * 32 + 32, r[1]);
          tmem_ld_wait();
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int c = c2 + h2;
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int j0 = 32 * c + 2 * j;
              const float p0 = j0 <= kmax ? ex2(fmaf(__uint_as_float(r[h2][2 * j]), P.scale_log2, -m_ref)) : 0.f;
              const float p1 = j0 + 1 <= kmax ? ex2(fmaf(__uint_as_float(r[h2][2 * j + 1]), P.scale_log2, -m_ref)) : 0.f;
              l += p0 + p1;
              w[j] = pack_bf16(p0, p1);
            }
            tmem_st16(tS(u) + lb + c * 16, w);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[S_PREADY + (u & 1)]);
      }
      if (!ok) break;
      // hand the row's maximum and sum to the output group (which has read the previous item's)
      if (k >= 1 && !(ok = __all_sync(0xffffffffu, wait(S_LEMPTY, k - 1)))) break;
      stat_m[row] = m_ref;
      stat_l[row] = l;
      mbar_arrive(&bar[S_LFULL]);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ output: O / rowsum, log-sum-exp
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    bool ok = true;
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, take(k, item))) || item < 0) break;
      int qt, bh, nt;
      sm_item(P, item, qt, bh, nt);
      const int b = bh / P.H, h = bh % P.H, qrow = 128 * qt + (int)row;
      const uint32_t tO = tOut(k);
      if (!(ok = __all_sync(0xffffffffu, wait(S_OFULL + (k & 1), k >> 1) && wait(S_LFULL, k)))) break;
      tc_fence_after();
      const float m = stat_m[row], l = stat_l[row];
      mbar_arrive(&bar[S_LEMPTY]);
      const float inv = 1.f / l;
      const bool valid = qrow < P.Tq;
      __nv_bfloat16 *dst = P.o + (int64_t)b * P.osb + (int64_t)h * P.osh + (int64_t)qrow * P.ost;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float x[32];
        uint32_t r[32];
        tmem_ld32(tO + lb + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]) * inv;
        if (valid) st_row_chunk(dst + 32 * c, x, P.wide != 0);
      }
      if (valid && P.lse) P.lse[(int64_t)bh * P.Tq + qrow] = (m + log2f(l)) * 0.6931471805599453f;
      tc_fence_before();
      mbar_arrive(&bar[S_OEMPTY + (k & 1)]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(P.counter + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(P.counter, 0);
      atomicExch(P.counter + 1, 0);
    }
  }
  if (warp == 1) tmem_dealloc(tmem, 512);
}

bool tmap_seq(const void *base, int B, int H, int T, int64_t sb, int64_t sh, int64_t st, CUtensorMap *m) {
  const uint64_t dims[4] = {128, (uint64_t)T, (uint64_t)H, (uint64_t)B};
  const uint64_t strides[3] = {(uint64_t)st * 2, (uint64_t)sh * 2, (uint64_t)sb * 2};
  return make_tmap_bf16(m, base, dims, strides);
}

}  // namespace

cudaError_t softmax_segment(const SoftmaxProblem &p, const void *q, const void *k, const void *v, void *o, float *lse,
                            int *status, cudaStream_t s) {
  alignas(64) CUtensorMap mq, mk, mv;
  if (!status || !tmap_seq(q, p.B, p.H, p.Tq, p.qsb, p.qsh, p.qst, &mq) ||
      !tmap_seq(k, p.B, p.H, p.Tk, p.ksb, p.ksh, p.kst, &mk) || !tmap_seq(v, p.B, p.H, p.Tk, p.ksb, p.ksh, p.kst, &mv))
    return cudaErrorInvalidValue;
  SoftmaxParams S;
  S.B = p.B; S.H = p.H; S.Tq = p.Tq; S.Tk = p.Tk; S.off = p.Tk - p.Tq;
  S.nqt = (p.Tq + 127) / 128;
  S.nitems = S.nqt * p.B * p.H;
  S.scale_log2 = p.scale * 1.4426950408889634f;
  S.o = static_cast<__nv_bfloat16 *>(o);
  S.osb = p.qsb; S.osh = p.qsh; S.ost = p.qst;
  S.lse = lse;
  auto a32 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 31u) == 0; };
  S.wide = a32(o) && (p.qsb * 2) % 32 == 0 && (p.qsh * 2) % 32 == 0 && (p.qst * 2) % 32 == 0;
  S.status = status;
  S.counter = status + kCounterSoftmax;
  const int grid = S.nitems < p.num_sms ? S.nitems : p.num_sms;
  cudaError_t e = cudaFuncSetAttribute(softmax_segment_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmSmem);
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_SOFTMAX_SEGMENT, s);
  softmax_segment_kernel<<<grid, kSmThreads, kSmSmem, s>>>(mq, mk, mv, S);
  return cudaGetLastError();
}

}  // namespace linattn
