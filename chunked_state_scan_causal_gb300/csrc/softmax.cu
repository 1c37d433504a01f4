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
// Persistent CTAs draw items of two adjacent query tiles of one sequence at
// run time, sequence by sequence (so that the keys and values of the sequences
// in flight stay in L2) and, within a sequence, longest (most key tiles) first.
// The two query tiles share every K and V tile and keep a score buffer and an
// output region each, so the tensor pipe alternates between them: while the
// softmax of one tile is formed, the other tile's products run.  Warp roles:
//   warp 0       TMA producer (one thread): the item's two Q tiles, then K and V
//                tiles through one ring of 32 KiB slots (K of a tile frees after
//                both score products, V after both output products)
//   warp 1       TMEM allocator and MMA issuer (the whole warp; one elected lane
//                issues each product)
//   warps 2..5   softmax and output of the first query tile, one thread per row
//   warps 6..9   the same for the second query tile
// (a warp reaches the TMEM lanes 32 (warp mod 4) .. +31, so each group of four
// consecutive warps covers the 128 rows).  Every wait is bounded.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace linattn {
namespace {

constexpr int kSmThreads = 320;
constexpr int kKvSlots = 5;                                // ring of K and V tiles (32 KiB each)
constexpr uint32_t kSmOffKv = 2 * kTileBytes;              // after the two Q tiles
constexpr uint32_t kSmOffBar = kSmOffKv + kKvSlots * kTileBytes;
constexpr size_t kSmSmem = kSmOffBar + 256 + 1024;         // (+ 1024: alignment of the tiles)
static_assert(kSmSmem + 128 <= 232448, "tiles, barriers and static shared memory fit 227 KB");

enum { S_QFULL = 0, S_QEMPTY, S_FULL, S_EMPTY = S_FULL + kKvSlots, S_SFULL = S_EMPTY + kKvSlots,
       S_PREADY = S_SFULL + 2, S_OFULL = S_PREADY + 2, S_OEMPTY = S_OFULL + 2, S_COUNT = S_OEMPTY + 2 };
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

// pairs of fp32 values in one 64-bit register: the packed FMA and add of sm_100 and later
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// the maximum of three fp32 values in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Whether the phases of the given parities of four mbarriers have all completed
// (never blocks): the four tests issue back to back, so their latencies overlap.
__device__ __forceinline__ bool mbar_test4(uint64_t *b0, int p0, uint64_t *b1, int p1, uint64_t *b2, int p2,
                                           uint64_t *b3, int p3) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred q0, q1, q2, q3;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q3, [%7], %8;\n\t"
      "and.pred q0, q0, q1;\n\tand.pred q2, q2, q3;\n\tand.pred q0, q0, q2;\n\t"
      "selp.u32 %0, 1, 0, q0;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(b0)), "r"(p0 & 1), "r"(smem_u32(b1)), "r"(p1 & 1), "r"(smem_u32(b2)), "r"(p2 & 1),
        "r"(smem_u32(b3)), "r"(p3 & 1)
      : "memory");
  return ok != 0;
}

// The row's maximum over the 128 scores of a tile (all visible), and over the
// columns up to kmax.
__device__ __forceinline__ float row_max(const uint32_t (&r)[4][32]) {
  float mc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    mc[c] = __uint_as_float(r[c][0]);
#pragma unroll
    for (int j = 1; j < 31; j += 2) mc[c] = max3(mc[c], __uint_as_float(r[c][j]), __uint_as_float(r[c][j + 1]));
    mc[c] = fmaxf(mc[c], __uint_as_float(r[c][31]));
  }
  return max3(fmaxf(mc[0], mc[1]), mc[2], mc[3]);
}
__device__ __forceinline__ float row_max_masked(const uint32_t (&r)[4][32], int kmax) {
  float m = -INFINITY;
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (32 * c + j <= kmax) m = fmaxf(m, __uint_as_float(r[c][j]));
  return m;
}

// p = exp2(cs - m) of the row's 128 scores s (0 past column kmax when MASKED), written
// as bf16 pairs into the first 64 columns of the score buffer at taddr (chunk c of 32
// scores to columns 16c .. 16c+15); returns the row's sum of p.  Pairs of scores go
// through the packed fp32 FMA and add; the sum keeps two packed partial sums.
template <bool MASKED>
__device__ __forceinline__ float probs_to_tmem(const uint32_t (&r)[4][32], float c, float m, int kmax,
                                               uint32_t taddr) {
  const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-m, -m);
  uint64_t l2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float p0, p1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(r[q][2 * j]), __uint_as_float(r[q][2 * j + 1])), c2, nm2), p0, p1);
      p0 = ex2(p0);
      p1 = ex2(p1);
      if (MASKED) {
        const int j0 = 32 * q + 2 * j;
        p0 = j0 <= kmax ? p0 : 0.f;
        p1 = j0 + 1 <= kmax ? p1 : 0.f;
      }
      l2[j & 1] = f2_add(l2[j & 1], f2_pack(p0, p1));
      w[j] = pack_bf16(p0, p1);
    }
    tmem_st16(taddr + 16 * q, w);
  }
  float a0, a1, b0, b1;
  f2_unpack(l2[0], a0, a1);
  f2_unpack(l2[1], b0, b1);
  return (a0 + a1) + (b0 + b1);
}

// item -> (pair of query tiles, sequence), sequence-major: the items that run at the
// same time share one or two sequences' keys and values, which then stay in L2 (every
// query tile of a sequence reads its whole key prefix); inside a sequence the pairs
// with the most key tiles come first.  qt = the pair's first query tile (the second
// is qt + 1, possibly past the end: its rows are then not stored); nt = key tiles up
// to the second tile's diagonal (the first tile masks the extra one)
__device__ __forceinline__ void sm_item(const SoftmaxParams &P, int item, int &qt, int &bh, int &nt) {
  const int npair = (P.nqt + 1) / 2;
  qt = 2 * (npair - 1 - item % npair);
  bh = item / npair;
  const int kend = min(P.Tk, P.off + 128 * qt + 256);  // keys up to the pair's last query
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
  __shared__ int abort_flag;
  __shared__ int ring_item[kRingS];
  __shared__ uint64_t ring_bar[2 * kRingS];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int *const detail = P.status ? P.status + 1 + warp : nullptr;
  uint64_t *ring_full = ring_bar, *ring_empty = ring_bar + kRingS;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar[S_QFULL], 1);
    mbar_init(&bar[S_QEMPTY], 1);
    for (int s = 0; s < kKvSlots; ++s) {
      mbar_init(&bar[S_FULL + s], 1);
      mbar_init(&bar[S_EMPTY + s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar[S_SFULL + x], 1);
      mbar_init(&bar[S_PREADY + x], 128);
      mbar_init(&bar[S_OFULL + x], 1);
      mbar_init(&bar[S_OEMPTY + x], 128);
    }
    for (int i = 0; i < kRingS; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 32 + 2 * 128);  // readers: the MMA warp, the two softmax groups
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
  // query tile x (0, 1) of an item: score buffer and output region
  auto tS = [&](int x) { return tmem + (uint32_t)x * 128u; };
  auto tO = [&](int x) { return tmem + 256u + (uint32_t)x * 128u; };
  auto sQ = [&](int x) { return smem_u32(smem) + (uint32_t)x * kTileBytes; };
  // ring slot of the i-th K/V tile loaded (K of key tile t and V of key tile t in turn)
  auto slot_addr = [&](int i) { return smem_u32(smem + kSmOffKv) + (uint32_t)(i % kKvSlots) * kTileBytes; };
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
      int li = 0, nq = 0;  // K/V tiles and Q tile pairs loaded
      bool ok = true;
      auto load = [&](const CUtensorMap *m, int row, int h, int b) {
        const int s = li % kKvSlots, u = li / kKvSlots;
        if (u > 0 && !(ok = wait(S_EMPTY + s, u - 1))) return;
        uint8_t *dst = smem + kSmOffKv + s * kTileBytes;
        mbar_arrive_expect_tx(&bar[S_FULL + s], kTileBytes);
        tma_load_4d(m, &bar[S_FULL + s], dst, 0, row, h, b, kPolicyEvictLast);
        tma_load_4d(m, &bar[S_FULL + s], dst + kTileHalfBytes, 64, row, h, b, kPolicyEvictLast);
        ++li;
      };
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
        mbar_arrive_expect_tx(&bar[S_QFULL], 2 * kTileBytes);
        for (int q = 0; q < 2; ++q) {
          uint8_t *dst = smem + q * kTileBytes;
          tma_load_4d(&mq, &bar[S_QFULL], dst, 0, 128 * (qt + q), h, b, kPolicyEvictFirst);
          tma_load_4d(&mq, &bar[S_QFULL], dst + kTileHalfBytes, 64, 128 * (qt + q), h, b, kPolicyEvictFirst);
        }
        ++nq;
        for (int t = 0; t < nt && ok; ++t) {
          load(&mk, 128 * t, h, b);
          if (ok) load(&mv, 128 * t, h, b);
        }
        if (!ok) break;
      }
      // time-bounded drain of the loads in flight (also after an abort)
      volatile int no_abort = 0;
      if (nq > 0) mbar_wait(&bar[S_QFULL], (nq - 1) & 1, &no_abort, P.status);
      for (int s = 0; s < kKvSlots; ++s) {
        const int uses = li > s ? (li - 1 - s) / kKvSlots + 1 : 0;
        if (uses > 0) mbar_wait(&bar[S_FULL + s], (uses - 1) & 1, &no_abort, P.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per key tile t, for the item's two query tiles in turn: O_x += P_x V_t (once the
    // softmax of x is done), then S_x = Q_x K_{t+1}^T -- so each tile's next scores are
    // issued right behind its output product, while the other tile's softmax runs.
    // The whole warp runs this loop (one elected lane issues each product).
    {
      const uint32_t id_qk = idesc_bf16(128, 128, false, false);  // Q K^T
      const uint32_t id_pv = idesc_bf16(128, 128, false, true);   // P V (P from TMEM)
      int li = 0, u = 0;  // K/V tiles consumed in load order; key tiles (both query tiles in step)
      bool ok = true;
      auto wait_all = [&](int idx, int parity) { return __all_sync(0xffffffffu, wait(idx, parity)); };
      auto qk = [&](int x, int ik) {
        const uint32_t K = slot_addr(ik);
#pragma unroll
        for (uint32_t ks = 0; ks < 8; ++ks)
          mma_ss_warp(tS(x), desc_kmajor(sQ(x), ks), desc_kmajor(K, ks), id_qk, ks > 0);
        mma_commit_warp(&bar[S_SFULL + x]);
      };
      for (int k = 0, item; ok; ++k) {
        if (!(ok = __all_sync(0xffffffffu, take(k, item))) || item < 0) break;
        int qt, bh, nt;
        sm_item(P, item, qt, bh, nt);
        if (!(ok = wait_all(S_QFULL, k) && wait_all(S_FULL + li % kKvSlots, li / kKvSlots))) break;
        tc_fence_after();
        qk(0, li);
        qk(1, li);
        mma_commit_warp(&bar[S_EMPTY + li % kKvSlots]);
        if (nt == 1) mma_commit_warp(&bar[S_QEMPTY]);
        for (int t = 0; t < nt && ok; ++t, ++u, li += 2) {
          const int iv = li + 1, ik1 = li + 2;  // V of this tile, K of the next
          for (int x = 0; x < 2 && ok; ++x) {
            // everything the two products of tile x need: its probabilities, its output region
            // (first key tile of an item), V of this key tile, K of the next; tested together,
            // then waited for one by one only when one of them is not yet there
            const bool first = t == 0 && k > 0, more = t + 1 < nt;
            const bool ready = __all_sync(
                0xffffffffu, mbar_test4(&bar[S_PREADY + x], u, &bar[first ? S_OEMPTY + x : S_PREADY + x],
                                        first ? k - 1 : u, &bar[S_FULL + iv % kKvSlots], iv / kKvSlots,
                                        &bar[S_FULL + (more ? ik1 : iv) % kKvSlots], (more ? ik1 : iv) / kKvSlots));
            if (!ready && !(ok = wait_all(S_PREADY + x, u) && (!first || wait_all(S_OEMPTY + x, k - 1)) &&
                                 wait_all(S_FULL + iv % kKvSlots, iv / kKvSlots)))
              break;
            tc_fence_after();
            const uint32_t V = slot_addr(iv);
#pragma unroll
            for (uint32_t ks = 0; ks < 8; ++ks)
              mma_ts_warp(tO(x), tS(x) + ks * 8, desc_mnmajor(V, ks), id_pv, (t > 0 || ks > 0) ? 1u : 0u);
            if (t + 1 == nt) mma_commit_warp(&bar[S_OFULL + x]);
            if (x == 1) mma_commit_warp(&bar[S_EMPTY + iv % kKvSlots]);
            if (more) {
              if (!ready) {
                if (!(ok = wait_all(S_FULL + ik1 % kKvSlots, ik1 / kKvSlots))) break;
                tc_fence_after();
              }
              qk(x, ik1);
              if (x == 1) {
                mma_commit_warp(&bar[S_EMPTY + ik1 % kKvSlots]);
                if (t + 2 == nt) mma_commit_warp(&bar[S_QEMPTY]);
              }
            }
          }
        }
      }
    }
  } else if (warp >= 2 && warp < 10) {
    // ------------------------------------------------------------ softmax and output of query tile x:
    // one query row per thread
    const int x = (warp - 2) >> 2;
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    int u = 0;
    bool ok = true;
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, take(k, item))) || item < 0) break;
      int qt, bh, nt;
      sm_item(P, item, qt, bh, nt);
      const int qtile = qt + x;
      const int qabs = P.off + 128 * qtile + (int)row;  // this row's query position in the prefix
      float m_ref = -INFINITY, l = 0.f;
      for (int t = 0; t < nt; ++t, ++u) {
        if (!(ok = __all_sync(0xffffffffu, wait(S_SFULL + x, u)))) break;
        tc_fence_after();
        // the row's 128 scores (all four loads in flight) and their masked maximum
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS(x) + lb + 32 * c, r[c]);
        tmem_ld_wait();
        const int kmax = qabs - 128 * t;  // the last key column this row may see
        // every column is visible to every row of the warp (the warp's first row sees them all)
        const bool full = __shfl_sync(0xffffffffu, kmax, 0) >= 127;
        // Past the first key tile, the probabilities are formed with the current reference
        // maximum first: every p of the tile is at most the tile's sum, so a sum of at most
        // 2^8 shows that the tile does not raise the row's maximum by more than 8, and the
        // reference stays.  Only otherwise is the tile's maximum taken and the tile redone.
        bool fast = t > 0 && full, move = false;
        float f = 1.f, s_tile = 0.f;
        if (fast) {
          s_tile = probs_to_tmem<false>(r, P.scale_log2, m_ref, kmax, tS(x) + lb);
          fast = !__any_sync(0xffffffffu, s_tile > 256.f);
          if (!fast) tmem_st_wait();  // overwritten below
        }
        if (!fast) {
          const float mt = (full ? row_max(r) : row_max_masked(r, kmax)) * P.scale_log2;
          // move the reference maximum only when this tile raises the row's maximum by more
          // than 8; O and the row sum are then scaled by f
          move = t == 0 || mt > m_ref + 8.f;
          f = t > 0 && move ? ex2(m_ref - mt) : 1.f;
          if (move) m_ref = mt;
          s_tile = full ? probs_to_tmem<false>(r, P.scale_log2, m_ref, kmax, tS(x) + lb)
                        : probs_to_tmem<true>(r, P.scale_log2, m_ref, kmax, tS(x) + lb);
        }
        l = l * f + s_tile;
        // the rescale of O: the output product of the previous key tile is complete (it
        // was issued before this tile's score product), this tile's is not yet issued
        if (t > 0 && __any_sync(0xffffffffu, move)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(tO(x) + lb + 32 * c, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
            tmem_st32(tO(x) + lb + 32 * c, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[S_PREADY + x]);
      }
      if (!ok) break;
      // output: O / rowsum as bf16, the log-sum-exp; then the region is free for the next item
      if (!(ok = __all_sync(0xffffffffu, wait(S_OFULL + x, k)))) break;
      tc_fence_after();
      const int b = bh / P.H, h = bh % P.H;
      const float inv = 1.f / l;
      const bool valid = qtile * 128 + (int)row < P.Tq;
      __nv_bfloat16 *dst = P.o + (int64_t)b * P.osb + (int64_t)h * P.osh + (int64_t)(qtile * 128 + (int)row) * P.ost;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float y[32];
        uint32_t o[32];
        tmem_ld32(tO(x) + lb + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(o[j]) * inv;
        if (valid) st_row_chunk(dst + 32 * c, y, P.wide != 0);
      }
      if (valid && P.lse) P.lse[(int64_t)bh * P.Tq + qtile * 128 + row] = (m_ref + log2f(l)) * 0.6931471805599453f;
      tc_fence_before();
      mbar_arrive(&bar[S_OEMPTY + x]);
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
  S.nitems = (S.nqt + 1) / 2 * p.B * p.H;
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
