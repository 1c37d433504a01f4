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

// ============================================================================ backward
// The gradients for an output gradient dO, with the forward's log-sum-exp per
// query row (lse) and delta_i = dO_i . o_i (the softmax Jacobian's row term):
//   p_ij  = exp(scale q_i . k_j - lse_i)         (the row's softmax weights, recomputed)
//   ds_ij = p_ij (dO_i . v_j - delta_i)
//   dv_j  = sum_i p_ij dO_i,  dk_j = scale sum_i ds_ij q_i,  dq_i = scale sum_j ds_ij k_j
// over the visible pairs j <= offset + i, in two launches, so that every output row is
// owned by one item and nothing is accumulated with atomics:
//   dK/dV (softmax_bwd_kernel): an item is one 128-key tile (X = K, V); it streams
//          the query tiles that see it (Y = Q, dO): S^T = K Q^T and dP^T = V dO^T into
//          TMEM, the elementwise warps write p and ds back as bf16, then dV += P^T dO
//          and dK += dS^T Q read them from TMEM as the A operand;
//   dQ (softmax_bwd_dq2_kernel, below): an item is a pair of 128-query tiles.
// Warp roles as in the forward: warp 0 the TMA producer, warp 1 the MMA issuer,
// warps 2..5 and 6..9 the elementwise work on the score columns 0..63 and 64..127
// of a tile (one row per thread), and the epilogue.  The bf16 results of a column
// half go to that half's own TMEM columns (64 g .. 64 g + 31), so neither half
// writes columns that the other still reads.  Every wait is bounded.
constexpr int kBwThreads = 320;
constexpr int kBwSlots = 4;                                  // ring of Y tiles (32 KiB each)
constexpr uint32_t kBwOffY = 2 * kTileBytes;                 // after the item's two X tiles
constexpr uint32_t kBwOffBar = kBwOffY + kBwSlots * kTileBytes;
constexpr size_t kBwSmem = kBwOffBar + 256 + 1024;
static_assert(kBwSmem + 2048 + 128 <= 232448, "tiles, barriers, column statistics and static shared memory fit");

enum { B_XFULL = 0, B_XEMPTY, B_FULL, B_EMPTY = B_FULL + kBwSlots, B_SFULL = B_EMPTY + kBwSlots, B_DPFULL,
       B_PREADY, B_DSREADY = B_PREADY + 2, B_AFULL = B_DSREADY + 2, B_AEMPTY, B_STAT, B_COUNT = B_STAT + 2 };
static_assert(B_COUNT * 8 + 4 <= 256, "backward barriers and the TMEM slot fit their 256 bytes");

struct BwdParams {
  int B, H, Tq, Tk, off, nqt, nkt, nitems;
  float scale_log2;             // softmax scale times log2(e)
  float scale;
  const float *lse2, *delta;    // [B*H][nqt*128]: lse_i log2(e) and dO_i . o_i (+inf and 0 past Tq)
  __nv_bfloat16 *out1, *out2;   // dK/dV launch: dv, dk;  dQ launch: dq
  int64_t osb, osh, ost;        // element strides of the outputs
  int wide;                     // every output row starts on a 32-byte boundary
  int *status;
  int *counter;                 // [2] item counter and finished CTAs (zero at launch)
};

// item -> (sequence, key tile, first query tile, query tiles), sequence-major (the
// items in flight share their sequences' query tiles in L2) and longest first inside
// a sequence: key tiles in ascending order (a key tile is seen by the query tiles
// from the one holding position key - offset on)
__device__ __forceinline__ void bw_item(const BwdParams &P, int item, int &bh, int &xt, int &lo, int &ns) {
  bh = item / P.nkt;
  xt = item % P.nkt;
  lo = max(0, 128 * xt - P.off) / 128;
  ns = P.nqt - lo;
}

__global__ void __launch_bounds__(kBwThreads, 1)
    softmax_bwd_kernel(const __grid_constant__ CUtensorMap mx1, const __grid_constant__ CUtensorMap mx2,
                       const __grid_constant__ CUtensorMap my1, const __grid_constant__ CUtensorMap my2, BwdParams P) {
  constexpr int kSlots = kBwSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kBwOffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + B_COUNT);
  __shared__ int abort_flag;
  __shared__ int ring_item[kRingS];
  __shared__ uint64_t ring_bar[2 * kRingS];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int *const detail = P.status ? P.status + 1 + warp : nullptr;
  uint64_t *ring_full = ring_bar, *ring_empty = ring_bar + kRingS;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar[B_XFULL], 1);
    mbar_init(&bar[B_XEMPTY], 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bar[B_FULL + s], 1);
      mbar_init(&bar[B_EMPTY + s], 1);
    }
    mbar_init(&bar[B_SFULL], 1);
    mbar_init(&bar[B_DPFULL], 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar[B_PREADY + x], 128);
      mbar_init(&bar[B_DSREADY + x], 128);
      mbar_init(&bar[B_STAT + x], 128);
    }
    mbar_init(&bar[B_AFULL], 1);
    mbar_init(&bar[B_AEMPTY], 256);
    for (int i = 0; i < kRingS; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 32 + 256);  // readers: the MMA warp, the eight elementwise warps
    }
    fence_mbar_init();
    prefetch_tensormap(&mx1);
    prefetch_tensormap(&mx2);
    prefetch_tensormap(&my1);
    prefetch_tensormap(&my2);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // TMEM: S^T (p in place as bf16), dP^T (ds in place), dV, dK
  const uint32_t tS = tmem, tP = tmem + 128u, tA1 = tmem + 256u, tA2 = tmem + 384u;
  // dK/dV: the current step's column statistics (lse2, delta) per column half, two buffers
  __shared__ float4 colstat[2][2][2][16];  // [step parity][half][lse2 | delta][16 x 4 columns]
  auto sX = [&](int x) { return smem_u32(smem) + (uint32_t)x * kTileBytes; };
  auto slot_addr = [&](int i) { return smem_u32(smem + kBwOffY) + (uint32_t)(i % kSlots) * kTileBytes; };
  auto wait = [&](int idx, int parity) { return mbar_wait(&bar[idx], parity & 1, &abort_flag, P.status, detail); };
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
      int li = 0, nx = 0;  // Y tiles and X tile pairs loaded
      bool ok = true;
      auto load = [&](const CUtensorMap *m, int row, int h, int b) {
        const int s = li % kSlots, u = li / kSlots;
        if (u > 0 && !(ok = wait(B_EMPTY + s, u - 1))) return;
        uint8_t *dst = smem + kBwOffY + s * kTileBytes;
        mbar_arrive_expect_tx(&bar[B_FULL + s], kTileBytes);
        tma_load_4d(m, &bar[B_FULL + s], dst, 0, row, h, b, kPolicyEvictLast);
        tma_load_4d(m, &bar[B_FULL + s], dst + kTileHalfBytes, 64, row, h, b, kPolicyEvictLast);
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
        int bh, xt, lo, ns;
        bw_item(P, item, bh, xt, lo, ns);
        const int b = bh / P.H, h = bh % P.H;
        if (k > 0 && !(ok = wait(B_XEMPTY, k - 1))) break;  // the previous item's score products read X
        mbar_arrive_expect_tx(&bar[B_XFULL], 2 * kTileBytes);
        tma_load_4d(&mx1, &bar[B_XFULL], smem, 0, 128 * xt, h, b, kPolicyEvictFirst);
        tma_load_4d(&mx1, &bar[B_XFULL], smem + kTileHalfBytes, 64, 128 * xt, h, b, kPolicyEvictFirst);
        tma_load_4d(&mx2, &bar[B_XFULL], smem + kTileBytes, 0, 128 * xt, h, b, kPolicyEvictFirst);
        tma_load_4d(&mx2, &bar[B_XFULL], smem + kTileBytes + kTileHalfBytes, 64, 128 * xt, h, b, kPolicyEvictFirst);
        ++nx;
        for (int n = 0; n < ns && ok; ++n) {
          load(&my1, 128 * (lo + n), h, b);
          if (ok) load(&my2, 128 * (lo + n), h, b);
        }
        if (!ok) break;
      }
      // time-bounded drain of the loads in flight (also after an abort)
      volatile int no_abort = 0;
      if (nx > 0) mbar_wait(&bar[B_XFULL], (nx - 1) & 1, &no_abort, P.status);
      for (int s = 0; s < kSlots; ++s) {
        const int uses = li > s ? (li - 1 - s) / kSlots + 1 : 0;
        if (uses > 0) mbar_wait(&bar[B_FULL + s], (uses - 1) & 1, &no_abort, P.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the whole warp)
    // Per step n (one query tile): dP(n), dV(n), S(n+1), dK(n).  The products of step n run
    // while the elementwise warps form its p and ds, and the next tile's scores run while
    // they form its ds; S(0) of an item opens its first step.
    // The products read the bf16 p and ds from TMEM right where the elementwise warps
    // wrote them, so every product that overwrites a score tile is issued after the one
    // that reads it (the products of a CTA run in issue order).
    const uint32_t id_ss = idesc_bf16(128, 128, false, false);  // X Y^T
    const uint32_t id_ts = idesc_bf16(128, 128, false, true);   // (bf16 tile in TMEM) Y
    int li = 0, u = 0;
    bool ok = true;
    auto wait_all = [&](int idx, int parity) { return __all_sync(0xffffffffu, wait(idx, parity)); };
    auto score = [&](uint32_t d, uint32_t x, uint32_t y) {
#pragma unroll
      for (uint32_t ks = 0; ks < 8; ++ks) mma_ss_warp(d, desc_kmajor(x, ks), desc_kmajor(y, ks), id_ss, ks > 0);
    };
    // the accumulation over the Y rows of one column half g (k-steps 4g .. 4g+3)
    auto accum = [&](uint32_t d, uint32_t a, uint32_t y, int g, bool first) {
#pragma unroll
      for (uint32_t kk = 0; kk < 4; ++kk) {
        const uint32_t ks = 4u * g + kk;
        mma_ts_warp(d, a + 64u * g + 8u * kk, desc_mnmajor(y, ks), id_ts, (!first || ks > 0) ? 1u : 0u);
      }
    };
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, take(k, item))) || item < 0) break;
      int bh, xt, lo, ns;
      bw_item(P, item, bh, xt, lo, ns);
      if (!(ok = wait_all(B_XFULL, k))) break;
      for (int n = 0; n < ns && ok; ++n, ++u, li += 2) {
        const int i1 = li, i2 = li + 1, i3 = li + 2;  // Y1, Y2 of this step, Y1 of the next
        if (!(ok = wait_all(B_FULL + i1 % kSlots, i1 / kSlots) && wait_all(B_FULL + i2 % kSlots, i2 / kSlots)))
          break;
        tc_fence_after();
        const uint32_t Y1 = slot_addr(i1), Y2 = slot_addr(i2);
        if (n == 0) {
          score(tS, sX(0), Y1);
          mma_commit_warp(&bar[B_SFULL]);
        }
        score(tP, sX(1), Y2);
        mma_commit_warp(&bar[B_DPFULL]);
        if (n + 1 == ns) mma_commit_warp(&bar[B_XEMPTY]);
        // the accumulators are free once the previous item's epilogue has read them
        if (n == 0 && k > 0 && !(ok = wait_all(B_AEMPTY, k - 1))) break;
        // dV += P^T dO, each column half as soon as its p are in TMEM
        for (int g = 0; g < 2 && ok; ++g) {
          if (!(ok = wait_all(B_PREADY + g, u))) break;
          tc_fence_after();
          accum(tA1, tS, Y2, g, n == 0);
        }
        if (!ok) break;
        if (n + 1 < ns) {
          // (the elementwise warps have read this step's scores, waited above, before the
          // next ones complete: a barrier phase never runs two ahead of its waiters)
          if (!(ok = wait_all(B_FULL + i3 % kSlots, i3 / kSlots))) break;
          tc_fence_after();
          score(tS, sX(0), slot_addr(i3));
          mma_commit_warp(&bar[B_SFULL]);
        }
        // dK += dS^T Q, each column half as soon as its ds are in TMEM
        for (int g = 0; g < 2 && ok; ++g) {
          if (!(ok = wait_all(B_DSREADY + g, u))) break;
          tc_fence_after();
          accum(tA2, tP, Y1, g, n == 0);
        }
        if (!ok) break;
        mma_commit_warp(&bar[B_EMPTY + i1 % kSlots]);
        mma_commit_warp(&bar[B_EMPTY + i2 % kSlots]);
        if (n + 1 == ns) mma_commit_warp(&bar[B_AFULL]);
      }
    }
  } else if (warp >= 2 && warp < 10) {
    // ------------------------------------------------------------ p and ds for a column half, epilogue
    const int g = (warp - 2) >> 2;
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    const int gt = threadIdx.x - 64 - 128 * g;  // 0..127 within the column half's warps
    int u = 0;
    bool ok = true;
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, take(k, item))) || item < 0) break;
      int bh, xt, lo, ns;
      bw_item(P, item, bh, xt, lo, ns);
      const float *L2 = P.lse2 + (int64_t)bh * P.nqt * 128, *DL = P.delta + (int64_t)bh * P.nqt * 128;
      // this thread's column statistic of a step (one value per thread: 64 columns x two
      // arrays per half), loaded one step ahead so that its latency is not on the step's path
      const int sc = gt & 63, which = gt >> 6;
      const float *stat = (which ? DL : L2) + 64 * g + sc;
      float sv = stat[128 * lo];
      for (int n = 0; n < ns; ++n, ++u) {
        const int yt = lo + n;
        float4 *cs = &colstat[u & 1][g][0][0];
        {
          // this step's 64 column statistics of the half into shared memory, published
          // through the half's mbarrier (a thread rewrites a buffer two steps later, after
          // every thread of the half has arrived for the step between)
          reinterpret_cast<float *>(cs)[64 * which + sc] = sv;
          mbar_arrive(&bar[B_STAT + g]);
          if (n + 1 < ns) sv = stat[128 * (yt + 1)];
        }
        if (!(ok = __all_sync(0xffffffffu, wait(B_SFULL, u) && wait(B_STAT + g, u)))) break;
        tc_fence_after();
        // key 128 xt + row sees the query columns c >= lim of this tile
        const int lim = 128 * (xt - yt) + (int)row - P.off;
        // every row of the warp sees every column of the half: no masks
        const bool full = __all_sync(0xffffffffu, lim <= 64 * g);
        // phase 1: p of the half's 64 columns (kept in registers, and into TMEM as bf16)
        float p[64];
        {
          uint32_t sr[2][32];
          tmem_ld32(tS + lb + 64 * g, sr[0]);
          tmem_ld32(tS + lb + 64 * g + 32, sr[1]);
          tmem_ld_wait();
#pragma unroll
          for (int j4 = 0; j4 < 16; ++j4) {
            const float4 l4 = cs[j4];
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = 4 * j4 + e;
              p[j] = ex2(fmaf(__uint_as_float(sr[j >> 5][j & 31]), P.scale_log2, -lv[e]));
            }
          }
          if (!full) {
#pragma unroll
            for (int j = 0; j < 64; ++j)
              if (64 * g + j < lim) p[j] = 0.f;
          }
        }
        // p into TMEM for the dV product
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t wp[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) wp[jj] = pack_bf16(p[32 * hh + 2 * jj], p[32 * hh + 2 * jj + 1]);
          tmem_st16(tS + lb + 64 * g + 16 * hh, wp);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[B_PREADY + g]);
        // phase 2: ds = p (dp - delta) into the dP tile as bf16
        if (!(ok = __all_sync(0xffffffffu, wait(B_DPFULL, u)))) break;
        tc_fence_after();
        {
          uint32_t dr[2][32];
          tmem_ld32(tP + lb + 64 * g, dr[0]);
          tmem_ld32(tP + lb + 64 * g + 32, dr[1]);
          tmem_ld_wait();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t wd[16];
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 d4 = cs[16 + 8 * hh + j4];
              const float dl[4] = {d4.x, d4.y, d4.z, d4.w};
              const int j = 4 * j4;
              wd[2 * j4] = pack_bf16(p[32 * hh + j] * (__uint_as_float(dr[hh][j]) - dl[0]),
                                     p[32 * hh + j + 1] * (__uint_as_float(dr[hh][j + 1]) - dl[1]));
              wd[2 * j4 + 1] = pack_bf16(p[32 * hh + j + 2] * (__uint_as_float(dr[hh][j + 2]) - dl[2]),
                                         p[32 * hh + j + 3] * (__uint_as_float(dr[hh][j + 3]) - dl[3]));
            }
            tmem_st16(tP + lb + 64 * g + 16 * hh, wd);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[B_DSREADY + g]);
      }
      if (!ok) break;
      // epilogue: the first half stores the dv row, the second the dk row (times the scale)
      if (!(ok = __all_sync(0xffffffffu, wait(B_AFULL, k)))) break;
      tc_fence_after();
      const int b = bh / P.H, h = bh % P.H, r = 128 * xt + (int)row;
      const bool valid = r < P.Tk;
      __nv_bfloat16 *dst = (g == 1 ? P.out2 : P.out1) + (int64_t)b * P.osb + (int64_t)h * P.osh + (int64_t)r * P.ost;
      const uint32_t src = (g == 0 ? tA1 : tA2) + lb;
      const float f = g == 0 ? 1.f : P.scale;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float y[32];
        uint32_t o[32];
        tmem_ld32(src + 32 * c, o);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(o[j]) * f;
        if (valid) st_row_chunk(dst + 32 * c, y, P.wide != 0);
      }
      tc_fence_before();
      mbar_arrive(&bar[B_AEMPTY]);
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

// dQ with two adjacent query tiles per CTA (A, B): each K and V tile serves both, and
// while one tile's p or ds are formed the other tile's products run.  Per tile one
// TMEM region holds S, then dP once p is in registers, then ds as bf16 (the A
// operand of dQ += dS K), and a dQ accumulator (4 x 128 columns).  Per key tile t:
//   S_x(t) -> p (elementwise) -> dP_x(t) -> ds -> dQ_x(t) -> S_x(t+1) ...
// issued as dP_A, dP_B, dQ_A, S_A(t+1), dQ_B, S_B(t+1).  Shared memory: the item's
// Q and dO tiles of A and B, K tiles alternating between two slots, V tiles in a third.
constexpr uint32_t kQ2OffY = 4 * kTileBytes;
constexpr uint32_t kQ2OffBar = kQ2OffY + 3 * kTileBytes;
constexpr size_t kQ2Smem = kQ2OffBar + 256 + 1024;
static_assert(kQ2Smem + 128 <= 232448, "tiles, barriers and static shared memory fit 227 KB");
enum { Q2_XFULL = 0, Q2_XEMPTY, Q2_FULL, Q2_EMPTY = Q2_FULL + 3, Q2_SFULL = Q2_EMPTY + 3, Q2_SREAD = Q2_SFULL + 2,
       Q2_DPFULL = Q2_SREAD + 2, Q2_DSREADY = Q2_DPFULL + 2, Q2_AFULL = Q2_DSREADY + 2, Q2_AEMPTY = Q2_AFULL + 2,
       Q2_COUNT = Q2_AEMPTY + 2 };
static_assert(Q2_COUNT * 8 + 4 <= 256, "dQ barriers and the TMEM slot fit their 256 bytes");

// item -> (sequence, first query tile of the pair, key tiles up to the second tile's
// diagonal), sequence-major and longest first inside a sequence (as the forward)
__device__ __forceinline__ void q2_item(const BwdParams &P, int item, int &bh, int &qt, int &nt) {
  const int npair = (P.nqt + 1) / 2;
  qt = 2 * (npair - 1 - item % npair);
  bh = item / npair;
  nt = (min(P.Tk, P.off + 128 * qt + 256) + 127) / 128;
}

__global__ void __launch_bounds__(kBwThreads, 1)
    softmax_bwd_dq2_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mdo,
                           const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                           BwdParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kQ2OffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + Q2_COUNT);
  __shared__ int abort_flag;
  __shared__ int ring_item[kRingS];
  __shared__ uint64_t ring_bar[2 * kRingS];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int *const detail = P.status ? P.status + 1 + warp : nullptr;
  uint64_t *ring_full = ring_bar, *ring_empty = ring_bar + kRingS;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar[Q2_XFULL], 1);
    mbar_init(&bar[Q2_XEMPTY], 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&bar[Q2_FULL + s], 1);
      mbar_init(&bar[Q2_EMPTY + s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar[Q2_SFULL + x], 1);
      mbar_init(&bar[Q2_SREAD + x], 128);
      mbar_init(&bar[Q2_DPFULL + x], 1);
      mbar_init(&bar[Q2_DSREADY + x], 128);
      mbar_init(&bar[Q2_AFULL + x], 1);
      mbar_init(&bar[Q2_AEMPTY + x], 128);
    }
    for (int i = 0; i < kRingS; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 32 + 256);  // readers: the MMA warp, the eight elementwise warps
    }
    fence_mbar_init();
    prefetch_tensormap(&mq);
    prefetch_tensormap(&mdo);
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
  auto tR = [&](int x) { return tmem + 128u * (uint32_t)x; };         // S / dP / ds of tile x
  auto tQ = [&](int x) { return tmem + 256u + 128u * (uint32_t)x; };  // dQ of tile x
  // smem: Q_A, dO_A, Q_B, dO_B, then the K slots 0, 1 and the V slot 2
  auto sXq = [&](int x) { return smem_u32(smem) + (uint32_t)(2 * x) * kTileBytes; };
  auto sXo = [&](int x) { return smem_u32(smem) + (uint32_t)(2 * x + 1) * kTileBytes; };
  auto sY = [&](int slot) { return smem_u32(smem + kQ2OffY) + (uint32_t)slot * kTileBytes; };
  auto wait = [&](int idx, int parity) { return mbar_wait(&bar[idx], parity & 1, &abort_flag, P.status, detail); };
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
      int nk = 0, nv = 0, nx = 0;  // K tiles, V tiles and X tile sets loaded
      bool ok = true;
      for (int k = 0;; ++k) {
        const int s = k % kRingS;
        if (k >= kRingS && !(ok = mbar_wait(&ring_empty[s], (k / kRingS - 1) & 1, &abort_flag, P.status, detail)))
          break;
        const int x = atomicAdd(P.counter, 1), item = x < P.nitems ? x : -1;
        *reinterpret_cast<volatile int *>(&ring_item[s]) = item;
        mbar_arrive(&ring_full[s]);
        if (item < 0) break;
        int bh, qt, nt;
        q2_item(P, item, bh, qt, nt);
        const int b = bh / P.H, h = bh % P.H;
        if (k > 0 && !(ok = wait(Q2_XEMPTY, k - 1))) break;  // the previous item's products read X
        mbar_arrive_expect_tx(&bar[Q2_XFULL], 4 * kTileBytes);
        for (int x = 0; x < 2; ++x) {
          uint8_t *dq = smem + (2 * x) * kTileBytes, *dd = smem + (2 * x + 1) * kTileBytes;
          tma_load_4d(&mq, &bar[Q2_XFULL], dq, 0, 128 * (qt + x), h, b, kPolicyEvictFirst);
          tma_load_4d(&mq, &bar[Q2_XFULL], dq + kTileHalfBytes, 64, 128 * (qt + x), h, b, kPolicyEvictFirst);
          tma_load_4d(&mdo, &bar[Q2_XFULL], dd, 0, 128 * (qt + x), h, b, kPolicyEvictFirst);
          tma_load_4d(&mdo, &bar[Q2_XFULL], dd + kTileHalfBytes, 64, 128 * (qt + x), h, b, kPolicyEvictFirst);
        }
        ++nx;
        for (int t = 0; t < nt && ok; ++t) {
          // K(t) into slot nk & 1 (its previous K released after that step's dQ products),
          // V(t) into slot 2 (the previous V released after that step's dP products)
          const int ks = nk & 1;
          if (nk >= 2 && !(ok = wait(Q2_EMPTY + ks, (nk >> 1) - 1))) break;
          mbar_arrive_expect_tx(&bar[Q2_FULL + ks], kTileBytes);
          uint8_t *dk = smem + kQ2OffY + ks * kTileBytes;
          tma_load_4d(&mk, &bar[Q2_FULL + ks], dk, 0, 128 * t, h, b, kPolicyEvictLast);
          tma_load_4d(&mk, &bar[Q2_FULL + ks], dk + kTileHalfBytes, 64, 128 * t, h, b, kPolicyEvictLast);
          ++nk;
          if (nv >= 1 && !(ok = wait(Q2_EMPTY + 2, nv - 1))) break;
          mbar_arrive_expect_tx(&bar[Q2_FULL + 2], kTileBytes);
          uint8_t *dv = smem + kQ2OffY + 2 * kTileBytes;
          tma_load_4d(&mv, &bar[Q2_FULL + 2], dv, 0, 128 * t, h, b, kPolicyEvictLast);
          tma_load_4d(&mv, &bar[Q2_FULL + 2], dv + kTileHalfBytes, 64, 128 * t, h, b, kPolicyEvictLast);
          ++nv;
        }
        if (!ok) break;
      }
      // time-bounded drain of the loads in flight (also after an abort)
      volatile int no_abort = 0;
      if (nx > 0) mbar_wait(&bar[Q2_XFULL], (nx - 1) & 1, &no_abort, P.status);
      for (int s = 0; s < 2; ++s) {
        const int uses = nk > s ? (nk - 1 - s) / 2 + 1 : 0;
        if (uses > 0) mbar_wait(&bar[Q2_FULL + s], (uses - 1) & 1, &no_abort, P.status);
      }
      if (nv > 0) mbar_wait(&bar[Q2_FULL + 2], (nv - 1) & 1, &no_abort, P.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the whole warp)
    const uint32_t id_ss = idesc_bf16(128, 128, false, false);  // X Y^T
    const uint32_t id_ts = idesc_bf16(128, 128, false, true);   // (ds in TMEM) K
    int nk = 0, nv = 0, u = 0;
    bool ok = true;
    auto wait_all = [&](int idx, int parity) { return __all_sync(0xffffffffu, wait(idx, parity)); };
    auto score = [&](uint32_t d, uint32_t x, uint32_t y) {
#pragma unroll
      for (uint32_t ks = 0; ks < 8; ++ks) mma_ss_warp(d, desc_kmajor(x, ks), desc_kmajor(y, ks), id_ss, ks > 0);
    };
    auto dq = [&](int x, uint32_t K, bool first) {
#pragma unroll
      for (uint32_t ks = 0; ks < 8; ++ks)
        mma_ts_warp(tQ(x), tR(x) + 8u * ks, desc_mnmajor(K, ks), id_ts, (!first || ks > 0) ? 1u : 0u);
    };
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, take(k, item))) || item < 0) break;
      int bh, qt, nt;
      q2_item(P, item, bh, qt, nt);
      if (!(ok = wait_all(Q2_XFULL, k) && wait_all(Q2_FULL + (nk & 1), nk >> 1))) break;
      tc_fence_after();
      // the item's first scores
      for (int x = 0; x < 2; ++x) {
        score(tR(x), sXq(x), sY(nk & 1));
        mma_commit_warp(&bar[Q2_SFULL + x]);
      }
      for (int t = 0; t < nt && ok; ++t, ++u, ++nk, ++nv) {
        const uint32_t K = sY(nk & 1), V = sY(2);
        if (!(ok = wait_all(Q2_FULL + 2, nv))) break;
        // dP of both tiles once their p are in registers (the region is then free)
        for (int x = 0; x < 2 && ok; ++x) {
          if (!(ok = wait_all(Q2_SREAD + x, u))) break;
          tc_fence_after();
          score(tR(x), sXo(x), V);
          mma_commit_warp(&bar[Q2_DPFULL + x]);
        }
        if (!ok) break;
        mma_commit_warp(&bar[Q2_EMPTY + 2]);
        if (t + 1 == nt) mma_commit_warp(&bar[Q2_XEMPTY]);
        if (t == 0 && k > 0 && !(ok = wait_all(Q2_AEMPTY, k - 1) && wait_all(Q2_AEMPTY + 1, k - 1))) break;
        // dQ of each tile once its ds are in TMEM, then that tile's next scores
        const bool more = t + 1 < nt;
        if (more && !(ok = wait_all(Q2_FULL + ((nk + 1) & 1), (nk + 1) >> 1))) break;
        for (int x = 0; x < 2 && ok; ++x) {
          if (!(ok = wait_all(Q2_DSREADY + x, u))) break;
          tc_fence_after();
          dq(x, K, t == 0);
          if (x == 1) mma_commit_warp(&bar[Q2_EMPTY + (nk & 1)]);
          if (t + 1 == nt) mma_commit_warp(&bar[Q2_AFULL + x]);
          if (more) {
            score(tR(x), sXq(x), sY((nk + 1) & 1));
            mma_commit_warp(&bar[Q2_SFULL + x]);
          }
        }
      }
    }
  } else if (warp >= 2 && warp < 10) {
    // ------------------------------------------------------------ p, ds and the dq rows of tile x
    const int x = (warp - 2) >> 2;
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    int u = 0;
    bool ok = true;
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, take(k, item))) || item < 0) break;
      int bh, qt, nt;
      q2_item(P, item, bh, qt, nt);
      const int qtile = qt + x, i = 128 * qtile + (int)row;
      // this row's statistics (a second tile past the end has none: p = 0)
      const bool in = qtile < P.nqt;
      const float lrow = in ? P.lse2[(int64_t)bh * P.nqt * 128 + i] : INFINITY;
      const float drow = in ? P.delta[(int64_t)bh * P.nqt * 128 + i] : 0.f;
      for (int t = 0; t < nt; ++t, ++u) {
        if (!(ok = __all_sync(0xffffffffu, wait(Q2_SFULL + x, u)))) break;
        tc_fence_after();
        // key column c of this tile is visible to the row when c <= lim
        const int lim = P.off + i - 128 * t;
        const bool full = __all_sync(0xffffffffu, lim >= 127);
        // p as bf16 pairs (the registers of a thread hold at most 168 values here)
        uint32_t pw[64];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t sr[2][32];
          tmem_ld32(tR(x) + lb + 64 * cc, sr[0]);
          tmem_ld32(tR(x) + lb + 64 * cc + 32, sr[1]);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int j = 64 * cc + 2 * jj;
            float p0 = ex2(fmaf(__uint_as_float(sr[jj >> 4][(2 * jj) & 31]), P.scale_log2, -lrow));
            float p1 = ex2(fmaf(__uint_as_float(sr[jj >> 4][(2 * jj + 1) & 31]), P.scale_log2, -lrow));
            if (!full) {
              p0 = j > lim ? 0.f : p0;
              p1 = j + 1 > lim ? 0.f : p1;
            }
            pw[32 * cc + jj] = pack_bf16(p0, p1);
          }
        }
        tc_fence_before();
        mbar_arrive(&bar[Q2_SREAD + x]);  // the scores are in registers: dP may overwrite them
        if (!(ok = __all_sync(0xffffffffu, wait(Q2_DPFULL + x, u)))) break;
        tc_fence_after();
        // ds = p (dp - delta), chunk by chunk into the region's first 64 columns (chunk c's
        // bf16 pairs overwrite dp columns that earlier chunks have already read)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t dr[32], wd[16];
          tmem_ld32(tR(x) + lb + 32 * c, dr);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const uint32_t pp = pw[16 * c + jj];
            wd[jj] = pack_bf16(bf16lo(pp) * (__uint_as_float(dr[2 * jj]) - drow),
                               bf16hi(pp) * (__uint_as_float(dr[2 * jj + 1]) - drow));
          }
          tmem_st16(tR(x) + lb + 16 * c, wd);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[Q2_DSREADY + x]);
      }
      if (!ok) break;
      // the dq row (times the scale)
      if (!(ok = __all_sync(0xffffffffu, wait(Q2_AFULL + x, k)))) break;
      tc_fence_after();
      const int b = bh / P.H, h = bh % P.H;
      const bool valid = i < P.Tq;
      __nv_bfloat16 *dst = P.out1 + (int64_t)b * P.osb + (int64_t)h * P.osh + (int64_t)i * P.ost;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float y[32];
        uint32_t o[32];
        tmem_ld32(tQ(x) + lb + 32 * c, o);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(o[j]) * P.scale;
        if (valid) st_row_chunk(dst + 32 * c, y, P.wide != 0);
      }
      tc_fence_before();
      mbar_arrive(&bar[Q2_AEMPTY + x]);
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

// The per-query statistics of the backward, one warp per padded query row:
// lse2 = lse log2(e) and delta = dO . o (fp32 from the bf16 rows); past Tq +inf and 0.
__global__ void __launch_bounds__(256) softmax_bwd_prep_kernel(const __nv_bfloat16 *o, const __nv_bfloat16 *dO,
                                                               const float *lse, int H, int Tq, int rows_pad,
                                                               int64_t sb, int64_t sh, int64_t st, int64_t nrows,
                                                               float *lse2, float *delta) {
  const int64_t r = ((int64_t)blockIdx.x * 256 + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (r >= nrows) return;
  const int64_t bh = r / rows_pad;
  const int i = (int)(r % rows_pad);
  if (i >= Tq) {
    if (lane == 0) {
      lse2[r] = INFINITY;
      delta[r] = 0.f;
    }
    return;
  }
  const int64_t off = (bh / H) * sb + (bh % H) * sh + (int64_t)i * st + 4 * lane;
  const uint2 a = *reinterpret_cast<const uint2 *>(o + off), c = *reinterpret_cast<const uint2 *>(dO + off);
  const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a), *c2 = reinterpret_cast<const __nv_bfloat162 *>(&c);
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(c2[e]);
    acc = fmaf(x.x, y.x, acc);
    acc = fmaf(x.y, y.y, acc);
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (lane == 0) {
    lse2[r] = lse[bh * Tq + i] * 1.4426950408889634f;
    delta[r] = acc;
  }
}

// Zero rows of 128 bf16 (the key gradients when no query is given), one warp per row.
__global__ void __launch_bounds__(256) zero_rows_kernel(__nv_bfloat16 *x, int H, int T, int64_t sb, int64_t sh,
                                                        int64_t st, int64_t nrows) {
  const int64_t r = ((int64_t)blockIdx.x * 256 + threadIdx.x) / 32;
  if (r >= nrows) return;
  const int64_t bh = r / T, i = r % T;
  *reinterpret_cast<uint2 *>(x + (bh / H) * sb + (bh % H) * sh + i * st + 4 * (threadIdx.x % 32)) = make_uint2(0u, 0u);
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


size_t softmax_bwd_stats_bytes(int B, int H, int Tq) {
  return 2 * align256((size_t)B * H * ((Tq + 127) / 128) * 128 * sizeof(float));
}

cudaError_t softmax_segment_bwd(const SoftmaxProblem &p, const void *q, const void *k, const void *v, const void *o,
                                const void *dO, const float *lse, void *dq, void *dk, void *dv, float *stats,
                                int *status, cudaStream_t s) {
  const int64_t BH = (int64_t)p.B * p.H;
  if (!status) return cudaErrorInvalidValue;
  if (p.Tq == 0) {
    // no queries: every key gradient is zero
    const int64_t nrows = BH * p.Tk;
    if (nrows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((nrows * 32 + 255) / 256);
    TimedLaunch t(K_SOFTMAX_BWD_PREP, s);
    zero_rows_kernel<<<blocks, 256, 0, s>>>(static_cast<__nv_bfloat16 *>(dk), p.H, p.Tk, p.ksb, p.ksh, p.kst, nrows);
    zero_rows_kernel<<<blocks, 256, 0, s>>>(static_cast<__nv_bfloat16 *>(dv), p.H, p.Tk, p.ksb, p.ksh, p.kst, nrows);
    return cudaGetLastError();
  }
  alignas(64) CUtensorMap mq, mk, mv, mdo;
  if (!tmap_seq(q, p.B, p.H, p.Tq, p.qsb, p.qsh, p.qst, &mq) || !tmap_seq(dO, p.B, p.H, p.Tq, p.qsb, p.qsh, p.qst, &mdo) ||
      !tmap_seq(k, p.B, p.H, p.Tk, p.ksb, p.ksh, p.kst, &mk) || !tmap_seq(v, p.B, p.H, p.Tk, p.ksb, p.ksh, p.kst, &mv))
    return cudaErrorInvalidValue;
  BwdParams P;
  P.B = p.B; P.H = p.H; P.Tq = p.Tq; P.Tk = p.Tk; P.off = p.Tk - p.Tq;
  P.nqt = (p.Tq + 127) / 128;
  P.nkt = (p.Tk + 127) / 128;
  P.scale_log2 = p.scale * 1.4426950408889634f;
  P.scale = p.scale;
  const int64_t nrows = BH * P.nqt * 128;
  float *lse2 = stats, *delta = stats + align256((size_t)nrows * sizeof(float)) / sizeof(float);
  P.lse2 = lse2;
  P.delta = delta;
  P.status = status;
  cudaError_t e;
  {
    TimedLaunch t(K_SOFTMAX_BWD_PREP, s);
    softmax_bwd_prep_kernel<<<(unsigned)((nrows * 32 + 255) / 256), 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dO), lse, p.H, p.Tq, P.nqt * 128,
        p.qsb, p.qsh, p.qst, nrows, lse2, delta);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  auto a32 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 31u) == 0; };
  // dK, dV: items over the key tiles
  {
    BwdParams K = P;
    K.nitems = (int)(P.nkt * BH);
    K.out1 = static_cast<__nv_bfloat16 *>(dv);
    K.out2 = static_cast<__nv_bfloat16 *>(dk);
    K.osb = p.ksb; K.osh = p.ksh; K.ost = p.kst;
    K.wide = a32(dk) && a32(dv) && (p.ksb * 2) % 32 == 0 && (p.ksh * 2) % 32 == 0 && (p.kst * 2) % 32 == 0;
    K.counter = status + kCounterSoftmaxKV;
    if ((e = cudaFuncSetAttribute(softmax_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kBwSmem)) != cudaSuccess)
      return e;
    TimedLaunch t(K_SOFTMAX_BWD_KV, s);
    softmax_bwd_kernel<<<K.nitems < p.num_sms ? K.nitems : p.num_sms, kBwThreads, kBwSmem, s>>>(mk, mv, mq, mdo, K);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // dQ: items over pairs of query tiles
  BwdParams Q = P;
  Q.nitems = (int)((P.nqt + 1) / 2 * BH);
  Q.out1 = static_cast<__nv_bfloat16 *>(dq);
  Q.out2 = nullptr;
  Q.osb = p.qsb; Q.osh = p.qsh; Q.ost = p.qst;
  Q.wide = a32(dq) && (p.qsb * 2) % 32 == 0 && (p.qsh * 2) % 32 == 0 && (p.qst * 2) % 32 == 0;
  Q.counter = status + kCounterSoftmaxQ;
  if ((e = cudaFuncSetAttribute(softmax_bwd_dq2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kQ2Smem)) != cudaSuccess)
    return e;
  TimedLaunch t(K_SOFTMAX_BWD_Q, s);
  softmax_bwd_dq2_kernel<<<Q.nitems < p.num_sms ? Q.nitems : p.num_sms, kBwThreads, kQ2Smem, s>>>(mq, mdo, mk, mv,
                                                                                                 Q);
  return cudaGetLastError();
}

}  // namespace linattn
