// Tensor-core kernels (tcgen05 + TMEM + TMA) for bf16 sequences with d = 128.
//
// Both kernels are persistent (one CTA per SM, items taken round-robin) and
// warp-specialised:
//   warp 0        TMA producer (one thread)
//   warp 1        TMEM allocator and MMA issuer (one thread)
//   warps 4..7    epilogue group A (TMEM -> registers -> shared / global)
//   warps 8..11   epilogue group B
// Every wait is a bounded mbarrier wait (see ptx.cuh); a timeout records an
// error in the status word and unwinds the kernel instead of hanging.
//
// A "block" is 128 tokens, i.e. two chunks of 64: the M = 128 tcgen05 MMA is
// the natural tile, and chunking at 128 instead of 64 changes only the
// rounding order (the chunked form equals the definition for any chunk
// length).  All operands are SW128 tiles (ptx.cuh).
#include <cstdlib>

#include "internal.h"
#include "ptx.cuh"

namespace linattn {

bool tc_supported(const Problem &p) { return p.dtype == 0 && p.d == 128 && p.T >= 1; }

int tc_group_len(const Problem &p) {
  // Enough (group, sequence) items for ~8 per SM, but groups of at least 512
  // tokens so that the per-group fp32 state (64 KiB) stays small next to the
  // group's own data (256 KiB of q, k, v per 512 tokens).
  const int64_t BH = (int64_t)p.B * p.H;
  const int64_t target = 8 * (int64_t)p.num_sms;
  int64_t L = (p.T * BH + target - 1) / target;
  L = (L + 127) / 128 * 128;
  if (L < 512) L = 512;
  const int64_t Tr = ((int64_t)p.T + 127) / 128 * 128;
  if (L > Tr) L = Tr;
  return (int)L;
}

namespace {

constexpr int kThreads = 384;

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Multiply one 128-element bf16 row of an SW128 tile by w (rounded back to bf16).
__device__ __forceinline__ void scale_tile_row(uint32_t tile, uint32_t row, float w) {
#pragma unroll 4
  for (uint32_t c = 0; c < 16; ++c) {
    const uint32_t addr = tile + sw128_offset(row, c);
    uint32_t x0, x1, x2, x3;
    ld_shared_v4(addr, x0, x1, x2, x3);
    x0 = pack_bf16(bf16lo(x0) * w, bf16hi(x0) * w);
    x1 = pack_bf16(bf16lo(x1) * w, bf16hi(x1) * w);
    x2 = pack_bf16(bf16lo(x2) * w, bf16hi(x2) * w);
    x3 = pack_bf16(bf16lo(x3) * w, bf16hi(x3) * w);
    st_shared_v4(addr, x0, x1, x2, x3);
  }
}

// Store 32 fp32 values (columns 32c .. 32c+31 of `row`) as bf16 into an SW128 tile.
__device__ __forceinline__ void store_row_chunk_bf16(uint32_t tile, uint32_t row, uint32_t c,
                                                     const float (&x)[32]) {
#pragma unroll
  for (uint32_t q = 0; q < 4; ++q) {
    st_shared_v4(tile + sw128_offset(row, 4 * c + q), pack_bf16(x[8 * q + 0], x[8 * q + 1]),
                 pack_bf16(x[8 * q + 2], x[8 * q + 3]), pack_bf16(x[8 * q + 4], x[8 * q + 5]),
                 pack_bf16(x[8 * q + 6], x[8 * q + 7]));
  }
}

__device__ __forceinline__ void ld_chunk(uint32_t taddr, float (&x)[32]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
}

// ============================================================================ segment aggregates
struct AggParams {
  int B, H, T, L, G, nitems, reverse;
  const float *decay;
  float *out;
  int *status;
};

template <bool DECAY>
__global__ void __launch_bounds__(kThreads, 1)
    tc_agg_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap my,
                  AggParams P) {
  constexpr int NS = 3;              // stages of (X tile, Y tile)
  constexpr uint32_t kStage = 2 * kTileBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NS * kStage);
  uint64_t *full = bars, *scaled = bars + NS, *empty = bars + 2 * NS;
  uint64_t *accf = bars + 3 * NS, *acce = accf + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(acce + 2);
  __shared__ int abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int BH = P.B * P.H;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&scaled[s], 128);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf[a], 1);
      mbar_init(&acce[a], 128);
    }
    fence_mbar_init();
    prefetch_tensormap(&mx);
    prefetch_tensormap(&my);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < P.nitems && ok; item += gridDim.x) {
        const int g = item / BH, bh = item % BH, b = bh / P.H, h = bh % P.H;
        const int s0 = g * P.L, s1 = min(P.T, s0 + P.L);
        for (int t0 = s0; t0 < s1; t0 += 128, ++it) {
          const int s = it % NS, u = it / NS;
          if (u > 0 && !(ok = mbar_wait(&empty[s], (u - 1) & 1, &abort_flag, P.status))) break;
          uint8_t *xs = smem + s * kStage;
          mbar_arrive_expect_tx(&full[s], kStage);
          tma_load_4d(&mx, &full[s], xs, 0, t0, h, b, kPolicyEvictFirst);
          tma_load_4d(&mx, &full[s], xs + kTileHalfBytes, 64, t0, h, b, kPolicyEvictFirst);
          tma_load_4d(&my, &full[s], xs + kTileBytes, 0, t0, h, b, kPolicyEvictFirst);
          tma_load_4d(&my, &full[s], xs + kTileBytes + kTileHalfBytes, 64, t0, h, b, kPolicyEvictFirst);
        }
      }
      // never leave with copies in flight: wait (time-bounded, even after an
      // abort) for the last load of every stage
      volatile int no_abort = 0;
      for (int s = 0; s < NS; ++s) {
        const int uses = it > s ? (it - 1 - s) / NS + 1 : 0;
        if (uses > 0) mbar_wait(&full[s], (uses - 1) & 1, &no_abort, P.status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, ai = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16(128, 128, true, true);
      for (int item = blockIdx.x; item < P.nitems && ok; item += gridDim.x) {
        const int g = item / BH;
        const int s0 = g * P.L, s1 = min(P.T, s0 + P.L);
        const int a = ai & 1, ua = ai >> 1;
        if (ua > 0 && !(ok = mbar_wait(&acce[a], (ua - 1) & 1, &abort_flag, P.status))) break;
        tc_fence_after();
        const uint32_t dt = tmem + a * 128;
        bool first = true;
        for (int t0 = s0; t0 < s1; t0 += 128, ++it) {
          const int s = it % NS, u = it / NS;
          if (!(ok = mbar_wait(DECAY ? &scaled[s] : &full[s], u & 1, &abort_flag, P.status))) break;
          tc_fence_after();
          const uint32_t xs = smem_u32(smem + s * kStage), ys = xs + kTileBytes;
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks)
            mma_ss(dt, desc_mnmajor(xs, ks), desc_mnmajor(ys, ks), idesc, (first && ks == 0) ? 0u : 1u);
          first = false;
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&accf[a]);
        ++ai;
      }
    }
  } else if (warp >= 4 && warp < 8) {
    if (DECAY) {
      // scale X rows in place by the token weights before the MMA reads them
      const uint32_t row = threadIdx.x - 128;
      int it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < P.nitems && ok; item += gridDim.x) {
        const int g = item / BH, h = (item % BH) % P.H;
        const int s0 = g * P.L, s1 = min(P.T, s0 + P.L);
        const float l2 = log2f(P.decay[h]);
        for (int t0 = s0; t0 < s1; t0 += 128, ++it) {
          const int s = it % NS, u = it / NS;
          if (!(ok = mbar_wait(&full[s], u & 1, &abort_flag, P.status))) break;
          const int tok = t0 + (int)row;
          float w = 0.f;
          if (tok < s1) w = exp2f(l2 * (float)(P.reverse ? (tok - s0 + 1) : (s1 - 1 - tok)));
          scale_tile_row(smem_u32(smem + s * kStage), row, w);
          fence_proxy_async_smem();
          mbar_arrive(&scaled[s]);
        }
      }
    }
  } else if (warp >= 8) {
    const uint32_t quad = warp & 3, row = quad * 32 + lane;
    int ai = 0;
    for (int item = blockIdx.x; item < P.nitems; item += gridDim.x, ++ai) {
      const int g = item / BH, bh = item % BH;
      const int a = ai & 1, ua = ai >> 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&accf[a], ua & 1, &abort_flag, P.status))) break;
      tc_fence_after();
      float *dst = P.out + ((int64_t)g * BH + bh) * 16384 + row * 128;
#pragma unroll 1
      for (uint32_t c = 0; c < 4; ++c) {
        float x[32];
        ld_chunk(tmem + a * 128 + ((quad * 32) << 16) + c * 32, x);
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4 *>(dst + c * 32 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
      }
      tc_fence_before();
      mbar_arrive(&acce[a]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// ============================================================================ per-group chunked kernel
struct MainParams {
  int B, H, T, L, G, nitems, init_t;
  const float *decay;
  const float *ginit;  // not fused: exclusive state of every group [G][BH][d][d]
  const float *init;   // fused: state before the first group of the chain [BH][d][d], or null
  float *final_state;  // forward: state after the last token [BH][d][d], or null
  float *dinit;        // fused reverse: state one step before the first token [BH][d][d], or null
  float *states_out;   // fused: exclusive state of every group [G][BH][d][d], or null
  float *agg, *incl;   // fused: look-back aggregates / inclusive prefixes [G][BH][d][d]
  unsigned *flags;     // fused: [G][BH] 0 empty, 1 aggregate, 2 inclusive (zeroed before launch)
  int *status;
};

constexpr int kSlots = 5;
constexpr uint32_t kOffPs = kSlots * kTileBytes;          // P (then O staging) tile
constexpr uint32_t kOffSh = kOffPs + kTileBytes;          // bf16 state tile
constexpr uint32_t kOffBar = kOffSh + kTileBytes;
constexpr size_t kMainSmem = kOffBar + 256 + 1024;

// barrier indices
enum { B_FULL = 0, B_EMPTY = kSlots, B_PFULL = 2 * kSlots, B_PEMPTY, B_OFULL, B_OEMPTY, B_SFULL, B_PRE,
       B_PSFULL, B_UFULL, B_UEMPTY, B_SCALED, B_K1FULL = B_SCALED + 4, B_COUNT = B_K1FULL + 4 };
static_assert(B_COUNT * 8 + 4 <= 256, "barrier area");

// Decay mask of one 32-column chunk of a score row: keep j <= i (causal) or
// j >= i (anti-causal) and weight by lambda^{|i-j|}; walks j so that the
// weight only ever shrinks (no overflow for any lambda in (0, 1]).
template <bool DECAY, bool REV>
__device__ __forceinline__ void mask_chunk(float (&x)[32], int i, int c, float lam, float l2) {
  if (!DECAY) {
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const int j = c * 32 + jj;
      x[jj] = (REV ? (j >= i) : (j <= i)) ? x[jj] : 0.f;
    }
    return;
  }
  if (!REV) {
    const int e0 = i - (c * 32 + 31);  // exponent at jj = 31
    float w = e0 >= 0 ? exp2f(l2 * (float)e0) : 0.f;
#pragma unroll
    for (int jj = 31; jj >= 0; --jj) {
      const int j = c * 32 + jj;
      if (j == i) w = 1.f;
      x[jj] = (j <= i) ? x[jj] * w : 0.f;
      w *= lam;
    }
  } else {
    const int e0 = c * 32 - i;  // exponent at jj = 0
    float w = e0 >= 0 ? exp2f(l2 * (float)e0) : 0.f;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const int j = c * 32 + jj;
      if (j == i) w = 1.f;
      x[jj] = (j >= i) ? x[jj] * w : 0.f;
      w *= lam;
    }
  }
}

// One work item: group g of sequence bh (tokens [s0, s1), nb 128-token blocks).
// Fused reverse-time launches walk the groups from the end so that every
// look-back predecessor (g + 1) is taken before its successor.
struct Item {
  int g, bh, b, h, s0, s1, nb;
};
template <bool REV, bool FUSED>
__device__ __forceinline__ Item item_of(const MainParams &P, int item) {
  const int BH = P.B * P.H;
  Item it;
  const int gi = item / BH;
  it.g = (FUSED && REV) ? P.G - 1 - gi : gi;
  it.bh = item % BH;
  it.b = it.bh / P.H;
  it.h = it.bh % P.H;
  it.s0 = it.g * P.L;
  it.s1 = min(P.T, it.s0 + P.L);
  it.nb = (it.s1 - it.s0 + 127) / 128;
  return it;
}
// fused: does the group hand a prefix to a successor, and does it need its own aggregate?
template <bool REV>
__device__ __forceinline__ bool has_succ(const MainParams &P, int g) { return REV ? g > 0 : g < P.G - 1; }
template <bool REV, bool FUSED>
__device__ __forceinline__ bool has_pass1(const MainParams &P, int g) {
  return FUSED && (has_succ<REV>(P, g) || (REV && g == 0 && P.dinit != nullptr));
}

template <bool DECAY, bool REV, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
    tc_main_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo,
                   MainParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + B_COUNT);
  __shared__ int abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int BH = P.B * P.H;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bar[B_FULL + s], 1);
      mbar_init(&bar[B_EMPTY + s], 1);
    }
    mbar_init(&bar[B_PFULL], 1);
    mbar_init(&bar[B_PEMPTY], 128);
    mbar_init(&bar[B_OFULL], 1);
    mbar_init(&bar[B_OEMPTY], 128);
    mbar_init(&bar[B_SFULL], 1);
    mbar_init(&bar[B_PRE], 128);
    mbar_init(&bar[B_PSFULL], 128);
    mbar_init(&bar[B_UFULL], 1);
    mbar_init(&bar[B_UEMPTY], 128);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar[B_SCALED + s], 64);
      mbar_init(&bar[B_K1FULL + s], 1);
    }
    fence_mbar_init();
    prefetch_tensormap(&mq);
    prefetch_tensormap(&mk);
    prefetch_tensormap(&mv);
    prefetch_tensormap(&mo);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tS = tmem, tP = tmem + 128, tO = tmem + 256, tU = tmem + 384;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sPs = sbase + kOffPs, sSh = sbase + kOffSh;
  auto slot_addr = [&](int t) { return sbase + (uint32_t)(t % kSlots) * kTileBytes; };
  // token offset of block n of pass 2 (walk order) and of pass 1 (the opposite
  // order, so pass 2 starts on the tiles pass 1 touched last)
  auto p2_t0 = [&](const Item &it, int n) { return it.s0 + 128 * (REV ? it.nb - 1 - n : n); };
  auto p1_t0 = [&](const Item &it, int n) { return it.s0 + 128 * (REV ? n : it.nb - 1 - n); };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int tc = 0, k1 = 0;
      bool ok = true;
      // With decay, pass-1 key tiles are completed on their own barrier ring
      // (K1FULL, indexed by the pass-1 key tile count): the weight warps wait on
      // every phase of that ring in order, never on a slot's FULL barrier whose
      // phases also advance with tiles they skip (a parity wait is only sound
      // one phase ahead).  The slot's FULL barrier gets a plain arrive so that
      // its phase count stays in step with the slot's uses.
      auto load = [&](const CUtensorMap *m, int t0, const Item &it, uint64_t policy, bool k1tile) -> bool {
        const int t = tc++, s = t % kSlots, u = t / kSlots;
        if (u > 0 && !mbar_wait(&bar[B_EMPTY + s], (u - 1) & 1, &abort_flag, P.status,
                                P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr))
          return false;
        uint8_t *dst = smem + s * kTileBytes;
        uint64_t *done = &bar[B_FULL + s];
        if (DECAY && FUSED && k1tile) {
          done = &bar[B_K1FULL + (k1 & 3)];
          ++k1;
          mbar_arrive(&bar[B_FULL + s]);
        }
        mbar_arrive_expect_tx(done, kTileBytes);
        tma_load_4d(m, done, dst, 0, t0, it.h, it.b, policy);
        tma_load_4d(m, done, dst + kTileHalfBytes, 64, t0, it.h, it.b, policy);
        return true;
      };
      for (int item = blockIdx.x; item < P.nitems && ok; item += gridDim.x) {
        const Item it = item_of<REV, FUSED>(P, item);
        if (has_pass1<REV, FUSED>(P, it.g))
          for (int n = 0; n < it.nb && ok; ++n)
            ok = load(&mk, p1_t0(it, n), it, kPolicyEvictLast, true) &&
                 load(&mv, p1_t0(it, n), it, kPolicyEvictLast, false);
        for (int n = 0; n < it.nb && ok; ++n) {
          const int t0 = p2_t0(it, n);
          ok = load(&mq, t0, it, kPolicyEvictFirst, false) && load(&mk, t0, it, kPolicyEvictFirst, false) &&
               load(&mv, t0, it, kPolicyEvictFirst, false);
        }
      }
      // time-bounded drain of the loads in flight (also after an abort)
      volatile int no_abort = 0;
      for (int s = 0; s < kSlots; ++s) {
        const int uses = tc > s ? (tc - 1 - s) / kSlots + 1 : 0;
        if (uses > 0) mbar_wait(&bar[B_FULL + s], (uses - 1) & 1, &no_abort, P.status);
      }
      for (int j = 0; j < 4; ++j) {
        const int uses = k1 > j ? (k1 - 1 - j) / 4 + 1 : 0;
        if (uses > 0) mbar_wait(&bar[B_K1FULL + j], (uses - 1) & 1, &no_abort, P.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16(128, 128, false, false);  // Q K^T
      const uint32_t id_qs = idesc_bf16(128, 128, false, true);   // Q S,  P V
      const uint32_t id_kv = idesc_bf16(128, 128, true, true);    // K^T V
      int tc = 0, blk = 0, ui = 0, k1 = 0;
      bool ok = true;
      auto full = [&](int t) {
        return mbar_wait(&bar[B_FULL + t % kSlots], (t / kSlots) & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr);
      };
      for (int item = blockIdx.x; item < P.nitems && ok; item += gridDim.x) {
        const Item it = item_of<REV, FUSED>(P, item);
        if (has_pass1<REV, FUSED>(P, it.g)) {
          // pass 1: the group's aggregate U = K'^T V into its own TMEM columns
          if (ui > 0 && !(ok = mbar_wait(&bar[B_UEMPTY], (ui - 1) & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr))) break;
          for (int n = 0; n < it.nb && ok; ++n) {
            const int tk = tc++, tv = tc++;
            ok = (DECAY ? mbar_wait(&bar[B_SCALED + (k1 & 3)], (k1 >> 2) & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr) : full(tk)) &&
                 full(tv);
            ++k1;
            if (!ok) break;
            tc_fence_after();
            const uint32_t K = slot_addr(tk), V = slot_addr(tv);
#pragma unroll
            for (uint32_t ks = 0; ks < 8; ++ks)
              mma_ss(tU, desc_mnmajor(K, ks), desc_mnmajor(V, ks), id_kv, (n > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&bar[B_EMPTY + tk % kSlots]);
            mma_commit(&bar[B_EMPTY + tv % kSlots]);
          }
          if (!ok) break;
          mma_commit(&bar[B_UFULL]);
          ++ui;
        }
        for (int n = 0; n < it.nb; ++n, ++blk) {
          const int tq = tc++, tk = tc++, tv = tc++;
          const uint32_t Q = slot_addr(tq), K = slot_addr(tk), V = slot_addr(tv);
          // scores: P = Q K^T
          ok = full(tq) && full(tk) &&
               (blk == 0 || mbar_wait(&bar[B_PEMPTY], (blk - 1) & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) mma_ss(tP, desc_kmajor(Q, ks), desc_kmajor(K, ks), id_qk, ks > 0);
          mma_commit(&bar[B_PFULL]);
          // inter-block term: O = Q' S   (Q' = decay-weighted rows)
          ok = mbar_wait(&bar[B_PRE], blk & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr) &&
               (blk == 0 || mbar_wait(&bar[B_OEMPTY], (blk - 1) & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) mma_ss(tO, desc_kmajor(Q, ks), desc_mnmajor(sSh, ks), id_qs, ks > 0);
          mma_commit(&bar[B_EMPTY + tq % kSlots]);
          // state update: S += K'^T V
          if (!(ok = full(tv))) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) mma_ss(tS, desc_mnmajor(K, ks), desc_mnmajor(V, ks), id_kv, 1u);
          mma_commit(&bar[B_EMPTY + tk % kSlots]);
          mma_commit(&bar[B_SFULL]);
          // intra-block term: O += P V
          if (!(ok = mbar_wait(&bar[B_PSFULL], blk & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr))) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) mma_ss(tO, desc_kmajor(sPs, ks), desc_mnmajor(V, ks), id_qs, 1u);
          mma_commit(&bar[B_EMPTY + tv % kSlots]);
          mma_commit(&bar[B_OFULL]);
        }
      }
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ pass-1 key weights (fused, decay)
    if (DECAY && FUSED) {
      const int t64 = threadIdx.x - 64;
      int tc = 0, k1 = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < P.nitems && ok; item += gridDim.x) {
        const Item it = item_of<REV, FUSED>(P, item);
        const float l2 = log2f(P.decay[it.h]);
        if (has_pass1<REV, FUSED>(P, it.g)) {
          for (int n = 0; n < it.nb; ++n) {
            const int tk = tc;
            tc += 2;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_K1FULL + (k1 & 3)], (k1 >> 2) & 1, &abort_flag,
                                                   P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr));
            if (!ok) break;
            const int t0 = p1_t0(it, n);
            for (int r = t64; r < 128; r += 64) {
              const int tok = t0 + r;
              // forward: lambda^{end - s};  reverse: lambda^{s - start + 1}
              const float w = tok < it.s1 ? exp2f(l2 * (float)(REV ? tok - it.s0 + 1 : it.s1 - 1 - tok)) : 0.f;
              scale_tile_row(slot_addr(tk), (uint32_t)r, w);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bar[B_SCALED + (k1 & 3)]);
            ++k1;
          }
        }
        tc += 3 * it.nb;
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ group A: scores and outputs
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    const bool leader = threadIdx.x == 128;
    int blk = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < P.nitems && ok; item += gridDim.x) {
      const Item it = item_of<REV, FUSED>(P, item);
      const float lam = DECAY ? P.decay[it.h] : 1.f;
      const float l2 = DECAY ? log2f(lam) : 0.f;
      for (int n = 0; n < it.nb; ++n, ++blk) {
        const int t0 = p2_t0(it, n);
        ok = group_all(mbar_wait(&bar[B_PFULL], blk & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr), 2, 128);
        if (!ok) break;
        tc_fence_after();
        // the P tile buffer is free once the previous output store has read it
        if (leader) bulk_wait_read_all();
        named_bar_sync(1, 128);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float x[32];
          ld_chunk(tP + lb + c * 32, x);
          mask_chunk<DECAY, REV>(x, (int)row, c, lam, l2);
          store_row_chunk_bf16(sPs, row, c, x);
        }
        tc_fence_before();
        mbar_arrive(&bar[B_PEMPTY]);
        fence_proxy_async_smem();
        mbar_arrive(&bar[B_PSFULL]);
        // outputs
        ok = group_all(mbar_wait(&bar[B_OFULL], blk & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr), 2, 128);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float x[32];
          ld_chunk(tO + lb + c * 32, x);
          store_row_chunk_bf16(sPs, row, c, x);
        }
        tc_fence_before();
        mbar_arrive(&bar[B_OEMPTY]);
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          tma_store_4d_hint(&mo, smem + kOffPs, 0, t0, it.h, it.b, kPolicyEvictFirst);
          tma_store_4d_hint(&mo, smem + kOffPs + kTileHalfBytes, 64, t0, it.h, it.b, kPolicyEvictFirst);
          bulk_commit();
        }
      }
    }
    if (leader) bulk_wait_all();
  } else if (warp >= 8) {
    // ------------------------------------------------------------ group B: state tile, look-back, decay weights
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    const bool leader = threadIdx.x == 256;
    int blk = 0, tc = 0, ui = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < P.nitems && ok; item += gridDim.x) {
      const Item it = item_of<REV, FUSED>(P, item);
      const int g = it.g, bh = it.bh;
      const bool p1 = has_pass1<REV, FUSED>(P, g);
      const int tc2 = tc + (p1 ? 2 * it.nb : 0);  // first pass-2 tile of the item
      tc = tc2 + 3 * it.nb;
      const float lam = DECAY ? P.decay[it.h] : 1.f;
      const float l2 = DECAY ? log2f(lam) : 0.f;
      auto nvalid = [&](int n) { return min(128, it.s1 - p2_t0(it, n)); };
      // Decay weights of pass-2 block n (global block counter bb) with nv valid rows:
      // forward q_i *= lambda^{i+1}, k_j *= lambda^{nv-1-j};
      // reverse q_i *= lambda^{nv-1-i}, k_j *= lambda^{j+1}.
      auto weigh = [&](int n, int bb) -> bool {
        if (!group_all(mbar_wait(&bar[B_PFULL], bb & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr), 3, 128)) return false;
        const int r = (int)row, nv = nvalid(n);
        float wq = 0.f, wk = 0.f;
        if (r < nv) {
          wq = exp2f(l2 * (float)(REV ? nv - 1 - r : r + 1));
          wk = exp2f(l2 * (float)(REV ? r + 1 : nv - 1 - r));
        }
        scale_tile_row(slot_addr(tc2 + 3 * n), row, wq);
        scale_tile_row(slot_addr(tc2 + 3 * n + 1), row, wk);
        return true;
      };
      const size_t gslot = ((size_t)g * BH + bh) * 16384 + (size_t)row * 128;
      // ---- the state entering the group
      const float dec0 = DECAY ? exp2f(l2 * (float)nvalid(0)) : 1.f;
      auto put_state = [&](int c, const float (&x)[32]) {
        store_row_chunk_bf16(sSh, row, c, x);
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j] * dec0);
        tmem_st32(tS + lb + c * 32, r);
      };
      if (!FUSED) {
        const float *src = P.ginit + gslot - (size_t)row * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float x[32];
          if (!P.init_t) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 v4 = __ldg(reinterpret_cast<const float4 *>(src + row * 128 + c * 32 + j));
              x[j] = v4.x; x[j + 1] = v4.y; x[j + 2] = v4.z; x[j + 3] = v4.w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __ldg(src + (c * 32 + j) * 128 + row);
          }
          put_state(c, x);
        }
      } else {
        const bool first = REV ? g == P.G - 1 : g == 0;
        const bool succ = has_succ<REV>(P, g);
        const float decL = DECAY ? exp2f(l2 * (float)(it.s1 - it.s0)) : 1.f;  // lambda^{group length}
        if (p1) {
          ok = group_all(mbar_wait(&bar[B_UFULL], ui & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr), 3, 128);
          if (!ok) break;
          tc_fence_after();
          if (succ && !first) {
            // publish the aggregate at once so that successors need not wait for this group's look-back
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              float u[32];
              ld_chunk(tU + lb + c * 32, u);
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(P.agg + gslot + c * 32 + j) = make_float4(u[j], u[j + 1], u[j + 2], u[j + 3]);
            }
            __threadfence();
            group_all(true, 3, 128);
            if (leader) st_release_gpu(P.flags + (size_t)g * BH + bh, 1u);
          }
        }
        // exclusive state: the chain's initial state, or a decoupled look-back over predecessors
        bool got = true;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float x[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = 0.f;
          if (first) {
            if (P.init) {
              const float *src = P.init + (size_t)bh * 16384;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                x[j] = P.init_t ? __ldg(src + (c * 32 + j) * 128 + row) : __ldg(src + row * 128 + c * 32 + j);
            }
          } else if (got) {
            float fac = 1.f;
            int pg = REV ? g + 1 : g - 1;
#pragma unroll 1
            while (true) {
              const unsigned f = wait_flag(P.flags + (size_t)pg * BH + bh, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr);
              if (f == 0) {
                got = false;
                break;
              }
              const float *src = (f == 2 ? P.incl : P.agg) + ((size_t)pg * BH + bh) * 16384 + (size_t)row * 128 + c * 32;
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                const float4 v4 = __ldcg(reinterpret_cast<const float4 *>(src + j));
                x[j] = fmaf(fac, v4.x, x[j]);
                x[j + 1] = fmaf(fac, v4.y, x[j + 1]);
                x[j + 2] = fmaf(fac, v4.z, x[j + 2]);
                x[j + 3] = fmaf(fac, v4.w, x[j + 3]);
              }
              if (f == 2) break;
              if (DECAY) fac *= exp2f(l2 * (float)(min(P.T, (pg + 1) * P.L) - pg * P.L));
              pg = REV ? pg + 1 : pg - 1;
            }
          }
          if (P.states_out) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4 *>(P.states_out + gslot + c * 32 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
          }
          if (p1) {
            // inclusive prefix handed on: lambda^{L_g} S + U
            float u[32];
            ld_chunk(tU + lb + c * 32, u);
#pragma unroll
            for (int j = 0; j < 32; ++j) u[j] = fmaf(decL, x[j], u[j]);
            float *dst = succ ? P.incl + gslot : (P.dinit + (size_t)bh * 16384 + (size_t)row * 128);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4 *>(dst + c * 32 + j) = make_float4(u[j], u[j + 1], u[j + 2], u[j + 3]);
          }
          put_state(c, x);
        }
        ok = group_all(got, 3, 128);
        if (!ok) break;
        if (p1) {
          tc_fence_before();
          mbar_arrive(&bar[B_UEMPTY]);
          ++ui;
        }
        if (succ) {
          __threadfence();
          group_all(true, 3, 128);
          if (leader) st_release_gpu(P.flags + (size_t)g * BH + bh, 2u);
        }
      }
      tmem_st_wait();
      if (DECAY && !(ok = weigh(0, blk))) break;
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&bar[B_PRE]);
      for (int n = 0; n < it.nb; ++n, ++blk) {
        ok = group_all(mbar_wait(&bar[B_SFULL], blk & 1, &abort_flag, P.status, P.status ? P.status + 1 + (threadIdx.x / 32) : nullptr), 3, 128);
        if (!ok) break;
        tc_fence_after();
        if (n + 1 < it.nb) {
          const float dec = DECAY ? exp2f(l2 * (float)nvalid(n + 1)) : 1.f;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float x[32];
            ld_chunk(tS + lb + c * 32, x);
            store_row_chunk_bf16(sSh, row, c, x);
            if (DECAY) {
              uint32_t r[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j] * dec);
              tmem_st32(tS + lb + c * 32, r);
            }
          }
          if (DECAY) tmem_st_wait();
          if (DECAY && !(ok = weigh(n + 1, blk + 1))) break;
          tc_fence_before();
          fence_proxy_async_smem();
          mbar_arrive(&bar[B_PRE]);
        } else if (P.final_state && !REV && g == P.G - 1) {
          float *dst = P.final_state + (int64_t)bh * 16384 + row * 128;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float x[32];
            ld_chunk(tS + lb + c * 32, x);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4 *>(dst + c * 32 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
          }
          tc_fence_before();
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

bool seq_tmap(const Problem &p, const void *base, CUtensorMap *m) {
  const uint64_t dims[4] = {(uint64_t)p.d, (uint64_t)p.T, (uint64_t)p.H, (uint64_t)p.B};
  const uint64_t strides[3] = {(uint64_t)p.st * 2, (uint64_t)p.sh * 2, (uint64_t)p.sb * 2};
  return make_tmap_bf16(m, base, dims, strides);
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t tc_segment_states(const Problem &p, int seg_len, const void *X, const void *Y, bool reverse,
                              float *out, int *status, cudaStream_t s) {
  alignas(64) CUtensorMap mx, my;
  if (!seq_tmap(p, X, &mx) || !seq_tmap(p, Y, &my)) return cudaErrorInvalidValue;
  AggParams A;
  A.B = p.B; A.H = p.H; A.T = p.T; A.L = seg_len;
  A.G = (p.T + seg_len - 1) / seg_len;
  A.nitems = A.G * p.B * p.H;
  A.reverse = reverse ? 1 : 0;
  A.decay = p.decay; A.out = out; A.status = status;
  const size_t smem = 3 * 2 * kTileBytes + 1024 + 256;
  const int grid = A.nitems < p.num_sms ? A.nitems : p.num_sms;
  cudaError_t e;
  TimedLaunch t(K_TC_AGG, s);
  if (p.decay) {
    if ((e = set_smem(tc_agg_kernel<true>, smem)) != cudaSuccess) return e;
    tc_agg_kernel<true><<<grid, kThreads, smem, s>>>(mx, my, A);
  } else {
    if ((e = set_smem(tc_agg_kernel<false>, smem)) != cudaSuccess) return e;
    tc_agg_kernel<false><<<grid, kThreads, smem, s>>>(mx, my, A);
  }
  return cudaGetLastError();
}

namespace {
MainParams main_params(const Problem &p, int group_len, bool init_transposed, int *status) {
  MainParams M = {};
  M.B = p.B; M.H = p.H; M.T = p.T; M.L = group_len;
  M.G = (p.T + group_len - 1) / group_len;
  M.nitems = M.G * p.B * p.H;
  M.init_t = init_transposed ? 1 : 0;
  M.decay = p.decay;
  M.status = status;
  return M;
}

template <bool FUSED>
cudaError_t launch_main(const Problem &p, bool reverse, const CUtensorMap &mq, const CUtensorMap &mk,
                        const CUtensorMap &mv, const CUtensorMap &mo, const MainParams &M, cudaStream_t s) {
  const int grid = M.nitems < p.num_sms ? M.nitems : p.num_sms;
  cudaError_t e;
  TimedLaunch t(FUSED ? (reverse ? K_TC_FUSED_REV : K_TC_FUSED_FWD) : (reverse ? K_TC_MAIN_REV : K_TC_MAIN_FWD), s);
#define LINATTN_LAUNCH_MAIN(DEC, REV)                                                      \
  do {                                                                                     \
    if ((e = set_smem(tc_main_kernel<DEC, REV, FUSED>, kMainSmem)) != cudaSuccess) return e; \
    tc_main_kernel<DEC, REV, FUSED><<<grid, kThreads, kMainSmem, s>>>(mq, mk, mv, mo, M);   \
  } while (0)
  if (p.decay) {
    if (reverse) LINATTN_LAUNCH_MAIN(true, true); else LINATTN_LAUNCH_MAIN(true, false);
  } else {
    if (reverse) LINATTN_LAUNCH_MAIN(false, true); else LINATTN_LAUNCH_MAIN(false, false);
  }
#undef LINATTN_LAUNCH_MAIN
  return cudaGetLastError();
}

bool seq_tmaps(const Problem &p, const void *q, const void *k, const void *v, const void *o, CUtensorMap *m) {
  return seq_tmap(p, q, &m[0]) && seq_tmap(p, k, &m[1]) && seq_tmap(p, v, &m[2]) && seq_tmap(p, o, &m[3]);
}
}  // namespace

cudaError_t tc_main(const Problem &p, int group_len, bool reverse, const void *q, const void *k,
                    const void *v, void *o, const float *group_init, bool init_transposed,
                    float *final_state, int *status, cudaStream_t s) {
  alignas(64) CUtensorMap m[4];
  if (!seq_tmaps(p, q, k, v, o, m)) return cudaErrorInvalidValue;
  MainParams M = main_params(p, group_len, init_transposed, status);
  M.ginit = group_init;
  M.final_state = final_state;
  return launch_main<false>(p, reverse, m[0], m[1], m[2], m[3], M, s);
}

int tc_fused_group_len(const Problem &p) {
  // Short groups keep pass 1's tiles in L2 until pass 2 re-reads them; long
  // groups make the 64 KiB look-back states cheap next to the group's data.
  int L = 1024;
  if (const char *env = getenv("LINATTN_GROUP_LEN")) {
    const int v = atoi(env);
    if (v >= 128 && v % 128 == 0) L = v;
  }
  const int64_t BH = (int64_t)p.B * p.H;
  while (L > 256 && ((p.T + L - 1) / L) * BH < 2 * (int64_t)p.num_sms) L /= 2;
  const int Tr = (p.T + 127) / 128 * 128;
  return L < Tr ? L : Tr;
}

size_t tc_fused_scratch_bytes(const Problem &p, int group_len) {
  const size_t items = (size_t)((p.T + group_len - 1) / group_len) * p.B * p.H;
  return align256(items * 4) + 2 * align256(items * 16384 * sizeof(float));
}

cudaError_t tc_fused(const Problem &p, int group_len, bool reverse, const void *q, const void *k,
                     const void *v, void *o, const float *init, bool init_transposed, float *final_state,
                     float *dinit, float *states_out, void *scratch, int *status, cudaStream_t s) {
  alignas(64) CUtensorMap m[4];
  if (!seq_tmaps(p, q, k, v, o, m)) return cudaErrorInvalidValue;
  MainParams M = main_params(p, group_len, init_transposed, status);
  const size_t items = (size_t)M.nitems;
  char *w = static_cast<char *>(scratch);
  M.flags = reinterpret_cast<unsigned *>(w);
  M.agg = reinterpret_cast<float *>(w + align256(items * 4));
  M.incl = reinterpret_cast<float *>(w + align256(items * 4) + align256(items * 16384 * sizeof(float)));
  M.init = init;
  M.final_state = final_state;
  M.dinit = dinit;
  M.states_out = states_out;
  cudaError_t e = cudaMemsetAsync(M.flags, 0, items * 4, s);
  if (e != cudaSuccess) return e;
  return launch_main<true>(p, reverse, m[0], m[1], m[2], m[3], M, s);
}

}  // namespace linattn
