// Tensor-core kernels (tcgen05 + TMEM + TMA) for bf16 sequences with d = 128.
//
// The kernels are persistent (one CTA per SM; (group, sequence) items drawn
// at run time, see ItemRing) and warp-specialised:
//   warp 0        TMA producer and item drawer (one thread)
//   warp 1        TMEM allocator and MMA issuer (the whole warp runs the issue
//                 loop, one elected lane issues each product; see mma_ss_warp)
//   warps 4..7    epilogue group A (TMEM -> registers -> shared / global)
//   warps 8..11   epilogue group B
// Every wait is a bounded mbarrier wait (see ptx.cuh); a timeout records an
// error in the status word and unwinds the kernel instead of hanging.
//
// A "block" is 128 tokens, i.e. two chunks of 64: the M = 128 tcgen05 MMA is
// the natural tile, and chunking at 128 instead of 64 changes only the
// rounding order (the chunked form equals the definition for any chunk
// length).  All operands are SW128 tiles (ptx.cuh).
#include <algorithm>

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace linattn {

bool tc_supported(const Problem &p) { return p.dtype == 0 && p.d == 128 && p.T >= 1; }

// The tail of short groups (tc_group_plan): the last kTailNum / kTailDen of a
// sequence in groups of L / kTailDiv tokens, from kTailMinWaves waves of items.
constexpr int kTailNum = 1, kTailDen = 10, kTailDiv = 2, kTailMinWaves = 3;

GroupPlan tc_group_plan(const Problem &p, int max_len) {
  // The persistent kernels hand out whole (group, sequence) items, so a launch
  // lasts about ceil(items / SMs) waves of one item each.  Pick the group count
  // G (at most 256 per sequence: the scan's column-parallel form) whose group
  // length L (a multiple of 128 tokens, at least 256) minimises
  //     waves(G) * (L / 128 + 1),
  // the "+ 1" standing for an item's fixed cost (its entering state, its
  // outputs at the end) in units of one 128-token block.  Ties go to longer
  // groups (fewer states).
  const int64_t BH = (int64_t)p.B * p.H, T = p.T, sms = p.num_sms > 0 ? p.num_sms : 1;
  const int64_t cap = max_len > 0 ? std::max<int64_t>(max_len, ((T + 255) / 256 + 127) / 128 * 128) : 0;
  int64_t bestL = 0, bestCost = 0;
  for (int64_t G = 1; G <= 256; ++G) {
    int64_t L = ((T + G - 1) / G + 127) / 128 * 128;
    if (L < 256) L = 256;
    const int64_t Ge = (T + L - 1) / L;
    if (Ge > 256 || (cap && L > cap)) continue;
    const int64_t waves = (BH * Ge + sms - 1) / sms;
    const int64_t cost = waves * (L / 128 + 1);
    if (bestL == 0 || cost < bestCost || (cost == bestCost && L > bestL)) {
      bestL = L;
      bestCost = cost;
    }
  }
  // (G = 256 always qualifies, so bestL is set)
  const int64_t Tr = (T + 127) / 128 * 128;
  const int L = (int)(bestL < Tr ? bestL : Tr);
  GroupPlan gp = GroupPlan::uniform((int)T, L);
  // CTAs do not all stream at the same rate (measured with a fixed share of
  // items per CTA: the last CTA of a launch ended up to 15 % after the median
  // one).  With items drawn at run time, cutting the last tenth of every
  // sequence into groups of half the length lets the faster CTAs take the short
  // items at the end.  Worth it only with several waves of items.
  const int64_t waves = (BH * gp.G + sms - 1) / sms;
  if (waves < kTailMinWaves) return gp;
  const int Ls = std::max(256, (L / kTailDiv + 127) / 128 * 128);
  const int kb = (int)(T * (kTailDen - kTailNum) / ((int64_t)kTailDen * L));
  if (Ls >= L || kb < 1) return gp;
  const int64_t rest = T - (int64_t)kb * L, Gs = (rest + Ls - 1) / Ls;
  if (kb + Gs > 256) return gp;
  gp.G = kb + (int)Gs;
  gp.kb = kb;
  gp.Ls = Ls;
  return gp;
}

namespace {

constexpr int kThreads = 384;

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ---------------------------------------------------------------------------- item order
// The (group, sequence) items of a persistent launch are handed out at run
// time: the producer thread draws the CTA's next item from a counter in global
// memory when it is ready to load it, and posts it in a small shared ring that
// every warp role reads in the same order (-1: no items left).  CTAs on SMs
// that get more memory bandwidth draw more items, instead of every CTA waiting
// for the slowest one's fixed share.  The last CTA of a launch to finish sets
// the counters back to zero for the next launch on the stream (items_done).
constexpr int kRing = 4;
struct ItemRing {
  int *item;        // [kRing]
  uint64_t *full;   // [kRing]: one arrival, the producer's
  uint64_t *empty;  // [kRing]: one arrival per reading thread
};

__device__ __forceinline__ void ring_init(const ItemRing &r, int readers) {
  for (int i = 0; i < kRing; ++i) {
    mbar_init(&r.full[i], 1);
    mbar_init(&r.empty[i], readers);
  }
}

struct NoSkip {
  __device__ bool operator()(int) const { return false; }
};

// Producer: draw and post this CTA's k-th item (items for which skip() holds
// are drawn and passed over).  False if a wait gave up.
template <class Skip = NoSkip>
__device__ __forceinline__ bool ring_post(const ItemRing &r, int k, int *counter, int nitems, int &item,
                                          volatile int *abort_flag, int *status, int *detail,
                                          Skip skip = Skip()) {
  const int s = k % kRing;
  if (k >= kRing && !mbar_wait(&r.empty[s], (k / kRing - 1) & 1, abort_flag, status, detail)) return false;
  int x = atomicAdd(counter, 1);
  while (x < nitems && skip(x)) x = atomicAdd(counter, 1);
  item = x < nitems ? x : -1;
  *reinterpret_cast<volatile int *>(&r.item[s]) = item;
  mbar_arrive(&r.full[s]);  // release: the item is visible to the readers of the phase
  return true;
}

// Reader: this CTA's k-th item.  False if the wait gave up.
__device__ __forceinline__ bool ring_take(const ItemRing &r, int k, int &item, volatile int *abort_flag,
                                          int *status, int *detail) {
  const int s = k % kRing;
  if (!mbar_wait(&r.full[s], (k / kRing) & 1, abort_flag, status, detail)) return false;
  item = *reinterpret_cast<volatile int *>(&r.item[s]);
  mbar_arrive(&r.empty[s]);
  return true;
}

// End of a CTA (after its last barrier): counter[0] counts items drawn,
// counter[1] finished CTAs; the last CTA out zeroes both.
__device__ __forceinline__ void items_done(int *counter) {
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(counter + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(counter, 0);
      atomicExch(counter + 1, 0);
    }
  }
}

// Per-head decays lambda >= kWeightedMin take the weighted-operand forms of
// the chunked kernels (rows weighted in shared memory, masks that reduce to a
// 0/1 pattern times one scalar per block, output rows weighted in the store):
// the mask scalars and the row weights then stay within lambda^{+-256}, i.e.
// 2^{+-83} at 0.8.  (The reverse aggregates' token weights lambda^{s-start+1}
// may underflow deep into a group, as they do in the aggregate kernel: those
// terms are far below the fp32 resolution of the group's first ones.)
constexpr float kWeightedMin = 0.8f;

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
  int B, H, T, nitems, reverse;
  GroupPlan gp;
  const float *decay;
  float *out;
  int *status;
  int *counter;  // [2] item counter and finished CTAs (zero at launch)
  const float *gC, *gtot;  // gates: group-local log2 cumulative sums [BH][T], group totals [G][BH]
  int skip_weighted;       // pass over the items of the weighted form (the dq pass has them): heads with
                           // lambda >= kWeightedMin, or gated items flagged in gflag
  const int *gflag;        // gates: per item [G][BH], nonzero for the weighted form
  int dout;                // rows and columns of the stored states: 128, or 64 (top-left blocks)
};

// GATE (with DECAY): token weights from the gates' cumulative sums instead of
// powers of lambda: exp2(tot_g - C_s) (forward), exp2(C_s) (reverse).
template <bool DECAY, bool GATE = false>
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
  __shared__ int ring_item[kRing];
  __shared__ uint64_t ring_bar[2 * kRing];
  const ItemRing ring{ring_item, ring_bar, ring_bar + kRing};
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int BH = P.B * P.H;
  int *const detail = P.status ? P.status + 1 + warp : nullptr;  // which wait gave up, per warp role

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
    ring_init(ring, 32 + (DECAY ? 128 : 0) + 128);  // readers: MMA warp, scaling warps, store warps
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
  // barriers, ring, TMEM and tensor maps are set up: wait for the kernel before on
  // the stream (its outputs are this kernel's inputs), then let the next one start
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int k = 0, item; ok; ++k) {
        auto skip = [&](int x) {
          if (!DECAY || !P.skip_weighted) return false;
          return GATE ? (P.gflag && P.gflag[x] != 0) : P.decay[(x % BH) % P.H] >= kWeightedMin;
        };
        if (!(ok = ring_post(ring, k, P.counter, P.nitems, item, &abort_flag, P.status, detail, skip)) || item < 0)
          break;
        const int g = item / BH, bh = item % BH, b = bh / P.H, h = bh % P.H;
        const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1));
        for (int t0 = s0; t0 < s1; t0 += 128, ++it) {
          const int s = it % NS, u = it / NS;
          if (u > 0 && !(ok = mbar_wait(&empty[s], (u - 1) & 1, &abort_flag, P.status, detail))) break;
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
    {  // the whole warp: one elected lane issues each product
      int it = 0, ai = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16(128, 128, true, true);
      for (int k = 0, item; ok; ++k) {
        if (!(ok = __all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail))) || item < 0) break;
        const int g = item / BH;
        const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1));
        const int a = ai & 1, ua = ai >> 1;
        if (ua > 0 && !(ok = mbar_wait_w(&acce[a], (ua - 1) & 1, &abort_flag, P.status, detail))) break;
        tc_fence_after();
        const uint32_t dt = tmem + a * 128;
        bool first = true;
        for (int t0 = s0; t0 < s1; t0 += 128, ++it) {
          const int s = it % NS, u = it / NS;
          if (!(ok = mbar_wait_w(DECAY ? &scaled[s] : &full[s], u & 1, &abort_flag, P.status, detail))) break;
          tc_fence_after();
          const uint32_t xs = smem_u32(smem + s * kStage), ys = xs + kTileBytes;
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks)
            mma_ss_warp(dt, desc_mnmajor(xs, ks), desc_mnmajor(ys, ks), idesc, (first && ks == 0) ? 0u : 1u);
          first = false;
          mma_commit_warp(&empty[s]);
        }
        if (!ok) break;
        mma_commit_warp(&accf[a]);
        ++ai;
      }
    }
  } else if (warp >= 4 && warp < 8) {
    if (DECAY) {
      // scale X rows in place by the token weights before the MMA reads them
      const uint32_t row = threadIdx.x - 128;
      int it = 0;
      bool ok = true;
      for (int k = 0, item; ok; ++k) {
        if (!(ok = __all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail))) || item < 0)
          break;
        const int g = item / BH, bh = item % BH, h = bh % P.H;
        const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1));
        const float l2 = GATE ? 0.f : log2f(P.decay[h]);
        const float *gc = GATE ? P.gC + (int64_t)bh * P.T : nullptr;
        const float gt = GATE ? P.gtot[(int64_t)g * BH + bh] : 0.f;
        for (int t0 = s0; t0 < s1; t0 += 128, ++it) {
          const int s = it % NS, u = it / NS;
          const int tok = t0 + (int)row;
          const float ct = (GATE && tok < s1) ? gc[tok] : 0.f;  // load before the wait
          if (!(ok = mbar_wait(&full[s], u & 1, &abort_flag, P.status, detail))) break;
          float w = 0.f;
          if (tok < s1)
            w = GATE ? exp2f(P.reverse ? ct : gt - ct)
                     : exp2f(l2 * (float)(P.reverse ? (tok - s0 + 1) : (s1 - 1 - tok)));
          scale_tile_row(smem_u32(smem + s * kStage), row, w);
          fence_proxy_async_smem();
          mbar_arrive(&scaled[s]);
        }
      }
    }
  } else if (warp >= 8) {
    const uint32_t quad = warp & 3, row = quad * 32 + lane;
    int ai = 0;
    for (int k = 0, item;; ++k, ++ai) {
      if (!__all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail)) || item < 0) break;
      const int g = item / BH, bh = item % BH;
      const int a = ai & 1, ua = ai >> 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&accf[a], ua & 1, &abort_flag, P.status, detail))) break;
      tc_fence_after();
      const int dout = P.dout;
      float *dst = P.out + ((int64_t)g * BH + bh) * dout * dout + (int64_t)row * dout;
#pragma unroll 1
      for (uint32_t c = 0; c < 4; ++c) {
        float x[32];
        ld_chunk(tmem + a * 128 + ((quad * 32) << 16) + c * 32, x);
        if ((int)row < dout && (int)c * 32 < dout) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4 *>(dst + c * 32 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&acce[a]);
    }
  }
  tc_fence_before();
  __syncthreads();
  items_done(P.counter);
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// ============================================================================ per-chunk states
// The exclusive state entering every chunk of C = 64 tokens, [B][H][ceil(T/64)][d][d]
// fp32: per (group, sequence) item, from the state entering the group (the scan's
// output), walking the group's chunks in order:
//   out[c] = S;   S <- lambda^64 S + (diag(lambda^{63-j}) K_c)^T V_c   (j: row in the chunk)
// The state stays in TMEM; each chunk's product contracts over the 64 rows of its
// half of the 128-token tile (four K = 16 steps).  The last chunk of a group needs
// no product (the next group starts from its own scanned state).
struct ChunkParams {
  int B, H, T, nitems, nch;  // nch = ceil(T / 64) chunks per sequence
  GroupPlan gp;
  const float *decay;
  const float *ginit;  // [G][BH][d][d] states entering the groups
  float *out;          // [BH][nch][dout][dout]
  int *status;
  int *counter;        // [2] item counter and finished CTAs (zero at launch)
  int dout;            // 128, or 64 for d = 64 run at d = 128 (the states' top-left blocks)
};

template <bool DECAY>
__global__ void __launch_bounds__(kThreads, 1)
    tc_chunk_states_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                           ChunkParams P) {
  constexpr int NS = 3;  // stages of (K tile, V tile)
  constexpr uint32_t kStage = 2 * kTileBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NS * kStage);
  uint64_t *full = bars, *scaled = bars + NS, *empty = bars + 2 * NS;
  uint64_t *crd = bars + 3 * NS, *cmma = crd + 1;  // chunk state read out; chunk product done
  uint32_t *tslot = reinterpret_cast<uint32_t *>(cmma + 1);
  __shared__ int abort_flag;
  __shared__ int ring_item[kRing];
  __shared__ uint64_t ring_bar[2 * kRing];
  const ItemRing ring{ring_item, ring_bar, ring_bar + kRing};
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int BH = P.B * P.H;
  int *const detail = P.status ? P.status + 1 + warp : nullptr;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&scaled[s], 128);
      mbar_init(&empty[s], 1);
    }
    mbar_init(crd, 128);
    mbar_init(cmma, 1);
    ring_init(ring, 32 + (DECAY ? 128 : 0) + 128);  // readers: MMA warp, weighting warps, state warps
    fence_mbar_init();
    prefetch_tensormap(&mk);
    prefetch_tensormap(&mv);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS = *tslot;
  auto range = [&](int item, int &s0, int &s1) {
    const int g = item / BH;
    s0 = P.gp.start(g);
    s1 = min(P.T, P.gp.start(g + 1));
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer: K, V tiles per block
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int k = 0, item; ok; ++k) {
        if (!(ok = ring_post(ring, k, P.counter, P.nitems, item, &abort_flag, P.status, detail)) || item < 0) break;
        const int bh = item % BH, b = bh / P.H, h = bh % P.H;
        int s0, s1;
        range(item, s0, s1);
        for (int t0 = s0; t0 < s1; t0 += 128, ++it) {
          const int s = it % NS, u = it / NS;
          if (u > 0 && !(ok = mbar_wait(&empty[s], (u - 1) & 1, &abort_flag, P.status, detail))) break;
          uint8_t *xs = smem + s * kStage;
          mbar_arrive_expect_tx(&full[s], kStage);
          tma_load_4d(&mk, &full[s], xs, 0, t0, h, b, kPolicyEvictFirst);
          tma_load_4d(&mk, &full[s], xs + kTileHalfBytes, 64, t0, h, b, kPolicyEvictFirst);
          tma_load_4d(&mv, &full[s], xs + kTileBytes, 0, t0, h, b, kPolicyEvictFirst);
          tma_load_4d(&mv, &full[s], xs + kTileBytes + kTileHalfBytes, 64, t0, h, b, kPolicyEvictFirst);
        }
      }
      volatile int no_abort = 0;
      for (int s = 0; s < NS; ++s) {
        const int uses = it > s ? (it - 1 - s) / NS + 1 : 0;
        if (uses > 0) mbar_wait(&full[s], (uses - 1) & 1, &no_abort, P.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer: one half-tile product per chunk
    {  // the whole warp: one elected lane issues each product
      const uint32_t idesc = idesc_bf16(128, 128, true, true);
      int it = 0, ck = 0;  // blocks and chunks seen by this CTA
      bool ok = true;
      for (int k = 0, item; ok; ++k) {
        if (!(ok = __all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail))) || item < 0) break;
        int s0, s1;
        range(item, s0, s1);
        const int nc = (s1 - s0 + 63) / 64;
        for (int c = 0; c < nc && ok; ++c, ++ck) {
          const int s = it % NS, u = it / NS;
          // the chunk's entering state has been read out (and decayed) from TMEM
          if (!(ok = mbar_wait_w(crd, ck & 1, &abort_flag, P.status, detail))) break;
          if (c + 1 < nc) {
            if ((c & 1) == 0 &&
                !(ok = mbar_wait_w(DECAY ? &scaled[s] : &full[s], u & 1, &abort_flag, P.status, detail)))
              break;
            tc_fence_after();
            const uint32_t xs = smem_u32(smem + s * kStage), ys = xs + kTileBytes;
#pragma unroll
            for (uint32_t j = 0; j < 4; ++j) {
              const uint32_t ks = 4 * (c & 1) + j;  // the chunk's 64 rows of the tile
              mma_ss_warp(tS, desc_mnmajor(xs, ks), desc_mnmajor(ys, ks), idesc, 1u);
            }
            mma_commit_warp(cmma);
          }
          // a block's stage is released after its second chunk, or the group's last
          if ((c & 1) == 1 || c + 1 == nc) {
            if (c + 1 == nc && (c & 1) == 0 &&
                !(ok = mbar_wait_w(DECAY ? &scaled[s] : &full[s], u & 1, &abort_flag, P.status, detail)))
              break;
            mma_commit_warp(&empty[s]);
            ++it;
          }
        }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    if (DECAY) {
      // key rows weighted in place: lambda^{63 - (row mod 64)}, before the products read them
      const uint32_t row = threadIdx.x - 128;
      int it = 0;
      bool ok = true;
      for (int k = 0, item; ok; ++k) {
        if (!(ok = __all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail))) || item < 0)
          break;
        const float l2 = log2f(P.decay[(item % BH) % P.H]);
        const float w = exp2f(l2 * (float)(63 - (int)(row & 63)));
        int s0, s1;
        range(item, s0, s1);
        for (int t0 = s0; t0 < s1; t0 += 128, ++it) {
          const int s = it % NS, u = it / NS;
          if (!(ok = mbar_wait(&full[s], u & 1, &abort_flag, P.status, detail))) break;
          scale_tile_row(smem_u32(smem + s * kStage), row, w);
          fence_proxy_async_smem();
          mbar_arrive(&scaled[s]);
        }
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ state warps: read out every chunk's state
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    int ck = 0;
    bool ok = true;
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail))) || item < 0)
        break;
      const int g = item / BH, bh = item % BH;
      int s0, s1;
      range(item, s0, s1);
      const int nc = (s1 - s0 + 63) / 64;
      const float dec = DECAY ? exp2f(log2f(P.decay[bh % P.H]) * 64.f) : 1.f;
      const int dout = P.dout, osz = dout * dout;
      const bool store_row = (int)row < dout;  // d = 64: rows 64..127 of the state are zero, not stored
      float *dst0 = P.out + ((int64_t)bh * P.nch + s0 / 64) * osz + (int64_t)row * dout;
      const float *src = P.ginit + ((int64_t)g * BH + bh) * 16384 + row * 128;
      for (int c = 0; c < nc && ok; ++c, ++ck) {
        float *dst = dst0 + (int64_t)c * osz;
        if (c > 0) {
          // chunk c-1's product is done: its result is chunk c's entering state
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(cmma, (ck - 1 - k) & 1, &abort_flag, P.status, detail))))
            break;
          tc_fence_after();
        }
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          float x[32];
          if (c == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 v4 = __ldg(reinterpret_cast<const float4 *>(src + q * 32 + j));
              x[j] = v4.x; x[j + 1] = v4.y; x[j + 2] = v4.z; x[j + 3] = v4.w;
            }
          } else {
            ld_chunk(tS + lb + q * 32, x);
          }
          if (store_row && q * 32 < dout) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              __stcs(reinterpret_cast<float4 *>(dst + q * 32 + j), make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]));
          }
          if ((c == 0 || DECAY) && c + 1 < nc) {
            // the state the chunk's product accumulates into: lambda^64 S
            uint32_t r[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j] * dec);
            tmem_st32(tS + lb + q * 32, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(crd);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  items_done(P.counter);
  if (warp == 1) tmem_dealloc(tS, 128);
}

// ============================================================================ per-group main kernel
struct MainParams {
  int B, H, T, nitems, init_t;
  GroupPlan gp;
  const float *decay;
  const float *ginit;  // [G][BH][d][d]
  float *final_state;  // [BH][d][d] or null
  float *agg_out;      // [G][BH][d][d]: per group sum_s x_s q_s^T (AGG instances)
  int *status;
  int *counter;        // [2] item counter and finished CTAs (zero at launch)
  const float *gC;     // GATE: group-local log2 cumulative sums of the gates [BH][T]
  const int *gflag;    // GATE, forward: per item [G][BH], nonzero: the weighted-operand form applies
  const __nv_bfloat16 *gq;  // GATE, dq pass: the true q (strides sb, sh, st) for gx = q . dq
  float *gx;           // GATE, dq pass: [BH][T] fp32 q_t . dq_t from the unrounded dq, or null
  int half_out;        // the output rows have 64 columns (d = 64 run at d = 128): one store box
  int64_t sb, sh, st;
};

constexpr int kSlots = 5;
constexpr uint32_t kOffPs = kSlots * kTileBytes;          // P (then O staging) tile
constexpr uint32_t kOffSh = kOffPs + kTileBytes;          // bf16 state tile
constexpr uint32_t kOffBar = kOffSh + kTileBytes;
constexpr uint32_t kOffGate = kOffBar + 256;               // GATE: a block's 128 sums, 128 column factors
constexpr size_t kMainSmem = kOffGate + 1024 + 1024;

// barrier indices
// B_KS / B_XS: the block's K (X) tile weighted in place, two barriers each by
// block parity (an arrival for block n + 2 can only follow the MMA thread's
// wait for block n).
enum { B_FULL = 0, B_EMPTY = kSlots, B_PFULL = 2 * kSlots, B_PEMPTY, B_OFULL, B_OEMPTY, B_SFULL, B_PRE,
       B_PSFULL, B_WEMPTY, B_KS, B_XS = B_KS + 2, B_COUNT = B_XS + 2 };
static_assert(B_COUNT * 8 + 4 <= 256, "chunked kernel barriers and the TMEM slot fit their 256 bytes");

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

// Cumulative gate sums of token t0 + r of a block of nv valid tokens (rows past
// the end take the last valid one: finite weights for zero rows).
__device__ __forceinline__ float gate_c(const float *gc, int t0, int r, int nv) {
  return gc[t0 + (r < nv ? r : nv - 1)];
}

// Gated mask of one 32-column chunk of a score row i: keep j <= i (causal) or
// j >= i (anti-causal) and weight by exp2(C_i - C_j) (exp2(C_j - C_i)), with cb
// the block's 128 cumulative sums.  The weight factors through the chunk's
// middle column m: exp2(C_i - C_m) per row times the column factor
// cw[j] = exp2(C_m - C_j) (anti-causal: exp2(C_m - C_i) and exp2(C_j - C_m)),
// one exponential per row and chunk instead of one per element.  Both factors
// stay within 2^+-100 when the chunk's sums span at most 100 (kept entries: the
// product is the weight, <= 1); a wider span (very small gates) takes the
// per-element form.  Entries outside the mask are set, never multiplied.
template <bool REV>
__device__ __forceinline__ void mask_chunk_gate(float (&x)[32], int i, int c, float ci, const float *cb,
                                                const float *cw) {
  const int j0 = c * 32;
  if (fabsf(cb[j0] - cb[j0 + 31]) <= 100.f) {
    const float cm = cb[j0 + 16];
    const float rf = exp2f(REV ? cm - ci : ci - cm);
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const int j = j0 + jj;
      const bool keep = REV ? (j >= i) : (j <= i);
      x[jj] = keep ? x[jj] * (rf * cw[j]) : 0.f;
    }
  } else {
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const int j = j0 + jj;
      const bool keep = REV ? (j >= i) : (j <= i);
      x[jj] = keep ? x[jj] * exp2f(REV ? cb[j] - ci : ci - cb[j]) : 0.f;
    }
  }
}

// Column factor of token r of a block (see mask_chunk_gate): exp2(C_m - C_r),
// or exp2(C_r - C_m) for the anti-causal mask, m the middle of r's chunk.
template <bool REV>
__device__ __forceinline__ float gate_colw(const float *gc, int t0, int r, int nv) {
  const float cr = gate_c(gc, t0, r, nv), cm = gate_c(gc, t0, (r & ~31) + 16, nv);
  return exp2f(REV ? cr - cm : cm - cr);
}

// sum_j x[j] * bf16(y[j] w) over columns 32c .. 32c+31 of a row of 128 bf16 y held
// in registers (16 x 8 bf16), rounded as dot32_bf16_w rounds them.
__device__ __forceinline__ float dot32_regs_w(const float (&x)[32], const uint4 (&y)[16], int c, float w) {
  float acc = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint4 u = y[4 * c + m];
    const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t z = pack_bf16(bf16lo(v[e]) * w, bf16hi(v[e]) * w);
      acc = fmaf(x[8 * m + 2 * e], bf16lo(z), acc);
      acc = fmaf(x[8 * m + 2 * e + 1], bf16hi(z), acc);
    }
  }
  return acc;
}

// sum_j x[j] * bf16(y[j] w) for 32 fp32 x and 32 bf16 y at src (64 contiguous
// bytes): the row y weighted and rounded as scale_tile_row weights a tile row.
__device__ __forceinline__ float dot32_bf16_w(const float (&x)[32], const __nv_bfloat16 *src, float w) {
  const uint4 *p = reinterpret_cast<const uint4 *>(src);
  float acc = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint4 u = __ldg(p + m);
    const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t y = pack_bf16(bf16lo(v[e]) * w, bf16hi(v[e]) * w);
      acc = fmaf(x[8 * m + 2 * e], bf16lo(y), acc);
      acc = fmaf(x[8 * m + 2 * e + 1], bf16hi(y), acc);
    }
  }
  return acc;
}

// sum_j x[j] * y[j] for 32 fp32 x and 32 bf16 y at src (64 contiguous bytes).
__device__ __forceinline__ float dot32_bf16(const float (&x)[32], const __nv_bfloat16 *src) {
  const uint4 *p = reinterpret_cast<const uint4 *>(src);
  float acc = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint4 u = __ldg(p + m);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(x[8 * m + 2 * e], bf16lo(w[e]), acc);
      acc = fmaf(x[8 * m + 2 * e + 1], bf16hi(w[e]), acc);
    }
  }
  return acc;
}


// With a decay, each (group, sequence) item takes one of two forms:
//  * weighted operands (lambda >= kWeightedMin; gated forward items that
//    gate_prep flags): group B weights the value rows (v_j *= lambda^{nv-1-j},
//    for the state update K^T V' and for P V'), so the scores Q K^T need no
//    weighted tile and take the causal 0/1 mask times lambda^{-nv}
//    (lambda^{-j-1} v_j = lambda^{-nv} v'_j), and the output accumulator takes
//    Q S and then P V', holding o_i / lambda^{i+1}, which the store multiplies
//    back;
//  * otherwise the inter-block term goes to the fourth TMEM region from the
//    unweighted q (O_inter = Q S), the mask is applied per element, the
//    epilogue adds lambda^{i+1} O_inter to the intra-block term, and the key
//    rows are weighted after the scores have read them, for the state update.
// AGG instances also load a fourth tile x per block and accumulate the group
// aggregate W = sum_s w_s x_s q_s^T in the fourth TMEM region (w_s =
// lambda^{s-start+1}, 1 without a decay; x rows weighted as they land),
// written per group to agg_out: for the dq launch (q := dO, x := q) that is
// the reverse group aggregate sum_s w_s q_s dO_s^T.  With a decay only the
// items of the weighted form do so (the fourth region holds O_inter in the
// others); gated items of that form weight the x rows by exp2(C_s).  Tiles are loaded in the order q, x, k, v and released as their
// last product completes.
// GATE (with DECAY) takes every weight from the gates' group-local cumulative
// sums C: o_i = exp2(C_i - C_prev) (Q S)_i + (P V)_i, mask exp2(C_i - C_j), key
// rows exp2(C_last - C_j), state decay exp2(C_last - C_prev) per block (C_prev:
// the token before the block, 0 at a group start); in the weighted form the
// mask scalar is exp2(C_prev - C_last) and the store's row weight
// exp2(C_i - C_prev).
template <bool DECAY, bool AGG = false, bool GATE = false>
__global__ void __launch_bounds__(kThreads, 1)
    tc_main_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo,
                   const __grid_constant__ CUtensorMap mx, MainParams P) {
  static_assert(!GATE || DECAY, "gates use the weighted code paths");
  constexpr int NT = AGG ? 4 : 3;  // tiles per block
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + B_COUNT);
  __shared__ int abort_flag;
  __shared__ int ring_item[kRing];
  __shared__ uint64_t ring_bar[2 * kRing];
  const ItemRing ring{ring_item, ring_bar, ring_bar + kRing};
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int BH = P.B * P.H;
  int *const detail = P.status ? P.status + 1 + warp : nullptr;  // which wait gave up, per warp role

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
    mbar_init(&bar[B_WEMPTY], 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[B_KS + i], 128);
      mbar_init(&bar[B_XS + i], 128);
    }
    ring_init(ring, 32 + 128 + 128);  // readers: MMA warp, groups A and B
    fence_mbar_init();
    prefetch_tensormap(&mq);
    prefetch_tensormap(&mk);
    prefetch_tensormap(&mv);
    prefetch_tensormap(&mo);
    if (AGG) prefetch_tensormap(&mx);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // barriers, ring, TMEM and tensor maps are set up: wait for the kernel before on
  // the stream (its outputs are this kernel's inputs), then let the next one start
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tS = tmem, tP = tmem + 128, tO = tmem + 256;
  const uint32_t tW = tmem + 384, tOi = tmem + 384;  // AGG: aggregate; DECAY: inter-block term
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sPs = sbase + kOffPs, sSh = sbase + kOffSh;
  auto slot_addr = [&](int t) { return sbase + (uint32_t)(t % kSlots) * kTileBytes; };
  // ring position of tile role r (0 q, 1 k, 2 v, 3 x) of block blk
  auto tile_of = [&](int blk, int r) {
    return NT * blk + (AGG ? (r == 0 ? 0 : (r == 3 ? 1 : r + 1)) : r);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int blk = 0;
      bool ok = true;
      for (int k = 0, item; ok; ++k) {
        if (!(ok = ring_post(ring, k, P.counter, P.nitems, item, &abort_flag, P.status, detail)) || item < 0) break;
        const int g = item / BH, bh = item % BH, b = bh / P.H, h = bh % P.H;
        const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1)), nb = (s1 - s0 + 127) / 128;
        bulk_prefetch_l2(P.ginit + ((int64_t)g * BH + bh) * 16384, 16384 * 4);  // the entering state
        for (int n = 0; n < nb && ok; ++n, ++blk) {
          const int t0 = s0 + 128 * n;
          for (int x = 0; x < NT; ++x) {
            const int t = NT * blk + x, s = t % kSlots, u = t / kSlots;
            if (u > 0 && !(ok = mbar_wait(&bar[B_EMPTY + s], (u - 1) & 1, &abort_flag, P.status, detail))) break;
            const CUtensorMap *m = AGG ? (x == 0 ? &mq : (x == 1 ? &mx : (x == 2 ? &mk : &mv)))
                                       : (x == 0 ? &mq : (x == 1 ? &mk : &mv));
            uint8_t *dst = smem + s * kTileBytes;
            mbar_arrive_expect_tx(&bar[B_FULL + s], kTileBytes);
            tma_load_4d(m, &bar[B_FULL + s], dst, 0, t0, h, b, kPolicyEvictFirst);
            tma_load_4d(m, &bar[B_FULL + s], dst + kTileHalfBytes, 64, t0, h, b, kPolicyEvictFirst);
          }
        }
      }
      // time-bounded drain of the loads in flight (also after an abort)
      const int ntile = NT * blk;
      volatile int no_abort = 0;
      for (int s = 0; s < kSlots; ++s) {
        const int uses = ntile > s ? (ntile - 1 - s) / kSlots + 1 : 0;
        if (uses > 0) mbar_wait(&bar[B_FULL + s], (uses - 1) & 1, &no_abort, P.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    {  // the whole warp: one elected lane issues each product
      const uint32_t id_qk = idesc_bf16(128, 128, false, false);  // Q K^T
      const uint32_t id_qs = idesc_bf16(128, 128, false, true);   // Q S,  P V
      const uint32_t id_kv = idesc_bf16(128, 128, true, true);    // K^T V
      const uint32_t id_xq = idesc_bf16(128, 128, true, true);    // X^T Q
      // steps of 16 over the head dimension: with d = 64 (run zero-padded) the last
      // four multiply zero columns only, so they are skipped
      const uint32_t nkd = P.half_out ? 4u : 8u;
      int blk = 0, ia = 0;  // ia: items that accumulated their group aggregate (phases of B_WEMPTY)
      bool ok = true;
      for (int k = 0, item; ok; ++k) {
        if (!(ok = __all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail))) || item < 0) break;
        const int g = item / BH;
        const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1)), nb = (s1 - s0 + 127) / 128;
        // weighted-operand form (K and X weighted as they land); the group
        // aggregate is accumulated here unless a decay takes the other form
        const bool wtd = DECAY && (GATE ? P.gflag && P.gflag[item] != 0
                                        : P.decay[(item % BH) % P.H] >= kWeightedMin);
        const bool aggw = AGG && (!DECAY || wtd);
        for (int n = 0; n < nb; ++n, ++blk) {
          const int tq = tile_of(blk, 0), tk = tile_of(blk, 1), tv = tile_of(blk, 2), tx = tile_of(blk, 3);
          const uint32_t Q = slot_addr(tq), K = slot_addr(tk), V = slot_addr(tv);
          const int wb = blk & 1, wp = (blk >> 1) & 1;
          // scores: P = Q K^T
          ok = mbar_wait_w(&bar[B_FULL + tq % kSlots], (tq / kSlots) & 1, &abort_flag, P.status, detail) &&
               mbar_wait_w(&bar[B_FULL + tk % kSlots], (tk / kSlots) & 1, &abort_flag, P.status, detail) &&
               (blk == 0 || mbar_wait_w(&bar[B_PEMPTY], (blk - 1) & 1, &abort_flag, P.status, detail));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks)
            if (ks < nkd) mma_ss_warp(tP, desc_kmajor(Q, ks), desc_kmajor(K, ks), id_qk, ks > 0);
          mma_commit_warp(&bar[B_PFULL]);
          // inter-block term: O = Q S (its own accumulator with a decay, unless weighted)
          ok = mbar_wait_w(&bar[B_PRE], blk & 1, &abort_flag, P.status, detail) &&
               (blk == 0 || mbar_wait_w(&bar[B_OEMPTY], (blk - 1) & 1, &abort_flag, P.status, detail));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks)
            if (ks < nkd)
              mma_ss_warp((DECAY && !wtd) ? tOi : tO, desc_kmajor(Q, ks), desc_mnmajor(sSh, ks), id_qs, ks > 0);
          if (aggw) {
            // group aggregate: W += X'^T Q (the previous group's W must have been read out;
            // with a decay X' has its rows weighted by lambda^{s - start + 1})
            ok = (DECAY ? mbar_wait_w(&bar[B_XS + wb], wp, &abort_flag, P.status, detail)
                        : mbar_wait_w(&bar[B_FULL + tx % kSlots], (tx / kSlots) & 1, &abort_flag, P.status, detail)) &&
                 (n > 0 || ia == 0 || mbar_wait_w(&bar[B_WEMPTY], (ia - 1) & 1, &abort_flag, P.status, detail));
            if (!ok) break;
            tc_fence_after();
            const uint32_t X = slot_addr(tx);
#pragma unroll
            for (uint32_t ks = 0; ks < 8; ++ks)
              mma_ss_warp(tW, desc_mnmajor(X, ks), desc_mnmajor(Q, ks), id_xq, (n > 0 || ks > 0) ? 1u : 0u);
          }
          // an X tile that no product reads is still waited for before its slot is released
          if (AGG && !aggw &&
              !(ok = mbar_wait_w(&bar[B_FULL + tx % kSlots], (tx / kSlots) & 1, &abort_flag, P.status, detail)))
            break;
          mma_commit_warp(&bar[B_EMPTY + tq % kSlots]);
          if (AGG) mma_commit_warp(&bar[B_EMPTY + tx % kSlots]);
          // state update: S += K'^T V (decay-weighted key rows), or K^T V' in the
          // weighted form (decay-weighted value rows, which P V reads too)
          ok = (!DECAY || mbar_wait_w(&bar[B_KS + wb], wp, &abort_flag, P.status, detail)) &&
               mbar_wait_w(&bar[B_FULL + tv % kSlots], (tv / kSlots) & 1, &abort_flag, P.status, detail);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) mma_ss_warp(tS, desc_mnmajor(K, ks), desc_mnmajor(V, ks), id_kv, 1u);
          mma_commit_warp(&bar[B_EMPTY + tk % kSlots]);
          mma_commit_warp(&bar[B_SFULL]);
          // intra-block term: O += P V
          if (!(ok = mbar_wait_w(&bar[B_PSFULL], blk & 1, &abort_flag, P.status, detail))) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks)
            mma_ss_warp(tO, desc_kmajor(sPs, ks), desc_mnmajor(V, ks), id_qs, (!DECAY || wtd || ks > 0) ? 1u : 0u);
          mma_commit_warp(&bar[B_EMPTY + tv % kSlots]);
          mma_commit_warp(&bar[B_OFULL]);
        }
        if (ok && aggw) ++ia;
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ group A: scores and outputs
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    const bool leader = threadIdx.x == 128;
    int blk = 0;
    bool ok = true;
    for (int k = 0, item; ok; ++k) {
      if (!(ok = group_all(ring_take(ring, k, item, &abort_flag, P.status, detail), 2, 128)) || item < 0) break;
      const int g = item / BH, bh = item % BH, b = bh / P.H, h = bh % P.H;
      const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1)), nb = (s1 - s0 + 127) / 128;
      const float lam = (DECAY && !GATE) ? P.decay[h] : 1.f;
      const float l2 = (DECAY && !GATE) ? log2f(lam) : 0.f;
      const bool wtd = DECAY && (GATE ? P.gflag && P.gflag[item] != 0 : lam >= kWeightedMin);
      const float *gc = GATE ? P.gC + (int64_t)bh * P.T : nullptr;
      for (int n = 0; n < nb; ++n, ++blk) {
        const int t0 = s0 + 128 * n, nv = min(128, s1 - t0);
        // weighted form: the scores of K' take lambda^{-nv} (gates: exp2(C_prev -
        // C_last)) inside the causal mask
        float wsc = 1.f;
        if (wtd) wsc = GATE ? exp2f((t0 > s0 ? gc[t0 - 1] : 0.f) - gc[t0 + nv - 1]) : exp2f(-l2 * (float)nv);
        float ci = 0.f, cprev = 0.f;
        // one buffer of sums and column factors: the previous block's readers passed
        // the output-store barrier of that block before this write
        float *cb = reinterpret_cast<float *>(smem + kOffGate), *cw = cb + 128;
        if (GATE) {
          ci = gate_c(gc, t0, (int)row, nv);
          cprev = t0 > s0 ? gc[t0 - 1] : 0.f;
          if (!wtd) {  // the per-element mask's sums and column factors
            cb[row] = ci;  // read by the whole group after the barrier below
            cw[row] = gate_colw<false>(gc, t0, (int)row, nv);
          }
        }
        // the q row for the epilogue's q . dq: in the weighted form loaded whole into
        // registers now (a thread's own row: a warp's loads touch 32 lines; their
        // latency passes while the block's products run), else two lines into L1
        uint4 qv[16];
        const bool qreg = GATE && wtd && P.gx && (int)row < nv;
        if (GATE && P.gx && (int)row < nv) {
          const __nv_bfloat16 *qr = P.gq + (int64_t)b * P.sb + (int64_t)h * P.sh + (int64_t)(t0 + (int)row) * P.st;
          if (qreg) {
#pragma unroll
            for (int m = 0; m < 16; ++m)  // (rows of 64 columns: the first 8 pieces)
              if (m < 8 || !P.half_out) qv[m] = __ldg(reinterpret_cast<const uint4 *>(qr) + m);
          } else {
            prefetch_l1(qr);
            if (!P.half_out) prefetch_l1(qr + 64);
          }
        }
        ok = group_all(mbar_wait(&bar[B_PFULL], blk & 1, &abort_flag, P.status, detail), 2, 128);
        if (!ok) break;
        tc_fence_after();
        // the P tile buffer is free once the previous output store has read it
        if (leader) bulk_wait_read_all();
        named_bar_sync(1, 128);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float x[32];
          ld_chunk(tP + lb + c * 32, x);
          if (GATE && !wtd) {
            mask_chunk_gate<false>(x, (int)row, c, ci, cb, cw);
          } else if (wtd) {
            mask_chunk<false, false>(x, (int)row, c, 1.f, 0.f);
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] *= wsc;
          } else {
            mask_chunk<DECAY, false>(x, (int)row, c, lam, l2);
          }
          store_row_chunk_bf16(sPs, row, c, x);
        }
        tc_fence_before();
        mbar_arrive(&bar[B_PEMPTY]);
        fence_proxy_async_smem();
        mbar_arrive(&bar[B_PSFULL]);
        // outputs
        ok = group_all(mbar_wait(&bar[B_OFULL], blk & 1, &abort_flag, P.status, detail), 2, 128);
        if (!ok) break;
        tc_fence_after();
        const float wq = GATE ? exp2f(ci - cprev) : (DECAY ? exp2f(l2 * (float)(row + 1)) : 0.f);
        const bool gx_row = GATE && P.gx && (int)row < nv;
        const __nv_bfloat16 *qrow = gx_row ? P.gq + (int64_t)b * P.sb + (int64_t)h * P.sh +
                                                  (int64_t)(t0 + (int)row) * P.st : nullptr;
        float gxacc = 0.f;
        if (GATE && wtd) {
          // gated, weighted form: the gate-gradient term q . dq takes the q row as the
          // dk/dv pass's products see it (bf16(q exp2(C_i - C_prev))) with the
          // accumulator (dq / exp2(C_i - C_prev)); then dq = accumulator x weight
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float x[32];
            ld_chunk(tO + lb + c * 32, x);
            if (qreg && (c < 2 || !P.half_out)) gxacc += dot32_regs_w(x, qv, c, wq);
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] *= wq;
            store_row_chunk_bf16(sPs, row, c, x);
          }
        } else {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float x[32];
          ld_chunk(tO + lb + c * 32, x);
          if (wtd) {
            // the accumulator holds o_i / lambda^{i+1} (gates: / exp2(C_i - C_prev))
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] *= wq;
          } else if (DECAY) {
            float y[32];
            ld_chunk(tOi + lb + c * 32, y);
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = fmaf(wq, y[j], x[j]);
          }
          if (gx_row && !wtd && (c < 2 || !P.half_out))
            gxacc += dot32_bf16(x, qrow + c * 32);  // q . dq before dq is rounded
          store_row_chunk_bf16(sPs, row, c, x);
        }
        }
        if (gx_row) P.gx[(int64_t)bh * P.T + t0 + row] = gxacc;
        tc_fence_before();
        mbar_arrive(&bar[B_OEMPTY]);
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          tma_store_4d_hint(&mo, smem + kOffPs, 0, t0, h, b, kPolicyEvictFirst);
          if (!P.half_out) tma_store_4d_hint(&mo, smem + kOffPs + kTileHalfBytes, 64, t0, h, b, kPolicyEvictFirst);
          bulk_commit();
        }
      }
    }
    if (leader) bulk_wait_all();
  } else if (warp >= 8) {
    // ------------------------------------------------------------ group B: state tile (+ decay weights)
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    int blk = 0;
    bool ok = true;
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail))) || item < 0)
        break;
      const int g = item / BH, bh = item % BH, h = bh % P.H;
      const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1)), nb = (s1 - s0 + 127) / 128;
      const float lam = (DECAY && !GATE) ? P.decay[h] : 1.f;
      const float l2 = (DECAY && !GATE) ? log2f(lam) : 0.f;
      const bool wtd = DECAY && (GATE ? P.gflag && P.gflag[item] != 0 : lam >= kWeightedMin);
      const bool aggw = AGG && (!DECAY || wtd);
      const float *gc = GATE ? P.gC + (int64_t)bh * P.T : nullptr;
      auto nvalid = [&](int n) { return min(128, s1 - (s0 + 128 * n)); };
      // weighted form: value rows lambda^{nv-1-j} (gates: exp2(C_last - C_j)); rows
      // of X (the group aggregate's left factor) lambda^{s-start+1}
      auto wk = [&](int n) {
        const int nv = nvalid(n), r = (int)row, t0 = s0 + 128 * n;
        if (r >= nv) return 0.f;
        return GATE ? exp2f(gc[t0 + nv - 1] - gc[t0 + r]) : exp2f(l2 * (float)(nv - 1 - r));
      };
      auto wx = [&](int n) {
        if ((int)row >= nvalid(n)) return 0.f;
        return GATE ? exp2f(gc[s0 + 128 * n + (int)row]) : exp2f(l2 * (float)(128 * n + (int)row + 1));
      };
      // weigh this thread's row of tile role r (2 V, 3 X) of CTA block b once it
      // has landed, then arrive on the barrier bar_idx + block parity
      auto weigh = [&](int b, int r, float w, int bar_idx) {
        const int t = tile_of(b, r);
        if (!__all_sync(0xffffffffu, mbar_wait(&bar[B_FULL + t % kSlots], (t / kSlots) & 1, &abort_flag, P.status,
                                               detail)))
          return false;
        scale_tile_row(slot_addr(t), row, w);
        fence_proxy_async_smem();
        mbar_arrive(&bar[bar_idx + (b & 1)]);
        return true;
      };
      // weighted form: the block's V (and X), with the value row's weight wkn
      // (loaded early: gates read it from global memory).  A tile's slot was
      // last filled by a tile of the block before (V: its k or, without AGG, its
      // q; X: its q), which the MMA thread waited for before that block's state
      // update, so the state barrier waited before this says the fill landed.
      // X first: its product comes earlier, and its slot frees earlier than V's.
      auto weigh_block = [&](int b, int n, float wkn) {
        return (!AGG || weigh(b, 3, wx(n), B_XS)) && weigh(b, 2, wkn, B_KS);
      };
      if (wtd && !(ok = weigh_block(blk, 0, wk(0)))) break;
      // state decay across block n: lambda^{nv}, or the product of its gates
      auto block_decay = [&](int n) {
        const int t0 = s0 + 128 * n, nv = nvalid(n);
        if (GATE) return exp2f(gc[t0 + nv - 1] - (t0 > s0 ? gc[t0 - 1] : 0.f));
        return DECAY ? exp2f(l2 * (float)nv) : 1.f;
      };
      // initial state of the group
      {
        const float *src = P.ginit + ((int64_t)g * BH + bh) * 16384;
        const float dec = block_decay(0);
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
          store_row_chunk_bf16(sSh, row, c, x);
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j] * dec);
          tmem_st32(tS + lb + c * 32, r);
        }
        tmem_st_wait();
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(&bar[B_PRE]);
      }
      for (int n = 0; n < nb; ++n, ++blk) {
        // the next block's state decay (gates: two loads), ahead of the waits below
        const float dec_next = n + 1 < nb ? block_decay(n + 1) : 1.f;
        const bool more = n + 1 < nb;
        const float wk_next = (wtd && more) ? wk(n + 1) : 0.f;  // ahead of the waits below
        if (DECAY && !wtd) {
          // key rows k_j *= lambda^{nv-1-j} (gates: exp2(C_last - C_j)) once the scores have read them
          const int nv = nvalid(n), r = (int)row, t0 = s0 + 128 * n;
          float w = 0.f;
          if (r < nv) w = GATE ? exp2f(gc[t0 + nv - 1] - gc[t0 + r]) : exp2f(l2 * (float)(nv - 1 - r));
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_PFULL], blk & 1, &abort_flag, P.status, detail))))
            break;
          scale_tile_row(slot_addr(tile_of(blk, 1)), row, w);
          fence_proxy_async_smem();
          mbar_arrive(&bar[B_KS + (blk & 1)]);
          if (AGG) mbar_arrive(&bar[B_XS + (blk & 1)]);  // one phase per block in either form
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_SFULL], blk & 1, &abort_flag, P.status, detail));
        if (!ok) break;
        tc_fence_after();
        if (more) {
          const float dec = dec_next;
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
          tc_fence_before();
          fence_proxy_async_smem();
          mbar_arrive(&bar[B_PRE]);
          // weighted form: the next block's V (and X), off the path to its scores
          if (wtd && !(ok = weigh_block(blk + 1, n + 1, wk_next))) break;
        } else if (aggw) {
          // the group's aggregate W (complete: its last product precedes the state update)
          float *dst = P.agg_out + ((int64_t)g * BH + bh) * 16384 + row * 128;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float x[32];
            ld_chunk(tW + lb + c * 32, x);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4 *>(dst + c * 32 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
          }
          tc_fence_before();
          mbar_arrive(&bar[B_WEMPTY]);
        } else if (P.final_state && g == P.gp.G - 1) {
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
  items_done(P.counter);
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ============================================================================ reverse-time dual kernel
// dv and dk of the backward in one pass over (k, q, dO, v), walking every
// group's blocks from its end.  With R the reverse state entering a block
// (R = sum over later tokens u of lambda^{u - block end} q_u dO_u^T) and rows
// i, j of the block (nv valid rows):
//   dv = diag(lambda^{nv-1-i}) K R   + (K Q^T  (.) M) dO
//   dk = diag(lambda^{nv-1-i}) V R^T + (V dO^T (.) M) Q
//   R <- lambda^{nv} R + Q^T diag(lambda^{j+1}) dO
// with the anti-causal decay mask M_ij = lambda^{j-i} [j >= i].  Both outputs
// share one TMEM state; R^T is the same bf16 tile read through a K-major
// descriptor.  The masked score tiles stay in TMEM: group A overwrites each
// fp32 score tile with its bf16 pairs, which the next product reads as its A
// operand (tcgen05 products issued by one thread run in issue order, so the
// following score product may overwrite them).  That leaves shared memory for
// six input tiles.  Warps 12..15 (group C) write dv and dk from registers.
struct DualParams {
  int B, H, T, nitems;
  GroupPlan gp;
  const float *decay;
  const float *ginit;  // [G][BH][d][d] reverse states entering each group
  __nv_bfloat16 *dk, *dv;
  int64_t sb, sh, st;  // element strides of dk and dv
  int wide;            // every row of dk and dv starts on a 32-byte boundary: 256-bit stores
  int *status;
  int *counter;        // [2] item counter and finished CTAs (zero at launch)
  const float *gC;     // GATE: group-local log2 cumulative sums of the gates [BH][T]
  const __nv_bfloat16 *gk;  // GATE: k (strides sb, sh, st) for gx -= k . dk
  float *gx;           // GATE: [BH][T] fp32, q . dq from the dq pass; k . dk (unrounded dk) subtracted
  const int *gflag;    // GATE: per item [G][BH], nonzero: the weighted-operand form (as in the dq pass)
  int half_out;        // dk, dv rows have 64 columns (d = 64 run at d = 128): chunks 0, 1 only
};

constexpr int kDualThreads = 512;
constexpr int kDualSlots = 6;
constexpr uint32_t kDualOffSh = kDualSlots * kTileBytes;  // bf16 state tile
constexpr uint32_t kDualOffBar = kDualOffSh + kTileBytes;
constexpr uint32_t kDualOffGate = kDualOffBar + 256;  // GATE: a block's 128 sums, 128 column factors
constexpr size_t kDualSmem = kDualOffGate + 1024 + 1024;
// D_KS, D_DS, D_VS: the K, dO and V tiles of a block weighted in place (two
// barriers each, by block parity, so that an arrival for block n + 2 can only
// follow the MMA thread's wait for block n).
enum { D_FULL = 0, D_EMPTY = kDualSlots, D_PFULL = 2 * kDualSlots, D_PSFULL, D_O1FULL, D_O1EMPTY, D_O2FULL,
       D_O2EMPTY, D_SFULL, D_PRE, D_KS, D_DS = D_KS + 2, D_VS = D_DS + 2, D_COUNT = D_VS + 2 };
static_assert(D_COUNT * 8 + 4 <= 256, "dual kernel barriers and the TMEM slot fit their 256 bytes");

// Per-head decays lambda >= kWeightedMin take the weighted-operand form of
// the dk/dv pass: only the rows of dO are weighted, by lambda^{j+1}, as soon as
// their tile lands (before any product reads it); the two accumulators hold
// dv and dk divided by the row weight w_i = lambda^{nv-1-i}, which the store
// multiplies back; and both score tiles need only the 0/1 anti-causal mask
// times the one scalar lambda^{-nv}:
//   dv_i = w_i [ (K R)_i + sum_j lambda^{-nv} [j >= i] (k_i.q_j) dO'_j ],
//   dk_i = w_i [ (V R^T)_i + sum_j lambda^{-nv} [j >= i] (v_i.dO'_j) q_j ],
// with dO'_j = lambda^{j+1} dO_j (expand: the products are lambda^{j-i}).
// The factors stay within lambda^{-128} .. lambda^{128}, i.e. 2^{+-42} for
// lambda >= kWeightedMin, far inside fp32 and bf16 range.  Smaller decays weight the
// rows of K, V and dO between the products (score tiles from unweighted
// operands, masks per element), which puts the weighting on the critical path
// of the block.

// Ring slot of tile x (0 K, 1 Q, 2 dO, 3 V) of the blk-th block a CTA
// processes, and how many loads that slot received before it.  Tiles are
// loaded in that order and released in the order K, dO, V, Q; each takes the
// slot freed six releases earlier, which repeats every four blocks:
//   slots  [0 1 2 3] [4 5 0 2] [3 1 4 0] [2 5 3 4]
// with 3, 2, 3, 3, 3, 2 loads of slots 0..5 per four blocks.
__device__ __forceinline__ void dual_slot(int blk, int x, int &slot, int &cnt) {
  constexpr uint64_t kSlot = 0x4352041320543210ull;  // 4 bits per (blk % 4, x)
  constexpr uint32_t kPrior = 0xa6955000u;           // 2 bits: loads of the slot earlier in the period
  constexpr uint32_t kPerPeriod = 0xbfbu;            // 2 bits per slot: loads per period
  const int i = 4 * (blk & 3) + x;
  slot = (int)((kSlot >> (4 * i)) & 15u);
  cnt = (blk >> 2) * (int)((kPerPeriod >> (2 * slot)) & 3u) + (int)((kPrior >> (2 * i)) & 3u);
}

// 32 fp32 values -> 64 contiguous bytes of bf16 in global memory (streaming
// stores).  WIDE: two 32-byte stores (dst 32-byte aligned), each a whole
// sector; else four 16-byte stores.  A warp's store covers 32 rows, so the
// 16-byte form leaves every sector to be completed by a second instruction;
// the 32-byte form took the dk/dv pass from 0.586 to 0.505 ms at B2 H16 T64K.
template <bool WIDE>
__device__ __forceinline__ void st_global_chunk_bf16(__nv_bfloat16 *dst, const float (&x)[32]) {
  if (WIDE) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 16 * q),
                   "r"(pack_bf16(x[16 * q + 0], x[16 * q + 1])), "r"(pack_bf16(x[16 * q + 2], x[16 * q + 3])),
                   "r"(pack_bf16(x[16 * q + 4], x[16 * q + 5])), "r"(pack_bf16(x[16 * q + 6], x[16 * q + 7])),
                   "r"(pack_bf16(x[16 * q + 8], x[16 * q + 9])), "r"(pack_bf16(x[16 * q + 10], x[16 * q + 11])),
                   "r"(pack_bf16(x[16 * q + 12], x[16 * q + 13])), "r"(pack_bf16(x[16 * q + 14], x[16 * q + 15]))
                   : "memory");
    }
    return;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 8 * q),
                 "r"(pack_bf16(x[8 * q + 0], x[8 * q + 1])), "r"(pack_bf16(x[8 * q + 2], x[8 * q + 3])),
                 "r"(pack_bf16(x[8 * q + 4], x[8 * q + 5])), "r"(pack_bf16(x[8 * q + 6], x[8 * q + 7]))
                 : "memory");
  }
}

// GATE (with DECAY): weights from the gates' group-local cumulative sums C:
// rows of K, V exp2(C_last - C_i), rows of dO exp2(C_j - C_prev), mask
// exp2(C_j - C_i), state decay exp2(C_last - C_prev) per block.
template <bool DECAY, bool GATE = false>
__global__ void __launch_bounds__(kDualThreads, 1)
    tc_dual_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mq,
                   const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                   DualParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kDualOffBar);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + D_COUNT);
  __shared__ int abort_flag;
  __shared__ int ring_item[kRing];
  __shared__ uint64_t ring_bar[2 * kRing];
  const ItemRing ring{ring_item, ring_bar, ring_bar + kRing};
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int BH = P.B * P.H;
  int *const detail = P.status ? P.status + 1 + warp : nullptr;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kDualSlots; ++s) {
      mbar_init(&bar[D_FULL + s], 1);
      mbar_init(&bar[D_EMPTY + s], 1);
    }
    mbar_init(&bar[D_PFULL], 1);
    mbar_init(&bar[D_PSFULL], 128);
    mbar_init(&bar[D_O1FULL], 1);
    mbar_init(&bar[D_O1EMPTY], 128);
    mbar_init(&bar[D_O2FULL], 1);
    mbar_init(&bar[D_O2EMPTY], 128);
    mbar_init(&bar[D_SFULL], 1);
    mbar_init(&bar[D_PRE], 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[D_KS + i], 128);
      mbar_init(&bar[D_DS + i], 128);
      mbar_init(&bar[D_VS + i], 128);
    }
    ring_init(ring, 32 + 3 * 128);  // readers: MMA warp, groups A, B and C
    fence_mbar_init();
    prefetch_tensormap(&mk);
    prefetch_tensormap(&mq);
    prefetch_tensormap(&mv);
    prefetch_tensormap(&mdo);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // barriers, ring, TMEM and tensor maps are set up: wait for the kernel before on
  // the stream (its outputs are this kernel's inputs), then let the next one start
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tR = tmem, tP = tmem + 128, tO1 = tmem + 256, tO2 = tmem + 384;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sSh = sbase + kDualOffSh;
  auto tile_addr = [&](int slot) { return sbase + (uint32_t)slot * kTileBytes; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int blk = 0;
      bool ok = true;
      int loads[kDualSlots] = {0, 0, 0, 0, 0, 0};
      for (int k = 0, item; ok; ++k) {
        if (!(ok = ring_post(ring, k, P.counter, P.nitems, item, &abort_flag, P.status, detail)) || item < 0) break;
        const int g = item / BH, bh = item % BH, b = bh / P.H, h = bh % P.H;
        const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1)), nb = (s1 - s0 + 127) / 128;
        bulk_prefetch_l2(P.ginit + ((int64_t)g * BH + bh) * 16384, 16384 * 4);  // the entering state
        for (int n = 0; n < nb && ok; ++n, ++blk) {
          const int t0 = s0 + 128 * (nb - 1 - n);
          for (int x = 0; x < 4; ++x) {
            int s, c;
            dual_slot(blk, x, s, c);
            if (c > 0 && !(ok = mbar_wait(&bar[D_EMPTY + s], (c - 1) & 1, &abort_flag, P.status, detail))) break;
            const CUtensorMap *m = x == 0 ? &mk : (x == 1 ? &mq : (x == 2 ? &mdo : &mv));
            uint8_t *dst = smem + s * kTileBytes;
            mbar_arrive_expect_tx(&bar[D_FULL + s], kTileBytes);
            tma_load_4d(m, &bar[D_FULL + s], dst, 0, t0, h, b, kPolicyEvictFirst);
            tma_load_4d(m, &bar[D_FULL + s], dst + kTileHalfBytes, 64, t0, h, b, kPolicyEvictFirst);
            ++loads[s];
          }
        }
      }
      volatile int no_abort = 0;
      for (int s = 0; s < kDualSlots; ++s)
        if (loads[s] > 0) mbar_wait(&bar[D_FULL + s], (loads[s] - 1) & 1, &no_abort, P.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    {  // the whole warp: one elected lane issues each product
      const uint32_t id_kk = idesc_bf16(128, 128, false, false);  // A K-major, B K-major
      const uint32_t id_km = idesc_bf16(128, 128, false, true);   // A K-major (or TMEM), B MN-major
      const uint32_t id_mm = idesc_bf16(128, 128, true, true);    // A MN-major, B MN-major
      // steps of 16 over the head dimension (d = 64 runs zero-padded: the last four
      // multiply zero columns only and are skipped)
      const uint32_t nkd = P.half_out ? 4u : 8u;
      int blk = 0;
      bool ok = true;
      auto wait = [&](int idx, int parity) {
        return mbar_wait_w(&bar[idx], parity & 1, &abort_flag, P.status, detail);
      };
      auto full = [&](int x) {
        int s, c;
        dual_slot(blk, x, s, c);
        return wait(D_FULL + s, c);
      };
      auto release = [&](int x) {
        int s, c;
        dual_slot(blk, x, s, c);
        mma_commit_warp(&bar[D_EMPTY + s]);
      };
      auto addr = [&](int x) {
        int s, c;
        dual_slot(blk, x, s, c);
        return tile_addr(s);
      };
      for (int k = 0, item; ok; ++k) {
        if (!(ok = __all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail))) || item < 0) break;
        const int g = item / BH;
        const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1)), nb = (s1 - s0 + 127) / 128;
        // weighted-operand form: dO is weighted before its first product
        // weighted-operand form: dO (gates: Q) is weighted before its first product
        const bool wtd = DECAY && (GATE ? P.gflag && P.gflag[item] != 0
                                        : P.decay[(item % BH) % P.H] >= kWeightedMin);
        const bool wq = GATE && wtd;  // the weighted tile is Q, read by P1 already
        // the decay-free order (R updated right after dv's state term)
        const bool early_r = !DECAY || wtd;
        for (int n = 0; n < nb && ok; ++n, ++blk) {
          const uint32_t K = addr(0), Q = addr(1), DO = addr(2), V = addr(3);
          const int u1 = 2 * blk, u2 = u1 + 1, wb = blk & 1, wp = blk >> 1;
          // P1 = K Q^T  (the previous block's P2~ has been consumed: issue order)
          if (!(ok = full(0) && (wq ? wait(D_DS + wb, wp) : full(1)))) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks)
            if (ks < nkd) mma_ss_warp(tP, desc_kmajor(K, ks), desc_kmajor(Q, ks), id_kk, ks > 0);
          mma_commit_warp(&bar[D_PFULL]);
          // dv = K' R   (R from the bf16 state tile, MN-major)
          ok = (!DECAY || wtd || wait(D_KS + wb, wp)) && wait(D_PRE, blk) && (blk == 0 || wait(D_O1EMPTY, blk - 1));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks)
            if (ks < nkd) mma_ss_warp(tO1, desc_kmajor(K, ks), desc_mnmajor(sSh, ks), id_km, ks > 0);
          release(0);
          if (early_r) {
            // R += Q^T dO' (the state tile is rewritten only after SFULL, below)
            if (!(ok = (wtd && !wq) ? wait(D_DS + wb, wp) : full(2))) break;
            tc_fence_after();
#pragma unroll
            for (uint32_t ks = 0; ks < 8; ++ks) mma_ss_warp(tR, desc_mnmajor(Q, ks), desc_mnmajor(DO, ks), id_mm, 1u);
          }
          // dv += P1~ dO   (P1~ in TMEM as bf16 pairs)
          if (!(ok = (early_r ? true : full(2)) && wait(D_PSFULL, u1))) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) mma_ts_warp(tO1, tP + ks * 8, desc_mnmajor(DO, ks), id_km, 1u);
          mma_commit_warp(&bar[D_O1FULL]);
          // P2 = V dO^T
          if (!(ok = full(3))) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks)
            if (ks < nkd) mma_ss_warp(tP, desc_kmajor(V, ks), desc_kmajor(DO, ks), id_kk, ks > 0);
          mma_commit_warp(&bar[D_PFULL]);
          if (early_r) release(2);
          // dk = V' R^T  (the state tile read K-major)
          ok = (early_r || wait(D_VS + wb, wp)) && (blk == 0 || wait(D_O2EMPTY, blk - 1));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks)
            if (ks < nkd) mma_ss_warp(tO2, desc_kmajor(V, ks), desc_kmajor(sSh, ks), id_kk, ks > 0);
          release(3);
          if (!early_r) {
            // R += Q^T dO'  (dO rows weighted together with V's)
#pragma unroll
            for (uint32_t ks = 0; ks < 8; ++ks) mma_ss_warp(tR, desc_mnmajor(Q, ks), desc_mnmajor(DO, ks), id_mm, 1u);
            release(2);
          }
          mma_commit_warp(&bar[D_SFULL]);
          // dk += P2~ Q
          if (!(ok = wait(D_PSFULL, u2))) break;
          tc_fence_after();
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) mma_ts_warp(tO2, tP + ks * 8, desc_mnmajor(Q, ks), id_km, 1u);
          mma_commit_warp(&bar[D_O2FULL]);
          release(1);
        }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ group A: masked score tiles
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    int blk = 0;
    bool ok = true;
    for (int k = 0, item; ok; ++k) {
      if (!(ok = group_all(ring_take(ring, k, item, &abort_flag, P.status, detail), 3, 128)) || item < 0) break;
      const int g = item / BH, bh = item % BH, h = bh % P.H;
      const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1)), nb = (s1 - s0 + 127) / 128;
      const float lam = (DECAY && !GATE) ? P.decay[h] : 1.f;
      const float l2 = (DECAY && !GATE) ? log2f(lam) : 0.f;
      const bool wtd = DECAY && (GATE ? P.gflag && P.gflag[item] != 0 : lam >= kWeightedMin);
      const float *gc = GATE ? P.gC + (int64_t)bh * P.T : nullptr;
      for (int n = 0; n < nb && ok; ++n, ++blk) {
        // weighted operands: both score tiles take lambda^{-nv} (gates: exp2(C_prev -
        // C_last), the factor of the dq pass's transposed tile) inside the mask
        float wsc = 1.f;
        if (wtd) {
          const int t0 = s0 + 128 * (nb - 1 - n), nv = min(128, s1 - t0);
          wsc = GATE ? exp2f((t0 > s0 ? gc[t0 - 1] : 0.f) - gc[t0 + nv - 1]) : exp2f(-l2 * (float)nv);
        }
        float ci = 0.f;
        float *cb = reinterpret_cast<float *>(smem + kDualOffGate), *cw = cb + 128;
        if (GATE && !wtd) {
          // the block's cumulative sums and column factors, shared by the group
          // (rewritten only after the barrier that ends the block below)
          const int t0 = s0 + 128 * (nb - 1 - n), nv = min(128, s1 - t0);
          ci = gate_c(gc, t0, (int)row, nv);
          cb[row] = ci;
          cw[row] = gate_colw<true>(gc, t0, (int)row, nv);
          named_bar_sync(3, 128);
        }
        for (int half = 0; half < 2 && ok; ++half) {
          const int u = 2 * blk + half;
          // group-uniform decision: the group also meets at named barrier 3
          if (!(ok = group_all(mbar_wait(&bar[D_PFULL], u & 1, &abort_flag, P.status, detail), 3, 128))) break;
          tc_fence_after();
          // chunk c's 32 scores become 16 columns of bf16 pairs at 16c: only
          // columns already read are overwritten
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float x[32];
            ld_chunk(tP + lb + c * 32, x);
            if (GATE && !wtd) {
              mask_chunk_gate<true>(x, (int)row, c, ci, cb, cw);
            } else if (wtd) {
              mask_chunk<false, true>(x, (int)row, c, 1.f, 0.f);
#pragma unroll
              for (int j = 0; j < 32; ++j) x[j] *= wsc;
            } else {
              mask_chunk<DECAY, true>(x, (int)row, c, lam, l2);
            }
            uint32_t r[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = pack_bf16(x[2 * j], x[2 * j + 1]);
            tmem_st16(tP + lb + c * 16, r);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bar[D_PSFULL]);
        }
        if (GATE && !wtd) named_bar_sync(3, 128);  // the block's sums are no longer read (ok, wtd group-uniform)
        if (GATE && wtd && ok) {
          // Gated items in the weighted form store their dv rows here, in fp32 times
          // the row weight exp2(C_last - C_i): the store warps keep the block for the dk
          // rows and the gate gradient's k . dk term.
          const int t0 = s0 + 128 * (nb - 1 - n), nv = min(128, s1 - t0);
          const bool valid = (int)row < nv;
          const float wrow = valid ? exp2f(gc[t0 + nv - 1] - gc[t0 + (int)row]) : 1.f;
          if (!(ok = group_all(mbar_wait(&bar[D_O1FULL], blk & 1, &abort_flag, P.status, detail), 3, 128))) break;
          tc_fence_after();
          __nv_bfloat16 *dst = P.dv + (int64_t)(bh / P.H) * P.sb + (int64_t)h * P.sh + (int64_t)(t0 + (int)row) * P.st;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float x[32];
            ld_chunk(tO1 + lb + c * 32, x);
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] *= wrow;
            if (valid && (c < 2 || !P.half_out)) {
              if (P.wide)
                st_global_chunk_bf16<true>(dst + c * 32, x);
              else
                st_global_chunk_bf16<false>(dst + c * 32, x);
            }
          }
          tc_fence_before();
          mbar_arrive(&bar[D_O1EMPTY]);
        }
      }
    }
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------ group B: state tile (+ decay weights)
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    int blk = 0;
    bool ok = true;
    auto wait = [&](int idx, int parity) {
      return __all_sync(0xffffffffu, mbar_wait(&bar[idx], parity & 1, &abort_flag, P.status, detail));
    };
    // Weight this thread's row of tile x (0 K, 2 dO, 3 V) of CTA block b once it
    // has landed, then arrive on the tile's barrier (bar_idx + block parity).
    auto weigh = [&](int b, int x, float w, int bar_idx) {
      int s, c;
      dual_slot(b, x, s, c);
      if (!wait(D_FULL + s, c)) return false;
      scale_tile_row(tile_addr(s), row, w);
      fence_proxy_async_smem();
      mbar_arrive(&bar[bar_idx + (b & 1)]);
      return true;
    };
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail))) || item < 0)
        break;
      const int g = item / BH, bh = item % BH, h = bh % P.H;
      const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1)), nb = (s1 - s0 + 127) / 128;
      const float lam = (DECAY && !GATE) ? P.decay[h] : 1.f;
      const float l2 = (DECAY && !GATE) ? log2f(lam) : 0.f;
      const bool wtd = DECAY && (GATE ? P.gflag && P.gflag[item] != 0 : lam >= kWeightedMin);
      const float *gc = GATE ? P.gC + (int64_t)bh * P.T : nullptr;
      auto nvalid = [&](int n) { return min(128, s1 - (s0 + 128 * (nb - 1 - n))); };
      auto start = [&](int n) { return s0 + 128 * (nb - 1 - n); };
      auto cprev = [&](int n) { return start(n) > s0 ? gc[start(n) - 1] : 0.f; };
      auto clast = [&](int n) { return gc[start(n) + nvalid(n) - 1]; };
      // state decay across walk block n: lambda^{nv}, or the product of its gates
      auto block_decay = [&](int n) {
        if (GATE) return exp2f(clast(n) - cprev(n));
        return DECAY ? exp2f(l2 * (float)nvalid(n)) : 1.f;
      };
      // weighted form: the weighted tile (dO; gates: Q) and this thread's row weight
      // in walk block n: lambda^{r+1}, or exp2(C_r - C_prev), the weight of the q row
      // in the dq pass's gate-gradient term (the same fp32 expression)
      const int wtile = GATE ? 1 : 2;
      auto wdo = [&](int n) {
        const int r = (int)row;
        if (r >= nvalid(n)) return 0.f;
        return GATE ? exp2f(gate_c(gc, start(n), r, nvalid(n)) - cprev(n)) : exp2f(l2 * (float)(r + 1));
      };
      // weighted form: that tile of a block, plus one (empty) phase of the K and V
      // weighting barriers, which every block completes whatever its form
      auto weigh_do = [&](int b, int n) {
        if (!weigh(b, wtile, wdo(n), D_DS)) return false;
        mbar_arrive(&bar[D_KS + (b & 1)]);
        mbar_arrive(&bar[D_VS + (b & 1)]);
        return true;
      };
      {
        const float *src = P.ginit + ((int64_t)g * BH + bh) * 16384;
        const float dec = block_decay(0);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float x[32];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 v4 = __ldg(reinterpret_cast<const float4 *>(src + row * 128 + c * 32 + j));
            x[j] = v4.x; x[j + 1] = v4.y; x[j + 2] = v4.z; x[j + 3] = v4.w;
          }
          store_row_chunk_bf16(sSh, row, c, x);
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j] * dec);
          tmem_st32(tR + lb + c * 32, r);
        }
        tmem_st_wait();
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(&bar[D_PRE]);
      }
      if (wtd && !(ok = weigh_do(blk, 0))) break;
      for (int n = 0; n < nb && ok; ++n, ++blk) {
        // the next walk block's state decay (gates: two loads), ahead of the waits below
        const float dec_next = n + 1 < nb ? block_decay(n + 1) : 1.f;
        const bool more = n + 1 < nb;
        if (DECAY && !wtd) {
          // weights between the products: K after P1; V and dO after P2
          // (which follows dv += P1~ dO)
          const int nv = nvalid(n), r = (int)row;
          float wx = 0.f, wy = 0.f;  // rows of K and V; rows of dO
          if (r < nv) {
            if (GATE) {
              const float cr = gc[start(n) + r];
              wx = exp2f(clast(n) - cr);
              wy = exp2f(cr - cprev(n));
            } else {
              wx = exp2f(l2 * (float)(nv - 1 - r));
              wy = exp2f(l2 * (float)(r + 1));
            }
          }
          int sk, sdo, sv, c;
          dual_slot(blk, 0, sk, c);
          dual_slot(blk, 2, sdo, c);
          dual_slot(blk, 3, sv, c);
          if (!(ok = wait(D_PFULL, 2 * blk))) break;
          scale_tile_row(tile_addr(sk), row, wx);
          fence_proxy_async_smem();
          mbar_arrive(&bar[D_KS + (blk & 1)]);
          if (!(ok = wait(D_PFULL, 2 * blk + 1))) break;
          scale_tile_row(tile_addr(sv), row, wx);
          scale_tile_row(tile_addr(sdo), row, wy);
          fence_proxy_async_smem();
          // every block completes one phase of each weighting barrier, whatever
          // the form (a CTA's items may mix both)
          mbar_arrive(&bar[D_DS + (blk & 1)]);
          mbar_arrive(&bar[D_VS + (blk & 1)]);
        }
        // weighted form, next block: dO as soon as it lands, unless this
        // block's state is ready first (the state goes first then, being on the
        // critical path)
        bool do_done = false;
        if (GATE && wtd && more) {
          // gates: the weighted tile is Q, which the next block's first product reads;
          // it lands a block or more ahead, so it goes first
          if (!(ok = weigh_do(blk + 1, n + 1))) break;
          do_done = true;
        } else if (wtd && more) {
          int s, c;
          dual_slot(blk + 1, wtile, s, c);
          // bounded poll of both events; the bounded waits below follow either way
#pragma unroll 1
          for (int i = 0; i < (1 << 20) && !abort_flag; ++i) {
            if (__any_sync(0xffffffffu, mbar_test_wait(&bar[D_SFULL], blk & 1))) break;
            if (__all_sync(0xffffffffu, mbar_test_wait(&bar[D_FULL + s], c & 1))) {
              do_done = true;
              break;
            }
          }
          if (do_done && !(ok = weigh_do(blk + 1, n + 1))) break;
        }
        if (!(ok = wait(D_SFULL, blk))) break;
        tc_fence_after();
        if (more) {
          const float dec = dec_next;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float x[32];
            ld_chunk(tR + lb + c * 32, x);
            store_row_chunk_bf16(sSh, row, c, x);
            if (DECAY) {
              uint32_t r[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j] * dec);
              tmem_st32(tR + lb + c * 32, r);
            }
          }
          if (DECAY) tmem_st_wait();
          tc_fence_before();
          fence_proxy_async_smem();
          mbar_arrive(&bar[D_PRE]);
          if (wtd && !do_done && !(ok = weigh_do(blk + 1, n + 1))) break;
        }
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ group C: dv and dk rows to global memory
    const uint32_t quad = warp & 3, row = quad * 32 + lane, lb = (quad * 32) << 16;
    int blk = 0;
    bool ok = true;
    for (int k = 0, item; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, ring_take(ring, k, item, &abort_flag, P.status, detail))) || item < 0)
        break;
      const int g = item / BH, bh = item % BH, b = bh / P.H, h = bh % P.H;
      const int s0 = P.gp.start(g), s1 = min(P.T, P.gp.start(g + 1)), nb = (s1 - s0 + 127) / 128;
      const float lam = (DECAY && !GATE) ? P.decay[h] : 1.f;
      const bool wtd = DECAY && (GATE ? P.gflag && P.gflag[item] != 0 : lam >= kWeightedMin);
      const float l2 = (wtd && !GATE) ? log2f(lam) : 0.f;
      const float *gc = GATE ? P.gC + (int64_t)bh * P.T : nullptr;
      for (int n = 0; n < nb && ok; ++n, ++blk) {
        const int t0 = s0 + 128 * (nb - 1 - n);
        const bool valid = t0 + (int)row < s1;
        // weighted form: the accumulators hold the rows divided by lambda^{nv-1-i}
        // (gates: exp2(C_last - C_i), the weight of the k row in the dq pass)
        float wrow = 1.f;
        if (wtd && valid) {
          const int nv = min(128, s1 - t0);
          wrow = GATE ? exp2f(gc[t0 + nv - 1] - gc[t0 + (int)row]) : exp2f(l2 * (float)(nv - 1 - (int)row));
        }
        if (GATE && P.gx && valid) {
          // the k row for k . dk: two 128-byte lines into L1 while dv drains
          const __nv_bfloat16 *kr = P.gk + (int64_t)b * P.sb + (int64_t)h * P.sh + (int64_t)(t0 + (int)row) * P.st;
          prefetch_l1(kr);
          if (!P.half_out) prefetch_l1(kr + 64);
        }
        // (gated items in the weighted form: the dv rows are stored by the score warps)
        for (int half = (GATE && wtd) ? 1 : 0; half < 2 && ok; ++half) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bar[half ? D_O2FULL : D_O1FULL], blk & 1, &abort_flag,
                                                 P.status, detail));
          if (!ok) break;
          tc_fence_after();
          __nv_bfloat16 *dst = (half ? P.dk : P.dv) + (int64_t)b * P.sb + (int64_t)h * P.sh +
                               (int64_t)(t0 + (int)row) * P.st;
          const uint32_t tO = half ? tO2 : tO1;
          const bool gx_row = GATE && half == 1 && P.gx && valid;
          const __nv_bfloat16 *krow = gx_row ? P.gk + (int64_t)b * P.sb + (int64_t)h * P.sh +
                                                   (int64_t)(t0 + (int)row) * P.st : nullptr;
          float gxacc = 0.f;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float x[32];
            ld_chunk(tO + lb + c * 32, x);
            // the gate-gradient term k . dk: in the weighted form, the k row as the dq
            // pass's products saw it (bf16(k exp2(C_last - C_i))) with the accumulator
            // (dk / exp2(C_last - C_i)), so that the intra-block terms of q . dq and
            // k . dk are the same products
            if (gx_row && wtd && (c < 2 || !P.half_out)) gxacc += dot32_bf16_w(x, krow + c * 32, wrow);
            if (wtd) {
#pragma unroll
              for (int j = 0; j < 32; ++j) x[j] *= wrow;
            }
            if (gx_row && !wtd && (c < 2 || !P.half_out))
              gxacc += dot32_bf16(x, krow + c * 32);  // k . dk before dk is rounded
            if (valid && (c < 2 || !P.half_out)) {
              if (P.wide)
                st_global_chunk_bf16<true>(dst + c * 32, x);
              else
                st_global_chunk_bf16<false>(dst + c * 32, x);
            }
          }
          if (gx_row) P.gx[(int64_t)bh * P.T + t0 + row] -= gxacc;
          tc_fence_before();
          mbar_arrive(&bar[half ? D_O2EMPTY : D_O1EMPTY]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  items_done(P.counter);
  if (warp == 1) tmem_dealloc(tmem, 512);
}

bool seq_tmap(const Problem &p, const void *base, CUtensorMap *m) {
  // with dcols = 64 the second 64-column box of every tile lies past the rows' end:
  // its loads fill zeros
  const uint64_t dims[4] = {(uint64_t)(p.dcols ? p.dcols : p.d), (uint64_t)p.T, (uint64_t)p.H, (uint64_t)p.B};
  const uint64_t strides[3] = {(uint64_t)p.st * 2, (uint64_t)p.sh * 2, (uint64_t)p.sb * 2};
  return make_tmap_bf16(m, base, dims, strides);
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t tc_segment_states(const Problem &p, const GroupPlan &gp, const void *X, const void *Y, bool reverse,
                              float *out, int *status, cudaStream_t s, bool skip_weighted, int dout) {
  alignas(64) CUtensorMap mx, my;
  if (!seq_tmap(p, X, &mx) || !seq_tmap(p, Y, &my)) return cudaErrorInvalidValue;
  AggParams A;
  A.B = p.B; A.H = p.H; A.T = p.T; A.gp = gp;
  A.nitems = gp.G * p.B * p.H;
  A.reverse = reverse ? 1 : 0;
  if (!status) return cudaErrorInvalidValue;
  A.decay = p.decay; A.out = out; A.status = status; A.counter = status + kCounterAgg;
  A.gC = p.gC; A.gtot = p.gtot;
  A.skip_weighted = skip_weighted ? 1 : 0;
  A.gflag = p.gflag;
  A.dout = dout;
  const size_t smem = 3 * 2 * kTileBytes + 1024 + 256;
  const int grid = A.nitems < p.num_sms ? A.nitems : p.num_sms;
  cudaError_t e;
  TimedLaunch t(K_TC_AGG, s);
  if (p.gC) {
    if ((e = set_smem(tc_agg_kernel<true, true>, smem)) != cudaSuccess) return e;
    e = launch_overlapped(tc_agg_kernel<true, true>, grid, kThreads, smem, s, mx, my, A);
  } else if (p.decay) {
    if ((e = set_smem(tc_agg_kernel<true>, smem)) != cudaSuccess) return e;
    e = launch_overlapped(tc_agg_kernel<true>, grid, kThreads, smem, s, mx, my, A);
  } else {
    if ((e = set_smem(tc_agg_kernel<false>, smem)) != cudaSuccess) return e;
    e = launch_overlapped(tc_agg_kernel<false>, grid, kThreads, smem, s, mx, my, A);
  }
  return e;
}

cudaError_t tc_chunk_states(const Problem &p, const GroupPlan &gp, const void *k, const void *v,
                            const float *group_init, float *out, int *status, cudaStream_t s) {
  alignas(64) CUtensorMap mk, mv;
  if (!status || !seq_tmap(p, k, &mk) || !seq_tmap(p, v, &mv)) return cudaErrorInvalidValue;
  ChunkParams C;
  C.B = p.B; C.H = p.H; C.T = p.T; C.gp = gp;
  C.nitems = gp.G * p.B * p.H;
  C.nch = (p.T + 63) / 64;
  C.decay = p.decay; C.ginit = group_init; C.out = out; C.status = status; C.counter = status + kCounterChunk;
  C.dout = p.dcols == 64 ? 64 : 128;
  const size_t smem = 3 * 2 * kTileBytes + 1024 + 256;
  const int grid = C.nitems < p.num_sms ? C.nitems : p.num_sms;
  cudaError_t e;
  TimedLaunch t(K_TC_CHUNK_STATES, s);
  if (p.decay) {
    if ((e = set_smem(tc_chunk_states_kernel<true>, smem)) != cudaSuccess) return e;
    tc_chunk_states_kernel<true><<<grid, kThreads, smem, s>>>(mk, mv, C);
  } else {
    if ((e = set_smem(tc_chunk_states_kernel<false>, smem)) != cudaSuccess) return e;
    tc_chunk_states_kernel<false><<<grid, kThreads, smem, s>>>(mk, mv, C);
  }
  return cudaGetLastError();
}

cudaError_t tc_dual(const Problem &p, const GroupPlan &gp, const void *q, const void *k, const void *v,
                    const void *dO, void *dk, void *dv, const float *group_init, int *status, cudaStream_t s) {
  alignas(64) CUtensorMap mk, mq, mv, mdo;
  if (!seq_tmap(p, k, &mk) || !seq_tmap(p, q, &mq) || !seq_tmap(p, v, &mv) || !seq_tmap(p, dO, &mdo))
    return cudaErrorInvalidValue;
  DualParams D;
  D.B = p.B; D.H = p.H; D.T = p.T; D.gp = gp;
  D.nitems = gp.G * p.B * p.H;
  D.decay = p.decay; D.ginit = group_init;
  D.dk = static_cast<__nv_bfloat16 *>(dk); D.dv = static_cast<__nv_bfloat16 *>(dv);
  if (!status) return cudaErrorInvalidValue;
  D.sb = p.sb; D.sh = p.sh; D.st = p.st; D.status = status; D.counter = status + kCounterDual;
  auto a32 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 31u) == 0; };
  D.wide = a32(dk) && a32(dv) && (p.sb * 2) % 32 == 0 && (p.sh * 2) % 32 == 0 && (p.st * 2) % 32 == 0;
  D.gC = p.gC;
  D.gk = static_cast<const __nv_bfloat16 *>(p.gk);
  D.gx = p.gx;
  D.gflag = p.gflag;
  D.half_out = p.dcols == 64;
  const int grid = D.nitems < p.num_sms ? D.nitems : p.num_sms;
  cudaError_t e;
  TimedLaunch t(K_TC_DUAL_REV, s);
  if (p.gC) {
    if ((e = set_smem(tc_dual_kernel<true, true>, kDualSmem)) != cudaSuccess) return e;
    e = launch_overlapped(tc_dual_kernel<true, true>, grid, kDualThreads, kDualSmem, s, mk, mq, mv, mdo, D);
  } else if (p.decay) {
    if ((e = set_smem(tc_dual_kernel<true>, kDualSmem)) != cudaSuccess) return e;
    e = launch_overlapped(tc_dual_kernel<true>, grid, kDualThreads, kDualSmem, s, mk, mq, mv, mdo, D);
  } else {
    if ((e = set_smem(tc_dual_kernel<false>, kDualSmem)) != cudaSuccess) return e;
    e = launch_overlapped(tc_dual_kernel<false>, grid, kDualThreads, kDualSmem, s, mk, mq, mv, mdo, D);
  }
  return e;
}

cudaError_t tc_main(const Problem &p, const GroupPlan &gp, const void *q, const void *k, const void *v, void *o,
                    const float *group_init, bool init_transposed, float *final_state, int *status,
                    cudaStream_t s, const void *x, float *agg_out) {
  if (x && !agg_out) return cudaErrorInvalidValue;
  alignas(64) CUtensorMap mq, mk, mv, mo, mx;
  if (!seq_tmap(p, q, &mq) || !seq_tmap(p, k, &mk) || !seq_tmap(p, v, &mv) || !seq_tmap(p, o, &mo) ||
      !seq_tmap(p, x ? x : q, &mx))
    return cudaErrorInvalidValue;
  MainParams M;
  M.B = p.B; M.H = p.H; M.T = p.T; M.gp = gp;
  M.nitems = gp.G * p.B * p.H;
  M.init_t = init_transposed ? 1 : 0;
  if (!status) return cudaErrorInvalidValue;
  M.decay = p.decay; M.ginit = group_init; M.final_state = final_state; M.status = status;
  M.counter = status + kCounterMain;
  M.agg_out = agg_out;
  M.gC = p.gC;
  M.gflag = p.gflag;
  M.half_out = p.dcols == 64;
  M.gq = static_cast<const __nv_bfloat16 *>(p.gq);
  M.gx = p.gx;
  M.sb = p.sb; M.sh = p.sh; M.st = p.st;
  const int grid = M.nitems < p.num_sms ? M.nitems : p.num_sms;
  cudaError_t e;
  TimedLaunch t(x ? K_TC_MAIN_AGG : K_TC_MAIN_FWD, s);
#define LINATTN_LAUNCH_MAIN(DEC, AGG, GATE)                                                    \
  do {                                                                                        \
    if ((e = set_smem(tc_main_kernel<DEC, AGG, GATE>, kMainSmem)) != cudaSuccess) return e;   \
    e = launch_overlapped(tc_main_kernel<DEC, AGG, GATE>, grid, kThreads, kMainSmem, s, mq, mk, mv, mo, mx, M); \
  } while (0)
  if (x && p.gC)
    LINATTN_LAUNCH_MAIN(true, true, true);
  else if (x && p.decay)
    LINATTN_LAUNCH_MAIN(true, true, false);
  else if (x)
    LINATTN_LAUNCH_MAIN(false, true, false);
  else if (p.gC)
    LINATTN_LAUNCH_MAIN(true, false, true);
  else if (p.decay)
    LINATTN_LAUNCH_MAIN(true, false, false);
  else
    LINATTN_LAUNCH_MAIN(false, false, false);
#undef LINATTN_LAUNCH_MAIN
  return e;
}

}  // namespace linattn
