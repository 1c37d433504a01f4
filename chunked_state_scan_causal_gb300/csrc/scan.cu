// Exclusive prefix scan of fp32 segment states -- the single-GPU counterpart
// of the All-Scan that hands every sequence-parallel rank exactly its initial
// state ("ZeCO: Zero Communication Overhead Sequence Parallelism for Linear
// Attention", abstract) and of LASP-2's one gather of length-independent
// memory states followed by a local combine ("LASP-2", abstract).
//
//   out[0] = init,  out[g] = a * out[g-1] + U[g-1]     (a = lambda^L per sequence)
//
// The combine of two neighbouring pieces is affine: (a2, X2) o (a1, X1) =
// (a1 a2, a2 X1 + X2), so the scan is associative and runs in parallel:
//  * a tile is 32 consecutive segments x 8 consecutive state elements; one
//    warp owns a tile, lane l holds segment l's 8 elements (one 32-byte
//    sector per lane, so every warp load is sector-complete);
//  * inside the tile: Kogge-Stone inclusive scan with warp shuffles;
//  * across tiles: decoupled look-back.  Tiles are taken from an atomic
//    ticket in segment-tile-major order, so every predecessor of a waiting
//    tile is already running; each tile publishes its aggregate at once and
//    its inclusive prefix after the look-back; waits are bounded.
// Up to kColumnMaxG segments a second, column-parallel form is used instead:
// every thread owns 4 consecutive state elements and walks the segments in
// order with several loads in flight, so every warp access is one contiguous
// 512-byte piece (the segment-per-lane tiles above touch 32 scattered sectors
// per warp access, which DRAM serves far less efficiently).  The look-back
// form remains for long scans, where it supplies the parallelism.
#include <cstdlib>
#include <mutex>

#include "../../include/linattn.h"
#include "internal.h"
#include "ptx.cuh"

namespace linattn {
namespace {

constexpr int kWarps = 8;
constexpr int kVec = 8;  // fp32 elements per lane

// lambda^len: exp2(len * log2 lambda) in fp32 (relative error about 1e-7 * |len * log2 lambda|),
// 1 for len = 0.  A double-precision pow per thread cost more than the scan's memory traffic.
__device__ __forceinline__ float pow_len(float lam, int len) { return len == 0 ? 1.f : exp2f(log2f(lam) * (float)len); }

struct ScanArgs {
  int G, BH, DD, H, seg_len, ntg, ncg, reverse;
  int kb, seg_len2;    // with decay_h (column form): groups kb.. have seg_len2 tokens
  const float *seg_decay, *decay_h, *local, *init;
  const float *glog2;  // [G][BH] log2 of each group's own multiplier (column form only), or null
  float *out, *total;
  unsigned *counter;  // ticket counter (zeroed before launch)
  unsigned *flags;    // [ntg * ncg] 0 empty, 1 aggregate, 2 inclusive (zeroed before launch)
  float *agg, *incl;  // [ntg * ncg][kVec]
  int *status;
  uint64_t limit_ns;  // bound of every look-back wait
  int withhold;       // diagnostics: this tile never publishes (-1: none)
};

constexpr unsigned kBatch = 16;  // tickets taken per atomic (look-back case)

__global__ void __launch_bounds__(kWarps * 32) scan_kernel(ScanArgs A) {
  const int lane = threadIdx.x & 31;
  const int64_t E = (int64_t)A.BH * A.DD;
  const unsigned ntiles = (unsigned)A.ntg * (unsigned)A.ncg;
  // Without look-back (one segment tile) tiles are independent: plain grid
  // stride.  With look-back, tickets come in order from an atomic counter, a
  // batch of kBatch per warp; a warp works through its batch in order, so
  // every tile a warp waits on belongs to a warp that is already running.
  const unsigned gwarp = blockIdx.x * kWarps + threadIdx.x / 32, nwarp = gridDim.x * kWarps;
  unsigned next = gwarp, end = 0;
  while (true) {
    unsigned ticket;
    if (A.ntg == 1) {
      ticket = next;
      next += nwarp;
    } else {
      if (next >= end) {
        unsigned base = 0;
        if (lane == 0) base = atomicAdd(A.counter, kBatch);
        next = __shfl_sync(0xffffffffu, base, 0);
        end = next + kBatch;
      }
      ticket = next++;
    }
    if (ticket >= ntiles) break;
    const int tg = (int)(ticket / A.ncg), cg = (int)(ticket % A.ncg);
    const int64_t e0 = (int64_t)cg * kVec;
    const int bh = (int)(e0 / A.DD);
    float a = 1.f;
    if (A.seg_decay) a = A.seg_decay[bh];
    else if (A.decay_h) a = pow_len(A.decay_h[bh % A.H], A.seg_len);

    // processing index p = tg*32 + lane; segment g = p (forward) or G-1-p (reverse)
    const int pidx = tg * 32 + lane;
    const bool valid = pidx < A.G;
    const int g = A.reverse ? A.G - 1 - pidx : pidx;
    float x[kVec];
    if (valid) {
      const float4 *src = reinterpret_cast<const float4 *>(A.local + (int64_t)g * E + e0);
      const float4 u0 = __ldg(src), u1 = __ldg(src + 1);
      x[0] = u0.x; x[1] = u0.y; x[2] = u0.z; x[3] = u0.w;
      x[4] = u1.x; x[5] = u1.y; x[6] = u1.z; x[7] = u1.w;
    } else {
#pragma unroll
      for (int i = 0; i < kVec; ++i) x[i] = 0.f;
    }
    // inclusive scan inside the tile: X_l = sum_{m<=l} a^{l-m} U_m
    float ad = a;  // a^d
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
      for (int i = 0; i < kVec; ++i) {
        const float y = __shfl_up_sync(0xffffffffu, x[i], d);
        if (lane >= d) x[i] = fmaf(ad, y, x[i]);
      }
      ad *= ad;
    }
    const float a32 = ad;  // a^32
    // prefix entering the tile (state after all earlier segments, incl. init)
    float pin[kVec];
    if (tg == 0) {
#pragma unroll
      for (int i = 0; i < kVec; ++i) pin[i] = A.init ? __ldg(A.init + e0 + i) : 0.f;
    } else {
      // publish the aggregate, then look back
      if (lane == 31 && ticket != (unsigned)A.withhold) {
        float4 *dst = reinterpret_cast<float4 *>(A.agg + (int64_t)ticket * kVec);
        dst[0] = make_float4(x[0], x[1], x[2], x[3]);
        dst[1] = make_float4(x[4], x[5], x[6], x[7]);
        __threadfence();
        st_release_gpu(A.flags + ticket, 1u);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < kVec; ++i) pin[i] = 0.f;
      float fac = 1.f;
      int pred = tg - 1;
      while (true) {
        const unsigned pt = (unsigned)pred * A.ncg + cg;
        unsigned f = 0;
        if (lane == 0) {
          f = ld_acquire_gpu(A.flags + pt);
          if (f == 0) {
            const uint64_t t0 = globaltimer_ns();
            while ((f = ld_acquire_gpu(A.flags + pt)) == 0) {
              if (globaltimer_ns() - t0 > A.limit_ns) {
                report_error(A.status, -6);
                f = 3;  // give up: treat as an inclusive prefix of zeros
                break;
              }
            }
          }
        }
        f = __shfl_sync(0xffffffffu, f, 0);
        if (f == 3) break;
        const float *src = (f == 2 ? A.incl : A.agg) + (int64_t)pt * kVec;
#pragma unroll
        for (int i = 0; i < kVec; ++i) pin[i] = fmaf(fac, __ldcg(src + i), pin[i]);
        if (f == 2) break;
        fac *= a32;
        if (--pred < 0) {
          // reached the first tile without an inclusive prefix: add the decayed init
          if (A.init) {
#pragma unroll
            for (int i = 0; i < kVec; ++i) pin[i] = fmaf(fac, __ldg(A.init + e0 + i), pin[i]);
          }
          break;
        }
      }
    }
    // publish the inclusive prefix of this tile
    if (tg + 1 < A.ntg && lane == 31 && ticket != (unsigned)A.withhold) {
      float4 *dst = reinterpret_cast<float4 *>(A.incl + (int64_t)ticket * kVec);
      float v[kVec];
#pragma unroll
      for (int i = 0; i < kVec; ++i) v[i] = fmaf(a32, pin[i], x[i]);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
      __threadfence();
      st_release_gpu(A.flags + ticket, 2u);
    }
    // exclusive outputs: out[p] = X_{l-1} + a^l * pin
    float al = 1.f;  // a^lane
    {
      float base = a;
      int n = lane;
#pragma unroll 1
      while (n) {
        if (n & 1) al *= base;
        base *= base;
        n >>= 1;
      }
    }
    float ex[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const float y = __shfl_up_sync(0xffffffffu, x[i], 1);
      ex[i] = fmaf(al, pin[i], lane == 0 ? 0.f : y);
    }
    if (valid) {
      float4 *dst = reinterpret_cast<float4 *>(A.out + (int64_t)g * E + e0);
      dst[0] = make_float4(ex[0], ex[1], ex[2], ex[3]);
      dst[1] = make_float4(ex[4], ex[5], ex[6], ex[7]);
      if (A.total && pidx == A.G - 1) {
        // value one step past the end: a * out[last] + U[last] = X_l + a^{l+1} pin
        float4 *tt = reinterpret_cast<float4 *>(A.total + e0);
        float v[kVec];
#pragma unroll
        for (int i = 0; i < kVec; ++i) v[i] = fmaf(al * a, pin[i], x[i]);
        tt[0] = make_float4(v[0], v[1], v[2], v[3]);
        tt[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  }
}

constexpr int kColumnMaxG = 256;
constexpr int kColumnDepth = 4;  // loads in flight per thread

__global__ void __launch_bounds__(256) scan_columns_kernel(ScanArgs A) {
  griddep_wait();  // the states come from the kernel before on the stream
  griddep_launch_dependents();
  const int64_t E = (int64_t)A.BH * A.DD, n4 = E / 4;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n4; c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e0 = c * 4;
    const int bh = (int)(e0 / A.DD);
    float a = 1.f, a2 = 1.f;  // multipliers across a group of seg_len, of seg_len2 tokens
    if (A.seg_decay) {
      a = a2 = A.seg_decay[bh];
    } else if (A.decay_h) {
      a = pow_len(A.decay_h[bh % A.H], A.seg_len);
      a2 = A.kb < A.G ? pow_len(A.decay_h[bh % A.H], A.seg_len2) : a;
    }
    float4 acc = A.init ? __ldg(reinterpret_cast<const float4 *>(A.init + e0)) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < A.G; i += kColumnDepth) {
      float4 u[kColumnDepth];
#pragma unroll
      for (int j = 0; j < kColumnDepth; ++j) {
        const int p = i + j, g = A.reverse ? A.G - 1 - p : p;
        if (p < A.G) u[j] = __ldg(reinterpret_cast<const float4 *>(A.local + (int64_t)g * E + e0));
      }
#pragma unroll
      for (int j = 0; j < kColumnDepth; ++j) {
        const int p = i + j, g = A.reverse ? A.G - 1 - p : p;
        if (p < A.G) {
          *reinterpret_cast<float4 *>(A.out + (int64_t)g * E + e0) = acc;
          // the combine across group g decays by that group's multiplier
          const float ag = A.glog2 ? exp2f(A.glog2[(int64_t)g * A.BH + bh]) : (g < A.kb ? a : a2);
          acc = make_float4(fmaf(ag, acc.x, u[j].x), fmaf(ag, acc.y, u[j].y), fmaf(ag, acc.z, u[j].z),
                            fmaf(ag, acc.w, u[j].w));
        }
      }
    }
    if (A.total) *reinterpret_cast<float4 *>(A.total + e0) = acc;
  }
}

}  // namespace

size_t scan_workspace_bytes(int G, int64_t E) {
  const int64_t ntg = (G + 31) / 32, ncg = E / kVec;
  const int64_t nt = ntg * ncg;
  return align256(256 + nt * 4) + 2 * align256(nt * kVec * 4);
}

namespace {
__global__ void fold_kernel(float *w, const float *d, const float *decay_h, int H, int DD, int len, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float a = decay_h ? pow_len(decay_h[(i / DD) % H], len) : 1.f;
    w[i] = fmaf(a, d[i], w[i]);
  }
}
}  // namespace

namespace {
__global__ void seg_decay_kernel(const float *decay_h, int H, int n, int len, float *out) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = pow_len(decay_h[i % H], len);
}
}  // namespace

cudaError_t segment_decay(const float *decay_h, int B, int H, int len, float *out, cudaStream_t s) {
  const int n = B * H;
  seg_decay_kernel<<<(n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024, 256, 0, s>>>(decay_h, H, n, len, out);
  return cudaGetLastError();
}

cudaError_t fold_state(float *w, const float *d, const float *decay_h, int H, int DD, int len, int64_t n,
                       cudaStream_t s) {
  const int64_t want = (n + 255) / 256;
  TimedLaunch t(K_SCAN, s);
  fold_kernel<<<(int)(want < 1024 ? want : 1024), 256, 0, s>>>(w, d, decay_h, H, DD, len, n);
  return cudaGetLastError();
}

uint64_t wait_limit_ns() {
  const char *e = getenv("LINATTN_LOOKBACK_LIMIT_MS");
  if (e && *e) {
    const double ms = strtod(e, nullptr);
    if (ms > 0 && ms < 6e4) return (uint64_t)(ms * 1e6);
  }
  return kWaitLimitNs;
}

cudaError_t state_scan(int G, int BH, int DD, const float *seg_decay, const float *decay_h, int H,
                       int seg_len, bool reverse, const float *local, const float *init, float *out,
                       float *total, void *ws, int *status, cudaStream_t s, const float *group_log2, int kb,
                       int seg_len2, uint64_t limit_ns, int withhold) {
  const int64_t E = (int64_t)BH * DD;
  if ((group_log2 || kb < G) && G > kColumnMaxG) return cudaErrorInvalidValue;
  ScanArgs A;
  A.G = G; A.BH = BH; A.DD = DD; A.H = H; A.seg_len = seg_len;
  A.kb = kb; A.seg_len2 = seg_len2;
  A.ntg = (G + 31) / 32;
  A.ncg = (int)(E / kVec);
  A.reverse = reverse ? 1 : 0;
  A.seg_decay = seg_decay; A.decay_h = decay_h; A.local = local; A.init = init; A.glog2 = group_log2;
  A.out = out; A.total = total; A.status = status;
  A.limit_ns = limit_ns ? limit_ns : wait_limit_ns();
  A.withhold = withhold;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (G <= kColumnMaxG && withhold < 0) {
    const int64_t n4 = E / 4, want = (n4 + 255) / 256, cap = (int64_t)sms * 8;
    TimedLaunch t(K_SCAN, s);
    return launch_overlapped(scan_columns_kernel, dim3((unsigned)(want < cap ? want : cap)), dim3(256), 0, s, A);
  }
  const int64_t nt = (int64_t)A.ntg * A.ncg;
  char *w = static_cast<char *>(ws);
  A.counter = reinterpret_cast<unsigned *>(w);
  A.flags = reinterpret_cast<unsigned *>(w + 256);
  const size_t head = align256(256 + nt * 4);
  A.agg = reinterpret_cast<float *>(w + head);
  A.incl = reinterpret_cast<float *>(w + head + align256(nt * kVec * 4));
  if (A.ntg > 1) {  // ticket counter and look-back flags start at zero
    cudaError_t e = cudaMemsetAsync(w, 0, head, s);
    if (e != cudaSuccess) return e;
  }
  const int64_t want = (nt + kWarps - 1) / kWarps;
  const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  TimedLaunch t(K_SCAN, s);
  scan_kernel<<<grid, kWarps * 32, 0, s>>>(A);
  return cudaGetLastError();
}

}  // namespace linattn

// ============================================================================
// Allocation-free entry point: the same scan with its scratch in a fixed
// static device array (see linattn_state_scan_noalloc in linattn.h).
namespace linattn {
namespace {
static_assert(LINATTN_NOALLOC_SCRATCH_BYTES == 256 + 4 * LINATTN_NOALLOC_MAX_TILES +
                                                   2 * LINATTN_NOALLOC_MAX_TILES * kVec * 4,
              "scratch size must cover the scan's workspace layout at the tile limit");
static __device__ __align__(256) unsigned char g_noalloc_scratch[LINATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch for the current device, looked up once per
// device (with that device current).  In host code the symbol itself is only a
// host-side stand-in, never a device address.
cudaError_t noalloc_scratch(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = p;
  }
  *ptr = g_noalloc_addr[dev];
  return cudaSuccess;
}
}  // namespace
namespace {
__global__ void clear_header_kernel(int *hdr, int n) {
  griddep_launch_dependents();  // the next kernel waits for this one before its first access
  griddep_wait();               // the header may still be in use by the kernel before
  for (int i = threadIdx.x; i < n; i += blockDim.x) hdr[i] = 0;
}
}  // namespace

cudaError_t clear_header(void *ws, size_t bytes, cudaStream_t s) {
  if (!ws || bytes % 4 || bytes > 1024) return cudaErrorInvalidValue;
  TimedLaunch t(K_CLEAR_STATUS, s);
  return launch_overlapped(clear_header_kernel, dim3(1), dim3(64), 0, s, static_cast<int *>(ws), (int)(bytes / 4));
}

}  // namespace linattn

extern "C" int32_t linattn_state_scan_noalloc(int32_t G, int32_t BH, int32_t dk, int32_t dv,
                                              const float *seg_decay, const float *local_states,
                                              const float *init, float *init_states, float *total,
                                              int32_t *device_status, void *stream) {
  using namespace linattn;
  if (G < 1 || BH < 1 || dk < 1 || dv < 1) return LINATTN_ERR_INVALID;
  const int64_t DD = (int64_t)dk * dv;
  if (DD % kVec) return LINATTN_ERR_UNSUPPORTED;
  if (!local_states || !init_states) return LINATTN_ERR_INVALID;
  for (const void *x : {(const void *)seg_decay, (const void *)local_states, (const void *)init,
                        (const void *)init_states, (const void *)total})
    if (reinterpret_cast<uintptr_t>(x) & 15u) return LINATTN_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(device_status) & 3u) return LINATTN_ERR_ALIGN;
  // Only the look-back form (more than kColumnMaxG segments) uses the scratch;
  // the column-parallel form touches none of it, so it has no size limit here.
  const int64_t ntiles = (int64_t)((G + 31) / 32) * ((int64_t)BH * DD / kVec);
  if (G > kColumnMaxG && ntiles > LINATTN_NOALLOC_MAX_TILES) return LINATTN_ERR_SCRATCH_LIMIT;
  int st = device_ok();
  if (st != LINATTN_OK) return st;
  void *scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return LINATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (device_status && cudaMemsetAsync(device_status, 0, sizeof(int32_t), s) != cudaSuccess)
    return LINATTN_ERR_CUDA;
  // state_scan clears the ticket counter and the look-back flags itself
  cudaError_t e = state_scan(G, BH, (int)DD, seg_decay, nullptr, 1, 1, false, local_states, init,
                             init_states, total, scratch, reinterpret_cast<int *>(device_status), s);
  return e == cudaSuccess ? LINATTN_OK : LINATTN_ERR_CUDA;
}
