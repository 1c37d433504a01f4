// C-ABI entry points of liblinattn: argument validation, workspace layout,
// TMA descriptor encoding and the choice between the tensor-core pipeline
// (bf16, d = 128) and the CUDA-core kernels (fp32 inputs, d = 64).  Every
// error is detected here before anything is enqueued.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>
#include <vector>

#include "../../include/linattn.h"
#include "internal.h"

namespace linattn {

// ------------------------------------------------------------------ device checks
int device_ok() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LINATTN_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return LINATTN_ERR_CUDA;
  return (major == 10 && minor == 3) ? LINATTN_OK : LINATTN_ERR_DEVICE;
}

static int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_tmap_bf16(void *map, const void *base, const uint64_t dims[4], const uint64_t strides[3]) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t gs[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(reinterpret_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void *>(base), gd, gs, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ per-kernel timing
namespace {
struct TimingState {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> pool;  // pairs (start, stop), reused across collections
  struct Rec { int kind; int slot; };
  std::vector<Rec> recs;
  int used = 0;
};
TimingState &timing() {
  static TimingState t;
  return t;
}
}  // namespace

TimedLaunch::TimedLaunch(int k, cudaStream_t s) : kind(k), slot(-1), stream(s) {
  TimingState &t = timing();
  std::lock_guard<std::mutex> g(t.mu);
  if (!t.on) return;
  if (t.used * 2 + 2 > (int)t.pool.size()) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return;
    if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); return; }
    t.pool.push_back(a);
    t.pool.push_back(b);
  }
  slot = t.used++;
  cudaEventRecord(t.pool[2 * slot], s);
}
TimedLaunch::~TimedLaunch() {
  if (slot < 0) return;
  TimingState &t = timing();
  std::lock_guard<std::mutex> g(t.mu);
  cudaEventRecord(t.pool[2 * slot + 1], stream);
  t.recs.push_back({kind, slot});
}

// ------------------------------------------------------------------ validation
static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int validate(const linattn_shape *s, Problem *p) {
  if (!s) return LINATTN_ERR_INVALID;
  if (s->abi_version != LINATTN_ABI_VERSION) return LINATTN_ERR_INVALID;
  if (s->B < 1 || s->H < 1 || s->T < 0 || s->dk < 1 || s->dv < 1 || s->chunk < 1)
    return LINATTN_ERR_INVALID;
  if (s->dtype != LINATTN_BF16 && s->dtype != LINATTN_F32) return LINATTN_ERR_INVALID;
  // an empty sequence reads nothing, so its strides are not checked
  if (s->T > 0 && (s->stride_b < 1 || s->stride_h < 1 || s->stride_t < s->dk)) return LINATTN_ERR_INVALID;
  if (s->chunk != 64) return LINATTN_ERR_UNSUPPORTED;
  if (s->dk != s->dv || (s->dk != 64 && s->dk != 128)) return LINATTN_ERR_UNSUPPORTED;
  const int64_t esz = s->dtype == LINATTN_BF16 ? 2 : 4;
  if (s->T > 0 && ((s->stride_t * esz) % 16 || (s->stride_h * esz) % 16 || (s->stride_b * esz) % 16))
    return LINATTN_ERR_ALIGN;
  if ((int64_t)s->B * s->H > (1 << 30)) return LINATTN_ERR_UNSUPPORTED;
  p->B = s->B;
  p->H = s->H;
  p->T = s->T;
  p->d = s->dk;
  p->dtype = s->dtype == LINATTN_BF16 ? 0 : 1;
  p->sb = s->stride_b;
  p->sh = s->stride_h;
  p->st = s->stride_t;
  p->decay = s->decay;
  p->num_sms = num_sms();
  return LINATTN_OK;
}

static int check_ptrs(std::initializer_list<const void *> required, std::initializer_list<const void *> optional) {
  for (const void *x : required) {
    if (!x) return LINATTN_ERR_INVALID;
    if (!aligned16(x)) return LINATTN_ERR_ALIGN;
  }
  for (const void *x : optional)
    if (x && !aligned16(x)) return LINATTN_ERR_ALIGN;
  return LINATTN_OK;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? LINATTN_OK : LINATTN_ERR_CUDA; }

// ------------------------------------------------------------------ workspace layout
constexpr size_t kHeader = 256;  // int32 status word at offset 0

struct FwdLayout {
  GroupPlan gp;
  int G = 0;
  size_t agg = 0, states = 0, scan = 0, total = kHeader;
};
static FwdLayout fwd_layout(const Problem &p, int max_len = 0) {
  FwdLayout w;
  if (!tc_supported(p) || p.T == 0) return w;
  w.gp = tc_group_plan(p, max_len);
  w.G = w.gp.G;
  const size_t st = (size_t)w.G * p.B * p.H * p.d * p.d * sizeof(float);
  w.agg = kHeader;
  w.states = w.agg + align256(st);
  w.scan = w.states + align256(st);
  w.total = w.scan + scan_workspace_bytes(w.G, (int64_t)p.B * p.H * p.d * p.d);
  return w;
}
struct BwdLayout {
  FwdLayout f;            // forward group aggregates / states (recomputed without a checkpoint)
  size_t wagg = 0, rbar = 0, total = kHeader;
};
static BwdLayout bwd_layout(const Problem &p) {
  BwdLayout w;
  w.f = fwd_layout(p);
  if (w.f.G == 0) return w;
  const size_t st = (size_t)w.f.G * p.B * p.H * p.d * p.d * sizeof(float);
  w.wagg = w.f.total;
  w.rbar = w.wagg + align256(st);
  w.total = w.rbar + align256(st);
  return w;
}

// bf16 with d = 64 runs on the d = 128 tensor-core kernels as the zero-padded
// problem, which is the same problem: the tiles' columns 64..127 of q, k, v load
// as zeros (the tensor maps give the rows 64 columns), so every q . k and every
// product with the state is unchanged, the state's rows and columns 64..127 stay
// zero, and only the first 64 output columns are stored (per-chunk states: their
// top-left 64 x 64 blocks).  The states go through zero-padded 128 x 128 copies
// (pad.cu), after the d = 128 workspace, whose status word stays at offset 0.
static bool padded(const Problem &p) { return p.dtype == 0 && p.d == 64 && p.T > 0; }
static Problem padded_problem(const Problem &p) {
  Problem q = p;
  q.d = 128;
  q.dcols = 64;
  return q;
}
static size_t pad_state_bytes(const Problem &p) { return align256((size_t)p.B * p.H * 128 * 128 * sizeof(float)); }

// Checkpoint of the forward group states: [G][BH][d][d] fp32 (tensor-core path only).
static size_t ckpt_bytes(const Problem &p) {
  if (padded(p)) return ckpt_bytes(padded_problem(p));
  const FwdLayout w = fwd_layout(p);
  return w.G == 0 ? 0 : (size_t)w.G * p.B * p.H * p.d * p.d * sizeof(float);
}
// workspace of linattn_fwd / linattn_bwd: the d = 128 layout, then the padded
// states (initial and final; or initial, final-state gradient and d_init)
static size_t fwd_ws_bytes(const Problem &p) {
  if (!padded(p)) return fwd_layout(p).total;
  return align256(fwd_layout(padded_problem(p)).total) + 2 * pad_state_bytes(p);
}
static size_t bwd_ws_bytes(const Problem &p) {
  if (!padded(p)) return bwd_layout(p).total;
  return align256(bwd_layout(padded_problem(p)).total) + 3 * pad_state_bytes(p);
}

// Gated layouts: the forward layout plus the gates' cumulative sums [BH][T],
// group totals [G][BH] and the forward's per-item weighting flags [G][BH]; the
// backward adds the reverse aggregates, the reverse
// group states and the per-token q . dq - k . dk of the gate gradient.  The gated checkpoint holds the
// group states and then the final state.
struct GatedLayout {
  FwdLayout f;
  size_t C = 0, tot = 0, wflag = 0, wagg = 0, rbar = 0, gx = 0, fwd_total = kHeader, bwd_total = kHeader;
};
// With gates the groups are kept to at most 2048 tokens: the gate gradient sums
// q.dq - k.dk inside a group (anchored exactly at the group ends), and those
// sums gather the error of every token of the group.
constexpr int kGatedMaxGroup = 2048;
static GatedLayout gated_layout(const Problem &p) {
  GatedLayout w;
  w.f = fwd_layout(p, kGatedMaxGroup);
  if (w.f.G == 0) return w;
  const int64_t BH = (int64_t)p.B * p.H;
  const size_t st = (size_t)w.f.G * BH * p.d * p.d * sizeof(float);
  w.C = w.f.total;
  w.tot = w.C + align256((size_t)BH * p.T * sizeof(float));
  w.wflag = w.tot + align256((size_t)w.f.G * BH * sizeof(float));
  w.fwd_total = w.wflag + align256((size_t)w.f.G * BH * sizeof(int));
  w.wagg = w.fwd_total;
  w.rbar = w.wagg + align256(st);
  w.gx = w.rbar + align256(st);
  w.bwd_total = w.gx + align256((size_t)BH * p.T * sizeof(float));
  return w;
}
static size_t ckpt_bytes_gated(const Problem &p);
// gated workspaces; bf16 d = 64 adds its padded states (initial; or final-state
// gradient and d_init) after the d = 128 layout
static size_t gated_fwd_ws_bytes(const Problem &p) {
  if (!padded(p)) return gated_layout(p).fwd_total;
  return align256(gated_layout(padded_problem(p)).fwd_total) + pad_state_bytes(p);
}
static size_t gated_bwd_ws_bytes(const Problem &p) {
  if (!padded(p)) return gated_layout(p).bwd_total;
  return align256(gated_layout(padded_problem(p)).bwd_total) + 2 * pad_state_bytes(p);
}
static size_t ckpt_bytes_gated(const Problem &p) {
  if (padded(p)) return ckpt_bytes_gated(padded_problem(p));
  const FwdLayout w = fwd_layout(p, kGatedMaxGroup);
  return w.G == 0 ? 0 : ((size_t)w.G + 1) * p.B * p.H * p.d * p.d * sizeof(float);
}

// Exclusive scan of group aggregates over the groups of a plan (per-head decay
// across each group by its own length; gates by group_log2).
static cudaError_t plan_scan(const Problem &p, const GroupPlan &gp, bool reverse, const float *local,
                             const float *init, float *out, float *total, void *ws, int *status, cudaStream_t s,
                             const float *group_log2 = nullptr) {
  return state_scan(gp.G, p.B * p.H, p.d * p.d, nullptr, group_log2 ? nullptr : p.decay, p.H, gp.L, reverse, local,
                    init, out, total, ws, status, s, group_log2, gp.kb, gp.Ls);
}

static int check_ws(void *ws, size_t bytes, size_t need) {
  if (!ws) return LINATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return LINATTN_ERR_WORKSPACE;
  if (bytes < need) return LINATTN_ERR_WORKSPACE;
  return LINATTN_OK;
}

}  // namespace linattn

using namespace linattn;

extern "C" {

int32_t linattn_abi_version(void) { return LINATTN_ABI_VERSION; }

const char *linattn_status_string(int32_t s) {
  switch (s) {
    case LINATTN_OK: return "ok";
    case LINATTN_ERR_INVALID: return "invalid argument";
    case LINATTN_ERR_UNSUPPORTED: return "unsupported shape or option";
    case LINATTN_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case LINATTN_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case LINATTN_ERR_CUDA: return "CUDA call failed";
    case LINATTN_ERR_DEVICE_TIMEOUT: return "device-side bounded wait timed out";
    case LINATTN_ERR_DEVICE: return "current device is not sm_103";
    case LINATTN_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of the allocation-free entry point";
    default: return "unknown status";
  }
}

int32_t linattn_workspace_size(const linattn_shape *shape, int32_t op, int32_t seg_len, size_t *bytes) {
  if (!bytes) return LINATTN_ERR_INVALID;
  Problem p;
  int st = validate(shape, &p);
  if (st) return st;
  if (op == LINATTN_OP_FWD) {
    *bytes = fwd_ws_bytes(p);
  } else if (op == LINATTN_OP_BWD) {
    *bytes = bwd_ws_bytes(p);
  } else if (op == LINATTN_OP_CHUNK_STATES) {
    if (seg_len < 1) return LINATTN_ERR_INVALID;
    *bytes = kHeader;
  } else if (op == LINATTN_OP_CHECKPOINT) {
    *bytes = ckpt_bytes(p);
  } else if (op == LINATTN_OP_FWD_GATED) {
    *bytes = gated_fwd_ws_bytes(p);
  } else if (op == LINATTN_OP_BWD_GATED) {
    *bytes = gated_bwd_ws_bytes(p);
  } else if (op == LINATTN_OP_CHECKPOINT_GATED) {
    *bytes = ckpt_bytes_gated(p);
  } else if (op == LINATTN_OP_SOFTMAX_SEGMENT) {
    *bytes = kHeader;
  } else if (op == LINATTN_OP_FWD_GATED_VEC || op == LINATTN_OP_BWD_GATED_VEC) {
    *bytes = kHeader + gated_vec_ws_bytes(p, op == LINATTN_OP_BWD_GATED_VEC);
  } else if (op == LINATTN_OP_CHECKPOINT_GATED_VEC) {
    *bytes = gated_vec_ckpt_bytes(p);
  } else if (op == LINATTN_OP_SOFTMAX_SEGMENT_BWD) {
    *bytes = kHeader + softmax_bwd_stats_bytes(p.B, p.H, p.T);
  } else {
    return LINATTN_ERR_INVALID;
  }
  return LINATTN_OK;
}

static int32_t fwd_impl(const linattn_shape *shape, const void *q, const void *k, const void *v, void *o,
                        const float *init_state, float *final_state, float *chunk_states, float *ckpt,
                        size_t ckpt_size, bool want_ckpt, void *workspace, size_t workspace_bytes, void *stream) {
  Problem p;
  int st = validate(shape, &p);
  if (st) return st;
  if (p.T > 0 && (st = check_ptrs({q, k, v, o}, {}))) return st;
  if ((st = check_ptrs({}, {init_state, final_state, chunk_states}))) return st;
  const bool pad = padded(p);
  const Problem pt = pad ? padded_problem(p) : p;  // the problem the kernels run
  const FwdLayout w = fwd_layout(pt);
  if ((st = check_ws(workspace, workspace_bytes, pad ? fwd_ws_bytes(p) : w.total))) return st;
  const size_t need_ckpt = want_ckpt ? ckpt_bytes(p) : 0;
  if (need_ckpt && (!ckpt || (reinterpret_cast<uintptr_t>(ckpt) & 255u) || ckpt_size < need_ckpt))
    return LINATTN_ERR_INVALID;
  if ((st = device_ok())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  int *status = reinterpret_cast<int *>(ws);
  if (clear_header(ws, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  const int64_t BH = (int64_t)p.B * p.H;
  const size_t state_bytes = (size_t)BH * p.d * p.d * sizeof(float);
  if (p.T == 0) {
    if (final_state) {
      cudaError_t e = init_state ? cudaMemcpyAsync(final_state, init_state, state_bytes,
                                                   cudaMemcpyDeviceToDevice, s)
                                 : cudaMemsetAsync(final_state, 0, state_bytes, s);
      return cuda_status(e);
    }
    return LINATTN_OK;
  }
  if (!tc_supported(pt))
    return cuda_status(simt_fwd(p, q, k, v, o, init_state, final_state, chunk_states, s));
  cudaError_t e = cudaSuccess;
  const void *qk[3] = {q, k, v};
  void *out = o;
  const float *init = init_state;
  float *fin = final_state;
  if (pad) {
    char *pb = ws + align256(w.total);
    if (init) {
      e = pad_state_d64(init_state, reinterpret_cast<float *>(pb), BH, s);
      init = reinterpret_cast<const float *>(pb);
    }
    if (fin) fin = reinterpret_cast<float *>(pb + pad_state_bytes(p));
  }
  // tensor-core path: chunk-group aggregates -> exclusive scan of the group states
  // -> chunked forward of every group from its entering state
  float *agg = reinterpret_cast<float *>(ws + w.agg);
  float *states = need_ckpt ? ckpt : reinterpret_cast<float *>(ws + w.states);
  if (e == cudaSuccess) e = tc_segment_states(pt, w.gp, qk[1], qk[2], false, agg, status, s);
  if (e == cudaSuccess) e = plan_scan(pt, w.gp, false, agg, init, states, nullptr, ws + w.scan, status, s);
  if (e == cudaSuccess) e = tc_main(pt, w.gp, qk[0], qk[1], qk[2], out, states, false, fin, status, s);
  // per-chunk (C = 64) exclusive states, when asked for: every group walked again
  // from its entering state, one state out per chunk
  if (e == cudaSuccess && chunk_states) e = tc_chunk_states(pt, w.gp, qk[1], qk[2], states, chunk_states, status, s);
  if (pad && fin && e == cudaSuccess) e = unpad_state_d64(fin, final_state, BH, s);
  return cuda_status(e);
}

int32_t linattn_fwd(const linattn_shape *shape, const void *q, const void *k, const void *v, void *o,
                    const float *init_state, float *final_state, float *chunk_states, void *workspace,
                    size_t workspace_bytes, void *stream) {
  return fwd_impl(shape, q, k, v, o, init_state, final_state, chunk_states, nullptr, 0, false, workspace,
                  workspace_bytes, stream);
}

int32_t linattn_fwd_ckpt(const linattn_shape *shape, const void *q, const void *k, const void *v, void *o,
                         const float *init_state, float *final_state, void *checkpoint,
                         size_t checkpoint_bytes, void *workspace, size_t workspace_bytes, void *stream) {
  return fwd_impl(shape, q, k, v, o, init_state, final_state, nullptr, static_cast<float *>(checkpoint),
                  checkpoint_bytes, true, workspace, workspace_bytes, stream);
}

static int32_t bwd_impl(const linattn_shape *shape, const void *q, const void *k, const void *v,
                        const void *dO, const float *init_state, const float *d_final, const float *ckpt,
                        size_t ckpt_size, bool use_ckpt, void *dq, void *dk, void *dv, float *d_init_state,
                        void *workspace, size_t workspace_bytes, void *stream) {
  Problem p;
  int st = validate(shape, &p);
  if (st) return st;
  if (p.T > 0 && (st = check_ptrs({q, k, v, dO, dq, dk, dv}, {}))) return st;
  if ((st = check_ptrs({}, {init_state, d_final, d_init_state}))) return st;
  const bool pad = padded(p);
  const Problem pt = pad ? padded_problem(p) : p;  // the problem the kernels run
  const BwdLayout w = bwd_layout(pt);
  if ((st = check_ws(workspace, workspace_bytes, pad ? bwd_ws_bytes(p) : w.total))) return st;
  const size_t need_ckpt = use_ckpt ? ckpt_bytes(p) : 0;
  if (need_ckpt && (!ckpt || (reinterpret_cast<uintptr_t>(ckpt) & 255u) || ckpt_size < need_ckpt))
    return LINATTN_ERR_INVALID;
  if ((st = device_ok())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  int *status = reinterpret_cast<int *>(ws);
  if (clear_header(ws, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  const int64_t BH = (int64_t)p.B * p.H;
  const size_t state_bytes = (size_t)BH * p.d * p.d * sizeof(float);
  if (p.T == 0) {
    // no tokens: the initial state is the final one
    if (d_init_state)
      return cuda_status(d_final ? cudaMemcpyAsync(d_init_state, d_final, state_bytes, cudaMemcpyDeviceToDevice, s)
                                 : cudaMemsetAsync(d_init_state, 0, state_bytes, s));
    return LINATTN_OK;
  }
  if (!tc_supported(pt))
    return cuda_status(simt_bwd(p, q, k, v, dO, init_state, d_final, dq, dk, dv, d_init_state, s));
  cudaError_t e = cudaSuccess;
  float *const user_dinit = d_init_state;
  if (pad) {
    char *sp = ws + align256(w.total);
    const size_t SB = pad_state_bytes(p);
    if (init_state) {
      e = pad_state_d64(init_state, reinterpret_cast<float *>(sp), BH, s);
      init_state = reinterpret_cast<const float *>(sp);
    }
    if (d_final && e == cudaSuccess) {
      e = pad_state_d64(d_final, reinterpret_cast<float *>(sp + SB), BH, s);
      d_final = reinterpret_cast<const float *>(sp + SB);
    }
    if (d_init_state) d_init_state = reinterpret_cast<float *>(sp + 2 * SB);
  }
  const GroupPlan &gp = w.f.gp;
  const int G = gp.G;
  float *agg = reinterpret_cast<float *>(ws + w.f.agg);
  float *wagg = reinterpret_cast<float *>(ws + w.wagg);
  float *rbar = reinterpret_cast<float *>(ws + w.rbar);
  // forward group states: from the checkpoint, or recomputed from k, v and init_state
  const float *states = ckpt;
  if (!need_ckpt) {
    float *st = reinterpret_cast<float *>(ws + w.f.states);
    if (e == cudaSuccess) e = tc_segment_states(pt, gp, k, v, false, agg, status, s);
    if (e == cudaSuccess) e = plan_scan(pt, gp, false, agg, init_state, st, nullptr, ws + w.f.scan, status, s);
    states = st;
  }
  // dq: the forward-time kernel with (q, k, v) := (dO, v, k), reading every
  // group's state transposed.  Reverse group states Rbar_g = sum_{u > group end}
  // lambda^{u-end} q_u dO_u^T come from group aggregates of q dO^T scanned from
  // the end (the value one step before token 0 is d_init = sum_t lambda^{t+1}
  // q_t dO_t^T).  The dq pass accumulates those aggregates too, for every head
  // without a decay or with one of at least 0.8; the aggregate pass computes
  // them for the heads with smaller decays and passes over the others.
  if (e == cudaSuccess) e = tc_main(pt, gp, dO, v, k, dq, states, true, nullptr, status, s, q, wagg);
  if (e == cudaSuccess && p.decay) e = tc_segment_states(pt, gp, q, dO, true, wagg, status, s, true);
  // A gradient D arriving at the final state enters the reverse scan across the
  // last group, whose length may be short of L: fold lambda^{len} D into that
  // group's aggregate, scan from zero, and give the last group D itself.
  const int64_t E = BH * pt.d * pt.d;
  if (e == cudaSuccess && d_final)
    e = fold_state(wagg + (int64_t)(G - 1) * E, d_final, p.decay, p.H, pt.d * pt.d, gp.len(G - 1, p.T), E, s);
  if (e == cudaSuccess) e = plan_scan(pt, gp, true, wagg, nullptr, rbar, d_init_state, ws + w.f.scan, status, s);
  if (e == cudaSuccess && d_final)
    e = cudaMemcpyAsync(rbar + (int64_t)(G - 1) * E, d_final, (size_t)E * sizeof(float), cudaMemcpyDeviceToDevice, s);
  // dv and dk in one reverse-time pass from the states Rbar
  if (e == cudaSuccess) e = tc_dual(pt, gp, q, k, v, dO, dk, dv, rbar, status, s);
  if (pad && user_dinit && e == cudaSuccess) e = unpad_state_d64(d_init_state, user_dinit, BH, s);
  return cuda_status(e);
}

int32_t linattn_bwd(const linattn_shape *shape, const void *q, const void *k, const void *v,
                    const void *dO, const float *init_state, const float *d_final_state, void *dq,
                    void *dk, void *dv, float *d_init_state, void *workspace, size_t workspace_bytes,
                    void *stream) {
  return bwd_impl(shape, q, k, v, dO, init_state, d_final_state, nullptr, 0, false, dq, dk, dv, d_init_state,
                  workspace, workspace_bytes, stream);
}

int32_t linattn_bwd_ckpt(const linattn_shape *shape, const void *q, const void *k, const void *v,
                         const void *dO, const float *init_state, const float *d_final_state,
                         const void *checkpoint, size_t checkpoint_bytes, void *dq, void *dk, void *dv,
                         float *d_init_state, void *workspace, size_t workspace_bytes, void *stream) {
  return bwd_impl(shape, q, k, v, dO, init_state, d_final_state, static_cast<const float *>(checkpoint),
                  checkpoint_bytes, true, dq, dk, dv, d_init_state, workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------------ data-dependent gates
static int gated_checks(const linattn_shape *shape, Problem *p, const float *log_gate, const void *ckpt,
                        size_t ckpt_size) {
  int st = validate(shape, p);
  if (st) return st;
  if (p->decay) return LINATTN_ERR_INVALID;  // gates replace the per-head decay
  if (p->T > 0 && (st = check_ptrs({log_gate}, {}))) return st;
  const size_t need = ckpt_bytes_gated(*p);
  if (need && (!ckpt || (reinterpret_cast<uintptr_t>(ckpt) & 255u) || ckpt_size < need)) return LINATTN_ERR_INVALID;
  return LINATTN_OK;
}

int32_t linattn_fwd_gated(const linattn_shape *shape, const void *q, const void *k, const void *v,
                          const float *log_gate, void *o, const float *init_state, float *final_state,
                          void *checkpoint, size_t checkpoint_bytes, void *workspace, size_t workspace_bytes,
                          void *stream) {
  Problem p;
  int st = gated_checks(shape, &p, log_gate, checkpoint, checkpoint_bytes);
  if (st) return st;
  if (p.T > 0 && (st = check_ptrs({q, k, v, o}, {}))) return st;
  if ((st = check_ptrs({}, {init_state, final_state}))) return st;
  const bool pad = padded(p);
  Problem pt = pad ? padded_problem(p) : p;  // the problem the kernels run
  const GatedLayout w = gated_layout(pt);
  if ((st = check_ws(workspace, workspace_bytes, gated_fwd_ws_bytes(p)))) return st;
  if ((st = device_ok())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  int *status = reinterpret_cast<int *>(ws);
  if (clear_header(ws, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  const int64_t BH = (int64_t)p.B * p.H;
  const size_t state_bytes = (size_t)BH * p.d * p.d * sizeof(float);
  if (p.T == 0) {
    if (final_state) {
      cudaError_t e = init_state ? cudaMemcpyAsync(final_state, init_state, state_bytes,
                                                   cudaMemcpyDeviceToDevice, s)
                                 : cudaMemsetAsync(final_state, 0, state_bytes, s);
      return cuda_status(e);
    }
    return LINATTN_OK;
  }
  // CUDA-core path (fp32 inputs): one sequential walk, no checkpoint
  if (!tc_supported(pt)) return cuda_status(simt_fwd(p, q, k, v, o, init_state, final_state, nullptr, s, log_gate));
  const GroupPlan &gp = w.f.gp;
  const int G = gp.G;
  float *C = reinterpret_cast<float *>(ws + w.C), *tot = reinterpret_cast<float *>(ws + w.tot);
  float *agg = reinterpret_cast<float *>(ws + w.f.agg);
  float *states = static_cast<float *>(checkpoint);
  float *fin = states + (size_t)G * BH * pt.d * pt.d;  // the checkpoint's final state
  int *wflag = reinterpret_cast<int *>(ws + w.wflag);
  cudaError_t e = gate_prep(pt, gp, log_gate, C, tot, wflag, s);
  const float *init = init_state;
  if (pad && init && e == cudaSuccess) {
    float *ip = reinterpret_cast<float *>(ws + align256(w.fwd_total));
    e = pad_state_d64(init_state, ip, BH, s);
    init = ip;
  }
  pt.gC = C;
  pt.gtot = tot;
  pt.gflag = wflag;  // the chunked forward may weight its operands
  if (e == cudaSuccess) e = tc_segment_states(pt, gp, k, v, false, agg, status, s);
  if (e == cudaSuccess) e = plan_scan(pt, gp, false, agg, init, states, nullptr, ws + w.f.scan, status, s, tot);
  if (e == cudaSuccess) e = tc_main(pt, gp, q, k, v, o, states, false, fin, status, s);
  if (e == cudaSuccess && final_state)
    e = pad ? unpad_state_d64(fin, final_state, BH, s)
            : cudaMemcpyAsync(final_state, fin, state_bytes, cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

int32_t linattn_bwd_gated(const linattn_shape *shape, const void *q, const void *k, const void *v,
                          const void *dO, const float *log_gate, const float *init_state,
                          const float *d_final_state, const void *checkpoint, size_t checkpoint_bytes, void *dq,
                          void *dk, void *dv, float *d_log_gate, float *d_init_state, void *workspace,
                          size_t workspace_bytes, void *stream) {
  Problem p;
  int st = gated_checks(shape, &p, log_gate, checkpoint, checkpoint_bytes);
  if (st) return st;
  if (p.T > 0 && (st = check_ptrs({q, k, v, dO, dq, dk, dv, d_log_gate}, {}))) return st;
  if ((st = check_ptrs({}, {init_state, d_final_state, d_init_state}))) return st;
  const bool pad = padded(p);
  Problem pt = pad ? padded_problem(p) : p;  // the problem the kernels run
  const GatedLayout w = gated_layout(pt);
  if ((st = check_ws(workspace, workspace_bytes, gated_bwd_ws_bytes(p)))) return st;
  if ((st = device_ok())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  int *status = reinterpret_cast<int *>(ws);
  if (clear_header(ws, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  const int64_t BH = (int64_t)p.B * p.H;
  const size_t user_state_bytes = (size_t)BH * p.d * p.d * sizeof(float);
  if (p.T == 0) {
    if (d_init_state)
      return cuda_status(d_final_state ? cudaMemcpyAsync(d_init_state, d_final_state, user_state_bytes,
                                                         cudaMemcpyDeviceToDevice, s)
                                       : cudaMemsetAsync(d_init_state, 0, user_state_bytes, s));
    return LINATTN_OK;
  }
  // CUDA-core path: recomputes the forward states from init_state (the checkpoint is empty)
  if (!tc_supported(pt))
    return cuda_status(simt_bwd(p, q, k, v, dO, init_state, d_final_state, dq, dk, dv, d_init_state, s, log_gate,
                                d_log_gate));
  const int64_t E = BH * pt.d * pt.d;
  const size_t state_bytes = (size_t)E * sizeof(float);
  const GroupPlan &gp = w.f.gp;
  const int G = gp.G;
  float *C = reinterpret_cast<float *>(ws + w.C), *tot = reinterpret_cast<float *>(ws + w.tot);
  float *wagg = reinterpret_cast<float *>(ws + w.wagg), *rbar = reinterpret_cast<float *>(ws + w.rbar);
  const float *states = static_cast<const float *>(checkpoint);
  const float *fin = states + (size_t)G * E;
  // per-item flags: the dq and dk/dv passes take the weighted-operand form together
  int *wflag = reinterpret_cast<int *>(ws + w.wflag);
  cudaError_t e = gate_prep(pt, gp, log_gate, C, tot, wflag, s);
  // bf16 d = 64: the final-state gradient in, d_init out through padded states
  const float *dfin = d_final_state;
  float *dinit = d_init_state;
  if (pad) {
    float *sp = reinterpret_cast<float *>(ws + align256(w.bwd_total));
    if (dfin && e == cudaSuccess) {
      e = pad_state_d64(d_final_state, sp, BH, s);
      dfin = sp;
    }
    if (dinit) dinit = reinterpret_cast<float *>(ws + align256(w.bwd_total) + pad_state_bytes(p));
  }
  pt.gC = C;
  pt.gtot = tot;
  pt.gflag = wflag;
  pt.gq = q;
  pt.gk = k;
  pt.gx = reinterpret_cast<float *>(ws + w.gx);
  // dq: forward-time kernel with (q, k, v) := (dO, v, k) from the group states (transposed),
  // which also accumulates the reverse group aggregates sum_s exp2(C_s) q_s dO_s^T of the
  // items in the weighted form; the aggregate pass forms those of the other items
  if (e == cudaSuccess) e = tc_main(pt, gp, dO, v, k, dq, states, true, nullptr, status, s, q, wagg);
  if (e == cudaSuccess) e = tc_segment_states(pt, gp, q, dO, true, wagg, status, s, true);
  // the final-state gradient folded across the last group, and the reverse scan with
  // every group's own multiplier
  if (e == cudaSuccess && dfin)
    e = fold_state_log2(wagg + (int64_t)(G - 1) * E, dfin, tot + (int64_t)(G - 1) * BH, pt.d * pt.d, E, s);
  if (e == cudaSuccess) e = plan_scan(pt, gp, true, wagg, nullptr, rbar, dinit, ws + w.f.scan, status, s, tot);
  if (e == cudaSuccess && dfin)
    e = cudaMemcpyAsync(rbar + (int64_t)(G - 1) * E, dfin, state_bytes, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = tc_dual(pt, gp, q, k, v, dO, dk, dv, rbar, status, s);
  if (e == cudaSuccess) e = gate_grad(pt, gp, pt.gx, rbar, states, dfin, fin, d_log_gate, s);
  if (pad && d_init_state && e == cudaSuccess) e = unpad_state_d64(dinit, d_init_state, BH, s);
  return cuda_status(e);
}

static int check_vec_ckpt(const Problem &p, const void *ckpt, size_t ckpt_size, bool use_ckpt) {
  const size_t need = use_ckpt ? gated_vec_ckpt_bytes(p) : 0;
  if (need && (!ckpt || (reinterpret_cast<uintptr_t>(ckpt) & 255u) || ckpt_size < need)) return LINATTN_ERR_INVALID;
  return LINATTN_OK;
}

static int32_t fwd_gated_vec_impl(const linattn_shape *shape, const void *q, const void *k, const void *v,
                                  const float *log_gate, void *o, const float *init_state, float *final_state,
                                  void *ckpt, size_t ckpt_size, bool use_ckpt, void *workspace,
                                  size_t workspace_bytes, void *stream) {
  Problem p;
  int st = validate(shape, &p);
  if (st) return st;
  if (p.decay) return LINATTN_ERR_INVALID;  // the gates replace the per-head decay
  if ((st = check_ptrs({}, {init_state, final_state}))) return st;
  if ((st = check_ws(workspace, workspace_bytes, kHeader + gated_vec_ws_bytes(p, false)))) return st;
  if ((st = check_vec_ckpt(p, ckpt, ckpt_size, use_ckpt))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.T == 0) {
    if (!final_state) return LINATTN_OK;
    const size_t bytes = (size_t)p.B * p.H * p.d * p.d * sizeof(float);
    return cuda_status(init_state ? cudaMemcpyAsync(final_state, init_state, bytes, cudaMemcpyDeviceToDevice, s)
                                  : cudaMemsetAsync(final_state, 0, bytes, s));
  }
  if ((st = check_ptrs({q, k, v, o, log_gate}, {}))) return st;
  if ((st = device_ok())) return st;
  if (clear_header(workspace, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  return cuda_status(gated_vec_fwd(p, q, k, v, log_gate, o, init_state, final_state,
                                   static_cast<char *>(workspace) + kHeader,
                                   use_ckpt && gated_vec_ckpt_bytes(p) ? ckpt : nullptr, s));
}

int32_t linattn_fwd_gated_vec(const linattn_shape *shape, const void *q, const void *k, const void *v,
                              const float *log_gate, void *o, const float *init_state, float *final_state,
                              void *workspace, size_t workspace_bytes, void *stream) {
  return fwd_gated_vec_impl(shape, q, k, v, log_gate, o, init_state, final_state, nullptr, 0, false, workspace,
                            workspace_bytes, stream);
}

int32_t linattn_fwd_gated_vec_ckpt(const linattn_shape *shape, const void *q, const void *k, const void *v,
                                   const float *log_gate, void *o, const float *init_state, float *final_state,
                                   void *checkpoint, size_t checkpoint_bytes, void *workspace,
                                   size_t workspace_bytes, void *stream) {
  return fwd_gated_vec_impl(shape, q, k, v, log_gate, o, init_state, final_state, checkpoint, checkpoint_bytes,
                            true, workspace, workspace_bytes, stream);
}

static int32_t bwd_gated_vec_impl(const linattn_shape *shape, const void *q, const void *k, const void *v,
                                  const void *dO, const float *log_gate, const float *init_state,
                                  const float *d_final_state, const void *ckpt, size_t ckpt_size, bool use_ckpt,
                                  void *dq, void *dk, void *dv, float *d_log_gate, float *d_init_state,
                                  void *workspace, size_t workspace_bytes, void *stream) {
  Problem p;
  int st = validate(shape, &p);
  if (st) return st;
  if (p.decay) return LINATTN_ERR_INVALID;
  if ((st = check_ptrs({}, {init_state, d_final_state, d_init_state}))) return st;
  if ((st = check_ws(workspace, workspace_bytes, kHeader + gated_vec_ws_bytes(p, true)))) return st;
  if ((st = check_vec_ckpt(p, ckpt, ckpt_size, use_ckpt))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.T == 0) {
    if (!d_init_state) return LINATTN_OK;
    const size_t bytes = (size_t)p.B * p.H * p.d * p.d * sizeof(float);
    return cuda_status(d_final_state
                           ? cudaMemcpyAsync(d_init_state, d_final_state, bytes, cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(d_init_state, 0, bytes, s));
  }
  if ((st = check_ptrs({q, k, v, dO, log_gate, dq, dk, dv, d_log_gate}, {}))) return st;
  if ((st = device_ok())) return st;
  if (clear_header(workspace, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  return cuda_status(gated_vec_bwd(p, q, k, v, dO, log_gate, init_state, d_final_state, dq, dk, dv, d_log_gate,
                                   d_init_state, static_cast<char *>(workspace) + kHeader,
                                   use_ckpt && gated_vec_ckpt_bytes(p) ? ckpt : nullptr, s));
}

int32_t linattn_bwd_gated_vec(const linattn_shape *shape, const void *q, const void *k, const void *v,
                              const void *dO, const float *log_gate, const float *init_state,
                              const float *d_final_state, void *dq, void *dk, void *dv, float *d_log_gate,
                              float *d_init_state, void *workspace, size_t workspace_bytes, void *stream) {
  return bwd_gated_vec_impl(shape, q, k, v, dO, log_gate, init_state, d_final_state, nullptr, 0, false, dq, dk, dv,
                            d_log_gate, d_init_state, workspace, workspace_bytes, stream);
}

int32_t linattn_bwd_gated_vec_ckpt(const linattn_shape *shape, const void *q, const void *k, const void *v,
                                   const void *dO, const float *log_gate, const float *init_state,
                                   const float *d_final_state, const void *checkpoint, size_t checkpoint_bytes,
                                   void *dq, void *dk, void *dv, float *d_log_gate, float *d_init_state,
                                   void *workspace, size_t workspace_bytes, void *stream) {
  return bwd_gated_vec_impl(shape, q, k, v, dO, log_gate, init_state, d_final_state, checkpoint, checkpoint_bytes,
                            true, dq, dk, dv, d_log_gate, d_init_state, workspace, workspace_bytes, stream);
}

int32_t linattn_decode(const linattn_shape *shape, const void *q, const void *k, const void *v, void *o,
                       float *state, void *stream) {
  Problem p;
  int st = validate(shape, &p);
  if (st) return st;
  if (p.T == 0) return LINATTN_OK;
  if ((st = check_ptrs({q, k, v, o, state}, {}))) return st;
  if ((st = device_ok())) return st;
  return cuda_status(decode(p, q, k, v, o, state, static_cast<cudaStream_t>(stream)));
}

static int32_t chunk_states_impl(const linattn_shape *shape, int32_t seg_len, const void *x, const void *y,
                                 bool reverse, float *out, void *workspace, size_t workspace_bytes, void *stream) {
  Problem p;
  int st = validate(shape, &p);
  if (st) return st;
  if (seg_len < 1) return LINATTN_ERR_INVALID;
  if (p.T < 1 || p.T % seg_len) return LINATTN_ERR_UNSUPPORTED;
  if ((st = check_ptrs({x, y, out}, {}))) return st;
  if ((st = check_ws(workspace, workspace_bytes, kHeader))) return st;
  if ((st = device_ok())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int *status = reinterpret_cast<int *>(workspace);
  if (clear_header(workspace, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  if (tc_supported(p) && seg_len % 128 == 0)
    return cuda_status(tc_segment_states(p, GroupPlan::uniform(p.T, seg_len), x, y, reverse, out, status, s));
  if (padded(p) && seg_len % 128 == 0)  // bf16 d = 64: the d = 128 kernel, 64 x 64 states stored
    return cuda_status(tc_segment_states(padded_problem(p), GroupPlan::uniform(p.T, seg_len), x, y, reverse, out,
                                         status, s, false, 64));
  return cuda_status(simt_segment_states(p, seg_len, x, y, reverse, out, s));
}

int32_t linattn_chunk_states(const linattn_shape *shape, int32_t seg_len, const void *k, const void *v,
                             float *local_states, void *workspace, size_t workspace_bytes, void *stream) {
  return chunk_states_impl(shape, seg_len, k, v, false, local_states, workspace, workspace_bytes, stream);
}

int32_t linattn_chunk_states_rev(const linattn_shape *shape, int32_t seg_len, const void *q, const void *dO,
                                 float *local_grad_states, void *workspace, size_t workspace_bytes,
                                 void *stream) {
  return chunk_states_impl(shape, seg_len, q, dO, true, local_grad_states, workspace, workspace_bytes, stream);
}

int32_t linattn_state_scan_workspace_size(int32_t G, int32_t BH, int32_t dk, int32_t dv, size_t *bytes) {
  if (!bytes || G < 1 || BH < 1 || dk < 1 || dv < 1) return LINATTN_ERR_INVALID;
  if (((int64_t)dk * dv) % 8) return LINATTN_ERR_UNSUPPORTED;
  *bytes = kHeader + scan_workspace_bytes(G, (int64_t)BH * dk * dv);
  return LINATTN_OK;
}

int32_t linattn_state_scan(int32_t G, int32_t BH, int32_t dk, int32_t dv, const float *seg_decay,
                           const float *local_states, const float *init, float *init_states,
                           float *total, void *workspace, size_t workspace_bytes, void *stream) {
  size_t need = 0;
  int st = linattn_state_scan_workspace_size(G, BH, dk, dv, &need);
  if (st) return st;
  if ((st = check_ptrs({local_states, init_states}, {seg_decay, init, total}))) return st;
  if ((st = check_ws(workspace, workspace_bytes, need))) return st;
  if ((st = device_ok())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  if (clear_header(ws, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  return cuda_status(state_scan(G, BH, dk * dv, seg_decay, nullptr, 1, 1, false, local_states, init,
                                init_states, total, ws + kHeader, reinterpret_cast<int *>(ws), s));
}

int32_t linattn_softmax_segment_fwd(const linattn_shape *q_shape, const linattn_shape *kv_shape, const void *q,
                                    const void *k, const void *v, void *o, float *lse, float softmax_scale,
                                    void *workspace, size_t workspace_bytes, void *stream) {
  Problem pq, pk;
  int st = validate(q_shape, &pq);
  if (st) return st;
  if ((st = validate(kv_shape, &pk))) return st;
  if (pq.B != pk.B || pq.H != pk.H || pq.d != pk.d || pq.dtype != pk.dtype || pk.T < pq.T) return LINATTN_ERR_INVALID;
  if (pq.decay || pk.decay) return LINATTN_ERR_INVALID;
  if (pq.dtype != 0 || pq.d != 128) return LINATTN_ERR_UNSUPPORTED;
  if (!(softmax_scale > 0.f) && softmax_scale != 0.f) return LINATTN_ERR_INVALID;
  if (pq.T > 0 && (st = check_ptrs({q, k, v, o}, {lse}))) return st;
  if ((st = check_ws(workspace, workspace_bytes, kHeader))) return st;
  if ((st = device_ok())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (clear_header(workspace, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  if (pq.T == 0) return LINATTN_OK;
  SoftmaxProblem sp;
  sp.B = pq.B; sp.H = pq.H; sp.Tq = pq.T; sp.Tk = pk.T;
  sp.qsb = pq.sb; sp.qsh = pq.sh; sp.qst = pq.st;
  sp.ksb = pk.sb; sp.ksh = pk.sh; sp.kst = pk.st;
  sp.scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf((float)pq.d);
  sp.num_sms = pq.num_sms;
  return cuda_status(softmax_segment(sp, q, k, v, o, lse, static_cast<int *>(workspace), s));
}

int32_t linattn_softmax_segment_bwd(const linattn_shape *q_shape, const linattn_shape *kv_shape, const void *q,
                                    const void *k, const void *v, const void *o, const void *dO, const float *lse,
                                    void *dq, void *dk, void *dv, float softmax_scale, void *workspace,
                                    size_t workspace_bytes, void *stream) {
  Problem pq, pk;
  int st = validate(q_shape, &pq);
  if (st) return st;
  if ((st = validate(kv_shape, &pk))) return st;
  if (pq.B != pk.B || pq.H != pk.H || pq.d != pk.d || pq.dtype != pk.dtype || pk.T < pq.T) return LINATTN_ERR_INVALID;
  if (pq.decay || pk.decay) return LINATTN_ERR_INVALID;
  if (pq.dtype != 0 || pq.d != 128) return LINATTN_ERR_UNSUPPORTED;
  if (!(softmax_scale > 0.f) && softmax_scale != 0.f) return LINATTN_ERR_INVALID;
  if (pq.T > 0 && (st = check_ptrs({q, k, v, o, dO, lse, dq, dk, dv}, {}))) return st;
  if (pq.T == 0 && pk.T > 0 && (st = check_ptrs({dk, dv}, {}))) return st;
  if ((st = check_ws(workspace, workspace_bytes, kHeader + softmax_bwd_stats_bytes(pq.B, pq.H, pq.T)))) return st;
  if ((st = device_ok())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (clear_header(workspace, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  SoftmaxProblem sp;
  sp.B = pq.B; sp.H = pq.H; sp.Tq = pq.T; sp.Tk = pk.T;
  sp.qsb = pq.sb; sp.qsh = pq.sh; sp.qst = pq.st;
  sp.ksb = pk.sb; sp.ksh = pk.sh; sp.kst = pk.st;
  sp.scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf((float)pq.d);
  sp.num_sms = pq.num_sms;
  char *ws = static_cast<char *>(workspace);
  return cuda_status(softmax_segment_bwd(sp, q, k, v, o, dO, lse, dq, dk, dv, reinterpret_cast<float *>(ws + kHeader),
                                         reinterpret_cast<int *>(ws), s));
}

int32_t linattn_segment_decay(const float *decay, int32_t B, int32_t H, int32_t seg_len, float *out,
                              void *stream) {
  if (B < 1 || H < 1 || seg_len < 0 || (int64_t)B * H > (1 << 30)) return LINATTN_ERR_INVALID;
  int st = check_ptrs({decay, out}, {});
  if (st) return st;
  if ((st = device_ok())) return st;
  return cuda_status(segment_decay(decay, B, H, seg_len, out, static_cast<cudaStream_t>(stream)));
}

int32_t linattn_diag_scan_withhold(int32_t G, int32_t BH, int32_t dk, int32_t dv, const float *local_states,
                                   float *init_states, int32_t withhold_tile, double wait_limit_ms,
                                   void *workspace, size_t workspace_bytes, void *stream) {
  size_t need = 0;
  int st = linattn_state_scan_workspace_size(G, BH, dk, dv, &need);
  if (st) return st;
  if ((st = check_ptrs({local_states, init_states}, {}))) return st;
  if ((st = check_ws(workspace, workspace_bytes, need))) return st;
  const int64_t ntiles = (int64_t)((G + 31) / 32) * ((int64_t)BH * dk * dv / 8);
  if (withhold_tile < 0 || withhold_tile >= ntiles || !(wait_limit_ms > 0 && wait_limit_ms <= 2000))
    return LINATTN_ERR_INVALID;
  if ((st = device_ok())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  if (clear_header(ws, kHeader, s) != cudaSuccess) return LINATTN_ERR_CUDA;
  return cuda_status(state_scan(G, BH, dk * dv, nullptr, nullptr, 1, 1, false, local_states, nullptr, init_states,
                                nullptr, ws + kHeader, reinterpret_cast<int *>(ws), s, nullptr, 1 << 30, 0,
                                (uint64_t)(wait_limit_ms * 1e6), withhold_tile));
}

int32_t linattn_device_status(const void *workspace, void *stream) {
  if (!workspace) return LINATTN_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int h = 0;
  if (cudaMemcpyAsync(&h, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return LINATTN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LINATTN_ERR_CUDA;
  return h;
}

int32_t linattn_timing_enable(int32_t on) {
  TimingState &t = timing();
  std::lock_guard<std::mutex> g(t.mu);
  t.on = on != 0;
  return LINATTN_OK;
}

int32_t linattn_timing_collect(int32_t max_kinds, int32_t *launches, float *total_ms) {
  if (max_kinds < 0 || (max_kinds > 0 && (!launches || !total_ms))) return LINATTN_ERR_INVALID;
  TimingState &t = timing();
  std::lock_guard<std::mutex> g(t.mu);
  for (int k = 0; k < max_kinds; ++k) {
    launches[k] = 0;
    total_ms[k] = 0.f;
  }
  int status = LINATTN_OK;
  for (const auto &r : t.recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(t.pool[2 * r.slot + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, t.pool[2 * r.slot], t.pool[2 * r.slot + 1]) != cudaSuccess) {
      status = LINATTN_ERR_CUDA;
      continue;
    }
    if (r.kind < max_kinds) {
      launches[r.kind] += 1;
      total_ms[r.kind] += ms;
    }
  }
  t.recs.clear();
  t.used = 0;
  return status == LINATTN_OK ? (int32_t)K_KINDS : status;
}

const char *linattn_kernel_name(int32_t kind) {
  static const char *names[K_KINDS] = {"simt_fwd", "simt_bwd", "simt_segment_states", "state_scan",
                                       "tc_segment_aggregate", "tc_chunked_fwd",
                                       "diag_mma", "decode", "tc_dual_rev", "tc_chunked_fwd_agg",
                                       "gate_prep_and_grad", "tc_chunk_states", "softmax_segment",
                                       "gated_vec_fwd", "gated_vec_bwd", "pad_d64", "softmax_bwd_prep",
                                       "softmax_bwd_dkdv", "softmax_bwd_dq", "clear_status"};
  return (kind >= 0 && kind < K_KINDS) ? names[kind] : "?";
}

int32_t linattn_diag_mma(int32_t mode, const void *A, const void *B, float *D, void *stream) {
  if (mode < 0 || mode > 4) return LINATTN_ERR_INVALID;
  int st = check_ptrs({A, B, D}, {});
  if (st) return st;
  if ((st = device_ok())) return st;
  return cuda_status(diag_mma(mode, A, B, D, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
