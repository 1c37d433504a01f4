// Internal declarations shared by the host entry points and the kernel files.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace linattn {

// Launches with programmatic stream serialization: the kernel may start (up to its
// griddep_wait, which every kernel launched this way calls before its first global
// memory access) while the kernel before it on the stream finishes, so that its
// prologue overlaps that kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// A validated request.  Sequence tensors are [B, H, T, d] with element strides
// (sb, sh, st); states are [B*H, d, d] fp32.
struct Problem {
  int B, H, T, d;
  int dtype;            // 0 bf16, 1 fp32
  int64_t sb, sh, st;   // element strides
  const float *decay;   // [H] device, or nullptr (lambda = 1)
  int num_sms;
  // data-dependent gates (tensor-core path): group-local log2 cumulative sums
  // [B*H][T] and group totals [G][B*H] for the group length in use, or nullptr
  const float *gC = nullptr, *gtot = nullptr;
  // gated forward: per (group, sequence) item [G][B*H], nonzero when every
  // 128-token block of the group keeps its cumulative sums, and the one before
  // it, within a span of kGateWeightedSpan (the weighted-operand form applies)
  const int *gflag = nullptr;
  // gates, backward: q and k (bf16, the request's strides) and gx [B*H][T] fp32,
  // which the dq pass fills with q_t . dq_t and the dk/dv pass reduces by k_t . dk_t
  const void *gq = nullptr, *gk = nullptr;
  float *gx = nullptr;
  // bf16 d = 64 on the d = 128 tensor-core kernels: the sequence tensors have 64
  // columns (their tensor maps say so: the tiles' columns 64..127 load as zeros,
  // and only the first 64 output columns are stored); 0 means d
  int dcols = 0;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------- chunk groups
// How a sequence of T tokens is cut into chunk groups (the units of the state
// scan and the items of the persistent kernels): kb groups of L tokens, then
// groups of Ls <= L tokens, the last one possibly shorter.  The long groups
// come first, so the items a launch hands out last are short ones.  A uniform
// cut has kb >= G.
struct GroupPlan {
  int G = 0, L = 0, kb = 0, Ls = 0;
  __host__ __device__ int start(int g) const { return g <= kb ? g * L : kb * L + (g - kb) * Ls; }
  __host__ __device__ int len(int g, int T) const {
    const int e = start(g + 1);
    return (e < T ? e : T) - start(g);
  }
  static GroupPlan uniform(int T, int L) {
    GroupPlan gp;
    gp.G = (T + L - 1) / L;
    gp.L = gp.Ls = L;
    gp.kb = gp.G;
    return gp;
  }
};

// LINATTN_OK when the current device is an sm_103 GPU (api.cu).
int device_ok();

// ---------------------------------------------------------------- per-kernel timing (api.cu)
enum KernelKind {
  K_SIMT_FWD = 0, K_SIMT_BWD, K_SIMT_SEGMENT, K_SCAN, K_TC_AGG, K_TC_MAIN_FWD, K_DIAG,
  K_DECODE, K_TC_DUAL_REV, K_TC_MAIN_AGG, K_GATE, K_TC_CHUNK_STATES, K_SOFTMAX_SEGMENT, K_GATED_VEC_FWD,
  K_GATED_VEC_BWD, K_PAD_D64, K_SOFTMAX_BWD_PREP, K_SOFTMAX_BWD_KV, K_SOFTMAX_BWD_Q, K_CLEAR_STATUS, K_KINDS
};
// Records timing events around one launch on `s` while timing is enabled.
struct TimedLaunch {
  TimedLaunch(int kind, cudaStream_t s);
  ~TimedLaunch();
  int kind, slot;
  cudaStream_t stream;
};

// Zeroes `bytes` (a multiple of 4, at most 1024) at the start of a workspace (its
// status word and item counters) on the stream.  A kernel rather than a memset, so
// that it takes part in the overlapped launches: it waits for the kernel before it,
// and the next kernel may start its prologue meanwhile.
cudaError_t clear_header(void *ws, size_t bytes, cudaStream_t s);

// ---------------------------------------------------------------- SIMT path (simt.cu)
// log_gate ([BH][T] fp32, natural log of the per-token gates) replaces the per-head
// decay when non-null; the backward then also writes d_log_gate ([BH][T] fp32).
cudaError_t simt_fwd(const Problem &p, const void *q, const void *k, const void *v, void *o,
                     const float *init, float *final_state, float *chunk_states, cudaStream_t s,
                     const float *log_gate = nullptr);
cudaError_t simt_bwd(const Problem &p, const void *q, const void *k, const void *v, const void *dO,
                     const float *init, const float *d_final, void *dq, void *dk, void *dv, float *dinit,
                     cudaStream_t s, const float *log_gate = nullptr, float *d_log_gate = nullptr);
// Segment sums of w_s x_s y_s^T: w_s = lambda^{end - s}, or lambda^{s - start + 1} when reverse.
cudaError_t simt_segment_states(const Problem &p, int seg_len, const void *x, const void *y, bool reverse,
                                float *out, cudaStream_t s);

// ---------------------------------------------------------------- state scan (scan.cu)
// Exclusive scan over G segments of E = BH * DD fp32 elements each ([G][BH][DD]).
// Per-(bh) multiplier: seg_decay[bh] if given; else decay_h[bh % H]^seg_len if
// decay_h is given; else 1.  reverse: scan from g = G-1 down to 0 (out[G-1] =
// init, out[g] = a * out[g+1] + local[g+1]).  total (optional) is the value one
// step past the end.
size_t scan_workspace_bytes(int G, int64_t E);
// group_log2 (optional, [G][BH], G <= 256): log2 of every group's own multiplier,
// replacing the uniform one (data-dependent gates).  With decay_h, groups from
// index kb on (G <= 256) have seg_len2 tokens instead of seg_len (a GroupPlan).
// limit_ns bounds every look-back wait (0: LINATTN_LOOKBACK_LIMIT_MS from the
// environment, else 2 s); withhold >= 0 (diagnostics) forces the look-back form
// and keeps that tile from ever publishing, so its successors' waits give up.
cudaError_t state_scan(int G, int BH, int DD, const float *seg_decay, const float *decay_h, int H,
                       int seg_len, bool reverse, const float *local, const float *init, float *out,
                       float *total, void *ws, int *status, cudaStream_t s, const float *group_log2 = nullptr,
                       int kb = 1 << 30, int seg_len2 = 0, uint64_t limit_ns = 0, int withhold = -1);
// Bound of the device-side waits on other CTAs' results (the scan's look-back):
// LINATTN_LOOKBACK_LIMIT_MS from the environment, else 2 s.
uint64_t wait_limit_ns();

// out[b * H + h] = decay_h[h]^len for b < B (the scan multiplier of a segment of len tokens).
cudaError_t segment_decay(const float *decay_h, int B, int H, int len, float *out, cudaStream_t s);

// w[i] += lambda_h^len d[i] over n = BH * DD elements (h = (i / DD) % H; lambda = 1
// without decay_h): folds a state entering across a segment of len tokens into
// that segment's aggregate.
cudaError_t fold_state(float *w, const float *d, const float *decay_h, int H, int DD, int len, int64_t n,
                       cudaStream_t s);

// ---------------------------------------------------------------- data-dependent gates (gate.cu)
// C[t] = log2(e) * sum of log_gate over the group of L tokens up to t ([B,H,T]);
// tot[g][bh] = C at the group's last token; wflag[g][bh] (if not null) =
// whether every 128-token block of the group, with the sum before it, spans
// at most kGateWeightedSpan.
constexpr float kGateWeightedSpan = 60.f;
cudaError_t gate_prep(const Problem &p, const GroupPlan &gp, const float *log_gate, float *C, float *tot,
                      int *wflag, cudaStream_t s);
// w[i] += exp2(tot_last[i / DD]) d[i], n elements.
cudaError_t fold_state_log2(float *w, const float *d, const float *tot_last, int DD, int64_t n, cudaStream_t s);
// d_log_gate [B,H,T]: reverse sums of gx [B*H][T] (q_t . dq_t - k_t . dk_t) inside each
// group, plus <rbar[g], states[g+1]> (<d_final, final_state> for the last group).
cudaError_t gate_grad(const Problem &p, const GroupPlan &gp, const float *gx, const float *rbar, const float *states,
                      const float *d_final, const float *final_state, float *dlg, cudaStream_t s);

// ---------------------------------------------------------------- tensor-core path (tc.cu)
// The persistent kernels take `status`, the start of the workspace's 256-byte
// header (zeroed by every entry point): int 0 is the status word, ints 1..16 a
// per-warp record of a wait that gave up, and each kernel kind keeps the two
// counters of its dynamic item order at these offsets (each launch leaves them
// zero again, so one call may launch a kind more than once).
constexpr int kCounterAgg = 32, kCounterMain = 34, kCounterDual = 36, kCounterChunk = 38, kCounterSoftmax = 40,
              kCounterSoftmaxKV = 42, kCounterSoftmaxQ = 44;
bool tc_supported(const Problem &p);   // bf16, d = 128
// The chunk groups of the tensor-core path (lengths multiples of 128, at most
// 256 groups); max_len > 0 caps the lengths where possible.
GroupPlan tc_group_plan(const Problem &p, int max_len = 0);
// Segment aggregates sum_s w_s x_s y_s^T over groups of seg_len tokens (seg_len
// a multiple of 128), written as [G][BH][d][d] fp32.
//   reverse == false: w_s = lambda^{end - s};  reverse == true: w_s = lambda^{s - start + 1}.
// skip_weighted: leave out the groups of heads whose decay takes the weighted
// form (lambda >= 0.8), whose aggregates the dq pass accumulates itself.
// dout: rows and columns of the stored states (64: the top-left blocks, for d = 64
// run at d = 128 and stored at d = 64).
cudaError_t tc_segment_states(const Problem &p, const GroupPlan &gp, const void *X, const void *Y, bool reverse,
                              float *out, int *status, cudaStream_t s, bool skip_weighted = false,
                              int dout = 128);
// Per-group causal chunked attention from the given group states
// [G][BH][d][d] (read transposed when init_transposed): o_i = lambda^{i+1}
// S^T q_i + intra-block terms, S the state entering the block.  final_state
// (optional) is the state after the last token.  x (optional, no gates): also
// writes agg_out[g] = sum_{s in group g} w_s x_s q_s^T ([G][BH][d][d]) from the
// same pass, w_s = lambda^{s - start + 1} (1 without a decay), for the groups
// of heads whose decay takes the weighted form (lambda >= 0.8, or none); the
// other groups are left to tc_segment_states.
cudaError_t tc_main(const Problem &p, const GroupPlan &gp, const void *q, const void *k, const void *v, void *o,
                    const float *group_init, bool init_transposed, float *final_state, int *status,
                    cudaStream_t s, const void *x = nullptr, float *agg_out = nullptr);

// The exclusive state entering every chunk of 64 tokens, out [BH][ceil(T/64)][d][d]
// fp32, walking each group of the plan from its entering state group_init
// ([G][BH][d][d], the scan's output) with one half-tile K^T V product per chunk.
cudaError_t tc_chunk_states(const Problem &p, const GroupPlan &gp, const void *k, const void *v,
                            const float *group_init, float *out, int *status, cudaStream_t s);

// The backward's dv and dk in one reverse-time pass over (k, q, dO, v) from the
// reverse group states [G][BH][d][d] (sum over later tokens u of
// lambda^{u - group end} q_u dO_u^T); equals tc_main(reverse) with roles
// (k, q, dO) for dv and (v, dO, q) with the transposed states for dk.
cudaError_t tc_dual(const Problem &p, const GroupPlan &gp, const void *q, const void *k, const void *v,
                    const void *dO, void *dk, void *dv, const float *group_init, int *status, cudaStream_t s);

// ---------------------------------------------------------------- softmax segment (softmax.cu)
// Causal softmax attention of the last Tq positions of a prefix of Tk tokens over
// that prefix (bf16, d = 128): q and o [B,H,Tq,128] with strides (qsb, qsh, qst),
// k and v [B,H,Tk,128] with strides (ksb, ksh, kst); lse [B,H,Tq] fp32 optional.
struct SoftmaxProblem {
  int B, H, Tq, Tk;
  int64_t qsb, qsh, qst, ksb, ksh, kst;
  float scale;
  int num_sms;
};
// States of bf16 d = 64 problems run at d = 128 (pad.cu): [n][64][64] <-> the
// top-left block of [n][128][128], zeros elsewhere.
cudaError_t pad_state_d64(const float *src, float *dst, int64_t n, cudaStream_t s);
cudaError_t unpad_state_d64(const float *src, float *dst, int64_t n, cudaStream_t s);
// Per-dimension gates (gate_vec.cu): one CTA per (chunk group, batch, head) walks its
// tokens, the groups joined by scans with per-row multipliers; log_gate and d_log_gate
// are [B*H][T][d] fp32.  Workspace bytes of the group path (0 when one group covers
// the sequence).
size_t gated_vec_ws_bytes(const Problem &p, bool bwd);
// bytes of the per-dimension checkpoint (the groups' entering states and log-gate
// sums; 0 with one group per sequence)
size_t gated_vec_ckpt_bytes(const Problem &p);
// ckpt: NULL, or gated_vec_ckpt_bytes of device memory the forward fills and the
// backward then reads instead of recomputing the groups' states
cudaError_t gated_vec_fwd(const Problem &p, const void *q, const void *k, const void *v, const float *log_gate,
                          void *o, const float *init, float *final_state, void *ws, void *ckpt, cudaStream_t s);
cudaError_t gated_vec_bwd(const Problem &p, const void *q, const void *k, const void *v, const void *dO,
                          const float *log_gate, const float *init, const float *d_final, void *dq, void *dk,
                          void *dv, float *d_log_gate, float *d_init, void *ws, const void *ckpt, cudaStream_t s);
cudaError_t softmax_segment(const SoftmaxProblem &p, const void *q, const void *k, const void *v, void *o, float *lse,
                            int *status, cudaStream_t s);
// The backward: dq (q strides), dk and dv (k strides) for the output gradient dO
// (q strides), with the forward's o and lse; stats: softmax_bwd_stats_bytes of
// device scratch for the per-query statistics.
size_t softmax_bwd_stats_bytes(int B, int H, int Tq);
cudaError_t softmax_segment_bwd(const SoftmaxProblem &p, const void *q, const void *k, const void *v, const void *o,
                                const void *dO, const float *lse, void *dq, void *dk, void *dv, float *stats,
                                int *status, cudaStream_t s);

// ---------------------------------------------------------------- TMA descriptors (api.cu)
// 4-D bf16 tiled tensor map, dims innermost first, strides in bytes for dims 1..3,
// box {64, 128, 1, 1} with the 128-byte swizzle (the SW128 tile half).
bool make_tmap_bf16(void *map, const void *base, const uint64_t dims[4], const uint64_t strides[3]);

// ---------------------------------------------------------------- recurrent decode (decode.cu)
// For t = 0..T-1: S <- lambda S + k_t v_t^T, o_t = S^T q_t; state [BH][d][d] in/out.
cudaError_t decode(const Problem &p, const void *q, const void *k, const void *v, void *o, float *state,
                   cudaStream_t s);

// ---------------------------------------------------------------- diagnostics (diag.cu)
cudaError_t diag_mma(int mode, const void *A, const void *B, float *D, cudaStream_t s);

}  // namespace linattn
