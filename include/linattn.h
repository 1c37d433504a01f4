/*
 * linattn -- chunked causal linear attention with a chunk-state prefix scan,
 * for one NVIDIA GB300 (sm_103a).  C ABI: plain pointers, sizes and a stream.
 *
 * The operation (the recurrent definition; the chunked evaluation below
 * reaches the same values up to rounding order):
 *
 *     S_t = lambda_h * S_{t-1} + k_t v_t^T        S_{-1} = init_state (or 0)
 *     o_t = S_t^T q_t                             S is d_k x d_v, fp32
 *
 * computed right-product-first in chunks ("LASP-2: Rethinking Sequence
 * Parallelism for Linear Attention and Its Hybrid", abstract): inside a chunk
 * ordinary masked attention (Q K^T * M) V, across chunks the kernel trick
 * Q . S_prev (related-paper entry "Lightning Attention-2" on the same page),
 * with the chunk states combined by a prefix scan -- the single-GPU reading of
 * the All-Scan that hands every rank its initial state ("ZeCO: Zero
 * Communication Overhead Sequence Parallelism for Linear Attention",
 * abstract) and of LASP-2's single gather of length-independent states.
 *
 * CONVENTIONS (every entry point)
 *  - Every data pointer is CALLER-OWNED DEVICE memory on the current device.
 *    The library never allocates, frees or synchronises (except
 *    linattn_device_status, which synchronises the given stream).
 *  - All work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *    the legacy default stream) and the call returns without waiting.
 *  - Host-side errors are returned BEFORE anything is enqueued.  A failed
 *    launch returns LINATTN_ERR_CUDA.  Device-side errors (a bounded wait that
 *    gave up) are written to the status word at the start of the workspace
 *    and read back by linattn_device_status.  Every entry point that takes a
 *    workspace clears that word first, so it reports the last call only.
 *  - Re-entrant and stateless: concurrent calls need distinct workspaces.
 *  - Sequence tensors q, k, v, o (and dO, dq, dk, dv) are [B, H, T, d] with the
 *    last dimension contiguous and the element strides of linattn_shape.
 *    Their base pointers and row strides must be 16-byte aligned.  With
 *    T == 0 they are not read and may be NULL; the final state is then the
 *    initial state (or zeros) and d_init_state is zero.
 *  - States are fp32, row-major [.., d_k, d_v] (row index = key dimension).
 *  - Paths: bf16 with d = 128 runs on the tensor-core kernels (chunk groups
 *    processed in parallel, states joined by the scan).  bf16 with d = 64
 *    runs on the same kernels as the zero-padded d = 128 problem (exact: the
 *    tiles' columns past 64 load as zeros and are not stored; the states go
 *    through padded copies in the workspace), for linattn_fwd / _ckpt,
 *    linattn_bwd / _ckpt, linattn_fwd_gated / linattn_bwd_gated and
 *    linattn_chunk_states(_rev) with segments of a multiple of 128 tokens.
 *    fp32 inputs and segment states of other segment lengths run on CUDA-core
 *    kernels that walk every sequence serially, one CTA per (batch, head):
 *    correct for any length but far slower on long sequences (meant for fp32
 *    checks).
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LINATTN_ABI_VERSION 2

/* Status codes (return values and device status word). */
enum {
  LINATTN_OK = 0,
  LINATTN_ERR_INVALID = -1,        /* null pointer, negative size, bad op code       */
  LINATTN_ERR_UNSUPPORTED = -2,    /* valid request outside what is implemented      */
  LINATTN_ERR_ALIGN = -3,          /* pointer or stride not 16-byte aligned          */
  LINATTN_ERR_WORKSPACE = -4,      /* workspace missing, too small or not 256-B aligned */
  LINATTN_ERR_CUDA = -5,           /* a CUDA runtime / driver call failed            */
  LINATTN_ERR_DEVICE_TIMEOUT = -6, /* device status: a bounded wait gave up          */
  LINATTN_ERR_DEVICE = -7,         /* current device is not an sm_103 GPU            */
  LINATTN_ERR_SCRATCH_LIMIT = -8   /* request exceeds the fixed scratch of linattn_state_scan_noalloc */
};

/* Element type of the sequence tensors (states are always fp32). */
enum { LINATTN_BF16 = 0, LINATTN_F32 = 1 };

/* Workspace / checkpoint queries. */
enum { LINATTN_OP_FWD = 1, LINATTN_OP_BWD = 2, LINATTN_OP_CHUNK_STATES = 3, LINATTN_OP_CHECKPOINT = 4,
       LINATTN_OP_FWD_GATED = 5, LINATTN_OP_BWD_GATED = 6, LINATTN_OP_CHECKPOINT_GATED = 7,
       LINATTN_OP_SOFTMAX_SEGMENT = 8, LINATTN_OP_SOFTMAX_SEGMENT_BWD = 9, LINATTN_OP_FWD_GATED_VEC = 10,
       LINATTN_OP_BWD_GATED_VEC = 11, LINATTN_OP_CHECKPOINT_GATED_VEC = 12 };

typedef struct {
  int32_t abi_version;  /* must be LINATTN_ABI_VERSION                              */
  int32_t B, H, T;      /* batch, heads, tokens; B, H >= 1, T >= 0                  */
  int32_t dk, dv;       /* head dims; this version: dk == dv, both 64 or 128        */
  int32_t chunk;        /* chunk length C of the chunk-state outputs; must be 64    */
  int32_t dtype;        /* LINATTN_BF16 or LINATTN_F32 for every sequence tensor    */
  int64_t stride_b;     /* element strides of every sequence tensor; > 0 (unchecked when T == 0) */
  int64_t stride_h;
  int64_t stride_t;     /* >= dk; the last dimension is contiguous                  */
  const float *decay;   /* [H] device fp32 per-head lambda_h in (0, 1], or NULL for 1 */
} linattn_shape;

/* Library ABI version (LINATTN_ABI_VERSION of the build). */
int32_t linattn_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *linattn_status_string(int32_t status);

/* Workspace bytes needed by linattn_fwd (op=LINATTN_OP_FWD), linattn_bwd
 * (LINATTN_OP_BWD) or linattn_chunk_states / linattn_chunk_states_rev
 * (LINATTN_OP_CHUNK_STATES, with its seg_len; ignored otherwise) for this
 * shape on the current device.  With
 * op=LINATTN_OP_CHECKPOINT: bytes of the checkpoint of linattn_fwd_ckpt (may
 * be 0 when the shape takes the CUDA-core path, which recomputes instead).
 * Writes *bytes and returns a status; the workspace must be 256-byte aligned. */
int32_t linattn_workspace_size(const linattn_shape *shape, int32_t op, int32_t seg_len,
                               size_t *bytes);

/* Forward.  Computes o for every token (steps: intra-chunk masked attention,
 * inter-chunk query-times-state, state update, prefix scan of chunk-group
 * states; "Lightning Attention-2" entry and abstract of the LASP-2 page).
 *   q, k  [B,H,T,dk], v, o [B,H,T,dv]  (dtype of the shape)
 *   init_state   [B,H,dk,dv] fp32 state before token 0, or NULL (zeros)
 *   final_state  [B,H,dk,dv] fp32 state after token T-1, or NULL
 *   chunk_states [B,H,ceil(T/chunk),dk,dv] fp32 state ENTERING every chunk
 *                (exclusive: entry 0 is init_state), or NULL; on the
 *                tensor-core path they cost one more pass over k, v
 *                (every chunk group walked again from its scanned state)
 * Returns a status. */
int32_t linattn_fwd(const linattn_shape *shape, const void *q, const void *k, const void *v,
                    void *o, const float *init_state, float *final_state, float *chunk_states,
                    void *workspace, size_t workspace_bytes, void *stream);

/* Backward of linattn_fwd for an upstream gradient dO [B,H,T,dv]:
 *   dq_t = S_t dO_t,   dk_t = R_t v_t,   dv_t = R_t^T k_t,
 *   R_t = sum_{u>=t} lambda^{u-t} q_u dO_u^T + lambda^{T-1-t} D
 *         (reverse state, scanned backwards),
 *   d_init_state = lambda R_0 (= D when T = 0)   ([B,H,dk,dv] fp32, or NULL),
 * where D = d_final_state ([B,H,dk,dv] fp32, or NULL for zero) is the gradient
 * arriving at the state after token T-1 -- nonzero when the sequence goes on
 * in a later segment that started from this final state (the sequence-parallel
 * split of the ZeCO and LASP-2 pages: the backward passes it from rank r+1 to
 * rank r, see linattn_chunk_states_rev).  dq, dk [B,H,T,dk] and dv [B,H,T,dv]
 * are written in the shape's dtype.  The forward states are recomputed from k,
 * v and init_state (no stored activations).  Returns a status. */
int32_t linattn_bwd(const linattn_shape *shape, const void *q, const void *k, const void *v,
                    const void *dO, const float *init_state, const float *d_final_state, void *dq,
                    void *dk, void *dv, float *d_init_state, void *workspace, size_t workspace_bytes,
                    void *stream);

/* Forward that also stores a checkpoint for linattn_bwd_ckpt: the fp32 state
 * entering every chunk group of every sequence (the group length is the
 * library's choice; size from linattn_workspace_size(.., LINATTN_OP_CHECKPOINT,
 * ..)).  Same results as linattn_fwd (per-chunk states are not offered here).
 * `checkpoint` is caller-owned device memory, 256-byte aligned.  Returns a
 * status. */
int32_t linattn_fwd_ckpt(const linattn_shape *shape, const void *q, const void *k, const void *v, void *o,
                         const float *init_state, float *final_state, void *checkpoint,
                         size_t checkpoint_bytes, void *workspace, size_t workspace_bytes, void *stream);

/* Backward that takes the forward states from a checkpoint written by
 * linattn_fwd_ckpt for the same shape, k, v and init_state, instead of
 * recomputing them.  init_state is the same as given to the forward (only the
 * CUDA-core path, whose checkpoint is empty, reads it).  Same outputs as
 * linattn_bwd.  Returns a status. */
int32_t linattn_bwd_ckpt(const linattn_shape *shape, const void *q, const void *k, const void *v,
                         const void *dO, const float *init_state, const float *d_final_state,
                         const void *checkpoint, size_t checkpoint_bytes, void *dq, void *dk, void *dv,
                         float *d_init_state, void *workspace, size_t workspace_bytes, void *stream);

/* Data-dependent gates (the gated variant the LASP-2 page names beside the
 * plain one): a decay alpha_t = exp(log_gate_t) per token and head instead of
 * the shape's per-head lambda,
 *   S_t = alpha_t S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t.
 * log_gate is [B,H,T] fp32, contiguous, 16-byte aligned (log of gates in
 * (0, 1]: values <= 0; positive values are taken as given but their weights may
 * overflow).  The shape's decay must be NULL.  bf16 runs on the tensor-core
 * kernels (d = 64 as the zero-padded problem); fp32 on the CUDA-core kernels.  The
 * checkpoint (size from LINATTN_OP_CHECKPOINT_GATED) keeps every chunk group's
 * entering state and the final state for linattn_bwd_gated; it is required
 * when that size is nonzero (the CUDA-core path has none: its backward
 * recomputes the states from init_state).  Workspace sizes:
 * LINATTN_OP_FWD_GATED / LINATTN_OP_BWD_GATED.  Returns a status. */
int32_t linattn_fwd_gated(const linattn_shape *shape, const void *q, const void *k, const void *v,
                          const float *log_gate, void *o, const float *init_state, float *final_state,
                          void *checkpoint, size_t checkpoint_bytes, void *workspace, size_t workspace_bytes,
                          void *stream);

/* Backward of linattn_fwd_gated (same shape, q, k, v, log_gate, init_state and
 * its checkpoint), for an upstream gradient dO and the gradient d_final_state
 * arriving at the final state (or NULL): dq, dk, dv as linattn_bwd with every
 * lambda power replaced by the product of the gates between the two tokens,
 * d_init_state = alpha_0 R_0, and the gradient of every log-gate
 *   d_log_gate[t] = sum_{u >= t} (q_u . dq_u - k_u . dk_u)  + <d_final, S_final>
 * ([B,H,T] fp32, contiguous; derived from dL/d(cumulative log-gate) of the
 * chunked form).  Returns a status. */
int32_t linattn_bwd_gated(const linattn_shape *shape, const void *q, const void *k, const void *v,
                          const void *dO, const float *log_gate, const float *init_state,
                          const float *d_final_state, const void *checkpoint, size_t checkpoint_bytes, void *dq,
                          void *dk, void *dv, float *d_log_gate, float *d_init_state, void *workspace,
                          size_t workspace_bytes, void *stream);

/* Per-dimension gates (the vector form of the data-dependent gate: "Gated
 * Linear Attention ..." on the LASP-2 page's related list): a decay per token,
 * head and KEY dimension, alpha_t[i] = exp(log_gate_t[i]),
 *   S_t = diag(alpha_t) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t
 * (row i of the state decays by the gate of key dimension i).  log_gate is
 * [B,H,T,d] fp32, contiguous, 16-byte aligned; the shape's decay must be NULL.
 * Runs on CUDA-core kernels (fp32 state in registers, no device-side waits):
 * each sequence is cut into chunk groups, one CTA per (group, batch, head)
 * walks its tokens, and the groups are joined by scans whose multipliers are
 * per state row (the product of a group's gates of that key dimension); with
 * few tokens, one CTA per (batch, head) walks the whole sequence.  The
 * per-token gates above have the tensor-core path.  Workspace:
 * LINATTN_OP_FWD_GATED_VEC bytes (the groups' states).  Returns a status. */
int32_t linattn_fwd_gated_vec(const linattn_shape *shape, const void *q, const void *k, const void *v,
                              const float *log_gate, void *o, const float *init_state, float *final_state,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Backward of linattn_fwd_gated_vec for an upstream gradient dO and the
 * gradient d_final_state arriving at the final state (or NULL): dq, dk, dv,
 * d_init_state = diag(alpha_0) R_0 (R the state gradient), and the gradient of
 * every log-gate ([B,H,T,d] fp32, contiguous)
 *   d_log_gate[t][i] = sum_{u >= t} (q_u[i] dq_u[i] - k_u[i] dk_u[i]) + sum_j D[i][j] S_final[i][j].
 * The forward states are recomputed from init_state.  Workspace:
 * LINATTN_OP_BWD_GATED_VEC bytes.  Returns a status. */
int32_t linattn_bwd_gated_vec(const linattn_shape *shape, const void *q, const void *k, const void *v,
                              const void *dO, const float *log_gate, const float *init_state,
                              const float *d_final_state, void *dq, void *dk, void *dv, float *d_log_gate,
                              float *d_init_state, void *workspace, size_t workspace_bytes, void *stream);

/* linattn_fwd_gated_vec that also keeps a checkpoint for
 * linattn_bwd_gated_vec_ckpt: every chunk group's entering state and the sums
 * of its log-gates per key dimension (size from linattn_workspace_size(..,
 * LINATTN_OP_CHECKPOINT_GATED_VEC, ..); 0 when every sequence is one group, in
 * which case checkpoint may be NULL).  `checkpoint` is caller-owned device
 * memory, 256-byte aligned.  Same outputs as linattn_fwd_gated_vec.  Returns a
 * status (LINATTN_ERR_INVALID for a missing, misaligned or short checkpoint). */
int32_t linattn_fwd_gated_vec_ckpt(const linattn_shape *shape, const void *q, const void *k, const void *v,
                                   const float *log_gate, void *o, const float *init_state, float *final_state,
                                   void *checkpoint, size_t checkpoint_bytes, void *workspace,
                                   size_t workspace_bytes, void *stream);

/* linattn_bwd_gated_vec that takes the forward's group states from a checkpoint
 * written by linattn_fwd_gated_vec_ckpt for the same shape, k, v, log_gate and
 * init_state, instead of recomputing them (one pass over k, v and the gates
 * less).  init_state is the one given to the forward (read only when every
 * sequence is one group).  Same outputs as linattn_bwd_gated_vec.  Returns a
 * status. */
int32_t linattn_bwd_gated_vec_ckpt(const linattn_shape *shape, const void *q, const void *k, const void *v,
                                   const void *dO, const float *log_gate, const float *init_state,
                                   const float *d_final_state, const void *checkpoint, size_t checkpoint_bytes,
                                   void *dq, void *dk, void *dv, float *d_log_gate, float *d_init_state,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* Recurrent decode of T new tokens per sequence (constant-memory inference:
 * LASP-2 page, abstract): for t = 0..T-1
 *   S <- lambda S + k_t v_t^T,   o_t = S^T q_t,
 * with `state` ([B,H,dk,dv] fp32 device memory) read at the start and the
 * updated state written back in place.  q, k, v, o follow the shape (T >= 0;
 * meant for a few tokens per call -- the tokens of one call are processed in
 * order by every CTA, so long T belongs to linattn_fwd with init/final
 * states).  No workspace.  Returns a status. */
int32_t linattn_decode(const linattn_shape *shape, const void *q, const void *k, const void *v, void *o,
                       float *state, void *stream);

/* Segment-local states (what each sequence-parallel rank computes from its
 * own contiguous segment before the exchange; LASP-2 page, abstract):
 *   local_states[g,b,h] = sum_{s in segment g} lambda^{end_g - s} k_s v_s^T
 * for G = T / seg_len segments of seg_len tokens (seg_len >= 1 and a divisor
 * of T; T >= 1).  local_states is [G,B,H,dk,dv] fp32.  Returns a status. */
int32_t linattn_chunk_states(const linattn_shape *shape, int32_t seg_len, const void *k,
                             const void *v, float *local_states, void *workspace,
                             size_t workspace_bytes, void *stream);

/* Segment-local gradient states, the backward's counterpart of
 * linattn_chunk_states (what each sequence-parallel rank contributes to the
 * reverse scan that hands every rank the gradient at its final state):
 *   local_grad_states[g,b,h] = sum_{s in segment g} lambda^{s - start_g + 1} q_s dO_s^T
 * for G = T / seg_len segments (seg_len >= 1 and a divisor of T; T >= 1),
 * [G,B,H,dk,dv] fp32.  With every segment's value, the gradient arriving at
 * the final state of segment g is D_g = sum_{g' > g} a^{g'-g-1} W_g' (a =
 * lambda^seg_len; linattn_state_scan over the segments in reverse order), and
 * linattn_bwd of segment g with d_final_state = D_g gives that segment's part
 * of the whole sequence's gradients.  Workspace as for linattn_chunk_states.
 * Returns a status. */
int32_t linattn_chunk_states_rev(const linattn_shape *shape, int32_t seg_len, const void *q,
                                 const void *dO, float *local_grad_states, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* Softmax-attention segment of a hybrid model (LASP-2 page, abstract: LASP-2H
 * carries the one-gather exchange over to the softmax attention layers: one
 * gather hands every sequence-parallel rank the keys and values of every
 * position up to the end of its segment).  The queries are the LAST Tq
 * positions of a prefix of Tk >= Tq tokens (offset = Tk - Tq), attending
 * causally over the prefix with standard scaled dot-product softmax attention:
 *   o_i   = sum_{j <= offset+i} softmax_j(scale q_i . k_j) v_j
 *   lse_i = log sum_{j <= offset+i} exp(scale q_i . k_j)
 * (blockwise with a running maximum and sum per row; the full row softmax is
 * never formed).  The gradients are linattn_softmax_segment_bwd.
 *   q_shape:  B, H, T = Tq and the element strides of q and o
 *   kv_shape: B, H, T = Tk and the element strides of k and v
 *   both: bf16, dk = dv = 128, chunk = 64, decay NULL (else INVALID/UNSUPPORTED)
 *   q, o [B,H,Tq,128]; k, v [B,H,Tk,128]; lse [B,H,Tq] fp32 contiguous or NULL
 *   softmax_scale > 0, or 0 for 1/sqrt(128)
 *   workspace: LINATTN_OP_SOFTMAX_SEGMENT bytes (status word and item counters)
 * Returns a status. */
int32_t linattn_softmax_segment_fwd(const linattn_shape *q_shape, const linattn_shape *kv_shape, const void *q,
                                    const void *k, const void *v, void *o, float *lse, float softmax_scale,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* Gradients of the softmax-attention segment (the training step of the hybrid's
 * softmax layers): for an output gradient dO, with the forward's o and lse,
 *   p_ij  = exp(scale q_i . k_j - lse_i),   delta_i = dO_i . o_i,
 *   ds_ij = p_ij (dO_i . v_j - delta_i),
 *   dv_j  = sum_i p_ij dO_i,  dk_j = scale sum_i ds_ij q_i,  dq_i = scale sum_j ds_ij k_j
 * over the visible pairs j <= offset + i (offset = Tk - Tq).  p and ds enter the
 * products as bf16 (fp32 accumulation); delta is taken from the bf16 o.
 *   q_shape:  B, H, T = Tq and the element strides of q, o, dO and dq
 *   kv_shape: B, H, T = Tk and the element strides of k, v, dk and dv
 *   both: bf16, dk = dv = 128, decay NULL (else INVALID/UNSUPPORTED)
 *   lse [B,H,Tq] fp32 contiguous (the forward's); softmax_scale as in the forward
 *   workspace: LINATTN_OP_SOFTMAX_SEGMENT_BWD bytes for q_shape (status word, item
 *   counters and two fp32 statistics per query row)
 * Every output row is written (Tq = 0: dk and dv are zero).  Returns a status. */
int32_t linattn_softmax_segment_bwd(const linattn_shape *q_shape, const linattn_shape *kv_shape, const void *q,
                                    const void *k, const void *v, const void *o, const void *dO, const float *lse,
                                    void *dq, void *dk, void *dv, float softmax_scale, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* Workspace bytes for linattn_state_scan. */
int32_t linattn_state_scan_workspace_size(int32_t G, int32_t BH, int32_t dk, int32_t dv,
                                          size_t *bytes);

/* Exclusive prefix scan of segment states (ZeCO page, abstract: All-Scan
 * hands every rank exactly its initial state):
 *   init_states[0] = init (or 0),
 *   init_states[g] = a_bh * init_states[g-1] + local_states[g-1],
 *   total          = a_bh * init_states[G-1] + local_states[G-1]   (or NULL)
 * local_states / init_states [G,BH,dk,dv] fp32 (they must not overlap),
 * init / total [BH,dk,dv] fp32 or NULL, seg_decay [BH] fp32 (a_bh = lambda^L
 * of the segment length) or NULL for 1.  G >= 1, BH >= 1, dk*dv % 8 == 0.
 * Implemented as a warp-shuffle scan over 32 segments per warp with a
 * decoupled look-back across 32-segment tiles.  Returns a status. */
int32_t linattn_state_scan(int32_t G, int32_t BH, int32_t dk, int32_t dv, const float *seg_decay,
                           const float *local_states, const float *init, float *init_states,
                           float *total, void *workspace, size_t workspace_bytes, void *stream);

/* Allocation-free variant of linattn_state_scan (the pages have no
 * counterpart; this is a deployment convenience).  Some callers cannot call
 * cudaMalloc at all: code embedded in a host application whose device memory
 * is entirely owned by that application's own allocator or pool, and
 * latency-critical paths where an allocation (which may synchronise the
 * device) is not allowed.  Such callers cannot provide a workspace, so this
 * entry point takes none: its scratch (ticket counter, look-back flags,
 * per-tile aggregates and inclusive prefixes) is a fixed static device array
 * of LINATTN_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits.  Nothing is allocated:
 * no cudaMalloc, cudaFree or allocating library routine is called.
 *   - Same operands and results as linattn_state_scan.
 *   - Limit: up to 256 segments the scan runs column-parallel and uses none of
 *     the scratch (no size limit beyond the operands); with more segments
 *     ceil(G/32) * (BH*dk*dv/8) must be <= LINATTN_NOALLOC_MAX_TILES (65536),
 *     e.g. 1024 segments of one 128x128 state (32 x 2048 tiles); larger requests return
 *     LINATTN_ERR_SCRATCH_LIMIT before anything is enqueued.
 *   - device_status: optional device int32 (NULL allowed; 4-byte aligned) that
 *     is zeroed and then receives LINATTN_ERR_DEVICE_TIMEOUT if a bounded
 *     look-back wait gives up; there is no workspace status word in this variant.
 *   - The first call on a device looks up the scratch's device address once
 *     (cudaGetSymbolAddress, with that device current) and keeps it for the
 *     life of the process; make that first call before any stream capture.  A
 *     reset of the device's context (cudaDeviceReset) makes the kept address
 *     stale: do not call this entry point again in that process after one.
 *   - Every call uses the same scratch and leaves the last call's contents in
 *     it; the call clears what must start at zero (counter, flags) on
 *     `stream`.  Calls that overlap on the GPU (other streams, other host
 *     threads) race on the scratch: serialise them.  Returns a status. */
#define LINATTN_NOALLOC_MAX_TILES 65536
#define LINATTN_NOALLOC_SCRATCH_BYTES (256 + 4 * LINATTN_NOALLOC_MAX_TILES + 64 * LINATTN_NOALLOC_MAX_TILES)
int32_t linattn_state_scan_noalloc(int32_t G, int32_t BH, int32_t dk, int32_t dv, const float *seg_decay,
                                   const float *local_states, const float *init, float *init_states,
                                   float *total, int32_t *device_status, void *stream);

/* Scan multipliers of segments of seg_len tokens: out[b*H + h] = decay[h]^seg_len
 * for b < B (the seg_decay operand of linattn_state_scan for a sequence split into
 * segments of seg_len tokens; ZeCO page, abstract: All-Scan over the ranks'
 * segments).  decay [H] and out [B*H] are device fp32, 16-byte aligned;
 * seg_len >= 0 (0 gives 1).  Returns a status. */
int32_t linattn_segment_decay(const float *decay, int32_t B, int32_t H, int32_t seg_len, float *out,
                              void *stream);

/* Synchronises `stream`, then returns the device status word of `workspace`
 * (LINATTN_OK, or e.g. LINATTN_ERR_DEVICE_TIMEOUT) or LINATTN_ERR_CUDA. */
int32_t linattn_device_status(const void *workspace, void *stream);

/* Per-kernel timing (diagnostics for measurement, not part of the method).
 * While enabled for the process, every kernel the library launches is
 * bracketed by two CUDA timing events recorded on its launch stream (the
 * events come from a pool created on first use; no device memory is
 * allocated).  linattn_timing_collect synchronises the recorded events, writes
 * for every kernel kind k < max_kinds its launch count and summed device time
 * (ms), clears the record and returns the number of kinds
 * (LINATTN_KERNEL_KINDS), or a negative status. */
#define LINATTN_KERNEL_KINDS 20
int32_t linattn_timing_enable(int32_t on);
int32_t linattn_timing_collect(int32_t max_kinds, int32_t *launches, float *total_ms);
/* Name of kernel kind k (static string; "?" when out of range). */
const char *linattn_kernel_name(int32_t kind);

/* Bounded device waits.  Every device-side wait on another CTA's result (the
 * scan's look-back, the chained group states of the forward) gives up after
 * LINATTN_LOOKBACK_LIMIT_MS milliseconds (environment variable, read at every
 * call; default 2000), records LINATTN_ERR_DEVICE_TIMEOUT in the status word
 * and lets the kernel finish instead of hanging.
 *
 * Diagnostic for that path (not part of the method): linattn_state_scan in its
 * look-back form, except that look-back tile `withhold_tile` (tile index =
 * segment tile * (BH*dk*dv/8) + element group) never publishes its aggregate
 * or prefix, so every successor that looks back to it waits wait_limit_ms
 * (0 < wait_limit_ms <= 2000), gives up and reports LINATTN_ERR_DEVICE_TIMEOUT
 * in the workspace status word (read it with linattn_device_status).  The
 * outputs past the withheld tile are then wrong by design.  Workspace as for
 * linattn_state_scan.  Returns a status. */
int32_t linattn_diag_scan_withhold(int32_t G, int32_t BH, int32_t dk, int32_t dv, const float *local_states,
                                   float *init_states, int32_t withhold_tile, double wait_limit_ms,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* Diagnostic (not part of the method): one 128x128x128 bf16 tensor-core
 * product through the same shared-memory layouts the kernels use, written as
 * fp32 D[128][128].  A and B are 128x128 bf16 row-major device arrays.
 *   mode 0: D = A   B^T     mode 1: D = A^T B     mode 2: D = A B
 *   mode 3: D = A^T B^T     mode 4: D = A B with A staged through tensor memory
 * Returns a status (LINATTN_ERR_DEVICE off sm_103). */
int32_t linattn_diag_mma(int32_t mode, const void *A, const void *B, float *D, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* LINATTN_H */
