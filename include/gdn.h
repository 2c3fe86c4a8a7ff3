/*
 * gdn.h — C ABI of the GB300 (sm_103a) chunked Gated DeltaNet library.
 *
 * The library computes the gated delta rule over a packed batch of documents,
 * forward and backward. For document i = tokens [cu_seqlens[i], cu_seqlens[i+1])
 * and value head h (key head hk = h / (H_v / H_k)), the per-head state
 * S in R^{d_k x d_v} (d_k = d_v = 128) evolves as
 *     S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,   o_t = S_t^T q_t
 * ("How to Speed Up GDN Kernels for Qwen Models", section "What GDN actually
 * computes": S in R^{d_k x d_v}, alpha_t = e^{g_t}, the erase-then-write factor;
 * "Musings on long-context fine-tuning", section "Isolating the recurrent
 * layers": decay first, then correct the decayed memory's prediction; the query
 * reads the updated matrix). The state restarts at every document boundary and
 * may instead start from a pool entry or from another document's final state
 * (same page: a continuation receives the shared prefix's final state through
 * initial_state, with boundaries given by cu_seqlens). Work is done in chunks
 * of 64 tokens (the chunked formulation of the first page, same section).
 *
 * Conventions for every entry point below:
 *  - All tensor pointers are DEVICE pointers, token-major and contiguous:
 *      q, k      : bf16 [T, H_k, 128]   (fp16 with GDN_FLAG_FP16_INPUTS)
 *      v         : bf16 [T, H_v, 128]   (fp16 with GDN_FLAG_FP16_INPUTS)
 *      out       : bf16 [T, H_v, 128]
 *      g, beta   : fp32 [T, H_v]        (g = log-decay, expected <= 0; beta in [0, 1])
 *      cu_seqlens: int32 [N + 1]        (0 = cu[0] <= cu[1] <= ... <= cu[N] = T)
 *      init_idx  : int32 [N] or NULL    (NULL = every document starts from zero)
 *                  -1           : zero state
 *                  0..n_init-1  : initial_state[init_idx[i]]
 *                  n_init + j   : the final state of document j < i of this same call
 *      initial_state : fp32 [n_init, H_v, 128, 128] or NULL when n_init == 0
 *      final_state   : fp32 [N, H_v, 128, 128]  (layout [d_k][d_v] per head)
 *    q, k, v, out and every gradient of them must be 16-byte aligned. Gradients are fp32:
 *    dq reaches magnitudes where one bf16 rounding step exceeds the accuracy the library
 *    keeps for it, so the caller decides when to round.
 *  - Ownership: the caller owns all memory, including the workspace. The library
 *    never allocates, frees or synchronises; every kernel is enqueued on `stream`.
 *    Inputs are read-only; outputs are overwritten in full.
 *  - Errors: an int status is returned and nothing is thrown across the ABI.
 *    Argument errors the host can see are reported before any launch. Errors that
 *    need the device data (bad cu_seqlens / init_idx, an expired bounded wait) are
 *    written to a status word in the workspace; read it with gdn_workspace_status().
 *    After a device-side error the outputs are unspecified.
 *  - GPUs: built for sm_103a (GB300) only; any other GPU returns
 *    GDN_ERR_UNSUPPORTED ("Using it, and the fine print": the kernels refuse
 *    hardware they were not built for). The device is the one that holds the
 *    workspace. Every non-null pointer must be device memory of that GPU (or
 *    managed memory); a host, pinned-host or unregistered pointer, or one on
 *    another GPU, returns GDN_ERR_INVALID_ARG before anything is launched.
 *    An entry point may switch to the workspace's GPU while it enqueues work,
 *    and always gives the calling thread its own current device back.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gdn_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum gdn_status_code {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = -1, /* bad shapes, pointers, alignment, cu_seqlens or init_idx */
  GDN_ERR_UNSUPPORTED = -2, /* head_dim != 128, or the GPU is not sm_103 */
  GDN_ERR_CUDA = -3,        /* a CUDA launch or runtime call failed */
  GDN_ERR_TIMEOUT = -4,     /* a bounded device-side wait ran out */
  GDN_ERR_WORKSPACE = -5    /* the workspace is smaller than the size query returned */
};

/* gdn_options.flags: a training step keeps the forward's per-chunk records for its backward. */
enum gdn_flags {
  GDN_FLAG_SAVE_FOR_BWD = 1, /* forward: also leave in the workspace everything the backward recomputes
                                (the intra-chunk factors, the chunk-start states and V' = U - W S, in the
                                compensated precision of the backward's recompute), and form o from those
                                records. The workspace must then be of gdn_bwd_workspace_size() bytes
                                (gdn_fwd_workspace_size() returns that size when this flag is set).
                                Exact mode only. */
  GDN_FLAG_TEST_WITHHOLD_FORK = 4, /* forward, for testing the bounded waits only: no document of the call
                                      publishes its final state to the documents that fork from it, so
                                      their waits run out (after gdn_options.flag_wait_us) and the call
                                      reports GDN_ERR_TIMEOUT through the status word; outputs are then
                                      unspecified. Rejected by the backward (GDN_ERR_INVALID_ARG). */
  GDN_FLAG_L2NORM_QK = 8,    /* q and k come unnormalised: each (token, key head) row is first scaled to unit
                                L2 norm, y = x / sqrt(x . x + 1e-6) ("Musings on long-context fine-tuning",
                                "Triton autotuning in the first backward pass": the normalisation the model
                                applies right before the op), then opt->scale multiplies the normalised q.
                                The backward's dq and dk are the gradients with respect to the unnormalised
                                inputs. The workspace also holds the normalised copies (the size queries
                                count them); forward and backward of a training step must both set it. */
  GDN_FLAG_FP16_INPUTS = 16, /* q, k, v (and dout) are IEEE fp16 instead of bf16 ("Using it, and the fine
                                print": bf16 or fp16 inputs). The kernels' matrix operands are bf16: each
                                input is rounded once to bf16 (relative error at most 2^-9, as for any other
                                operand) into workspace copies that the size queries count; accumulation
                                stays fp32. Gradients stay fp32. Combines with GDN_FLAG_L2NORM_QK. */
  GDN_FLAG_REUSE_FWD = 2     /* backward: the workspace holds the records of a forward run with
                                GDN_FLAG_SAVE_FOR_BWD on the same inputs, options and stream order, and
                                nothing has written it since; the backward then skips its recompute
                                (it rebuilds only the chunk and segment maps). Records that do not
                                belong to these inputs give wrong gradients, not a fault. */
};

enum gdn_mode {
  GDN_MODE_EXACT = 0,   /* default: long documents split into segments, exact cross-segment fix-up */
  GDN_MODE_TRUNCATE = 1 /* opt-in: segment carries rebuilt from a warmup window ("Lever 1") */
};

typedef struct gdn_options {
  int32_t mode;              /* gdn_mode */
  float trunc_log_threshold; /* truncation mode: warmup window ends once the summed log-decay < this (-10) */
  int32_t segment_chunks;    /* segment length in 64-token chunks; 0 = automatic, < 0 = never split */
  float scale;               /* multiplies q (1.0: inputs already scaled) */
  int32_t flags;             /* gdn_flags, 0 = none */
  void* stage_events;        /* optional profiling hook: NULL, or a cudaEvent_t[2 * GDN_NUM_STAGES] array;
                                events 2s and 2s+1 are recorded on `stream` right before and right after
                                stage s (both at the same point when the stage has nothing to launch);
                                NULL entries are skipped */
  int32_t flag_wait_us;      /* limit of each wait of one work item for a state another item publishes
                                (a fork source's final state, a previous segment's end state), in
                                microseconds at the maximum SM clock; 0 = about two seconds. A wait that
                                runs out stops the call with GDN_ERR_TIMEOUT in the status word. */
} gdn_options;

/* Stages of a call (indices into gdn_options.stage_events). A backward call runs stages 0-3
 * (the forward recompute; stage 0 alone with GDN_FLAG_REUSE_FWD), then 4, 5, 7 and 6 in that order.
 * A forward with GDN_FLAG_SAVE_FOR_BWD runs stages 0-3 and 8. With GDN_FLAG_L2NORM_QK stage 9 runs
 * first in both directions and the backward ends with stage 10. */
enum gdn_fwd_stage {
  GDN_STAGE_PLAN = 0,      /* chunk / segment maps */
  GDN_STAGE_KKT_SOLVE = 1, /* intra-chunk K K^T, triangular solve, WY factors */
  GDN_STAGE_SPLIT = 2,     /* exact split, pass 1: segment transitions and local end states */
  GDN_STAGE_CHAIN = 3,     /* state chain fused with the output (records states in the backward) */
  GDN_STAGE_REV_CHAIN = 4, /* backward: reverse state-gradient chain */
  GDN_STAGE_GRADS = 5,     /* backward: per-chunk dk, dv, dbeta, dg (all but its q S dO term) */
  GDN_STAGE_DINIT = 6,     /* backward: d(initial_state) sums over documents sharing a pool entry */
  GDN_STAGE_DQ = 7,        /* backward: per-chunk dq; adds the q S dO term of dg */
  GDN_STAGE_OUT = 8,       /* forward with GDN_FLAG_SAVE_FOR_BWD: o from the records */
  GDN_STAGE_L2NORM = 9,    /* GDN_FLAG_L2NORM_QK: the normalised copies of q and k (both directions) */
  GDN_STAGE_L2NORM_BWD = 10, /* GDN_FLAG_L2NORM_QK, backward: dq, dk back to the unnormalised inputs */
  GDN_NUM_STAGES = 11
};

/* Fill `opt` with the defaults: exact mode, threshold -10, automatic segments, scale 1, no flags,
 * no events, the default wait limit. */
void gdn_default_options(gdn_options* opt);

/* Workspace bytes gdn_chunk_fwd needs for these sizes (opt may be NULL for defaults; with
 * GDN_FLAG_SAVE_FOR_BWD the backward's size). Returns 0 for invalid sizes. The value depends on the
 * current device's SM count. */
size_t gdn_fwd_workspace_size(int N, int T, int H_k, int H_v, const gdn_options* opt);

/* Workspace bytes gdn_chunk_bwd needs (opt->mode is ignored: the backward is exact). */
size_t gdn_bwd_workspace_size(int N, int T, int H_k, int H_v, const gdn_options* opt);

/*
 * Forward: out[t, h, :] = o_t for every token and value head; final_state[i, h] = state
 * after the last token of document i (its start state if the document is empty).
 * n_init: number of pool entries in initial_state (0 allowed).
 * head_dim must be 128. workspace: device memory of at least gdn_fwd_workspace_size() bytes,
 * 256-byte aligned; its contents need no initialisation.
 * opt->flags: GDN_FLAG_SAVE_FOR_BWD runs the forward of a training step (the backward's recompute,
 * with o formed from its records) and needs exact mode; GDN_FLAG_REUSE_FWD is rejected
 * (GDN_ERR_INVALID_ARG).
 */
int gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                  const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim,
                  const int32_t* init_idx, const float* initial_state, int n_init, void* out,
                  float* final_state, void* workspace, size_t ws_bytes, const gdn_options* opt,
                  gdn_stream_t stream);

/*
 * Backward of gdn_chunk_fwd for the loss sum(dout * out) + sum(dfinal_state * final_state).
 * dout: bf16 [T, H_v, 128] (fp16 with GDN_FLAG_FP16_INPUTS); dfinal_state: fp32 [N, H_v, 128, 128] or NULL (zero).
 * Outputs, all fp32: dq, dk [T, H_k, 128] (summed over the value heads of each key head);
 * dv [T, H_v, 128]; dg, dbeta [T, H_v]; dinitial_state [n_init, H_v, 128, 128]
 * (summed over every document that starts from the same pool entry; NULL allowed when n_init == 0).
 * A document forked from document j of the same call sends its gradient back into j
 * ("Musings on long-context fine-tuning", section "Backward through P").
 * The backward is always that of the exact forward: opt->mode is ignored (truncation is a
 * forward-only option), the other options apply. Long documents are split into segments in
 * both directions, with an exact fix-up of the state and of its gradient at each boundary.
 * opt->flags: GDN_FLAG_REUSE_FWD skips the recompute (see gdn_flags); GDN_FLAG_SAVE_FOR_BWD is
 * rejected (GDN_ERR_INVALID_ARG).
 */
int gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                  const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim,
                  const int32_t* init_idx, const float* initial_state, int n_init, const void* dout,
                  const float* dfinal_state, float* dq, float* dk, float* dv, float* dg, float* dbeta,
                  float* dinitial_state, void* workspace, size_t ws_bytes, const gdn_options* opt,
                  gdn_stream_t stream);

/* Forward without a workspace argument, for callers that cannot allocate device memory (a host
 * program with no device allocator of its own, or a plugin inside a framework whose memory pool
 * owns all device memory). The pages have no counterpart to this entry point. It runs the same
 * kernels as gdn_chunk_fwd with the scratch in a fixed array of gdn_noalloc_scratch_bytes() bytes
 * (160 MiB: room for one 32768-token document at 8 value heads) compiled into the library: every
 * GPU that loads the library holds that array until the process exits, and every call shares it.
 * Problems whose gdn_fwd_workspace_size() exceeds it return GDN_ERR_WORKSPACE before any launch.
 * The tensors' GPU is used (same pointer rules as gdn_chunk_fwd). Calls that overlap on the GPU
 * race on the array: order them on one stream. The array needs no clearing (the forward rewrites
 * everything it reads). The first call on each device looks up the array's device address; make
 * it before any stream capture. Device-side errors: read them with gdn_noalloc_status(). */
int gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                          const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim,
                          const int32_t* init_idx, const float* initial_state, int n_init, void* out,
                          float* final_state, const gdn_options* opt, gdn_stream_t stream);

/* Size in bytes of the array gdn_chunk_fwd_noalloc uses. */
size_t gdn_noalloc_scratch_bytes(void);

/* Device status word of the last gdn_chunk_fwd_noalloc call on CUDA device `device` (synchronises
 * `stream`, which must belong to that device): GDN_OK or its first device-side error, as
 * gdn_workspace_status() reports for a caller's workspace. GDN_ERR_INVALID_ARG if no such call has
 * run on that device. */
int gdn_noalloc_status(int device, gdn_stream_t stream);

/*
 * Decode: advance B sequences by one token each, in place on a pool of states ("How to Speed Up
 * GDN Kernels for Qwen Models", FAQ "Does this help decode too?"; the recurrence of section "What
 * GDN actually computes"). For sequence b and value head h (key head h / (H_v / H_k)), with
 * S = state_pool[state_idx[b], h]:
 *     S' = exp(g) S,  p = S'^T k,  d = beta (v - p),  S = S' + k d^T  (stored back),  out = scale S^T q.
 * This equals gdn_chunk_fwd on B one-token documents whose initial states are those pool entries.
 *   q, k  : bf16 [B, H_k, 128];  v, out : bf16 [B, H_v, 128];  g, beta : fp32 [B, H_v]
 *   state_idx  : int32 [B], pairwise distinct entries of [0, n_pool) (two sequences on one entry race)
 *   state_pool : fp32 [n_pool, H_v, 128, 128], read and overwritten in place (16-byte aligned)
 *   status     : device int32 or NULL; a sequence whose index is out of range is skipped (its out row
 *                is zero, its pool entry untouched) and GDN_ERR_INVALID_ARG is written here (never
 *                cleared: the caller zeroes it)
 * opt may be NULL; opt->scale and the GDN_FLAG_L2NORM_QK and GDN_FLAG_FP16_INPUTS bits of opt->flags
 * are used (q and k unnormalised, scaled to unit norm in fp32 first; q, k, v in fp16; out stays bf16). Same device rules as gdn_chunk_fwd (the pool's GPU);
 * nothing is allocated, everything runs on `stream`. B = 0 is a no-op.
 */
int gdn_decode_step(const void* q, const void* k, const void* v, const float* g, const float* beta, int B, int H_k,
                    int H_v, int head_dim, const int32_t* state_idx, float* state_pool, int n_pool, void* out,
                    int32_t* status, const gdn_options* opt, gdn_stream_t stream);

/*
 * Width-4 causal depthwise convolution over packed documents, the short convolution in front of the
 * recurrence ("Musings on long-context fine-tuning", section "Isolating the recurrent layers": it
 * reads the current input and the three before it; documents do not read each other; a continuation
 * forked from a prefix reads the prefix's last three inputs first; section "Backward through P": the
 * gradients through those inputs sum into the prefix). Per channel c, document i with inputs x[0..n-1]:
 *     E = (init[0], init[1], init[2], x[0], ..., x[n-1]),  y[p] = bias[c] + sum_m w[c][m] E[p + m],
 *     final_tail[i] = (E[n], E[n+1], E[n+2]).
 * init_idx has the encoding of gdn_chunk_fwd: -1 zeros, 0..n_init-1 conv_init[x], n_init + j the
 * final tail of document j < i of the same call (a fork). Layouts (device, contiguous):
 *   x, y, dy : bf16 [T, C] (C a multiple of 8);  w : fp32 [C, 4];  bias : fp32 [C] or NULL (zero)
 *   conv_init : bf16 [n_init, 3, C] or NULL;  final_tail : bf16 [N, 3, C] (copies of inputs)
 *   dfinal_tail : fp32 [N, 3, C] or NULL;  dx : fp32 [T, C];  dw : fp32 [C, 4];  dbias : fp32 [C] or NULL
 *   dconv_init : fp32 [n_init, 3, C] (summed over the documents that start from each entry)
 * The backward is that of the loss sum(dy * y) + sum(dfinal_tail * final_tail); forks send their
 * gradient into the forked document's last inputs. Every sum is formed in a fixed order
 * (deterministic). workspace: gdn_conv_workspace_size(N, T, C, backward) bytes, 256-byte aligned;
 * bad cu_seqlens / init_idx are reported in its status word (gdn_workspace_status). Same device and
 * ownership rules as gdn_chunk_fwd; nothing is allocated.
 */
size_t gdn_conv_workspace_size(int N, int T, int C, int backward);
int gdn_conv_fwd(const void* x, const float* w, const float* bias, const int32_t* cu_seqlens, int N, int T, int C,
                 const int32_t* init_idx, const void* conv_init, int n_init, void* y, void* final_tail,
                 void* workspace, size_t ws_bytes, gdn_stream_t stream);
int gdn_conv_bwd(const void* x, const float* w, const float* bias, const int32_t* cu_seqlens, int N, int T, int C,
                 const int32_t* init_idx, const void* conv_init, int n_init, const void* dy,
                 const float* dfinal_tail, float* dx, float* dw, float* dbias, float* dconv_init, void* workspace,
                 size_t ws_bytes, gdn_stream_t stream);

/* Copy the workspace's device status word to the host (synchronises `stream`) and return it:
 * GDN_OK or the first device-side error of the last call that used this workspace. */
int gdn_workspace_status(const void* workspace, gdn_stream_t stream);

/* Every host-side check gdn_chunk_fwd / gdn_chunk_bwd makes before its first launch (sizes,
 * options, null pointers, alignment, the memory kind and GPU of each pointer, the GPU's
 * architecture, the workspace size), with the same arguments minus the stream; returns the status
 * the entry point would return at that point, GDN_OK when it would go on to launch. Launches
 * nothing, reads and writes no buffer, leaves the caller's current device as it was. */
int gdn_fwd_check_args(const void* q, const void* k, const void* v, const float* g, const float* beta,
                       const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim,
                       const int32_t* init_idx, const float* initial_state, int n_init, void* out,
                       float* final_state, void* workspace, size_t ws_bytes, const gdn_options* opt);
int gdn_bwd_check_args(const void* q, const void* k, const void* v, const float* g, const float* beta,
                       const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim,
                       const int32_t* init_idx, const float* initial_state, int n_init, const void* dout,
                       const float* dfinal_state, float* dq, float* dk, float* dv, float* dg, float* dbeta,
                       float* dinitial_state, void* workspace, size_t ws_bytes, const gdn_options* opt);

/* Human-readable name of a status code (static string). */
const char* gdn_status_string(int status);

/* Host-side planner, exported for inspection and tests: given HOST copies of cu_seqlens
 * (int32[N+1]) and init_idx (int32[N] or NULL), fill the chunk and segment maps exactly as the
 * device planner does. Arrays (host memory, caller-owned):
 *   chunk_seq, chunk_tok0, chunk_len : int32[max_chunks]   (max_chunks >= T/64 + N)
 *   seg_info : int32[max_segs * 4]  (per segment: sequence, first chunk, chunk count, dependency)
 * num_sms: SM count to plan for. Returns the number of chunks in out_counts[0], segments in
 * out_counts[1], chosen segment length (chunks) in out_counts[2]; status as the return value. */
int gdn_plan_host(const int32_t* cu_seqlens, int N, int T, int H_v, const int32_t* init_idx, int n_init,
                  const gdn_options* opt, int num_sms, int32_t* chunk_seq, int32_t* chunk_tok0,
                  int32_t* chunk_len, int max_chunks, int32_t* seg_info, int max_segs, int32_t* out_counts);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
