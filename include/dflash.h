/*
 * dflash.h: C ABI of the GB300 (sm_103a) DFlash2 low-rank candidate selector.
 *
 * The method comes from the page "vllm.models.beam.nvidia.dflash2" (DFlash2 draft model
 * for Beam targets). For request r and block position (step) p, the selector:
 *   1. takes the top-K vocabulary candidates of the drafter's logits and their logits
 *      ("unary" scores)                  DFlash2BeamForCausalLM.compute_candidates
 *   2. projects the drafter hidden state to the codebook rank,
 *      h_p = W_proj . hidden[r, p]       DFlash2BeamCandidateSelector.__init__ / forward
 *   3. scores every candidate c against every candidate q one position back,
 *      E[r,p,q,c] = unary[r,p,c] + <pred_cb[cand[r,p-1,q]] * h_p, succ_cb[cand[r,p,c]]>,
 *      where the predecessor at p = 0 is the request's anchor token.
 *                                        DFlash2BeamCandidateSelector (class docstring)
 * Around these: step 1 straight from the LM head without logits in memory
 * (dflash_lmhead_topk, dflash_selector_lmhead), steps 2 and 3 on given candidates
 * (dflash_selector_forward), and the best path through E (dflash_best_path, a reading: the
 * page does not show what consumes E).
 *
 * Conventions for every entry point:
 *   - Pointers are caller-owned DEVICE memory on the current CUDA device, unless a
 *     comment says otherwise. Tensors are contiguous and row-major, in the shapes given.
 *     bf16 tensors are passed as uint16_t bit patterns.
 *   - Every pointer must be 16-byte aligned (vector loads and TMA), or the call returns
 *     DFLASH_INVALID_ARGUMENT. The exceptions are `logits` (the top-k finds the 16-byte
 *     boundaries itself), `anchors`, `cand_ids`, `unary`, `edges` and the best path's
 *     `path`, `tokens` and `score` (accessed one element at a time, or staged with copies
 *     as wide as their alignment allows): their natural
 *     4-byte alignment suffices, so a slice of requests out of larger arrays stays valid.
 *     `hidden`, `h_out`, the weights and the workspace stay 16-byte aligned.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream). They
 *     allocate no device memory and do not synchronise the device; dflash_device_status,
 *     dflash_trace_end and dflash_selftest_wait_timeout are the exceptions, and say so. A
 *     non-OK status means nothing was launched, except DFLASH_CUDA_ERROR, which reports a
 *     launch failure.
 *   - Supported sizes: R, S >= 1; 1 <= K <= 32 and K <= V; V < 2^31; H a multiple of 8;
 *     rank a multiple of 8 in [8, 256]. Out-of-range sizes give DFLASH_INVALID_ARGUMENT
 *     (bad values) or DFLASH_UNSUPPORTED (valid but not implemented, for example K > 32).
 *   - Token ids are int32. Anchor ids outside [0, V) are caller errors. The kernels
 *     check every gathered id: a bad id never reaches memory, its scores are NaN, and
 *     the device status word records DFLASH_DEVICE_BAD_ID (see dflash_device_status).
 *   - Calls that overlap on the GPU must not share an output or a workspace.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t. */
typedef struct CUstream_st* dflash_stream_t;

typedef enum {
    DFLASH_OK = 0,
    DFLASH_INVALID_ARGUMENT = 1,    /* null or misaligned pointer, size out of range      */
    DFLASH_UNSUPPORTED = 2,         /* valid request outside the implemented envelope     */
    DFLASH_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below the *_workspace_bytes query  */
    DFLASH_CUDA_ERROR = 4,          /* a CUDA runtime call or a launch failed             */
    DFLASH_NO_DEVICE = 5            /* the current device is not a GB300 (sm_103a), or none */
} dflash_status;

/* Bits of the device status word (dflash_device_status). */
#define DFLASH_DEVICE_BAD_ID 0x1u       /* a gathered token id was outside [0, V)        */
#define DFLASH_DEVICE_TIMEOUT 0x2u      /* a bounded wait inside a kernel gave up        */

/* A static string naming a status code. Never NULL. */
const char* dflash_status_string(int status);

/* A detail message for the last non-OK status returned on this host thread ("" if none).
 * The pointer stays valid until the next library call on this thread. */
const char* dflash_last_error(void);

/* ------------------------------------------------------------------------------------
 * Step 1: top-K candidates.
 * Source: DFlash2BeamForCausalLM.compute_candidates ("the selector's top-k candidate
 * ids and their logits at each position").
 *
 * logits    [R, S, V] float32   the drafter's vocabulary logits, one row per (r, p)
 * softcap, scale                the logits processor's options (second page,
 *                               DFlash2BeamForCausalLM.__init__: LogitsProcessor(soft_cap,
 *                               scale=output_multiplier)). The reported unary value is
 *                               scale * softcap * tanh(x / softcap), the cap first; softcap = 0
 *                               means no cap. scale must be > 0, so the map is increasing,
 *                               and candidates are selected and ordered on the raw logits.
 *                               Pass 0 and 1 for raw logits.
 * cand_ids  [R, S, K] int32     out: the K best token ids of each row, in candidate order
 * unary     [R, S, K] float32   out: their (processed) logits
 * workspace                     caller-owned device scratch of at least
 *                               dflash_topk_workspace_bytes(R, S, V, K) bytes. Its
 *                               contents on entry do not matter. The call overwrites it.
 *
 * Candidate order: logit descending; equal logits go to the lower token id; -0 equals
 * +0. A NaN with the sign bit clear ranks above +inf, and one with the sign set below
 * -inf. The unary value of a -0 logit is returned as +0.
 * ---------------------------------------------------------------------------------- */
size_t dflash_topk_workspace_bytes(int R, int S, int V, int K);

dflash_status dflash_topk_candidates(const float* logits, int R, int S, int V, int K,
                                     float softcap, float scale, int32_t* cand_ids,
                                     float* unary, void* workspace, size_t workspace_bytes,
                                     dflash_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Top-K candidates without a workspace argument. The pages have no counterpart to this
 * call; it exists for callers that must not allocate device memory. Examples are a
 * plugin running inside an inference engine that has already claimed all device memory
 * for its own pool, and code that may not call cudaMalloc because the allocation would
 * synchronise the device or is forbidden at that point.
 *
 * Same inputs, outputs and results as dflash_topk_candidates with softcap = 0 and
 * scale = 1 (raw logits). The scratch is a fixed
 * 4 MiB array in device memory that the library holds on every GPU that loads it, until
 * the process exits. A call whose scratch need (about R*S*4 bytes of counters plus
 * 512 bytes per streaming warp) exceeds 4 MiB returns DFLASH_UNSUPPORTED and launches
 * nothing; use dflash_topk_candidates with a workspace then.
 * - The call allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * - The first call on a device looks up the array's device address. Make that first call
 *   before any stream capture on the device. A lookup that fails is not remembered: the
 *   call returns DFLASH_CUDA_ERROR and the next call tries again.
 * - Every call on a device shares the one array. Each call clears the counters it needs
 *   (a memset on `stream`) before its kernel runs. Calls that overlap on the GPU (on
 *   different streams, or from several threads) race on the array: serialise them.
 * ---------------------------------------------------------------------------------- */
dflash_status dflash_topk_candidates_noalloc(const float* logits, int R, int S, int V, int K,
                                             int32_t* cand_ids, float* unary,
                                             dflash_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Step 1 from the LM head: the candidate head without materialised logits.
 * Source: DFlash2BeamForCausalLM.compute_candidates, which calls
 * LogitsProcessor.get_top_k_tokens(lm_head, hidden_states, top_k).
 *
 * hidden    [R, S, H] bf16   drafter hidden states
 * lm_head   [V, H]    bf16   the LM head weight (vocabulary rows)
 * cand_ids  [R, S, K] int32  out: the K best token ids of each row, in candidate order
 * unary     [R, S, K] float  out: their (processed) logits
 * workspace                  at least dflash_lmhead_topk_workspace_bytes(R, S, V, K) bytes;
 *                            its contents on entry do not matter.
 *
 * logits[r,p,v] = sum_i hidden[r,p,i] * lm_head[v,i] are fp32 sums taken by the tensor
 * cores (tcgen05, operands staged by TMA). They never leave the chip. The candidate order,
 * softcap and scale are those of dflash_topk_candidates. Where two logits differ by less
 * than their fp32 accumulation error, their order may differ from an exact computation.
 * Requires H a multiple of 8.
 * ---------------------------------------------------------------------------------- */
size_t dflash_lmhead_topk_workspace_bytes(int R, int S, int V, int K);

dflash_status dflash_lmhead_topk(const uint16_t* hidden, const uint16_t* lm_head, int R, int S,
                                 int H, int V, int K, float softcap, float scale,
                                 int32_t* cand_ids, float* unary, void* workspace,
                                 size_t workspace_bytes, dflash_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Step 2: hidden projection, h = hidden . W_proj^T with no bias.
 * Source: DFlash2BeamCandidateSelector.__init__ (hidden_projection: a bias-free linear
 * map hidden_size -> rank, in params_dtype) and forward (hidden must be bf16).
 *
 * hidden  [R, S, H]    bf16   drafter hidden states
 * w_proj  [rank, H]    bf16   projection weight, in the Linear [out, in] convention
 * h_out   [R, S, rank] bf16   out: fp32 accumulation, rounded to bf16 (nearest-even)
 * Runs on the tensor cores (tcgen05, operands staged by TMA). Like every compute call of
 * this library it needs a GB300 (compute capability 10.3): the library is built for
 * sm_103a only, and other devices get DFLASH_NO_DEVICE.
 * ---------------------------------------------------------------------------------- */
dflash_status dflash_hidden_projection(const uint16_t* hidden, const uint16_t* w_proj,
                                       int R, int S, int H, int rank, uint16_t* h_out,
                                       dflash_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Step 3: edge scores.
 * Source: DFlash2BeamCandidateSelector (class docstring and forward): "[requests,
 * steps, top_k (predecessor), top_k]".
 *
 * pred_cb, succ_cb  [V, rank]     bf16    predecessor / successor codebooks
 * cand_ids          [R, S, K]     int32   candidates (step 1's output)
 * unary             [R, S, K]     float32 their logits
 * h                 [R, S, rank]  bf16    projected hidden states (step 2's output)
 * anchors           [R]           int32   anchor (bonus) token of each request
 * edges             [R, S, K, K]  float32 out: E[r, p, q, c], with q the predecessor
 *                                         index and c the candidate index
 *
 * E[r,p,q,c] = unary[r,p,c] + sum_j pred_cb[pid, j] * h[r,p,j] * succ_cb[cand[r,p,c], j],
 * with pid = cand[r,p-1,q] for p > 0 and pid = anchors[r] (every q) for p = 0. The
 * products and sums are taken in fp32.
 * ---------------------------------------------------------------------------------- */
dflash_status dflash_candidate_edges(const uint16_t* pred_cb, const uint16_t* succ_cb,
                                     const int32_t* cand_ids, const float* unary,
                                     const uint16_t* h, const int32_t* anchors, int R, int S,
                                     int K, int V, int rank, float* edges,
                                     dflash_stream_t stream);

/* ------------------------------------------------------------------------------------
 * The whole selector in one call, with no host round trip. All three steps run on `stream`,
 * each kernel launched as the programmatic dependent of the one before it: a large projection
 * (step 2, more than 8 GFLOP) is launched first and the top-k (step 1) runs beside it; a
 * smaller projection is launched after the top-k and runs on the SMs the top-k's first
 * finished CTAs leave. The edges (step 3) take the SMs the top-k leaves as it finishes,
 * scoring each (r, p) tile as soon as the top-k has written the rows it needs and the
 * projection is done. The results do not depend on the order.
 * The call returns once everything is enqueued; later work on `stream` sees all outputs. It is
 * safe to capture in a CUDA graph; make one call on the device before capturing. The
 * workspace holds the top-k's and the edge tiles' bookkeeping (its size query includes
 * both; its contents on entry do not matter). The outputs, softcap and scale are as in the
 * three calls above; the edge scores use the processed unary values.
 * Source: the draft step captures the candidate head and the selector together
 * (module docstring of the page).
 * ---------------------------------------------------------------------------------- */
size_t dflash_selector_workspace_bytes(int R, int S, int V, int K);

dflash_status dflash_selector(const float* logits, const uint16_t* hidden,
                              const uint16_t* w_proj, const uint16_t* pred_cb,
                              const uint16_t* succ_cb, const int32_t* anchors, int R, int S,
                              int K, int V, int H, int rank, float softcap, float scale,
                              int32_t* cand_ids, float* unary, uint16_t* h_out, float* edges,
                              void* workspace, size_t workspace_bytes, dflash_stream_t stream);

/* ------------------------------------------------------------------------------------
 * The selector's forward pass: steps 2 and 3 on candidates the caller already has.
 * Source: DFlash2BeamCandidateSelector.forward(candidate_ids, unary_logits, hidden_states,
 * anchor_token_ids), which scores the candidates with candidate_edges on the projected
 * hidden states and returns the edge scores [requests, steps, top_k (predecessor), top_k].
 *
 * cand_ids, unary, anchors, pred_cb, succ_cb, K, V, rank, edges  as in dflash_candidate_edges
 * hidden, w_proj, H, h_out                                      as in dflash_hidden_projection
 *
 * The projection writes h_out, then the edges read it; both run on `stream` and the call
 * returns once they are enqueued. No workspace. The ranges are those of the two calls. It
 * is not traced by dflash_trace_begin, which traces the calls that include step 1. It can be
 * captured in a CUDA graph; make one call on the device before capturing.
 * ---------------------------------------------------------------------------------- */
dflash_status dflash_selector_forward(const int32_t* cand_ids, const float* unary,
                                      const uint16_t* hidden, const int32_t* anchors,
                                      const uint16_t* w_proj, const uint16_t* pred_cb,
                                      const uint16_t* succ_cb, int R, int S, int K, int V, int H,
                                      int rank, uint16_t* h_out, float* edges,
                                      dflash_stream_t stream);

/* ------------------------------------------------------------------------------------
 * The draft step from the LM head: steps 1 to 3 in one call, with step 1 taken straight
 * from the LM head as in dflash_lmhead_topk, so no logits are ever written.
 * Source: DFlash2BeamForCausalLM.compute_candidates takes the candidates from
 * get_top_k_tokens(lm_head, hidden, top_k), and the selector's forward scores them with the
 * same hidden states (DFlash2BeamCandidateSelector.forward).
 *
 * hidden, lm_head, H, softcap, scale, cand_ids, unary   as in dflash_lmhead_topk
 * w_proj, pred_cb, succ_cb, anchors, rank, h_out, edges as in dflash_selector
 * workspace  at least dflash_selector_lmhead_workspace_bytes(R, S, V, K) bytes; its contents
 *            on entry do not matter.
 *
 * The kernels run one after another on `stream`: projection, LM-head top-k, edges. The
 * LM-head top-k holds one CTA on every SM, so nothing runs beside it. The call returns once
 * everything is enqueued. The candidates may differ from an exact computation only where two
 * logits differ by less than their fp32 accumulation error (see dflash_lmhead_topk); the edge
 * scores are those of the candidates returned. Requires the ranges of dflash_selector and
 * H a multiple of 8. A traced call (dflash_trace_begin) records the same four events. It can
 * be captured in a CUDA graph; make one call on the device before capturing (the first call
 * sets the kernels' shared-memory limits).
 * ---------------------------------------------------------------------------------- */
size_t dflash_selector_lmhead_workspace_bytes(int R, int S, int V, int K);

dflash_status dflash_selector_lmhead(const uint16_t* hidden, const uint16_t* lm_head,
                                     const uint16_t* w_proj, const uint16_t* pred_cb,
                                     const uint16_t* succ_cb, const int32_t* anchors, int R,
                                     int S, int K, int V, int H, int rank, float softcap,
                                     float scale, int32_t* cand_ids, float* unary,
                                     uint16_t* h_out, float* edges, void* workspace,
                                     size_t workspace_bytes, dflash_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Best path through the edge scores: one candidate per step for every request.
 * Reading: the pages say the selector rescores each position's top-k tokens against the
 * token before it (page "vllm.models.beam.nvidia.dflash2", module docstring) but show no
 * consumer of the scores. This call takes the plainest one: the path that maximises the sum
 * over p of E[r,p,c_{p-1},c_p], the predecessor row at p = 0 being q = 0 (every q row there
 * is the anchor's).
 *
 * edges     [R, S, K, K] float  edge scores as dflash_candidate_edges writes them
 * cand_ids  [R, S, K]    int32  the candidates
 * path      [R, S]       int32  out: the chosen candidate index c_p at each step
 * tokens    [R, S]       int32  out: cand_ids[r, p, c_p], the drafted tokens
 * score     [R]          float  out: the path's score
 *
 * Max-sum dynamic programming in fp32, in a fixed order: V_0[c] = E[r,0,0,c]; V_p[c] is the
 * running maximum over q = 0..K-1 of V_{p-1}[q] + E[r,p,q,c], replaced only by a strictly
 * larger sum (ties keep the lower q; IEEE compares, so a NaN never replaces and is never
 * replaced); the last candidate is the running maximum of V_{S-1}, same rule, and the path
 * follows the kept predecessors back. The result is therefore exactly reproducible.
 * Requires 1 <= K <= 32 and S <= 256 (DFLASH_UNSUPPORTED beyond). No workspace.
 * ---------------------------------------------------------------------------------- */
dflash_status dflash_best_path(const float* edges, const int32_t* cand_ids, int R, int S, int K,
                               int32_t* path, int32_t* tokens, float* score,
                               dflash_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Device status word. Reads the DFLASH_DEVICE_* bits that kernels on the current device
 * have set since the last clear. Clears them if `clear` is non-zero. Synchronises the
 * device. `flags` is a host pointer.
 * ---------------------------------------------------------------------------------- */
dflash_status dflash_device_status(uint32_t* flags, int clear);

/* ------------------------------------------------------------------------------------
 * Self-check of the wait limit. There is no counterpart on the pages; this is a test aid for
 * the failure path. It launches one thread that waits on an mbarrier nothing ever arrives
 * on, through the same bounded wait the pipelined kernels use (projection, LM-head top-k),
 * then one edge CTA that waits in the fused selector's ready queue for a tile nothing ever
 * pushes. Each wait gives up after about one second, sets DFLASH_DEVICE_TIMEOUT in the status
 * word, and the kernel returns: nothing traps or faults, nothing is written, and the context
 * stays usable. Synchronises the device; read and clear the bit with dflash_device_status.
 * ---------------------------------------------------------------------------------- */
dflash_status dflash_selftest_wait_timeout(void);

/* ------------------------------------------------------------------------------------
 * Stage tracing for dflash_selector and dflash_selector_lmhead. There is no counterpart on
 * the pages; this is a profiling aid.
 * dflash_trace_begin(n) creates 4 timing events for each of the next n selector calls
 * made from this process on the current device. Each traced call records them: at its
 * start, when the projection is done, when the top-k is done and when the edges are done,
 * and its kernels then run one after another (untraced, dflash_selector overlaps them), so
 * that each can be timed. dflash_trace_end waits for the events. It writes up to max_calls
 * rows of 3 stage times (ms) into `stage_ms` (a host array of 3 * max_calls floats): the
 * projection, the top-k and the edges, each the time between two events. It stores the row
 * count in *n_calls, then releases the events.
 * ---------------------------------------------------------------------------------- */
dflash_status dflash_trace_begin(int n_calls);
dflash_status dflash_trace_end(float* stage_ms, int max_calls, int* n_calls);

/* Library version, "major.minor.patch". */
const char* dflash_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
