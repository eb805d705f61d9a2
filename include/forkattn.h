/*
 * forkattn.h - C ABI of the GB300 ForkAttention token-mixing layer.
 *
 * The layer is the data-parallel hot path of Flide ("Flide: Accelerating
 * Decision Inference with Exact State Forking"): a round of R requests
 * r = (s, q_1..q_n) is packed into one unpadded flat token stream, every
 * token carries device-resident metadata (request j, branch c, position t),
 * and the token mixers (fork-masked attention, two-call Gated DeltaNet) plus
 * the options readout run over that stream.
 *
 * Conventions shared by every entry point
 *   - All pointers named d_* or described as "device" are CUDA device
 *     pointers; the caller allocates and owns every buffer (metadata,
 *     workspace, inputs, outputs).  The library allocates no device memory
 *     and keeps no global state between calls, with one exception:
 *     fork_attn_noalloc takes its scratch from a file-scope device array that
 *     the library owns (and caches that array's device address per device).
 *     The host-side forest planner uses host scratch of its own, freed before
 *     it returns.
 *   - bf16 tensors are passed as uint16_t bit patterns (bfloat16), row-major
 *     with the layout stated per argument.  Every base pointer must be
 *     16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous and stream-ordered; none synchronises the host except
 *     fork_read_status (and fork_build_forest_meta given pageable host memory,
 *     whose copy waits for the stream), so a sequence of calls can be captured
 *     in a CUDA graph.  Grid sizes depend only on the capacities fixed at metadata
 *     build time (T_cap, max_req, max_q) and on the shape arguments.
 *   - Return value: FORK_OK or a host-detected error code (nothing is
 *     launched then).  Errors found on the device (an inconsistent
 *     descriptor) set bits of the status word inside the metadata and turn
 *     every later kernel of the round into a no-op; fork_read_status reads it.
 *     No kernel traps, asserts or waits without a bound.
 *   - Requires an sm_103 device (FORK_EUNSUPPORTED otherwise).
 */
#ifndef FORKATTN_H
#define FORKATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes (host) */
#define FORK_OK 0
#define FORK_EINVAL 1       /* null pointer, bad shape or size, misaligned buffer */
#define FORK_ECAPACITY 2    /* round larger than the metadata capacities */
#define FORK_EUNSUPPORTED 3 /* device is not sm_103 */
#define FORK_ECUDA 4        /* a CUDA runtime/driver call or launch failed */

/* Device status word bits (fork_read_status) */
#define FORK_STATUS_BAD_DESC 0x1   /* descriptor lengths inconsistent (negative, q_len < 1, ...) */
#define FORK_STATUS_CAPACITY 0x2   /* descriptor's stream longer than T_cap */
#define FORK_STATUS_BAD_CKPT 0x4   /* checkpoint position outside [prefix_len, P] */
#define FORK_STATUS_TIMEOUT 0x8    /* a bounded wait inside a kernel gave up */
#define FORK_STATUS_BAD_PREFIX 0x10 /* a request's prefix rows lie outside the prefix buffers or
                                       the resume state/window buffers are missing */
#define FORK_STATUS_CHECK 0x20      /* a FORK_CHECKS bounds check failed (the work was skipped) */

/* Flags */
#define FORK_DETERMINISTIC 0x1u /* bitwise identical results for a question under any round
                                   composition.  Every kernel here already computes each output
                                   from segment-aligned tiles and chunks in a fixed order, so the
                                   flag is accepted and changes nothing. */
#define FORK_CHECKS 0x2u        /* bounds checks on the device: fork_build_meta verifies the tables
                                   it built; fork_attn and fork_gdn_* check that every row range
                                   and state index a CTA is about to use lies inside the round;
                                   fork_readout checks the option offsets.  A failed check sets
                                   FORK_STATUS_CHECK and the CTA skips that work (no trap). */
#define FORK_WARP_MMA 0x4u      /* fork_attn, fork_gdn_*: run the warp-level mma.sync kernels instead
                                   of the tcgen05 ones (same results within rounding; for
                                   comparisons; d = 64 GDN always uses them) */
#define FORK_FOREST 0x8u        /* fork_attn: the metadata describes a token forest (built by
                                   fork_forest_plan); every node sees its ancestors' rows and
                                   its own (see "Token forests" below).  d = 128, no prefix
                                   rows, not with FORK_WARP_MMA. */
#define FORK_TEST_STALL 0x100u  /* test hook of the bounded waits (fork_attn, fork_gdn_* with
                                   d = 128): one role of every CTA waits on a barrier that
                                   nothing completes, so the wait runs out after
                                   fork_meta.wait_us; the CTA then drains its own copies and
                                   products, frees its tensor memory and exits, and the call
                                   reports FORK_STATUS_TIMEOUT.  Never set in normal use. */

/* ------------------------------------------------------------------------
 * Metadata (Flide pages: onedev summary "무엇과 다른가" - per-token (j, c, t),
 * question positions continue from P; rainbus summary "方法步骤详情" steps 1
 * and 3 - stream order s(1)|s(2)|...|q1(1)|..., segment lengths, positions,
 * key ranges and state indices written to device buffers; onedev "어떻게 쓰나").
 * ------------------------------------------------------------------------ */

/* Host-side handle of a metadata buffer.  Plain data, filled by
 * fork_meta_init and passed by pointer to every later call; the library
 * derives every launch shape from these capacities, never from the buffer
 * contents (so nothing has to be read back before a launch). */
typedef struct fork_meta {
  void* d_buf;         /* device buffer of at least fork_meta_bytes(...) bytes */
  size_t bytes;        /* its size */
  int32_t T_cap;       /* stream capacity in tokens */
  int32_t max_req;     /* most requests a round may hold */
  int32_t max_q;       /* most questions a round may hold */
  int32_t tile_tokens; /* tokens per attention work item: 256 / (Hq / Hkv) (two 128-row
                          query tiles per CTA), or 128 / (Hq / Hkv) (one tile) */
  uint32_t wait_us;    /* limit of every bounded wait inside the tensor-core kernels, in
                          microseconds (0 = 2 s); a wait that runs out sets
                          FORK_STATUS_TIMEOUT.  fork_meta_init sets 0; the caller may
                          change it between calls. */
} fork_meta;

/* Bytes of the metadata buffer for a stream capacity T_cap (tokens), at most
 * max_req requests and max_q questions per round.  Returns 0 for invalid
 * capacities (T_cap < 1 or > 1<<20, max_req < 1 or > 1<<16, max_q < 0 or
 * > 1<<18). */
size_t fork_meta_bytes(int32_t T_cap, int32_t max_req, int32_t max_q);

/* Fill *m (host only, no CUDA call).  tile_tokens in {8,16,32,64,128,256}.
 * Errors: FORK_EINVAL (null, invalid capacity, buffer too small or not
 * 16-byte aligned). */
int fork_meta_init(fork_meta* m, void* d_buf, size_t bytes, int32_t T_cap, int32_t max_req,
                   int32_t max_q, int32_t tile_tokens);

/* Build the round metadata on the device.
 *   d_desc   device int32 [4R + Nq]: R trunk lengths P_j (prefix included) |
 *            R question counts n_j | Nq question lengths (request order) |
 *            R prefix lengths (trunk tokens held outside the stream, from a
 *            checkpoint; 0 normally) | R checkpoint positions (-1 = none).
 *   R, Nq    counts (host ints); Nq must equal sum n_j (checked on device).
 * Produces: per-token request/branch/position (pad rows = -1); the segment
 * table (R trunk segments, then the Nq question segments in stream order)
 * with start, length, first position, request, branch, trunk start and
 * length, state index; per-request tables; the last stream row of every
 * question; the attention work list (segment, offset) of tile_tokens-token
 * tiles aligned to each segment's start, each segment's last tile first;
 * and the status word (cleared, then set if the descriptor is
 * inconsistent, in which case the round is empty for every later kernel).
 * Errors: FORK_EINVAL (null pointers, R < 0, Nq < 0), FORK_ECAPACITY
 * (R > max_req, Nq > max_q). */
int fork_build_meta(const fork_meta* m, const int32_t* d_desc, int32_t R, int32_t Nq,
                    uint32_t flags, void* stream);

/* Words of a fixed-capacity device descriptor for fork_build_meta_dev:
 * 2 + 4 * max_req + max_q (0 for invalid capacities). */
size_t fork_desc_capacity_words(int32_t max_req, int32_t max_q);

/* fork_build_meta with the request and question counts read on the device, so
 * that one captured CUDA graph serves every round up to the capacities (the
 * onedev summary's "어떻게 쓰나": one flat graph per capacity bucket, replayed for
 * any round that fits).
 *   d_desc   device int32 [fork_desc_capacity_words(max_req, max_q)]:
 *            R, Nq | max_req trunk lengths | max_req question counts | max_q
 *            question lengths | max_req prefix lengths | max_req checkpoint
 *            positions; entries past R (requests) or Nq (questions) are ignored.
 * Same results as fork_build_meta on the equivalent packed descriptor.  R or
 * Nq outside [0, max_req] / [0, max_q] sets FORK_STATUS_CAPACITY (round empty).
 * Errors: FORK_EINVAL (null pointer, invalid handle). */
int fork_build_meta_dev(const fork_meta* m, const int32_t* d_desc, uint32_t flags, void* stream);

/* cudaError_t value of the most recent CUDA runtime call of this library that
 * failed on the calling host thread (0 if none): the detail behind FORK_ECUDA. */
int fork_last_cuda_error(void);

/* Copy the device status word of a metadata buffer to *h_status.  Enqueues a
 * device-to-host copy on `stream` and synchronises that stream. */
int fork_read_status(const fork_meta* m, int32_t* h_status, void* stream);

/* ------------------------------------------------------------------------
 * Fork-masked attention (rainbus "方法步骤详情" step 2: key y is visible to
 * query x iff j_y = j_x, c_y in {0, c_x}, t_y <= t_x, and for a sliding
 * window layer t_x - t_y < W; onedev "무엇과 다른가": questions receive the
 * rotary positions they would have alone).
 * ------------------------------------------------------------------------ */

/* Workspace bytes fork_attn needs with these flags: with the rotary embedding,
 * rotated keys of the stream and of the prefix and two small rotary tables
 * (with FORK_WARP_MMA also rotated queries: the default kernel rotates its query
 * tiles in shared memory); for the default kernel, the values of the stream and
 * of the prefix as fp16 (its PV product multiplies fp16 exponentials by fp16
 * values; inputs beyond the fp16 range, |v| > 65504, are not supported) and
 * the counter through which its CTAs (one per SM) claim work items.
 * 0 only for FORK_WARP_MMA without the rotary embedding. */
size_t fork_attn_workspace_bytes(int32_t T_cap, int32_t prefix_rows, int32_t Hq, int32_t Hkv,
                                 int32_t d, float rope_theta, uint32_t flags);

/* o_x = sum_y softmax_y(<R(q_x,t_x), R(k_y,t_y)> * scale) v_y over visible y.
 *   q [T_cap, Hq, d], k and v [T_cap, Hkv, d] bf16 (stream rows; pad rows
 *   ignored); o [T_cap, Hq, d] bf16 (pad rows not written).  q-head h reads
 *   kv-head h / (Hq / Hkv).  d in {64, 128}; Hq / Hkv * tile_tokens is 256
 *   (each work item is two 128-row query tiles sharing every key tile: the fast
 *   configuration) or 128; FORK_WARP_MMA needs 128.
 *   window 0 = full attention, else W > 0.  rope_theta 0 = no rotary
 *   embedding, else rotate-half pairs (i, i + d/2) by t * theta^(-2i/d).
 *   scale: score scale (1/sqrt(d) in the workloads).
 *   prefix_k/prefix_v [prefix_rows, Hkv, d] bf16, un-rotated: keys/values of
 *   trunk positions 0..prefix_len_j-1 held outside the stream (incremental
 *   resume), request j's rows starting at the sum of earlier prefix lengths;
 *   NULL when no request has a prefix.
 *   workspace: device buffer of fork_attn_workspace_bytes(..., flags) bytes. */
int fork_attn(const fork_meta* m, const uint16_t* q, const uint16_t* k, const uint16_t* v,
              uint16_t* o, int32_t Hq, int32_t Hkv, int32_t d, int32_t window, float rope_theta,
              float scale, const uint16_t* prefix_k, const uint16_t* prefix_v, int32_t prefix_rows,
              void* workspace, size_t ws_bytes, uint32_t flags, void* stream);

/* fork_attn for callers that cannot allocate device memory.  The Flide pages
 * have no counterpart: this entry point exists for callers that hold only
 * pointers to their inputs and outputs and may not allocate (for example a
 * runtime that plans all device memory ahead and forbids allocation in its
 * serving loop, because cudaMalloc and cudaFree synchronise the device).
 * Arguments and results are those of fork_attn without the workspace: the
 * scratch fork_attn needs (rotated keys, rotary tables, fp16 values, the
 * work-item counter) is taken from an array
 * of FORK_NOALLOC_SCRATCH_BYTES bytes owned by the library, which every GPU
 * that loads the library keeps allocated until the process exits.
 *   - Returns FORK_ECAPACITY when fork_attn_workspace_bytes(T_cap,
 *     prefix_rows, Hq, Hkv, d, rope_theta, flags) exceeds
 *     FORK_NOALLOC_SCRATCH_BYTES (e.g. T_cap = 8192 with 16 q-heads,
 *     4 kv-heads, d = 128 fits (about 17 MB: rotated keys, fp16 values and
 *     tables); T_cap = 16384 with the same heads does not).
 *   - Calls no allocating routine (the array is the one piece of state the
 *     library keeps between calls).  The first call on a device looks up the
 *     array's device address (and loads the module there); make that first
 *     call before any stream capture.
 *   - Every call, on any stream, uses the same array and leaves its contents
 *     behind.  Nothing in it has to start at zero (each call writes every
 *     value it reads), but two calls that overlap on the GPU race on it:
 *     order them on one stream or with events. */
#define FORK_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int fork_attn_noalloc(const fork_meta* m, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      uint16_t* o, int32_t Hq, int32_t Hkv, int32_t d, int32_t window,
                      float rope_theta, float scale, const uint16_t* prefix_k,
                      const uint16_t* prefix_v, int32_t prefix_rows, uint32_t flags, void* stream);

/* ------------------------------------------------------------------------
 * Gated DeltaNet, two calls (onedev "무엇과 다른가"; rainbus "前置知识" and
 * "方法步骤详情" step 2: the first call processes every trunk segment and
 * emits each request's float32 state S_P and conv window; the second call
 * processes every question segment at once, each resuming from its own
 * S_P by index, the causal conv reading the trunk's last tokens).
 *
 * Per head, after a depthwise causal conv of width K (tap K-1 multiplies
 * the current token) and SiLU on the q, k, v channels and an L2
 * normalisation of q and k (x * (sum x^2 + 1e-6)^(-1/2)):
 *   S_t = alpha_t S_{t-1} (I - eta_t k_t k_t^T) + eta_t v_t k_t^T,  o_t = S_t q_t
 * with S of shape d x d (rows index v, columns index k).
 * Shared arguments:
 *   q, k, v [T_cap, H, d] bf16; alpha, eta [T_cap, H] float32 (gates after
 *   the sigmoid); conv_w [3 (q,k,v), H, d, K] float32; d = dk = dv in
 *   {64, 128}; K = 4; chunk = 64 (chunks are aligned to each segment's
 *   start); o [T_cap, H, d] bf16 (only the call's own segment rows written).
 * ------------------------------------------------------------------------ */

/* Call 1: every trunk segment.
 *   init_state [R, H, d, d] float32 and init_conv [R, K-1, 3, H, d] bf16:
 *   state and raw conv inputs at position prefix_len_j for requests with a
 *   prefix (a checkpoint being resumed); NULL when no request has a prefix.
 *   Outputs: S_P [R, H, d, d] float32 (state after the whole trunk);
 *   conv_win [R, K-1, 3, H, d] bf16 (raw q,k,v inputs of trunk positions
 *   P-K+1..P-1, zero before position 0); S_ckpt / conv_ckpt (same layouts,
 *   may be NULL when no request has a checkpoint): state after positions
 *   < m and raw inputs of positions m-K+1..m-1 for requests with ckpt_pos m.
 */
int fork_gdn_trunk(const fork_meta* m, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   const float* alpha, const float* eta, const float* conv_w, int32_t H, int32_t d,
                   int32_t K, int32_t chunk, const float* init_state, const uint16_t* init_conv,
                   float* S_P, uint16_t* conv_win, float* S_ckpt, uint16_t* conv_ckpt, uint16_t* o,
                   uint32_t flags, void* stream);

/* Call 2: every question segment; question i of request j starts from
 * S_P[j] and conv_win[j] (read by index, never copied). */
int fork_gdn_branches(const fork_meta* m, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      const float* alpha, const float* eta, const float* conv_w, int32_t H,
                      int32_t d, int32_t K, int32_t chunk, const float* S_P,
                      const uint16_t* conv_win, uint16_t* o, uint32_t flags, void* stream);

/* ------------------------------------------------------------------------
 * Token forests (rainbus summary "未来方向" (2): a tree of draft tokens has the
 * shape of the request tree and can run in the same flat stream; DFlash-TfM
 * summary "GDN을 위한 롤백 없는 트리 검증": the tree in topological order, the
 * recurrence in its chunked form).  A forest of N nodes, node k with parent
 * parent[k] (-1 for a root; parents precede their children) and node_len[k]
 * tokens of its own, stored node after node in one unpadded stream (node k's
 * rows start at the sum of the earlier nodes' lengths).  Node k's sequence is
 * its ancestors' tokens, root first, followed by its own: its first token has
 * position pos0_k = the sum of its ancestors' lengths.  Every result equals
 * that of the node's sequence run alone.
 *   - Attention (fork_attn with FORK_FOREST): key y is visible to query x iff
 *     y's node is x's node or one of its ancestors, t_y <= t_x and, for a
 *     sliding window, t_x - t_y < W.  The keys of every ancestor are read in
 *     place: no row is copied.
 *   - Gated DeltaNet (fork_gdn_forest, one call per depth): a node starts from
 *     its parent's end state and conv window, read by the parent's state index,
 *     and writes its own at its index.
 *   - Readout (fork_readout): the leaves are the questions, in node order.
 * ------------------------------------------------------------------------ */

#define FORK_FOREST_MAX_DEPTH 7 /* ancestors of a node, at most (8 levels) */
#define FORK_FOREST_MAX_LEVELS (FORK_FOREST_MAX_DEPTH + 1)
/* int32 words of the plan written by fork_forest_plan for N nodes */
#define FORK_FOREST_PLAN_WORDS(N) ((size_t)(N) + 2 + FORK_FOREST_MAX_LEVELS)

/* Plan a forest on the host (no CUDA call): fill h_image (fork_meta_bytes
 * bytes for m's capacities, host memory) with the metadata that fork_attn,
 * fork_gdn_forest and fork_readout read, and h_plan
 * [FORK_FOREST_PLAN_WORDS(N)] with:
 *   h_plan[0]           number of levels L (1 + the greatest depth);
 *   h_plan[1 + l]       first state index of level l, l = 0..L (h_plan[1 + L] = N);
 *   h_plan[2 + FORK_FOREST_MAX_LEVELS + k]  state index of node k.
 * State indices order the nodes by depth, then by node number; node k's end
 * state and conv window live at its state index in the caller's arrays.
 * The metadata holds one segment per node (in state-index order) with its
 * stream rows, pos0_k and the state index of its parent (-1 for a root), the
 * per-token positions (pad rows -1), the last row of every leaf (leaves in
 * node order) and the attention work list, tile_tokens-token tiles aligned to
 * each node's first row, launched in non-increasing order of visible keys.
 * m->d_buf is not touched (copy h_image there, or use fork_build_forest_meta).
 * Errors: FORK_EINVAL (null pointer, invalid handle, N < 1, a parent not
 * before its child, a negative length, a leaf without tokens), FORK_ECAPACITY
 * (N > max_req, more leaves than max_q, more than T_cap tokens, a node deeper
 * than FORK_FOREST_MAX_DEPTH). */
int fork_forest_plan(const fork_meta* m, const int32_t* parent, const int32_t* node_len, int32_t N,
                     int32_t* h_image, int32_t* h_plan);

/* fork_forest_plan, then a copy of h_image to m->d_buf on `stream`.  From
 * pageable host memory the copy first waits for the work already on the
 * stream and has read h_image when the call returns; from pinned memory it is
 * asynchronous: keep h_image unchanged until the copy has completed. */
int fork_build_forest_meta(const fork_meta* m, const int32_t* parent, const int32_t* node_len,
                           int32_t N, int32_t* h_image, int32_t* h_plan, void* stream);

/* Gated DeltaNet of the nodes with state indices [first, first + count) of a
 * forest (one level: their parents' states must be complete, i.e. the previous
 * level's call came earlier on the stream).  Shared arguments as for
 * fork_gdn_trunk, d = 128.  node_state [N, H, d, d] float32 and node_conv
 * [N, K-1, 3, H, d] bf16, indexed by state index: a node with pos0 > 0 starts
 * from its parent's entries, a node with pos0 = 0 from zero; every node writes
 * its end state and the raw conv inputs of its sequence's last K-1 positions
 * (zero before position 0) at its own index.  o: the nodes' rows.
 * Errors: FORK_EINVAL (null pointers, first < 0, count < 0, first + count >
 * max_req, d != 128, FORK_WARP_MMA). */
int fork_gdn_forest(const fork_meta* m, int32_t first, int32_t count, const uint16_t* q,
                    const uint16_t* k, const uint16_t* v, const float* alpha, const float* eta,
                    const float* conv_w, int32_t H, int32_t d, int32_t K, int32_t chunk,
                    float* node_state, uint16_t* node_conv, uint16_t* o, uint32_t flags,
                    void* stream);

/* ------------------------------------------------------------------------
 * Selective readout, eq. (1) (onedev "어떻게 동작하나"; rainbus "前置知识"):
 * p_i(o) = exp(w_o . h_i) / sum_{o' in O_i} exp(w_o' . h_i), h_i the hidden
 * row of question i's last token.
 *   h [T_cap, D] bf16 (the GDN output, heads flattened); w_opt [sum O, D]
 *   bf16; opt_off device int32 [Nq + 1] CSR offsets (opt_off[0] = 0, at
 *   least one option per question); p [sum O] float32.  Logits and the
 *   softmax are float32; D a multiple of 8, at most 16384.
 * ------------------------------------------------------------------------ */
int fork_readout(const fork_meta* m, const uint16_t* h, int32_t D, const uint16_t* w_opt,
                 const int32_t* opt_off, float* p, uint32_t flags, void* stream);

/* ------------------------------------------------------------------------
 * Selective readout with the last layer's pointwise block on the question
 * rows only (onedev "어떻게 쓰나": the MLP and what follows run only on each
 * question's last-token row, which changes no output).  The pages give no
 * form for the block; this one is a pre-norm SwiGLU MLP with a residual and a
 * final RMSNorm, rmsnorm(x) = x * (mean x^2 + 1e-6)^(-1/2):
 *   n_i = bf16(rmsnorm(h_i) * g1),  a_i = bf16(silu(W_gate n_i) * (W_up n_i)),
 *   y_i = h_i + W_down a_i,  z_i = rmsnorm(y_i) * g2,
 *   p_i(o) = exp(w_o . z_i) / sum_{o' in O_i} exp(w_o' . z_i).
 *   h [T_cap, D] bf16 (rows read at each question's last token); g1, g2 [D]
 *   float32; w_gate, w_up [F, D] and w_down [D, F] bf16, row-major; w_opt,
 *   opt_off, p as for fork_readout; h, g1, g2, the weights, w_opt and the
 *   workspace 16-byte aligned.  D a multiple of 64, at most 8192; F a
 *   multiple of 64, at most 65536.  Products on the tensor cores with bf16
 *   operands and float32 accumulation (tcgen05, 128 output columns per CTA,
 *   when D is a multiple of 128 and F of 256; else warp-level MMA); norms,
 *   SiLU and eq. (1) in float32.
 *   workspace: device buffer of fork_readout_mlp_workspace_bytes(max_q, D,
 *   F) bytes, 16-byte aligned, owned by the caller (the normalised rows
 *   [Mpad, D] bf16, the activations [Mpad, F] bf16, y [Mpad, D] float32 and,
 *   on the tcgen05 path, the partial products [Mpad, max(2F, 4D)] float32,
 *   each at a 256-byte-aligned offset, Mpad = max_q rounded up to 64).
 *   FORK_EINVAL for null pointers, bad sizes, misaligned buffers or a short
 *   workspace, with nothing launched.
 * ------------------------------------------------------------------------ */
size_t fork_readout_mlp_workspace_bytes(int32_t max_q, int32_t D, int32_t F);
int fork_readout_mlp(const fork_meta* m, const uint16_t* h, int32_t D, int32_t F, const float* g1,
                     const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                     const float* g2, const uint16_t* w_opt, const int32_t* opt_off, float* p,
                     void* workspace, size_t ws_bytes, uint32_t flags, void* stream);

/* The same pointwise block on every stream row (the cost the selective readout
 * avoids; onedev "어떻게 쓰나"): for each row r < T,
 *   z_r = bf16(rmsnorm(h_r + W_down a_r) * g2),  a_r = bf16(silu(W_gate n_r) * (W_up n_r)),
 *   n_r = bf16(rmsnorm(h_r) * g1);
 * fork_readout(m, z, ...) then gives eq. (1) from the questions' rows of z.
 *   z [T_cap, D] bf16 (pad rows not written); other arguments as for
 *   fork_readout_mlp; workspace of fork_pointwise_rows_workspace_bytes(T_cap,
 *   D, F) bytes (the same three buffers for T_cap rows). */
size_t fork_pointwise_rows_workspace_bytes(int32_t T_cap, int32_t D, int32_t F);
int fork_pointwise_rows(const fork_meta* m, const uint16_t* h, int32_t D, int32_t F, const float* g1,
                        const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                        const float* g2, uint16_t* z, void* workspace, size_t ws_bytes, uint32_t flags,
                        void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FORKATTN_H */
