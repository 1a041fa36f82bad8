/*
 * dflash.h -- C ABI of libdflash, the GB300 (sm_103a) hot path of DFlash-style
 * block-diffusion speculative drafting with target taps.
 *
 * Three stages, each behind one call:
 *   dflash_fuse_taps    tap planes -> fc -> hidden_norm -> fused ring rows,
 *                       then K/V injection into every drafter layer's cache
 *   dflash_draft_block  the drafter's block forward over anchor + 15 mask rows,
 *                       final norm, shared LM head, per-position top-k
 *   dflash_topk         vocab-wide top-k / argmax / temperature sampling
 *   dflash_verify       greedy longest-prefix + bonus, or speculative sampling
 *                       with residual correction
 * and the rows after them: dflash_draft_stop (min-p stop),
 * dflash_select_path (the DFlash2 candidate-path selector), dflash_tree_build
 * and dflash_tree_verify (tree drafting and greedy tree verification).
 *
 * Sources, cited by page title and section:
 *   [TF1851]  TensorFold pull request #1851, "qwen27 dflash: read and run the
 *             9B's DFlash drafter beside DFlash2", section "What this changes".
 *   [ST3457]  Strata pull request #3457, "Metal: opt-in --dflash DFlash2
 *             drafter in place of the MTP layer", sections "Approach" and
 *             "Validation".
 *   [EXPL]    "DFlash 解碼加速：原理、限制與 oMLX 實作" (a DFlash decoding
 *             explainer), sections 三 (how DFlash works), 四 (target
 *             verification) and 五 (DFlash 2).
 *   [PROT]    "Port the DFlash2 protocol, not its checkpoint", sections
 *             "What is portable" and "Golden replay before training".
 *
 * Conventions
 *   - Every function returns DFLASH_OK (0) or a negative DFLASH_E_* code, and
 *     never throws. dflash_strerror() names a code.
 *   - The caller owns all memory: weights, state memory, workspaces, inputs
 *     and outputs. The library never allocates device memory. Pointers named
 *     "device" must be device (or managed) memory of the handle's device;
 *     pointers named "host" are read on the host during the call and may be
 *     freed when it returns.
 *   - Every device-side step is enqueued asynchronously on the caller's
 *     stream (a cudaStream_t passed as dflash_stream_t; NULL = legacy default
 *     stream). Arguments are validated on the host before anything is
 *     enqueued; a call that returns an error has enqueued nothing.
 *   - bf16 tensors are IEEE bfloat16, row-major, densely packed unless a
 *     stride is given. Sums are fp32.
 *   - Faults only the device can see (an anchor id outside the vocabulary, a
 *     timed-out wait) set bits in the state's device status word; read it with
 *     dflash_device_status(). No kernel traps.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dflash_stream_t; /* a cudaStream_t */

/* ---------------------------------------------------------------- status */
enum {
  DFLASH_OK = 0,
  DFLASH_E_INVALID_ARG = -1,   /* NULL pointer, negative size, bad mode */
  DFLASH_E_TAPS_RANGE = -2,    /* tap count outside 1..8, or a tap past the target [TF1851 item 1] */
  DFLASH_E_TAPS_REPEATED = -3, /* the same target layer tapped twice [TF1851 item 1] */
  DFLASH_E_CAUSAL = -4,        /* a causal draft is refused [TF1851 item 1] */
  DFLASH_E_SHAPE = -5,         /* shapes this drafter cannot run */
  DFLASH_E_CAPACITY = -6,      /* a position past the ring / served span */
  DFLASH_E_WORKSPACE = -7,     /* workspace or state memory too small or misaligned */
  DFLASH_E_CUDA = -8,          /* a CUDA runtime / driver call failed */
  DFLASH_E_TIMEOUT = -9,       /* a device-side wait ran out (status word) */
  DFLASH_E_DEVICE_FAULT = -10, /* the device flagged bad data (status word) */
  DFLASH_E_UNSUPPORTED = -11   /* no sm_100-family device, or a missing driver entry point */
};

/* bits of the device status word */
enum {
  DFLASH_STATUS_BAD_TOKEN = 1,   /* an anchor id outside [0, vocab): row read as id 0 */
  DFLASH_STATUS_TIMEOUT = 2,     /* a bounded mbarrier wait expired; results invalid */
  DFLASH_STATUS_BAD_DRAFT = 4    /* a draft id outside [0, vocab) in dflash_verify */
};

#define DFLASH_MAX_TAPS 8
#define DFLASH_MAX_LAYERS 64
#define DFLASH_BLOCK 16 /* anchor + 15 mask rows [TF1851 item 1] */
#define DFLASH_MAX_TOPK 16

enum { DFLASH_LAYER_FULL = 0, DFLASH_LAYER_SLIDING = 1 };
enum { DFLASH_VARIANT_V1 = 1, DFLASH_VARIANT_2 = 2 };
enum { DFLASH_VERIFY_GREEDY = 0, DFLASH_VERIFY_SAMPLE = 1 };
#define DFLASH_MAX_SAMPLE_STREAMS 65535
enum { DFLASH_FUSE_INJECT_KV = 1 }; /* dflash_fuse_taps flags */

/* ---------------------------------------------------------------- config
 * The drafter's shape. [TF1851 item 1]: taps (up to eight), block, mask
 * token and layer kinds come from the drafter's config; its body is the qwen3
 * layer with eleven tensors. */
typedef struct dflash_config {
  int32_t variant;        /* DFLASH_VARIANT_V1 (fusing drafter, named "DFlash") or _2 ("DFlash2") */
  int32_t hidden;         /* H: hidden width of target taps and drafter */
  int32_t n_taps;         /* N: tap planes, 1..8 */
  int32_t tap_layers[DFLASH_MAX_TAPS]; /* target layer ids of the taps (first n_taps used) */
  int32_t target_layers;  /* number of target layers (taps must be < this) */
  int32_t n_layers;       /* L: drafter layers, 1..DFLASH_MAX_LAYERS */
  int32_t n_q_heads;      /* query heads */
  int32_t n_kv_heads;     /* key/value heads; n_q_heads % n_kv_heads == 0 */
  int32_t head_dim;       /* d: 32, 64 or 128 */
  int32_t ffn;            /* F: SwiGLU width */
  int32_t vocab;          /* V: target vocabulary (shared embedding / LM head), multiple of 128 */
  int32_t block;          /* must be 16 */
  int32_t mask_token;     /* id of the mask token, in [0, V) */
  int32_t causal;         /* must be 0: a causal draft is refused */
  int32_t sliding_window; /* W: window of sliding layers, > 0 if any layer slides */
  int32_t layer_kind[DFLASH_MAX_LAYERS]; /* DFLASH_LAYER_FULL or _SLIDING per layer */
  float rope_theta;       /* rotate-half RoPE base */
  float rms_eps;          /* RMSNorm epsilon */
  int32_t conv_groups;    /* 0, or the weight groups of DFlash2's two-tap dynamic
                             convolution over the block (variant 2 only; see
                             dflash_draft_conv) */
} dflash_config;

/* Check a config. Returns DFLASH_OK or the refusal: E_TAPS_RANGE (n_taps
 * outside 1..8, or a tap id outside [0, target_layers)), E_TAPS_REPEATED,
 * E_CAUSAL (causal != 0), E_SHAPE (block != 16; n_q_heads % n_kv_heads;
 * hidden != n_q_heads * head_dim; head_dim not 32/64/128; hidden, ffn or
 * n_kv_heads*head_dim not a multiple of 128; vocab not a multiple of 128;
 * mask token outside the vocabulary; a sliding layer with window <= 0;
 * variant not 1 or 2; conv_groups != 0 in a v1 drafter, whose layout has no
 * conv tensor; conv_groups outside 0..32 or hidden / conv_groups not a
 * multiple of 16), E_INVALID_ARG (NULL). [TF1851 item 1] */
int dflash_config_validate(const dflash_config* cfg);

/* "DFlash" for a v1 drafter, "DFlash2" otherwise, NULL for NULL. [TF1851
 * item 6: Config.kind() names the layout]. Static string. */
const char* dflash_kind(const dflash_config* cfg);

/* Prompt-memory price of one prompt row's taps, in bytes [TF1851 item 3]:
 * a v1 drafter holds its N planes, their row-major copy, fc's row and the
 * fused row, (2N + 2) * H * 2 (18 * H * 2 for eight taps); a DFlash2 drafter
 * keeps the N raw planes, N * H * 2. Returns -1 for NULL. (This library's
 * fc reads the planes in place, so it never builds the row-major copy.) */
int64_t dflash_tap_row_bytes(const dflash_config* cfg);

/* One fused ring row: H bf16 values, 8 KiB a token at hidden 4096
 * [TF1851 item 4]. Returns -1 for NULL. */
int64_t dflash_fused_row_bytes(const dflash_config* cfg);

/* ---------------------------------------------------------------- weights
 * Device pointers to bf16 tensors, row-major [out_features, in_features].
 * [TF1851 item 1]: eleven tensors a layer plus fc, hidden_norm and norm; the
 * embedding / LM head is the target's, shared and frozen [EXPL 三]. All base
 * addresses must be 16-byte aligned. The pointed-to memory must outlive the
 * handle. */
typedef struct dflash_layer_weights {
  const void* input_norm; /* [H] */
  const void* q_proj;     /* [n_q*d, H] */
  const void* k_proj;     /* [n_kv*d, H] */
  const void* v_proj;     /* [n_kv*d, H] */
  const void* o_proj;     /* [H, n_q*d] */
  const void* q_norm;     /* [d] per-head RMSNorm gain */
  const void* k_norm;     /* [d] */
  const void* post_norm;  /* [H] post-attention RMSNorm gain */
  const void* gate_proj;  /* [F, H] */
  const void* up_proj;    /* [F, H] */
  const void* down_proj;  /* [H, F] */
} dflash_layer_weights;

typedef struct dflash_weights {
  const void* fc;          /* [H, N*H]: concat of the N taps (tap 0 first) -> H */
  const void* hidden_norm; /* [H] */
  const void* norm;        /* [H] final norm */
  const void* embed;       /* [V, H] embedding, also the LM head */
  const dflash_layer_weights* layers; /* host array of n_layers entries (copied) */
  const void* conv_norm;   /* [H] two-tap convolution's RMSNorm gain (conv_groups > 0; else unused) */
  const void* conv_proj;   /* [2 * conv_groups, H]: row 2g + t = tap t of group g */
} dflash_weights;

typedef struct dflash_handle dflash_handle;
typedef struct dflash_state dflash_state;

/* Create a drafter handle on the current CUDA device. Validates cfg (same
 * codes as dflash_config_validate) and the weight pointers (E_INVALID_ARG for
 * NULL or unaligned), checks for an sm_100-family device (E_UNSUPPORTED), and
 * prepares the TMA descriptors of every weight. Host memory only; *out is set
 * on success. */
int dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_handle** out);
int dflash_destroy(dflash_handle* h); /* NULL is fine */

/* ---------------------------------------------------------------- state
 * Per-stream drafter state in caller-owned device memory: the fused ring
 * (served span of fused rows, [TF1851 item 4]), each layer's context K/V
 * cache (a full layer keeps the span, a sliding layer a ring of its window),
 * the committed length of every stream, RoPE tables and the status word.
 * ring_capacity R bounds every stream's length; positions >= R are refused
 * (E_CAPACITY), as a request past the served window is [TF1851 "Exactness"]. */
int dflash_state_bytes(const dflash_handle* h, int streams, int ring_capacity, size_t* bytes);

/* Carve a state out of dev_mem (>= dflash_state_bytes, 256-byte aligned),
 * upload its RoPE table (synchronously) and zero the lengths and status on
 * `stream`. All streams start empty. *out is host memory freed by
 * dflash_state_free (which does not touch dev_mem). */
int dflash_state_init(dflash_handle* h, void* dev_mem, size_t bytes, int streams, int ring_capacity,
                      dflash_stream_t stream, dflash_state** out);
int dflash_state_free(dflash_state* st);

/* Committed length of stream s as enqueued so far (host mirror). */
int dflash_state_length(const dflash_state* st, int s, int64_t* len);

/* Roll stream s back to new_len <= its length: rejected or cancelled rows
 * are dropped [PROT "What is portable": rollback of the rejected suffix].
 * Sliding-window cache slots that later rows overwrote are rebuilt from the
 * fused ring (needs ws of dflash_fuse_workspace_bytes(h, W) bytes). */
int dflash_state_truncate(dflash_handle* h, dflash_state* st, int s, int64_t new_len, void* ws,
                          size_t ws_bytes, dflash_stream_t stream);

/* Inspection of the state's device buffers (for checkpoints, tests and
 * tools; writing through them bypasses the length bookkeeping).
 * Ring: *ring = bf16 [streams][ring_capacity][H]; row p of stream s is the
 * fused row of position p. Layer l caches: *k, *v = bf16
 * [streams][n_kv_heads][cap][head_dim]; a full layer has cap = ring_capacity
 * and slot = position, a sliding layer cap = min(W, ring_capacity) and
 * slot = position % cap. */
int dflash_state_ring(const dflash_state* st, void** ring);
int dflash_state_cache(const dflash_state* st, int layer, void** k, void** v, int* cap);

/* Read and clear the state's device status word (synchronises `stream`).
 * *out receives DFLASH_STATUS_* bits. Returns E_TIMEOUT / E_DEVICE_FAULT when
 * the corresponding bits were set, DFLASH_OK when clear. */
int dflash_device_status(dflash_state* st, dflash_stream_t stream, int32_t* out);

/* Self-test of the bounded waits: one kernel waits on an mbarrier that
 * nothing arrives at, gives up after `cycles` SM cycles (0 .. 1e10; the hot
 * path's waits use 3e9) and sets DFLASH_STATUS_TIMEOUT in the state's status
 * word, exactly as an expired wait of the hot path does; the context stays
 * usable. Read the result with dflash_device_status (E_TIMEOUT). */
int dflash_state_wait_probe(dflash_state* st, int64_t cycles, dflash_stream_t stream);

/* ---------------------------------------------------------------- fusion
 * Tap fusion and context append [TF1851 item 4; ST3457 "Approach": each
 * prompt chunk and committed window injects its rows' features].
 * planes: host array of N device pointers; plane p is [rows, H] bf16 with a
 * row stride of plane_row_stride elements (>= H, multiple of 8); plane
 * bases 16-byte aligned. The rows are nseg segments in order: segment i holds
 * seg_rows[i] rows of stream seg_stream[i] at positions seg_start[i] ..
 * seg_start[i] + seg_rows[i] - 1 (host arrays). Each segment must start at
 * its stream's committed length (append only; a stream may appear once) and
 * end at or below the ring capacity (else E_CAPACITY).
 * For every row: y = concat(planes) * fc^T; fused = bf16(RMSNorm(y) *
 * hidden_norm) written to the ring. With DFLASH_FUSE_INJECT_KV, every layer l
 * also gets K = bf16(RoPE(k_norm(fused * k_proj_l^T), pos)) and V =
 * bf16(fused * v_proj_l^T) in its cache (context rows feed K and V only), and the stream
 * lengths advance. Without it only the ring is written and lengths stay
 * (fusion-only timing). Up to 1024 rows a call, a row's fused values and
 * K/V do not depend on which other rows share the call (a fill resumed after
 * dflash_state_truncate rebuilds the same cache). ws: >=
 * dflash_fuse_workspace_bytes(h, rows). */
int dflash_fuse_workspace_bytes(const dflash_handle* h, int rows, size_t* bytes);
int dflash_fuse_taps(dflash_handle* h, dflash_state* st, const void* const* planes, int64_t plane_row_stride,
                     int nseg, const int32_t* seg_stream, const int64_t* seg_start, const int32_t* seg_rows,
                     int flags, void* ws, size_t ws_bytes, dflash_stream_t stream);

/* ---------------------------------------------------------------- drafting
 * One block forward for streams s_begin .. s_begin + s_count - 1 of the state
 * [TF1851 item 1; EXPL 三]. For each stream, with C its committed length:
 * rows = [anchor_ids[i], mask x 15] at positions C..C+15; every layer:
 * h = RMSNorm(X); Q/K/V projections with per-head q_norm/k_norm and RoPE;
 * non-causal attention over the layer's visible context (full: positions
 * 0..C-1; sliding: C-W..C-1) plus the block's 16 rows; O-proj added to the
 * residual; RMSNorm; SwiGLU MLP added to the residual. Then RMSNorm (norm)
 * and the shared LM head on the 15 mask rows.
 * anchor_ids: device int32 [s_count]. logits_out: device bf16
 * [s_count*15, V] or NULL (then the logits live in ws). topk_ids (int32) and
 * topk_vals (fp32, the bf16 logit values): device [s_count*15, k], k in
 * 1..16, descending, ties to the lower id; either may be NULL to skip top-k.
 * Batch invariance [TF1851 "Exactness": concurrent equals solo]: with
 * s_count <= 4 a stream's logits and ids are bit-identical whichever streams
 * share the call (the reductions' split depends only on the weights' shapes
 * and the stream's own length); with more streams the GEMM split and the
 * attention split are chosen for throughput and the fp32 summation order,
 * hence the last bits, depend on s_count.
 * ws: >= dflash_draft_workspace_bytes(h, st, s_count, logits_out == NULL). */
int dflash_draft_workspace_bytes(const dflash_handle* h, const dflash_state* st, int s_count, int need_logits,
                                 size_t* bytes);
int dflash_draft_block(dflash_handle* h, dflash_state* st, int s_begin, int s_count, const int32_t* anchor_ids,
                       void* logits_out, int32_t* topk_ids, float* topk_vals, int k, void* ws, size_t ws_bytes,
                       dflash_stream_t stream);

/* The same block forward in stages, for staged execution and for
 * stage-isolated checks (each stage fed a reference input, so errors do not
 * compound). A layer is two stages, one per residual add [TF1851 item 1]:
 * stage 2l = layer l's input norm, Q/K/V, attention and O projection added
 * to the residual; stage 2l+1 = its post-attention norm and SwiGLU MLP added
 * to the residual. X is the fp32 residual stream, device [s_count*16, H],
 * row 16*i + j = row j (0 = anchor) of stream s_begin + i; 16-byte aligned.
 * dflash_draft_stages runs stages stage0 .. stage1-1 (0 <= stage0 <= stage1
 * <= 2L) on X in place, with the streams' K/V caches and lengths as
 * dflash_draft_block would; dflash_draft_head applies the final norm to the
 * 15 mask rows of every stream, the LM head (logits_out required) and the
 * optional top-k. Both take the workspace of
 * dflash_draft_workspace_bytes(h, st, s_count, 0). */
int dflash_draft_stages(dflash_handle* h, dflash_state* st, int s_begin, int s_count, int stage0, int stage1,
                        float* X, void* ws, size_t ws_bytes, dflash_stream_t stream);
int dflash_draft_head(dflash_handle* h, dflash_state* st, int s_count, const float* X, void* logits_out,
                      int32_t* topk_ids, float* topk_vals, int k, void* ws, size_t ws_bytes, dflash_stream_t stream);

/* ---------------------------------------------------------------- two-tap convolution
 * DFlash2's dynamic short convolution [EXPL 五 "Dynamic short convolution":
 * a two-tap dynamic convolution over adjacent positions of the block against
 * suffix decay; kernel size 2]. Reading: a dynamic convolution (Wu et al.
 * 2019: per-position kernel weights from the position's own input,
 * softmax-normalised over the taps, shared within a channel group) of kernel
 * size 2, causal inside the block, as a residual branch after the last layer:
 *   h = bf16(RMSNorm(X) * conv_norm); z_i = h_i . conv_proj^T  [groups, 2]
 *   a_i = softmax over the two taps of z_i (per group)
 *   X_i += a_i[g, 0] * h_{i-1} + a_i[g, 1] * h_i   (h_{-1} = 0; channel c in
 *          group c / (H / groups))
 * dflash_draft_block runs it before the final norm whenever conv_groups > 0.
 * dflash_draft_conv runs it alone on a caller residual X (device fp32
 * [16 * s_count, H], in place), for stage-by-stage checks; ws as for
 * dflash_draft_block. E_INVALID_ARG when the handle has no convolution. */
int dflash_draft_conv(dflash_handle* h, dflash_state* st, int s_count, float* X, void* ws, size_t ws_bytes,
                      dflash_stream_t stream);

/* ---------------------------------------------------------------- top-k
 * Per row of a bf16 logit matrix [rows, vocab] (device, rows contiguous):
 * the k largest logits (descending, ties to the lower id; ids int32, vals fp32
 * = the bf16 values) ["PROT" top candidates at each position]. With uniforms
 * (device fp32 [rows]) also one draw per row from softmax(logits / T) by
 * inverse CDF: the smallest id whose running sum in ascending id order exceeds
 * u * total (int32 [rows] in `sampled`). ids/vals may be NULL when k == 0;
 * sampled must be non-NULL iff uniforms is. vocab multiple of 8, T > 0. */
int dflash_topk(const void* logits, int rows, int vocab, int k, float temperature, const float* uniforms,
                int32_t* ids, float* vals, int32_t* sampled, dflash_stream_t stream);

/* ---------------------------------------------------------------- min-p stop
 * Where a draft stops [ST3457 "Problem and result": `--spec-min-p` stops a
 * draft where the confidence falls below it]. Reading (the v1 body has no
 * selector): the confidence of mask row i is the largest entry of
 * softmax(logits_i / temperature), and a stream's draft keeps its leading
 * rows whose confidence is at least min_p.
 *   logits:    device bf16 [streams * 15, vocab] (rows of a stream
 *              contiguous, as dflash_draft_block writes them), 16-byte
 *              aligned, vocab a multiple of 8.
 *   conf:      device fp32 [streams * 15] out.
 *   draft_len: device int32 [streams] out, in [0, 15].
 * temperature > 0, 0 <= min_p <= 1; otherwise DFLASH_E_INVALID_ARG and
 * nothing is enqueued. No workspace; asynchronous on `stream`. */
int dflash_draft_stop(const void* logits, int streams, int vocab, float temperature, float min_p, float* conf,
                      int32_t* draft_len, dflash_stream_t stream);

/* ---------------------------------------------------------------- candidate-path selector
 * The DFlash2 selector [EXPL 五 "Candidate path selector": keep the top-k
 * candidates of every position, score adjacent candidate pairs with a light
 * selector, choose one consistent path (selector_top_k 16, selector_rank 256
 * in the public DFlash2 config); TF1851 item 1: with no codebooks (rank 0)
 * the edge term is zero; PROT "What is portable": top candidates at each
 * position, then coherent candidate-path selection, then verification].
 * Reading: a path (candidate a_i at each position i) scores
 *   sum_i cand_vals[i][a_i] + sum_{i < P-1} <U[id(i, a_i)], W[id(i+1, a_{i+1})]>
 * (node scores: the drafter's logits, which rank paths as its
 * log-probabilities do); the chosen path maximises it, found by the max-sum
 * recursion over positions with ties to the lower candidate index at every
 * step. Edge dot products are fp32 sums in ascending rank order; path sums
 * fp32.
 *   cand_ids:   device int32 [streams, positions, k] (e.g. the top-k ids of
 *               dflash_draft_block or dflash_topk with positions = 15); an id
 *               outside [0, vocab) is not a candidate.
 *   cand_vals:  device fp32 [streams, positions, k] node scores.
 *   U, W:       device bf16 [vocab, rank] codebooks, 16-byte aligned (not
 *               read, and may be NULL, when rank == 0 or positions == 1).
 *   path_ids:   device int32 [streams, positions] out: the chosen ids.
 *   path_ranks: device int32 [streams, positions] out (may be NULL): their
 *               candidate indices.
 *   path_score: device fp32 [streams] out (may be NULL): the path's score.
 *   A stream with a position that has no valid candidate gets ids and ranks
 *   -1 and score -inf.
 * 1 <= positions <= 16, 1 <= k <= DFLASH_MAX_TOPK, 0 <= rank <=
 * DFLASH_MAX_SELECTOR_RANK with rank a multiple of 8; ws: device, 16-byte
 * aligned, >= dflash_select_path_workspace_bytes (0 bytes when positions ==
 * 1). Otherwise DFLASH_E_INVALID_ARG / DFLASH_E_WORKSPACE and nothing is
 * enqueued. Asynchronous on `stream`. */
#define DFLASH_MAX_SELECTOR_RANK 512
int dflash_select_path_workspace_bytes(int streams, int positions, int k, size_t* bytes);
int dflash_select_path(int streams, int positions, int k, int vocab, int rank, const int32_t* cand_ids,
                       const float* cand_vals, const void* U, const void* W, int32_t* path_ids, int32_t* path_ranks,
                       float* path_score, void* ws, size_t ws_bytes, dflash_stream_t stream);

/* ---------------------------------------------------------------- draft trees
 * Tree drafting and greedy tree verification [TF1851: streams draft
 * per-stream trees; with no codebooks (rank 0) the trees come from each
 * depth's marginals (item 1); EXPL 四: the greedy rule; PROT "Golden replay
 * before training": accepted prefix plus bonus]. Reading: the root (node 0,
 * depth 0) is the anchor; every node of depth j - 1 has as children the top
 * b_j candidates of mask row j (the drafter's marginal for position C + j),
 * in candidate order; nodes are numbered breadth first (children of earlier
 * nodes first), so a tree of widths b_1..b_D has
 * 1 + sum_j (b_1 * ... * b_j) nodes.
 *
 * dflash_tree_size: that node count. 1 <= depth <= 15, 1 <= b_j <= k <=
 * DFLASH_MAX_TOPK, at most DFLASH_MAX_TREE_NODES nodes; otherwise
 * DFLASH_E_INVALID_ARG. widths: host int32 [depth].
 *
 * dflash_tree_build: the trees of `streams` streams from their drafts.
 *   anchors:     device int32 [streams].
 *   topk_ids:    device int32 [streams * 15, k], the draft's per-row top-k
 *                ids (row s*15 + j - 1 is depth j of stream s), as
 *                dflash_draft_block writes them.
 *   node_tokens: device int32 [streams, N] out.
 *   node_parent: device int32 [streams, N] out, -1 for the root (may be NULL).
 *   node_depth:  device int32 [streams, N] out (may be NULL); a node's
 *                position is the stream's length C plus its depth.
 *   node_mask:   device uint32 [streams, N, ceil(N / 32)] out (may be NULL):
 *                bit m of row n is set iff node m is on the path from the
 *                root to n (the attention mask of a one-pass tree score).
 *
 * dflash_tree_verify: greedy verification of the trees. target_logits:
 * device bf16 [streams, N, vocab] (16-byte aligned, vocab a multiple of 8),
 * row n = the target's scores for the position after node n, having read the
 * path from the root to n. From the root, step to the child whose token is
 * the target's argmax at the current node (ties to the lowest id) while one
 * exists. accept_len: device int32 [streams] out (0..depth); out_tokens:
 * device int32 [streams, 16] out: the accepted path's tokens, the bonus (the
 * argmax at the last node reached), then -1; accept_node: device int32
 * [streams] out (may be NULL): the last node reached. ws: device, 16-byte
 * aligned, >= dflash_tree_verify_workspace_bytes. A single-branch tree (all
 * widths 1) verifies exactly as dflash_verify(GREEDY) on the chain. */
#define DFLASH_MAX_TREE_NODES 1024
int dflash_tree_size(int depth, const int32_t* widths, int k, int* nodes);
int dflash_tree_build(int streams, int depth, const int32_t* widths, int k, const int32_t* anchors,
                      const int32_t* topk_ids, int32_t* node_tokens, int32_t* node_parent, int32_t* node_depth,
                      uint32_t* node_mask, dflash_stream_t stream);
int dflash_tree_verify_workspace_bytes(int streams, int nodes, size_t* bytes);
int dflash_tree_verify(int streams, int depth, const int32_t* widths, int vocab, const int32_t* node_tokens,
                       const void* target_logits, int32_t* accept_len, int32_t* out_tokens, int32_t* accept_node,
                       void* ws, size_t ws_bytes, dflash_stream_t stream);

/* ---------------------------------------------------------------- verify
 * Target verification of S drafted blocks [EXPL 四; PROT "What is portable"].
 * draft_ids: device int32, d_{i+1} of stream s at draft_ids[(s*15 + i) * draft_ld]
 * (draft_ld = 1 for a dense [S, 15] array, k to read the top-1 column of a
 * [S*15, k] top-k output); target_logits: device bf16
 * [S, 16, V], row i = the target's scores for position C+i+1 (after reading
 * the anchor and d_1..d_i).
 * GREEDY: t_i = argmax row i (ties to the lowest id); a = length of the
 *   longest prefix with d_{i+1} == t_i; tokens = d_1..d_a, t_a.
 * SAMPLE: p_i = softmax(row i / T), q_{i+1} = softmax(draft_logits row i / T)
 *   (draft_logits: device bf16 [S, 15, V]); for i = 0..14 accept d_{i+1} iff
 *   u[s][i][0] * q(d) < p_i(d); at the first rejection draw from
 *   max(p_i - q_{i+1}, 0) (p_i if that is all zero); if none is rejected draw
 *   the bonus from p_15; draws use u[s][i][1] by inverse CDF. uniforms: device
 *   fp32 [S, 16, 2]. At most DFLASH_MAX_SAMPLE_STREAMS streams a call
 *   (E_INVALID_ARG above: a stream is one row of the kernels' grids).
 * Outputs: accept_len device int32 [S] (a in 0..15); out_tokens device int32
 * [S, 16]: the a+1 committed tokens then -1. A draft id outside [0, V) is
 * never accepted (and sets nothing else). ws: >= dflash_verify_workspace_bytes. */
int dflash_verify_workspace_bytes(int mode, int streams, int vocab, size_t* bytes);
int dflash_verify(int mode, int streams, int vocab, const int32_t* draft_ids, int draft_ld, const void* target_logits,
                  const void* draft_logits, const float* uniforms, float temperature, int32_t* accept_len,
                  int32_t* out_tokens, void* ws, size_t ws_bytes, dflash_stream_t stream);

/* ---------------------------------------------------------------- no-allocation variant
 * Sampling verification for callers that cannot allocate device memory (a
 * host framework that owns every allocation through its own pool, a plugin
 * inside another runtime, a serving loop that must not call the allocator
 * once running). Same arguments, rule and outputs as
 * dflash_verify(DFLASH_VERIFY_SAMPLE, ...), but the scratch lives in a
 * 248 KiB array inside the library (held on every GPU that loads it until
 * the process exits), so no workspace is passed. The pages have no
 * counterpart: this is an interface for such callers only.
 * - At most DFLASH_NOALLOC_MAX_STREAMS streams; more returns
 *   DFLASH_E_WORKSPACE and enqueues nothing.
 * - The first call on a device looks up the array's device address (once per
 *   device, with that device current). With lazy module loading (the CUDA
 *   default) that lookup may load the library's device code on that device,
 *   which allocates device memory for the module and may synchronise. So
 *   make one warm-up call per device at initialisation, before the loop
 *   that must not allocate and before any stream capture; later calls
 *   allocate nothing and never synchronise.
 * - All calls share the array: calls that overlap on the GPU (issued on
 *   different streams or from several host threads with nothing ordering
 *   them) race on it. Nothing in it needs to start at zero; each call writes
 *   every value it reads before reading it. */
#define DFLASH_NOALLOC_MAX_STREAMS 1024
int dflash_verify_sample_noalloc(int streams, int vocab, const int32_t* draft_ids, int draft_ld,
                                 const void* target_logits, const void* draft_logits, const float* uniforms,
                                 float temperature, int32_t* accept_len, int32_t* out_tokens,
                                 dflash_stream_t stream);

/* ---------------------------------------------------------------- misc */
const char* dflash_strerror(int code);
/* Kernel launches enqueued by this process so far (all entry points). */
int64_t dflash_launch_count(void);

/* Per-launch timing trace (process-wide). dflash_trace_enable(1) clears the
 * trace and starts recording: every kernel launch is then bracketed by two
 * CUDA events on its stream, with the launch's algorithmic bytes (each
 * weight, activation and output touched once) and flops. enable(0) stops.
 * dflash_trace_get waits for record i's end event and returns its label
 * (static string, e.g. "gemm.lm_head", "attention"), its duration in ms,
 * bytes and flops. Events cost a little GPU time; leave the trace off for
 * production timing. */
int dflash_trace_enable(int on);
int dflash_trace_count(void);
int dflash_trace_get(int i, const char** name, float* ms, double* bytes, double* flops);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
