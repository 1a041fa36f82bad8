"""Oracle: DFlash-style block-diffusion drafting, written from the pages' text.

TEST INFRASTRUCTURE ONLY -- imported by tests/, __graft_entry__.smoke() and the
bench's CPU-baseline leg, never by the product path.

Sources (cited by page title and section):

* TensorFold pull request #1851, "qwen27 dflash: read and run the 9B's DFlash
  drafter beside DFlash2" -- "What this changes", items 1 (drafter graph: qwen3
  body, eleven tensors a layer, fc, hidden_norm, norm, two residual adds, the
  fifteen mask rows, refusal of a causal draft), 3 (prompt-memory planner:
  18 x hidden x 2 bytes a prompt row for eight taps), 4 (fused ring rows of
  8 KiB a token; context rows appended as K and V only; sliding layers attend their
  own window, the full layer the whole span); "Exactness", the Precision
  bullet (bf16 activations, fp32 sums).
* Strata pull request #3457, "Metal: opt-in --dflash DFlash2 drafter in place
  of the MTP layer" -- "Approach" (each committed window injects its rows'
  features), "Validation" (native drafter checked against an f64 host
  reference).
* "DFlash 解碼加速：原理、限制與 oMLX 實作" (DFlash decoding explainer) --
  section 三 (features from several target depths fused by a projection and
  injected into every draft layer's K/V; one forward predicts all masked
  positions; shared, frozen embedding and LM head), section 四 (greedy rule;
  sampling acceptance with residual max(p_target - p_draft, 0)).
* "Port the DFlash2 protocol, not its checkpoint" -- "What is portable"
  (top candidates at each position, verification, accepted prefix plus bonus,
  rollback of the rejected suffix).

Precision reading. The drafter keeps bf16 activations and fp32 sums. The
oracle computes every sum in float64 and rounds to bf16 exactly where a
tensor is stored or handed to a matrix product: fused rows, the context K/V
caches, Q and the block's K/V, the normed inputs of the projections, the
attention output, the SwiGLU product, the final normed rows and the logits.
Everything in between (projection outputs before their norms, the residual
stream, norm statistics, the softmax) stays float64.

The same steps can also run with float32 arithmetic (``arithmetic(np.float32)``,
weights from ``weights_as(w, np.float32)``): a plain implementation of the
pages' precision (bf16 activations, fp32 sums; TensorFold #1851, "Exactness",
the Precision bullet), with the rotary angles still formed in float64 as any
careful implementation does. Its distance from the float64 run measures how
far two correct fp32 implementations of this method may drift apart after
several layers of bf16 rounding; the parity tests take their end-to-end
envelope for deep drafters from it. The default is float64.

Readings of points the pages leave open (each one is stated where used):
RMSNorm epsilon 1e-6; rotate-half RoPE with theta from the config; context
rows at absolute positions 0..C-1, the anchor at C and the mask rows at
C+1..C+15; a sliding layer sees context positions >= C - W plus all 16 block
rows; q_norm / k_norm are per-head RMSNorms over the head dimension; the LM
head runs on the 15 mask rows only; ties in argmax and top-k go to the lower
index; sampling accepts when u * q(x) < p(x) and draws by inverse CDF
(smallest j whose running sum exceeds u times the total, summed in ascending
index order), falling back to p when the residual is all zero.

Pins (tests/test_oracle_*.py): bf16 rounding against torch's converter on
fp32-representable values; RMSNorm and RoPE closed forms; brute-force
attention; window enumeration; fusion with an identity fc; byte constants and
tensor inventory printed on the pages; greedy fixtures (zero, partial, full
acceptance, ties); the sampling rule's output distribution equal to p
(exact enumeration) and a chi-square check of draws.
"""
from __future__ import annotations

import contextlib
import math

import numpy as np

FULL = 0
SLIDING = 1
BLOCK = 16  # anchor + 15 mask rows (TensorFold #1851, item 1)

__all__ = [
    "arithmetic",
    "weights_as",
    "BLOCK",
    "FULL",
    "SLIDING",
    "round_bf16",
    "to_f64",
    "weights_to_f64",
    "rms_norm",
    "rope",
    "fuse_taps",
    "context_kv",
    "visible_positions",
    "block_attention",
    "silu",
    "block_embed",
    "attention_half",
    "mlp_half",
    "draft_layer",
    "block_conv",
    "draft_head",
    "draft_block",
    "OracleStreams",
    "topk",
    "argmax_lowest",
    "greedy_verify",
    "softmax_t",
    "draft_confidence",
    "selector_edges",
    "path_score",
    "select_path",
    "tree_nodes",
    "tree_mask",
    "tree_greedy_verify",
    "draft_stop",
    "inverse_cdf",
    "sample_rows",
    "sampling_verify",
    "fused_row_bytes",
    "raw_plane_bytes",
    "tap_row_bytes",
    "drafter_tensor_count",
    "kind_name",
    "validate_config",
]

# ----------------------------------------------------------------------------
# arithmetic precision

_F = np.float64  # floating type of every sum, product and norm statistic below


@contextlib.contextmanager
def arithmetic(dtype):
    """Run the drafter's arithmetic (fusion, context K/V, the block forward
    and the head) in ``dtype`` (np.float64 or np.float32) inside the block.

    The bf16 rounding points stay where they are; only the type of the sums
    in between changes. Verification and sampling keep float64.
    """
    global _F
    old = _F
    _F = np.dtype(dtype).type
    try:
        yield
    finally:
        _F = old


def weights_as(w, dtype):
    """A copy of a weight dict (as from weights_to_f64) in another floating
    type; bf16 weights are exact in float32 and float64."""
    out = {k: np.asarray(v, dtype=dtype) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: np.asarray(v, dtype=dtype) for k, v in lw.items()} for lw in w["layers"]]
    return out


# ----------------------------------------------------------------------------
# number formats

_BF16_OVERFLOW = 2.0 ** 128


def round_bf16(x):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits and float32's exponent range. For x in
    [2^(e-1), 2^e) the spacing is 2^(e-8); below the smallest normal (2^-126)
    the spacing stays at the subnormal step 2^-133. Values that round to
    2^128 or beyond become infinities.
    """
    x = np.asarray(x)
    if x.dtype == np.float32:  # float32 arithmetic: round in float64, bf16 values are exact in float32
        return round_bf16(x.astype(np.float64)).astype(np.float32)
    x = x.astype(np.float64)
    _, e = np.frexp(x)
    q = np.maximum(e - 8, -133)
    r = np.ldexp(np.rint(np.ldexp(x, -q)), q)
    big = np.abs(r) >= _BF16_OVERFLOW
    if np.any(big):
        r = np.where(big, np.copysign(np.inf, x), r)
    return r


def to_f64(t):
    """A torch bf16/fp32 tensor (any device) or array -> float64 ndarray (exact)."""
    if hasattr(t, "detach"):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def weights_to_f64(w):
    """Convert a weight dict from the synthetic generator to float64 arrays."""
    out = {k: to_f64(v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: to_f64(v) for k, v in lw.items()} for lw in w["layers"]]
    return out


# ----------------------------------------------------------------------------
# operators


def rms_norm(x, g, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g."""
    x = np.asarray(x, dtype=_F)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope(x, pos, theta):
    """Rotate-half rotary embedding over the last axis (qwen3 convention).

    Dimension i < d/2 pairs with i + d/2 and turns by the angle
    pos * theta^(-2i/d). ``pos`` broadcasts against x's leading axes.
    """
    x = np.asarray(x, dtype=_F)
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-(np.arange(half, dtype=np.float64) * 2.0) / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv
    c, s = np.cos(ang).astype(_F), np.sin(ang).astype(_F)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


def fuse_taps(planes, fc, hidden_norm, eps):
    """Tap fusion: concat the N tap planes (tap 0 first), project with fc, RMSNorm.

    TensorFold #1851 item 4 (the taps pass runs fc and hidden_norm as a v1
    drafter's taps complete; a ring row is the fused row, 8 KiB a token at
    hidden 4096, so bf16) and the DFlash explainer section 三 (features from
    several depths fused by a projection). planes: list of [rows, H];
    fc: [H, N*H]. Returns the bf16 fused rows as float64 [rows, H].
    """
    x = np.concatenate([np.asarray(p, dtype=_F) for p in planes], axis=1)
    y = x @ np.asarray(fc, dtype=_F).T
    return round_bf16(rms_norm(y, hidden_norm, eps))


def context_kv(fused, positions, layer, model):
    """One drafter layer's K and V for fused context rows (context rows feed K and V only).

    TensorFold #1851 item 4 and the explainer's section 三 (KV injection into
    every draft layer). Reading: no input norm on context rows (they already
    went through hidden_norm); k_norm and RoPE apply to context keys as to
    block keys. fused: [n, H]; returns K, V as bf16 values [n, n_kv, d].
    """
    nkv, d = model["n_kv_heads"], model["head_dim"]
    n = fused.shape[0]
    k = (fused @ layer["k_proj"].T).reshape(n, nkv, d)
    v = (fused @ layer["v_proj"].T).reshape(n, nkv, d)
    k = rope(rms_norm(k, layer["k_norm"], model["rms_eps"]), np.asarray(positions)[:, None], model["rope_theta"])
    return round_bf16(k), round_bf16(v)


def visible_positions(kind, C, W):
    """Context positions a layer attends for a block drafted at length C.

    TensorFold #1851 item 4: a sliding layer attends its own window, the full
    layer the whole served span. Reading: the window is shared by the block
    (positions >= C - W), not per query row.
    """
    if kind == SLIDING:
        return np.arange(max(0, C - W), C)
    return np.arange(0, C)


def block_attention(q, k, v):
    """Non-causal attention of the block rows over context-plus-block keys.

    q: [16, n_q, d]; k, v: [n, n_kv, d] (context rows then the block's rows).
    Query head h reads kv head h // (n_q / n_kv). Scores use the explicit
    matrix Q K^T / sqrt(d) and a float64 softmax over every key (no mask: the
    pages refuse a causal draft, TensorFold #1851 item 1).
    """
    nq, d = q.shape[1], q.shape[2]
    nkv = k.shape[1]
    grp = nq // nkv
    out = np.empty((q.shape[0], nq, d), dtype=_F)
    for h in range(nq):
        kk = k[:, h // grp, :]
        vv = v[:, h // grp, :]
        s = q[:, h, :] @ kk.T / math.sqrt(d)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vv
    return out


def block_embed(model, w, anchor):
    """Residual rows of the block: the anchor token then fifteen mask tokens
    (TensorFold #1851 item 1: the fifteen mask rows), float64 copies of the
    shared embedding rows."""
    tokens = [int(anchor)] + [model["mask_token"]] * (BLOCK - 1)
    return w["embed"][tokens].astype(_F)


def attention_half(model, w, l, X, ctx_k, ctx_v, C):
    """First half of drafter layer l: input RMSNorm, Q/K/V with per-head
    norms and RoPE, non-causal attention over the layer's visible context
    plus the block, O projection added to the residual (TensorFold #1851
    item 1: each layer adds attention to the residual).

    ctx_k, ctx_v: [C, n_kv, d] bf16 K/V of this layer for positions 0..C-1.
    """
    nq, nkv, d = model["n_q_heads"], model["n_kv_heads"], model["head_dim"]
    eps, theta = model["rms_eps"], model["rope_theta"]
    lw = w["layers"][l]
    pos = C + np.arange(BLOCK)
    h = round_bf16(rms_norm(X, lw["input_layernorm"], eps))
    q = (h @ lw["q_proj"].T).reshape(BLOCK, nq, d)
    k = (h @ lw["k_proj"].T).reshape(BLOCK, nkv, d)
    v = (h @ lw["v_proj"].T).reshape(BLOCK, nkv, d)
    q = round_bf16(rope(rms_norm(q, lw["q_norm"], eps), pos[:, None], theta))
    k = round_bf16(rope(rms_norm(k, lw["k_norm"], eps), pos[:, None], theta))
    v = round_bf16(v)
    vis = visible_positions(model["layer_kinds"][l], C, model["sliding_window"])
    keys = np.concatenate([ctx_k[vis], k], axis=0)
    vals = np.concatenate([ctx_v[vis], v], axis=0)
    att = round_bf16(block_attention(q, keys, vals).reshape(BLOCK, nq * d))
    return X + att @ lw["o_proj"].T


def mlp_half(model, w, l, X):
    """Second half of drafter layer l: post-attention RMSNorm, SwiGLU MLP
    added to the residual (TensorFold #1851 item 1: each layer adds its MLP
    to the residual)."""
    lw = w["layers"][l]
    h2 = round_bf16(rms_norm(X, lw["post_attention_layernorm"], model["rms_eps"]))
    gate = h2 @ lw["gate_proj"].T
    up = h2 @ lw["up_proj"].T
    mid = round_bf16(silu(gate) * up)
    return X + mid @ lw["down_proj"].T


def draft_layer(model, w, l, X, ctx_k, ctx_v, C):
    """One drafter layer on the block's residual X [16, H] (qwen3 body:
    TensorFold #1851 item 1: two residual adds per layer)."""
    return mlp_half(model, w, l, attention_half(model, w, l, X, ctx_k, ctx_v, C))


def block_conv(model, w, X):
    """DFlash2's two-tap dynamic convolution over the block's rows.

    The explainer's section 五 ("Dynamic short convolution"): candidates
    further down the block are less accurate (suffix decay); DFlash 2 adds a
    two-tap dynamic convolution for the short-range dependencies between
    adjacent positions of the block; the public DFlash2 config gives kernel
    size 2. The pages give no more. Reading: a dynamic convolution in the
    published sense (Wu et al. 2019, "Pay Less Attention with Lightweight
    and Dynamic Convolutions": per-position kernel weights predicted from
    the position's own input by a linear map, normalised by a softmax over
    the kernel's taps, shared by the channels of a group), with kernel size
    2 and causal inside the block, so row i mixes rows i - 1 and i (row 0,
    the anchor, has no row before it). It is a residual branch on the
    normed rows after the last layer, before the final norm, as every
    other branch of the body:
        h = bf16(RMSNorm(X) * conv_norm)
        z_i = h_i . conv_proj^T, [groups, 2] (row 2g + t: tap t of group g)
        a_i = softmax over t of z_i (per group)
        X_i += a_i[g, 0] * h_{i-1} + a_i[g, 1] * h_i   (channel c in group
               c // (H / groups); h_{-1} = 0)
    X: [16, H]; returns the new residual.
    """
    G = model["conv_groups"]
    H = model["hidden"]
    h = round_bf16(rms_norm(X, w["conv_norm"], model["rms_eps"]))
    z = (h @ w["conv_proj"].T).reshape(X.shape[0], G, 2)
    z = z - z.max(axis=2, keepdims=True)
    a = np.exp(z)
    a = a / a.sum(axis=2, keepdims=True)
    prev = np.concatenate([np.zeros((1, H), dtype=h.dtype), h[:-1]], axis=0)
    gs = H // G
    return X + np.repeat(a[:, :, 0], gs, axis=1) * prev + np.repeat(a[:, :, 1], gs, axis=1) * h


def draft_head(model, w, X):
    """Final norm of the 15 mask rows and the shared LM head (the explainer's
    section 三: embedding and LM head are the target's). Returns bf16 logits
    [15, V] as float64."""
    z = round_bf16(rms_norm(X[1:], w["norm"], model["rms_eps"]))
    return round_bf16(z @ w["embed"].T)


def draft_block(model, w, ctx_k, ctx_v, C, anchor, keep_residuals=False):
    """One block forward of the drafter for one stream.

    TensorFold #1851 item 1 (qwen3 body; each layer adds attention and its MLP
    to the residual; the fifteen mask rows; fc / hidden_norm / norm), the
    explainer's section 三 (one forward predicts every masked position; the
    embedding and LM head are the target's, shared and frozen).

    ctx_k[l], ctx_v[l]: [C, n_kv, d] bf16 context K/V of layer l for positions
    0..C-1. anchor: token id at position C. Returns (logits [15, V] bf16 values
    of the mask rows, X final residual [16, H]); with keep_residuals, X is the
    list of residuals at every stage boundary: before layer 0, after layer
    0's attention add, after its MLP add, ..., after the last layer's MLP add
    (2L + 1 entries), then, for a drafter with the two-tap convolution
    (conv_groups > 0), after the convolution (2L + 2 entries).
    """
    X = block_embed(model, w, anchor)
    Xs = [X]
    for l in range(model["n_layers"]):
        X = attention_half(model, w, l, X, ctx_k[l], ctx_v[l], C)
        Xs.append(X)
        X = mlp_half(model, w, l, X)
        Xs.append(X)
    if model.get("conv_groups", 0):
        X = block_conv(model, w, X)
        Xs.append(X)
    logits = draft_head(model, w, X)
    assert logits.shape == (BLOCK - 1, w["embed"].shape[0]) and X.shape == (BLOCK, model["hidden"])
    return logits, (Xs if keep_residuals else X)


class OracleStreams:
    """Per-stream drafter state kept the plain way: every fused row and every
    layer's K/V for every committed position (no ring, no window storage).

    Appending rows is tap fusion followed by KV injection (Strata #3457
    "Approach": each committed window injects its rows' features); truncation
    drops the rejected suffix ("Port the DFlash2 protocol", rollback of every
    rejected cache and hidden-state suffix).
    """

    def __init__(self, model, w, streams):
        self.model = model
        self.w = w
        L = model["n_layers"]
        nkv, d, H = model["n_kv_heads"], model["head_dim"], model["hidden"]
        self.fused = [np.zeros((0, H), dtype=_F) for _ in range(streams)]
        self.k = [[np.zeros((0, nkv, d), dtype=_F) for _ in range(L)] for _ in range(streams)]
        self.v = [[np.zeros((0, nkv, d), dtype=_F) for _ in range(L)] for _ in range(streams)]

    def length(self, s):
        return self.fused[s].shape[0]

    def append(self, s, planes):
        m = self.model
        rows = fuse_taps(planes, self.w["fc"], self.w["hidden_norm"], m["rms_eps"])
        start = self.length(s)
        posn = np.arange(start, start + rows.shape[0])
        self.fused[s] = np.concatenate([self.fused[s], rows], axis=0)
        for l, lw in enumerate(self.w["layers"]):
            k, v = context_kv(rows, posn, lw, m)
            self.k[s][l] = np.concatenate([self.k[s][l], k], axis=0)
            self.v[s][l] = np.concatenate([self.v[s][l], v], axis=0)
        return rows

    def truncate(self, s, new_len):
        self.fused[s] = self.fused[s][:new_len]
        for l in range(self.model["n_layers"]):
            self.k[s][l] = self.k[s][l][:new_len]
            self.v[s][l] = self.v[s][l][:new_len]

    def draft(self, s, anchor, keep_residuals=False):
        return draft_block(self.model, self.w, self.k[s], self.v[s], self.length(s), anchor, keep_residuals)


# ----------------------------------------------------------------------------
# candidates and verification


def topk(row, k):
    """The k largest entries of a logit row, descending, ties to the lower index.

    "Port the DFlash2 protocol": top candidates at each position. Stable
    ordering on (value descending, index ascending).
    """
    row = np.asarray(row, dtype=np.float64)
    order = np.lexsort((np.arange(row.shape[0]), -row))[:k]
    return order.astype(np.int64), row[order]


def argmax_lowest(row):
    """Index of the largest entry; ties go to the lowest index."""
    return int(np.argmax(np.asarray(row, dtype=np.float64)))


def greedy_verify(draft_ids, target_logits):
    """Greedy verification: accept the longest matching prefix, then the bonus.

    The explainer's section 四 (greedy: accept the consecutive prefix that
    matches the target's argmax, then take the target's argmax at the first
    mismatch) and "Port the DFlash2 protocol" (accepted-prefix commit plus
    bonus token).

    draft_ids: the 15 drafted tokens d_1..d_15 (positions C+1..C+15).
    target_logits: [16, V], row i scored by the target after reading the
    anchor and d_1..d_i, i.e. its prediction for position C+i+1.
    Returns (a, tokens): a in [0, 15] accepted drafts; tokens[0..a] =
    d_1..d_a then the bonus t_a = argmax row a; the rest -1.
    """
    t = [argmax_lowest(target_logits[i]) for i in range(BLOCK)]
    a = 0
    while a < BLOCK - 1 and int(draft_ids[a]) == t[a]:
        a += 1
    out = [int(x) for x in draft_ids[:a]] + [t[a]] + [-1] * (BLOCK - 1 - a)
    return a, out


def softmax_t(row, T):
    """softmax(row / T) in float64."""
    z = np.asarray(row, dtype=np.float64) / T
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def draft_confidence(logits, T):
    """The drafter's confidence at each mask row: the top-1 probability of
    softmax(row / T).

    Strata pull request #3457, "Problem and result": `--spec-min-p` stops a
    draft where the confidence falls below it. Reading (the v1 body has no
    selector): a position's confidence is the largest entry of the drafter's
    softmax at that position. logits: [rows, V]; returns float64 [rows].
    """
    return np.asarray([softmax_t(r, T).max() for r in np.asarray(logits, dtype=np.float64)])


def draft_stop(conf, min_p):
    """Drafted tokens to send to verification, per stream: the number of
    leading positions whose confidence is at least min_p (the draft stops at
    the first position below it; Strata #3457, "Problem and result").

    conf: [S, 15]; returns int64 [S] in [0, 15].
    """
    conf = np.asarray(conf, dtype=np.float64).reshape(-1, BLOCK - 1)
    out = []
    for row in conf:
        n = 0
        while n < BLOCK - 1 and row[n] >= min_p:
            n += 1
        out.append(n)
    return np.asarray(out, dtype=np.int64)


# ----------------------------------------------------------------------------
# DFlash2 candidate-path selector


def selector_edges(cand_ids, U, W):
    """Edge scores of adjacent candidate pairs.

    The explainer's section 五 ("Candidate path selector"): DFlash 2 keeps
    the top-k candidates at every position and a light selector scores
    adjacent candidate pairs; the public DFlash2 config gives
    selector_top_k 16 and selector_rank 256. TensorFold #1851 item 1: with no
    codebooks (rank 0) the selector's edge term is zero. Reading: the pair
    score is a rank-r bilinear form of per-token codebooks U, W [V, r]:
    edge(i, a, b) = sum_j U[c(i, a), j] * W[c(i+1, b), j], where c(i, a) is
    candidate a of position i. An id outside [0, V) is not a candidate: its
    codebook rows count as zero.

    cand_ids: [P, k] ints; U, W: [V, r]. Returns float64 [P-1, k, k].
    """
    ids = np.asarray(cand_ids, dtype=np.int64)
    U = np.asarray(U, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    V = U.shape[0]
    valid = (ids >= 0) & (ids < V)
    safe = np.where(valid, ids, 0)
    Uc = U[safe] * valid[..., None]
    Wc = W[safe] * valid[..., None]
    return np.einsum("iar,ibr->iab", Uc[:-1], Wc[1:])


def path_score(ranks, cand_ids, cand_vals, U, W):
    """Score of one path (candidate index a_i at every position i): the node
    scores of its candidates plus the edge scores of its adjacent pairs."""
    vals = np.asarray(cand_vals, dtype=np.float64)
    ids = np.asarray(cand_ids, dtype=np.int64)
    V = np.asarray(U).shape[0]
    if any(not (0 <= ids[i, a] < V) for i, a in enumerate(ranks)):
        return -np.inf
    e = selector_edges(cand_ids, U, W)
    return float(sum(vals[i, a] for i, a in enumerate(ranks)) + sum(e[i, ranks[i], ranks[i + 1]] for i in range(len(ranks) - 1)))


def select_path(cand_ids, cand_vals, U, W):
    """The selector's choice: the one consistent path of highest score.

    The explainer's section 五: score adjacent candidate pairs, then choose a
    consistent path; "Port the DFlash2 protocol" ("What is portable"): top
    candidates at each position, then coherent candidate-path selection,
    then target verification. Reading: a path's score is the sum of its
    candidates' node scores (the drafter's logits; a position's
    log-probabilities differ from its logits by one constant, which moves
    every path's score alike) and of the edge scores of its adjacent pairs
    (selector_edges); the best path is found by the max-sum recursion over
    positions (Viterbi), ties going to the lower candidate index at every
    step. With rank 0 every edge is zero and the path is each position's
    highest candidate.

    cand_ids: [P, k] ints (candidate a of position i); cand_vals: [P, k]
    node scores; U, W: [V, r]. Returns (ranks [P], ids [P], score, margin):
    margin = score minus the best score of any path that differs from the
    chosen one (how far the choice is from flipping); ranks and ids are -1
    and score -inf when some position has no valid candidate.
    """
    ids = np.asarray(cand_ids, dtype=np.int64)
    vals = np.asarray(cand_vals, dtype=np.float64)
    P, k = ids.shape
    V = np.asarray(U).shape[0]
    node = np.where((ids >= 0) & (ids < V), vals, -np.inf)
    edge = selector_edges(ids, U, W)
    # forward: F[i][b] = best score of a path over positions 0..i ending in b
    F = np.empty((P, k))
    back = np.zeros((P, k), dtype=np.int64)
    F[0] = node[0]
    for i in range(1, P):
        for b in range(k):
            best, arg = -np.inf, 0
            for a in range(k):
                v = F[i - 1][a] + edge[i - 1][a][b]
                if v > best:
                    best, arg = v, a
            F[i][b] = node[i][b] + best
            back[i][b] = arg
    last, score = 0, -np.inf
    for b in range(k):
        if F[P - 1][b] > score:
            last, score = b, F[P - 1][b]
    if score == -np.inf:
        return [-1] * P, [-1] * P, -np.inf, 0.0
    ranks = [0] * P
    ranks[P - 1] = last
    for i in range(P - 1, 0, -1):
        ranks[i - 1] = int(back[i][ranks[i]])
    # backward: G[i][a] = best score of positions i+1..P-1 after a at i
    G = np.zeros((P, k))
    for i in range(P - 2, -1, -1):
        for a in range(k):
            G[i][a] = max(edge[i][a][b] + node[i + 1][b] + G[i + 1][b] for b in range(k))
    runner = -np.inf
    for i in range(P):
        for a in range(k):
            if a != ranks[i]:
                runner = max(runner, F[i][a] + G[i][a])
    return ranks, [int(ids[i][ranks[i]]) for i in range(P)], float(score), float(score - runner)


# ----------------------------------------------------------------------------
# tree drafting and tree verification


def tree_nodes(anchor, topk_ids, widths):
    """A stream's draft tree from each depth's marginals.

    TensorFold #1851: streams draft per-stream trees in the shared rounds,
    and with no codebooks (rank 0) the trees come from each depth's
    marginals (item 1). Reading: the root is the anchor (position C); every
    node at depth j - 1 has as children the top-b_j candidates of mask row j
    (the drafter's marginal for position C + j, one forward predicts every
    depth, so every parent gets the same candidates), in candidate order.
    Nodes are numbered breadth first, children of earlier nodes first.

    topk_ids: [15, k] the draft's per-row top candidates (row j - 1 is depth
    j); widths: b_1..b_D with 1 <= b_j <= k. Returns (tokens, parents,
    depths) lists, node 0 the root (parent -1, depth 0).
    """
    tokens, parents, depths = [int(anchor)], [-1], [0]
    level = [0]
    for j, b in enumerate(widths, start=1):
        nxt = []
        for p in level:
            for r in range(int(b)):
                tokens.append(int(topk_ids[j - 1][r]))
                parents.append(p)
                depths.append(j)
                nxt.append(len(tokens) - 1)
        level = nxt
    return tokens, parents, depths


def tree_mask(parents):
    """Ancestor-or-self relation of the tree's nodes, the attention mask a
    target applies when it scores the whole tree in one pass: mask[n][m] is
    True iff m lies on the path from the root to n."""
    N = len(parents)
    mask = np.zeros((N, N), dtype=bool)
    for n in range(N):
        m = n
        while m >= 0:
            mask[n][m] = True
            m = parents[m]
    return mask


def tree_greedy_verify(tokens, parents, target_logits):
    """Greedy verification of a draft tree.

    The explainer's section 四 (greedy: accept the drafted tokens that match
    the target's argmax, take the target's argmax at the first mismatch),
    applied along the tree: target_logits[n] is the target's prediction for
    the position after node n, having read the path from the root to n.
    From the root, step to the child whose token is the target's argmax at
    the current node (ties to the lowest id) while one exists; the accepted
    tokens are the path's, the bonus is the argmax at the last node reached
    ("Port the DFlash2 protocol": accepted prefix plus bonus).

    Returns (a, tokens16, node): a accepted drafts, the 16 committed-token
    slots (the a path tokens, the bonus, then -1), and the last node reached.
    """
    children = [[] for _ in tokens]
    for n, p in enumerate(parents):
        if p >= 0:
            children[p].append(n)
    cur, path = 0, []
    while True:
        t = argmax_lowest(target_logits[cur])
        nxt = [c for c in children[cur] if tokens[c] == t]
        if not nxt:
            break
        cur = nxt[0]
        path.append(tokens[cur])
    a = len(path)
    return a, path + [t] + [-1] * (BLOCK - 1 - a), cur


def inverse_cdf(wts, u):
    """Draw from unnormalised weights by inverse CDF.

    Returns (j, margin): j is the smallest index whose running sum (ascending
    index order) exceeds u * total; margin is the distance from u * total to
    the nearest running-sum boundary, relative to the total (how far the draw
    is from flipping to a neighbour).
    """
    wts = np.asarray(wts, dtype=np.float64)
    c = np.cumsum(wts)
    tot = c[-1]
    thr = u * tot
    j = int(np.searchsorted(c, thr, side="right"))
    if j >= wts.shape[0]:
        j = int(np.nonzero(wts > 0)[0][-1])
    lo = c[j - 1] if j > 0 else 0.0
    margin = min(abs(thr - lo), abs(c[j] - thr)) / tot if tot > 0 else 0.0
    return j, margin


def sample_rows(logits, T, uniforms):
    """One inverse-CDF draw from softmax(row / T) per row (draft-side sampling).

    Returns (ids, margins). Reading: the same inverse-CDF rule as the
    verifier's draws.
    """
    ids, margins = [], []
    for r in range(logits.shape[0]):
        j, m = inverse_cdf(softmax_t(logits[r], T), float(uniforms[r]))
        ids.append(j)
        margins.append(m)
    return np.asarray(ids, dtype=np.int64), np.asarray(margins)


def sampling_verify(draft_ids, target_logits, draft_logits, uniforms, T):
    """Speculative-sampling verification with residual correction.

    The explainer's section 四 (sampling: acceptance from the target and draft
    probabilities; on rejection draw from the residual max(p_target -
    p_draft, 0), renormalised; only then is the target's distribution kept).
    Acceptance is min(1, p/q), taken as u * q(x) < p(x).

    draft_ids [15]: d_1..d_15; target_logits [16, V]: p_i = softmax(row i / T)
    is the target's distribution for position C+i+1; draft_logits [15, V]:
    q_{i+1} = softmax(row i / T) is the drafter's distribution for the same
    position. uniforms [16, 2]: [i][0] for the test at i, [i][1] for the
    residual or bonus draw at i.
    Returns (a, tokens, margins): margins holds, for every decision taken,
    how far it was from flipping (relative), for near-tie reporting.
    """
    margins = []
    for i in range(BLOCK - 1):
        p = softmax_t(target_logits[i], T)
        q = softmax_t(draft_logits[i], T)
        x = int(draft_ids[i])
        lhs = float(uniforms[i][0]) * q[x]
        margins.append(abs(lhs - p[x]) / max(p[x], q[x], 1e-300))
        if lhs < p[x]:
            continue
        r = np.maximum(p - q, 0.0)
        if r.sum() <= 0.0:
            r = p
        j, m = inverse_cdf(r, float(uniforms[i][1]))
        margins.append(m)
        return i, [int(v) for v in draft_ids[:i]] + [j] + [-1] * (BLOCK - 1 - i), margins
    p = softmax_t(target_logits[BLOCK - 1], T)
    j, m = inverse_cdf(p, float(uniforms[BLOCK - 1][1]))
    margins.append(m)
    return BLOCK - 1, [int(v) for v in draft_ids] + [j], margins


# ----------------------------------------------------------------------------
# sizes, inventory and configuration rules


def fused_row_bytes(H):
    """One fused ring row: H bf16 values (8 KiB a token at hidden 4096)."""
    return H * 2


def raw_plane_bytes(N, H):
    """A token's raw tap planes: N planes of H bf16 values."""
    return N * H * 2


def tap_row_bytes(variant, N, H):
    """Prompt-memory price of a prompt row's taps (TensorFold #1851 item 3).

    A fusing (v1) drafter holds its N planes, the row-major copy of them,
    fc's output row and the fused row: (2N + 2) * H bf16 values, which is
    18 x hidden x 2 bytes for eight taps. A DFlash2 drafter keeps the raw
    planes only: N * H * 2.
    """
    if variant == 1:
        return (2 * N + 2) * H * 2
    return N * H * 2


def drafter_tensor_count(L):
    """Eleven tensors a layer plus fc, hidden_norm and norm (69 for six layers)."""
    return 11 * L + 3


def kind_name(variant):
    """A v1 (fusing, qwen3 body) drafter is named DFlash; the other DFlash2."""
    return "DFlash" if variant == 1 else "DFlash2"


def validate_config(model):
    """Refusals the pages name (TensorFold #1851 item 1): taps past the target
    or repeated, a causal draft; plus the shape rules this drafter needs.
    Returns None when accepted, else a short reason string."""
    N = model["n_taps"]
    taps = list(model["tap_layers"])[:N]
    if not (1 <= N <= 8):
        return "taps"
    if any(t < 0 or t >= model["target_layers"] for t in taps):
        return "taps past the target"
    if len(set(taps)) != len(taps):
        return "taps repeated"
    if model["causal"]:
        return "causal"
    if model["block"] != BLOCK:
        return "block"
    if model["n_q_heads"] % model["n_kv_heads"]:
        return "gqa"
    if model["hidden"] != model["n_q_heads"] * model["head_dim"]:
        return "hidden"
    for l in range(model["n_layers"]):
        if model["layer_kinds"][l] == SLIDING and model["sliding_window"] <= 0:
            return "window"
    G = model.get("conv_groups", 0)
    if G:
        # the v1 layout has no conv tensor (TensorFold #1851 item 1)
        if model["variant"] == 1:
            return "conv in a v1 drafter"
        if G < 0 or G > 32 or model["hidden"] % G or (model["hidden"] // G) % 16:
            return "conv groups"
    return None
