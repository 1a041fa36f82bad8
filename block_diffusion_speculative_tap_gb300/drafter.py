"""Thin object wrappers over the C ABI (marshalling only).

Device buffers are torch tensors; their data pointers and the current CUDA
stream are passed straight to libdflash. Workspaces are torch allocations
owned by the wrappers and reused across calls (so a CUDA graph captured over
a call stays valid).
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _abi as A
from ._abi import check, lib

__all__ = [
    "Drafter",
    "State",
    "config_validate",
    "kind",
    "tap_row_bytes",
    "fused_row_bytes",
    "topk",
    "verify_greedy",
    "verify_sample",
    "select_path",
    "tree_size",
    "tree_build",
    "tree_verify",
    "launch_count",
]


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else C.c_void_p(0)


def _need(t, dtype, what):
    if t.device.type != "cuda" or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{what}: expected a contiguous {dtype} CUDA tensor")


def config_validate(model: dict) -> int:
    """dflash_config_validate: 0 or a negative refusal code."""
    c = A.make_config(model)
    return lib.dflash_config_validate(C.byref(c))


def kind(model: dict) -> str:
    c = A.make_config(model)
    return lib.dflash_kind(C.byref(c)).decode()


def tap_row_bytes(model: dict) -> int:
    c = A.make_config(model)
    return lib.dflash_tap_row_bytes(C.byref(c))


def fused_row_bytes(model: dict) -> int:
    c = A.make_config(model)
    return lib.dflash_fused_row_bytes(C.byref(c))


def launch_count() -> int:
    return lib.dflash_launch_count()


class _Workspace:
    def __init__(self, device):
        self.device = device
        self.buf = None

    def get(self, nbytes):
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf


class Drafter:
    """A drafter handle (dflash_create) over bf16 weights on the GPU.

    weights: dict as produced by synthetic_inputs.make_weights (fc,
    hidden_norm, norm, embed, layers[l][name]); tensors must stay alive.
    """

    def __init__(self, model: dict, weights: dict):
        self.model = dict(model)
        self.cfg = A.make_config(model)
        self.weights = weights
        dev = weights["fc"].device
        if dev.type != "cuda":
            raise ValueError("weights must be CUDA tensors")
        self.device = dev
        for name in ("fc", "hidden_norm", "norm", "embed"):
            _need(weights[name], torch.bfloat16, name)
        L = model["n_layers"]
        self._layers = (A.LayerWeights * L)()
        keys = {
            "input_norm": "input_layernorm",
            "q_proj": "q_proj",
            "k_proj": "k_proj",
            "v_proj": "v_proj",
            "o_proj": "o_proj",
            "q_norm": "q_norm",
            "k_norm": "k_norm",
            "post_norm": "post_attention_layernorm",
            "gate_proj": "gate_proj",
            "up_proj": "up_proj",
            "down_proj": "down_proj",
        }
        for l in range(L):
            lw = weights["layers"][l]
            for field, key in keys.items():
                _need(lw[key], torch.bfloat16, f"layers[{l}].{key}")
                setattr(self._layers[l], field, lw[key].data_ptr())
        conv = (None, None)
        if model.get("conv_groups", 0):
            for name in ("conv_norm", "conv_proj"):
                _need(weights[name], torch.bfloat16, name)
            conv = (weights["conv_norm"].data_ptr(), weights["conv_proj"].data_ptr())
        self._w = A.Weights(
            weights["fc"].data_ptr(),
            weights["hidden_norm"].data_ptr(),
            weights["norm"].data_ptr(),
            weights["embed"].data_ptr(),
            C.cast(self._layers, C.POINTER(A.LayerWeights)),
            conv[0],
            conv[1],
        )
        h = C.c_void_p()
        with torch.cuda.device(dev):
            check(lib.dflash_create(C.byref(self.cfg), C.byref(self._w), C.byref(h)), "dflash_create")
        self.handle = h

    def close(self):
        if self.handle:
            lib.dflash_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def new_state(self, streams: int, ring: int) -> "State":
        return State(self, streams, ring)


class State:
    """Per-stream drafter state in a torch-allocated device buffer."""

    def __init__(self, drafter: Drafter, streams: int, ring: int):
        self.drafter = drafter
        self.streams = streams
        self.ring = ring
        nbytes = C.c_size_t()
        check(lib.dflash_state_bytes(drafter.handle, streams, ring, C.byref(nbytes)), "dflash_state_bytes")
        self.mem = torch.empty(nbytes.value, dtype=torch.uint8, device=drafter.device)
        st = C.c_void_p()
        check(
            lib.dflash_state_init(
                drafter.handle, _ptr(self.mem), nbytes.value, streams, ring, _stream(), C.byref(st)
            ),
            "dflash_state_init",
        )
        self.st = st
        self.ws_fuse = _Workspace(drafter.device)
        self.ws_draft = _Workspace(drafter.device)
        # argument marshalling kept between calls: workspace sizes by shape,
        # and the pointer array of the last validated list of tap planes
        self._ws_bytes = {}
        self._planes = None
        self._planes_arr = None

    def __del__(self):
        try:
            if self.st:
                lib.dflash_state_free(self.st)
                self.st = None
        except Exception:
            pass

    # ------------------------------------------------------------ queries
    def length(self, s: int) -> int:
        v = C.c_int64()
        check(lib.dflash_state_length(self.st, s, C.byref(v)), "dflash_state_length")
        return v.value

    def wait_probe(self, cycles: int):
        """Run the bounded-wait self-test (a wait nothing completes, given up
        after `cycles` SM cycles); read the outcome with status()."""
        check(lib.dflash_state_wait_probe(self.st, int(cycles), _stream()), "dflash_state_wait_probe")

    def status(self):
        """(rc, bits) of the device status word (synchronises the stream)."""
        v = C.c_int32()
        rc = lib.dflash_device_status(self.st, _stream(), C.byref(v))
        return rc, v.value

    # ------------------------------------------------------------ views
    def _view(self, ptr, shape, dtype):
        n = 1
        for x in shape:
            n *= x
        esz = torch.empty((), dtype=dtype).element_size()
        off = ptr - self.mem.data_ptr()
        assert 0 <= off and off + n * esz <= self.mem.numel()
        return self.mem[off : off + n * esz].view(dtype).view(*shape)

    def ring_view(self):
        """bf16 [streams, ring, H] view of the fused ring (shares memory)."""
        p = C.c_void_p()
        check(lib.dflash_state_ring(self.st, C.byref(p)), "dflash_state_ring")
        return self._view(p.value, (self.streams, self.ring, self.drafter.model["hidden"]), torch.bfloat16)

    def cache_view(self, layer):
        """(K, V) bf16 [streams, n_kv, cap, d] views of a layer's cache, and cap."""
        m = self.drafter.model
        k, v, cap = C.c_void_p(), C.c_void_p(), C.c_int()
        check(lib.dflash_state_cache(self.st, layer, C.byref(k), C.byref(v), C.byref(cap)), "dflash_state_cache")
        shape = (self.streams, m["n_kv_heads"], cap.value, m["head_dim"])
        return self._view(k.value, shape, torch.bfloat16), self._view(v.value, shape, torch.bfloat16), cap.value

    # ------------------------------------------------------------ calls
    def fuse_taps(self, planes, segments, inject=True):
        """planes: N bf16 CUDA tensors [rows, H] (same row stride);
        segments: list of (stream, start, rows)."""
        m = self.drafter.model
        cached = self._planes
        if (
            cached is not None
            and len(planes) == len(cached[0])
            and all(p is q for p, q in zip(planes, cached[0]))
            and [p.data_ptr() for p in planes] == cached[1]
        ):
            # the same tensors as the last call (a capture buffer reused every round)
            arr, stride = self._planes_arr
        else:
            if len(planes) != m["n_taps"]:
                raise ValueError("one plane per tap")
            stride = planes[0].stride(0)
            for p in planes:
                if p.dtype != torch.bfloat16 or p.device.type != "cuda" or p.stride(1) != 1 or p.stride(0) != stride:
                    raise ValueError("planes: bf16 CUDA [rows, H] with a common row stride")
            arr = (C.c_void_p * len(planes))(*[p.data_ptr() for p in planes])
            self._planes = (list(planes), [p.data_ptr() for p in planes])
            self._planes_arr = (arr, stride)
        rows = sum(r for _, _, r in segments)
        key = ("fuse", rows)
        nbytes = self._ws_bytes.get(key)
        if nbytes is None:
            nb = C.c_size_t()
            check(lib.dflash_fuse_workspace_bytes(self.drafter.handle, rows, C.byref(nb)), "fuse_workspace_bytes")
            nbytes = self._ws_bytes[key] = nb.value
        ws = self.ws_fuse.get(nbytes)
        n = len(segments)
        ss = (C.c_int32 * n)(*[s for s, _, _ in segments])
        st = (C.c_int64 * n)(*[b for _, b, _ in segments])
        rr = (C.c_int32 * n)(*[r for _, _, r in segments])
        flags = A.FUSE_INJECT_KV if inject else 0
        check(
            lib.dflash_fuse_taps(
                self.drafter.handle, self.st, arr, stride, n, ss, st, rr, flags, _ptr(ws), ws.numel(), _stream()
            ),
            "dflash_fuse_taps",
        )

    def truncate(self, s: int, new_len: int):
        W = max(1, self.drafter.model.get("sliding_window", 1))
        nb = C.c_size_t()
        check(lib.dflash_fuse_workspace_bytes(self.drafter.handle, min(W, self.ring), C.byref(nb)), "ws")
        ws = self.ws_fuse.get(nb.value)
        check(
            lib.dflash_state_truncate(self.drafter.handle, self.st, s, new_len, _ptr(ws), ws.numel(), _stream()),
            "dflash_state_truncate",
        )

    def draft_workspace_bytes(self, s_count, need_logits):
        nb = C.c_size_t()
        check(
            lib.dflash_draft_workspace_bytes(self.drafter.handle, self.st, s_count, int(need_logits), C.byref(nb)),
            "draft_workspace_bytes",
        )
        return nb.value

    def draft(self, anchors, s_begin=0, k=8, logits=None, want_logits=True, ids=None, vals=None):
        """One block forward for streams [s_begin, s_begin + len(anchors)).

        Returns (logits [S*15, V] bf16 or None, ids [S*15, k] int32, vals fp32)."""
        m = self.drafter.model
        _need(anchors, torch.int32, "anchors")
        S = anchors.numel()
        dev = self.drafter.device
        if logits is None and want_logits:
            logits = torch.empty(S * 15, m["vocab"], dtype=torch.bfloat16, device=dev)
        if k > 0:
            if ids is None:
                ids = torch.empty(S * 15, k, dtype=torch.int32, device=dev)
            if vals is None:
                vals = torch.empty(S * 15, k, dtype=torch.float32, device=dev)
        key = ("draft", S, logits is None)
        nbytes = self._ws_bytes.get(key)
        if nbytes is None:
            nbytes = self._ws_bytes[key] = self.draft_workspace_bytes(S, logits is None)
        ws = self.ws_draft.get(nbytes)
        check(
            lib.dflash_draft_block(
                self.drafter.handle,
                self.st,
                s_begin,
                S,
                _ptr(anchors),
                _ptr(logits),
                _ptr(ids) if k > 0 else C.c_void_p(0),
                _ptr(vals) if k > 0 else C.c_void_p(0),
                k,
                _ptr(ws),
                ws.numel(),
                _stream(),
            ),
            "dflash_draft_block",
        )
        return logits, ids, vals


    def draft_stages(self, X, g0, g1, s_begin=0):
        """Run stages [g0, g1) on the fp32 residual X [S*16, H] in place;
        stage 2l = layer l's attention half, 2l+1 = its MLP half."""
        _need(X, torch.float32, "X")
        S = X.shape[0] // 16
        ws = self.ws_draft.get(self.draft_workspace_bytes(S, False))
        check(
            lib.dflash_draft_stages(
                self.drafter.handle, self.st, s_begin, S, g0, g1, _ptr(X), _ptr(ws), ws.numel(), _stream()
            ),
            "dflash_draft_stages",
        )
        return X

    def draft_conv(self, X):
        """DFlash2's two-tap dynamic convolution on the fp32 residual X
        [S*16, H] in place (a drafter with conv_groups > 0)."""
        _need(X, torch.float32, "X")
        S = X.shape[0] // 16
        ws = self.ws_draft.get(self.draft_workspace_bytes(S, False))
        check(
            lib.dflash_draft_conv(self.drafter.handle, self.st, S, _ptr(X), _ptr(ws), ws.numel(), _stream()),
            "dflash_draft_conv",
        )
        return X

    def draft_head(self, X, k=8):
        """Final norm + LM head (+ top-k) of the fp32 residual X [S*16, H]."""
        _need(X, torch.float32, "X")
        S = X.shape[0] // 16
        dev = self.drafter.device
        logits = torch.empty(S * 15, self.drafter.model["vocab"], dtype=torch.bfloat16, device=dev)
        ids = torch.empty(S * 15, k, dtype=torch.int32, device=dev) if k > 0 else None
        vals = torch.empty(S * 15, k, dtype=torch.float32, device=dev) if k > 0 else None
        ws = self.ws_draft.get(self.draft_workspace_bytes(S, False))
        check(
            lib.dflash_draft_head(
                self.drafter.handle, self.st, S, _ptr(X), _ptr(logits), _ptr(ids), _ptr(vals), k, _ptr(ws),
                ws.numel(), _stream(),
            ),
            "dflash_draft_head",
        )
        return logits, ids, vals


# ---------------------------------------------------------------- free functions


def topk(logits, k, temperature=1.0, uniforms=None, ids=None, vals=None, sampled=None):
    """dflash_topk on a bf16 [rows, V] CUDA tensor. Returns (ids, vals, sampled)."""
    _need(logits, torch.bfloat16, "logits")
    rows, V = logits.shape
    dev = logits.device
    if k > 0:
        ids = ids if ids is not None else torch.empty(rows, k, dtype=torch.int32, device=dev)
        vals = vals if vals is not None else torch.empty(rows, k, dtype=torch.float32, device=dev)
    if uniforms is not None:
        _need(uniforms, torch.float32, "uniforms")
        sampled = sampled if sampled is not None else torch.empty(rows, dtype=torch.int32, device=dev)
    check(
        lib.dflash_topk(
            _ptr(logits),
            rows,
            V,
            k,
            float(temperature),
            _ptr(uniforms),
            _ptr(ids) if k > 0 else C.c_void_p(0),
            _ptr(vals) if k > 0 else C.c_void_p(0),
            _ptr(sampled),
            _stream(),
        ),
        "dflash_topk",
    )
    return ids, vals, sampled


def draft_stop(logits, min_p, temperature=1.0, conf=None, lens=None):
    """dflash_draft_stop on bf16 draft logits [S*15, V]: the per-row
    confidence (top-1 softmax probability) and, per stream, the number of
    leading drafted tokens whose confidence is at least min_p.
    Returns (conf fp32 [S*15], lens int32 [S])."""
    _need(logits, torch.bfloat16, "logits")
    rows, V = logits.shape
    if rows % 15:
        raise ValueError("logits: 15 rows a stream")
    S = rows // 15
    dev = logits.device
    conf = conf if conf is not None else torch.empty(rows, dtype=torch.float32, device=dev)
    lens = lens if lens is not None else torch.empty(S, dtype=torch.int32, device=dev)
    check(
        lib.dflash_draft_stop(_ptr(logits), S, V, float(temperature), float(min_p), _ptr(conf), _ptr(lens), _stream()),
        "dflash_draft_stop",
    )
    return conf, lens


def select_path(cand_ids, cand_vals, U, W, positions=15, path_ids=None, path_ranks=None, path_score=None, ws=None):
    """dflash_select_path: the DFlash2 selector's path through per-position
    candidates. cand_ids int32 / cand_vals fp32: [S * positions, k] (the
    top-k outputs of a draft) or [S, positions, k]; U, W: bf16 [V, rank]
    codebooks. Returns (path_ids [S, positions], path_ranks [S, positions],
    path_score [S])."""
    _need(cand_ids, torch.int32, "cand_ids")
    _need(cand_vals, torch.float32, "cand_vals")
    _need(U, torch.bfloat16, "U")
    _need(W, torch.bfloat16, "W")
    if U.shape != W.shape or U.dim() != 2:
        raise ValueError("U, W: bf16 [V, rank] of one shape")
    k = cand_ids.shape[-1]
    if cand_vals.shape != cand_ids.shape or cand_ids.numel() % (positions * k):
        raise ValueError("cand_ids / cand_vals: [S * positions, k] of one shape")
    S = cand_ids.numel() // (positions * k)
    V, rank = U.shape
    dev = cand_ids.device
    path_ids = path_ids if path_ids is not None else torch.empty(S, positions, dtype=torch.int32, device=dev)
    path_ranks = path_ranks if path_ranks is not None else torch.empty(S, positions, dtype=torch.int32, device=dev)
    path_score = path_score if path_score is not None else torch.empty(S, dtype=torch.float32, device=dev)
    nb = C.c_size_t()
    check(lib.dflash_select_path_workspace_bytes(S, positions, k, C.byref(nb)), "select_path_workspace_bytes")
    if ws is None:
        ws = torch.empty(max(nb.value, 256), dtype=torch.uint8, device=dev)
    check(
        lib.dflash_select_path(
            S, positions, k, V, rank, _ptr(cand_ids), _ptr(cand_vals), _ptr(U), _ptr(W), _ptr(path_ids),
            _ptr(path_ranks), _ptr(path_score), _ptr(ws), ws.numel(), _stream(),
        ),
        "dflash_select_path",
    )
    return path_ids, path_ranks, path_score


def _widths(widths):
    w = (C.c_int32 * len(widths))(*[int(x) for x in widths])
    return w, len(widths)


def tree_size(widths, k=16):
    """dflash_tree_size: nodes of a draft tree of these per-depth widths."""
    w, depth = _widths(widths)
    n = C.c_int()
    check(lib.dflash_tree_size(depth, w, k, C.byref(n)), "dflash_tree_size")
    return n.value


def tree_build(anchors, topk_ids, widths, want_mask=True):
    """dflash_tree_build: per-stream draft trees from a draft's top-k ids
    [S * 15, k]. Returns (tokens, parents, depths, mask) with [S, N] int32
    tables and mask uint32 [S, N, ceil(N / 32)] (as int32) or None."""
    _need(anchors, torch.int32, "anchors")
    _need(topk_ids, torch.int32, "topk_ids")
    S = anchors.numel()
    k = topk_ids.shape[-1]
    if topk_ids.numel() != S * 15 * k:
        raise ValueError("topk_ids: [S * 15, k]")
    N = tree_size(widths, k)
    w, depth = _widths(widths)
    dev = anchors.device
    tokens = torch.empty(S, N, dtype=torch.int32, device=dev)
    parents = torch.empty(S, N, dtype=torch.int32, device=dev)
    depths = torch.empty(S, N, dtype=torch.int32, device=dev)
    mask = torch.empty(S, N, (N + 31) // 32, dtype=torch.int32, device=dev) if want_mask else None
    check(
        lib.dflash_tree_build(S, depth, w, k, _ptr(anchors), _ptr(topk_ids), _ptr(tokens), _ptr(parents),
                              _ptr(depths), _ptr(mask), _stream()),
        "dflash_tree_build",
    )
    return tokens, parents, depths, mask


def tree_verify(node_tokens, target_logits, widths, accept=None, tokens=None, node=None, ws=None):
    """dflash_tree_verify: node_tokens [S, N] int32, target_logits [S, N, V]
    bf16 -> (accept [S], tokens [S, 16], last node [S])."""
    _need(node_tokens, torch.int32, "node_tokens")
    _need(target_logits, torch.bfloat16, "target_logits")
    S, N, V = target_logits.shape
    w, depth = _widths(widths)
    dev = target_logits.device
    accept = accept if accept is not None else torch.empty(S, dtype=torch.int32, device=dev)
    tokens = tokens if tokens is not None else torch.empty(S, 16, dtype=torch.int32, device=dev)
    node = node if node is not None else torch.empty(S, dtype=torch.int32, device=dev)
    nb = C.c_size_t()
    check(lib.dflash_tree_verify_workspace_bytes(S, N, C.byref(nb)), "tree_verify_workspace_bytes")
    if ws is None:
        ws = torch.empty(max(nb.value, 256), dtype=torch.uint8, device=dev)
    check(
        lib.dflash_tree_verify(S, depth, w, V, _ptr(node_tokens), _ptr(target_logits), _ptr(accept), _ptr(tokens),
                               _ptr(node), _ptr(ws), ws.numel(), _stream()),
        "dflash_tree_verify",
    )
    return accept, tokens, node


def _draft_ld(draft_ids):
    """Elements between consecutive draft positions: 1 for [S, 15], k for the
    top-1 column of a [S*15, k] top-k tensor."""
    if draft_ids.dtype != torch.int32 or draft_ids.device.type != "cuda" or not draft_ids.is_contiguous():
        raise ValueError("draft_ids: contiguous int32 CUDA tensor")
    if draft_ids.dim() == 2 and draft_ids.shape[1] != 15:
        return draft_ids.shape[1]
    return 1


def verify_greedy(draft_ids, target_logits, accept=None, tokens=None):
    """draft_ids [S, 15] int32 (or a [S*15, k] top-k id tensor: its top-1
    column is read in place); target_logits [S, 16, V] bf16 -> (accept [S],
    tokens [S, 16])."""
    dld = _draft_ld(draft_ids)
    _need(target_logits, torch.bfloat16, "target_logits")
    S, _, V = target_logits.shape
    dev = target_logits.device
    accept = accept if accept is not None else torch.empty(S, dtype=torch.int32, device=dev)
    tokens = tokens if tokens is not None else torch.empty(S, 16, dtype=torch.int32, device=dev)
    check(
        lib.dflash_verify(
            A.VERIFY_GREEDY, S, V, _ptr(draft_ids), dld, _ptr(target_logits), C.c_void_p(0), C.c_void_p(0), 1.0,
            _ptr(accept), _ptr(tokens), C.c_void_p(0), 0, _stream(),
        ),
        "dflash_verify",
    )
    return accept, tokens


def verify_sample(draft_ids, target_logits, draft_logits, uniforms, temperature=1.0, accept=None, tokens=None,
                  ws=None):
    """Speculative sampling verification; uniforms [S, 16, 2] fp32."""
    dld = _draft_ld(draft_ids)
    _need(target_logits, torch.bfloat16, "target_logits")
    _need(draft_logits, torch.bfloat16, "draft_logits")
    _need(uniforms, torch.float32, "uniforms")
    S, _, V = target_logits.shape
    dev = target_logits.device
    accept = accept if accept is not None else torch.empty(S, dtype=torch.int32, device=dev)
    tokens = tokens if tokens is not None else torch.empty(S, 16, dtype=torch.int32, device=dev)
    nb = C.c_size_t()
    check(lib.dflash_verify_workspace_bytes(A.VERIFY_SAMPLE, S, V, C.byref(nb)), "verify_workspace_bytes")
    if ws is None:
        ws = torch.empty(max(nb.value, 256), dtype=torch.uint8, device=dev)
    check(
        lib.dflash_verify(
            A.VERIFY_SAMPLE, S, V, _ptr(draft_ids), dld, _ptr(target_logits), _ptr(draft_logits), _ptr(uniforms),
            float(temperature), _ptr(accept), _ptr(tokens), _ptr(ws), ws.numel(), _stream(),
        ),
        "dflash_verify",
    )
    return accept, tokens
