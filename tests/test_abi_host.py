"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/dflash.h declares, and its host logic (config refusals,
byte prices, names, status strings) agrees with the pages."""
import json
import os
import re

import pytest

import oracle as O
import synthetic_inputs as SI

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def D():
    import block_diffusion_speculative_tap_gb300 as D

    return D


@pytest.fixture(scope="module")
def A():
    from block_diffusion_speculative_tap_gb300 import _abi as A

    return A


def declared_functions():
    with open(os.path.join(ROOT, "include", "dflash.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(A):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(A.lib, n), n
    assert set(names) == set(A.EXPORTED)


def test_refusals_match_the_oracle(D):
    m = SI.presets()["9b"]["model"]
    cases = [
        (dict(m), 0),
        (dict(m, tap_layers=[1, 5, 9, 13, 17, 21, 25, 32]), -2),
        (dict(m, tap_layers=[1, 5, 9, 13, 17, 21, 25, 25]), -3),
        (dict(m, causal=1), -4),
        (dict(m, n_taps=9), -2),
        (dict(m, n_taps=0), -2),
        (dict(m, block=8), -5),
        (dict(m, n_kv_heads=5), -5),
        (dict(m, layer_kinds=[1] * 6, sliding_window=0), -5),
        (dict(m, hidden=4224), -5),  # hidden != q heads x head dim
        (dict(m, conv_groups=16), -5),  # a v1 drafter has no convolution
        (dict(m, variant=2, conv_groups=16), 0),
        (dict(m, variant=2, conv_groups=3), -5),  # 4096 / 3
        (dict(m, variant=2, conv_groups=64), -5),  # more than 32 groups
    ]
    for cfg, code in cases:
        assert D.config_validate(cfg) == code, cfg
        why = O.validate_config(cfg)
        assert (why is None) == (code == 0)
    for name in SI.presets():
        assert D.config_validate(SI.presets()[name]["model"]) == 0


def test_byte_prices_and_names(D):
    with open(os.path.join(ROOT, "tests", "golden", "page_constants.json")) as f:
        c = json.load(f)
    m = SI.presets()["9b"]["model"]
    assert D.fused_row_bytes(m) == c["fused_row_bytes_at_4096"]
    assert D.tap_row_bytes(m) == c["tap_row_bytes_v1_eight_taps_factor"] * m["hidden"] * 2
    d2 = dict(m, variant=2, n_taps=5, tap_layers=[1, 5, 9, 13, 17])
    assert D.tap_row_bytes(d2) == 5 * m["hidden"] * 2
    assert D.kind(m) == c["kind_v1"] and D.kind(d2) == c["kind_dflash2"]
    for name in SI.presets():
        mm = SI.presets()[name]["model"]
        assert D.tap_row_bytes(mm) == O.tap_row_bytes(mm["variant"], mm["n_taps"], mm["hidden"])


def test_status_strings(A):
    for code in range(0, -12, -1):
        assert A.lib.dflash_strerror(code).decode() != "unknown status"
    assert A.lib.dflash_strerror(-99).decode() == "unknown status"


def test_null_arguments_are_refused(A):
    import ctypes as C

    assert A.lib.dflash_config_validate(None) == -1
    assert A.lib.dflash_tap_row_bytes(None) == -1
    assert A.lib.dflash_create(None, None, None) == -1
    assert A.lib.dflash_topk(None, 1, 8, 1, 1.0, None, None, None, None, None) == -1
    nb = C.c_size_t()
    assert A.lib.dflash_verify_workspace_bytes(1, 4, 4096, C.byref(nb)) == 0 and nb.value == 4 * 31 * 2 * 4
    assert A.lib.dflash_verify_workspace_bytes(7, 4, 4096, C.byref(nb)) == -1


def test_sampling_stream_limit_is_refused(A):
    """Sampling verification takes at most DFLASH_MAX_SAMPLE_STREAMS (65535)
    streams a call; more are refused before any device work (the pointers
    here are never dereferenced)."""
    import ctypes as C

    p = C.c_void_p(0x10000)
    args = lambda S: (1, S, 4096, p, 1, p, p, p, C.c_float(1.0), p, p, p, C.c_size_t(1 << 30), None)
    assert A.lib.dflash_verify(*args(65536)) == -1
    assert A.lib.dflash_verify(*args(1 << 20)) == -1


def test_kernel_shape_limits_are_refused(D):
    """Shapes the method allows but the kernels do not serve are refused
    up front (DFLASH_E_SHAPE), never run: query groups over 8 heads a kv head,
    head dims other than 32, 64, 128, widths and vocabularies off the 128-row
    tile, a mask token outside the vocabulary."""
    m = SI.presets()["9b"]["model"]
    for cfg in (
        dict(m, n_kv_heads=2),                            # 16 query heads a kv head
        dict(m, n_q_heads=16, head_dim=256),              # head dim 256
        dict(m, hidden=4096 + 64, n_q_heads=65, head_dim=64, n_kv_heads=13),  # width off the tile
        dict(m, ffn=12288 + 64),
        dict(m, vocab=151936 + 64, mask_token=151999),
        dict(m, mask_token=151936),
    ):
        assert D.config_validate(cfg) == -5, cfg


def test_tree_sizes_match_the_oracle_and_limits_are_refused(A):
    """dflash_tree_size counts the nodes of a tree of widths b_1..b_D as the
    oracle builds it (root plus b_1 * ... * b_j nodes at depth j, breadth
    first); depths outside 1..15, widths outside 1..k, k over
    DFLASH_MAX_TOPK and trees over DFLASH_MAX_TREE_NODES nodes are refused
    (DFLASH_E_INVALID_ARG)."""
    import ctypes as C

    import numpy as np

    def size(widths, k):
        n = C.c_int(-7)
        arr = (C.c_int32 * max(1, len(widths)))(*widths)
        rc = A.lib.dflash_tree_size(len(widths), arr, k, C.byref(n))
        return rc, n.value

    topk = np.arange(15 * 16, dtype=np.int64).reshape(15, 16)
    for widths in ([4, 2, 2, 1, 1, 1, 1], [1] * 15, [16, 8], [3, 3, 3, 3, 3], [2] * 9):
        tokens, parents, depths = O.tree_nodes(7, topk, widths)
        assert size(widths, 16) == (0, len(tokens)), widths
    assert size([4, 2, 2, 1, 1, 1, 1], 16) == (0, 93)  # the bench's tree
    for widths, k in (([], 16), ([1] * 16, 16), ([0, 2], 16), ([5], 4), ([2], 17), ([2], 0),
                      ([16, 16, 16], 16), ([2] * 10, 16)):
        rc, n = size(widths, k)
        assert rc == -1 and n == -7, (widths, k)
    assert A.lib.dflash_tree_size(2, None, 16, C.byref(C.c_int())) == -1
    assert A.lib.dflash_tree_size(2, (C.c_int32 * 2)(1, 1), 16, None) == -1


def test_path_and_tree_workspace_prices(A):
    """Workspace prices of the selector and of tree verification: the
    selector's pair-score table takes streams * (positions - 1) * k^2 fp32
    (nothing for one position), tree verification an arg-max id and value a
    node; shapes outside the documented ranges are refused."""
    import ctypes as C

    nb = C.c_size_t(123)
    assert A.lib.dflash_select_path_workspace_bytes(32, 15, 16, C.byref(nb)) == 0
    assert nb.value == 32 * 14 * 16 * 16 * 4
    assert A.lib.dflash_select_path_workspace_bytes(32, 1, 16, C.byref(nb)) == 0 and nb.value == 0
    for S, P, k in ((-1, 15, 16), (4, 0, 16), (4, 17, 16), (4, 15, 0), (4, 15, 17)):
        assert A.lib.dflash_select_path_workspace_bytes(S, P, k, C.byref(nb)) == -1, (S, P, k)
    assert A.lib.dflash_select_path_workspace_bytes(4, 15, 16, None) == -1
    assert A.lib.dflash_tree_verify_workspace_bytes(32, 93, C.byref(nb)) == 0 and nb.value == 32 * 93 * 8
    for S, N in ((-1, 93), (4, 0), (4, 1025)):
        assert A.lib.dflash_tree_verify_workspace_bytes(S, N, C.byref(nb)) == -1, (S, N)


def test_selector_tree_stop_and_topk_refusals(A):
    """Every refusal the header documents for the candidate-path selector,
    the draft trees, the min-p stop and the top-k scan happens on the host,
    before anything is enqueued (the device pointers below are never
    dereferenced: each call is refused, or has no rows, before any launch)."""
    import ctypes as C

    p = C.c_void_p(0x10000)        # a 16-byte-aligned stand-in, never read
    odd = C.c_void_p(0x10008)      # misaligned
    big = C.c_size_t(1 << 30)
    f = C.c_float
    w3 = (C.c_int32 * 3)(2, 2, 1)
    bad_w = (C.c_int32 * 3)(2, 0, 1)

    # selector: positions, k, vocab, rank (0..512, a multiple of 8), codebooks, workspace
    sel = lambda S, P, k, V, r, U=p, W=p, ws=p, wsb=big: A.lib.dflash_select_path(
        S, P, k, V, r, p, p, U, W, p, None, None, ws, wsb, None)
    assert sel(0, 15, 16, 4096, 256) == 0          # no streams: nothing to do
    for args in ((-1, 15, 16, 4096, 256), (4, 0, 16, 4096, 256), (4, 17, 16, 4096, 256), (4, 15, 0, 4096, 256),
                 (4, 15, 17, 4096, 256), (4, 15, 16, 0, 256), (4, 15, 16, 4096, -8), (4, 15, 16, 4096, 12),
                 (4, 15, 16, 4096, 520)):
        assert sel(*args) == -1, args
    assert sel(4, 15, 16, 4096, 256, U=None) == -1
    assert sel(4, 15, 16, 4096, 256, W=odd) == -1
    assert sel(4, 15, 16, 4096, 256, ws=None) == -7
    assert sel(4, 15, 16, 4096, 256, wsb=C.c_size_t(4 * 14 * 16 * 16 * 4 - 1)) == -7
    assert sel(4, 15, 16, 4096, 256, ws=odd) == -7
    assert A.lib.dflash_select_path(4, 15, 16, 4096, 256, None, p, p, p, p, None, None, p, big, None) == -1

    # trees: shape refusals before the stream count, null outputs, workspace
    assert A.lib.dflash_tree_build(-1, 3, w3, 16, p, p, p, None, None, None, None) == -1
    assert A.lib.dflash_tree_build(4, 3, bad_w, 16, p, p, p, None, None, None, None) == -1
    assert A.lib.dflash_tree_build(4, 0, w3, 16, p, p, p, None, None, None, None) == -1
    assert A.lib.dflash_tree_build(0, 3, w3, 16, p, p, p, None, None, None, None) == 0
    assert A.lib.dflash_tree_build(4, 3, w3, 16, None, p, p, None, None, None, None) == -1
    assert A.lib.dflash_tree_build(4, 3, w3, 16, p, p, None, None, None, None, None) == -1
    tv = lambda S, V, w=w3, logits=p, ws=p, wsb=big: A.lib.dflash_tree_verify(
        S, 3, w, V, p, logits, p, p, None, ws, wsb, None)
    assert tv(0, 4096) == 0
    assert tv(4, 4092) == -1 and tv(4, 4) == -1 and tv(-1, 4096) == -1
    assert tv(4, 4096, w=bad_w) == -1
    assert tv(4, 4096, logits=odd) == -1
    assert tv(4, 4096, ws=None) == -7
    assert tv(4, 4096, wsb=C.c_size_t(4 * 11 * 8 - 1)) == -7   # 11 nodes a stream (1 + 2 + 4 + 4)

    # min-p stop: temperature > 0, 0 <= min_p <= 1, vocab a multiple of 8
    stop = lambda S, V, T, mp, logits=p: A.lib.dflash_draft_stop(logits, S, V, f(T), f(mp), p, p, None)
    assert stop(0, 4096, 1.0, 0.5) == 0
    for args in ((4, 4096, 0.0, 0.5), (4, 4096, -1.0, 0.5), (4, 4096, float("nan"), 0.5), (4, 4096, 1.0, -0.01),
                 (4, 4096, 1.0, 1.01), (4, 4096, 1.0, float("nan")), (4, 4092, 1.0, 0.5), (-1, 4096, 1.0, 0.5)):
        assert stop(*args) == -1, args
    assert stop(4, 4096, 1.0, 0.5, logits=odd) == -1

    # top-k: k in 0..16, vocab a multiple of 8, uniforms and sampled together, T > 0 to sample
    tk = lambda rows, V, k, T=1.0, u=None, smp=None, ids=p, vals=p, logits=p: A.lib.dflash_topk(
        logits, rows, V, k, f(T), u, ids, vals, smp, None)
    assert tk(0, 4096, 8) == 0
    for args in ((4, 4092, 8), (4, 4096, 17), (4, 4096, -1), (-1, 4096, 8)):
        assert tk(*args) == -1, args
    assert tk(4, 4096, 8, ids=None) == -1
    assert tk(4, 4096, 8, u=p) == -1               # uniforms without an output for the draws
    assert tk(4, 4096, 8, smp=p) == -1             # an output for draws without uniforms
    assert tk(4, 4096, 8, T=0.0, u=p, smp=p) == -1
    assert tk(4, 4096, 8, logits=odd) == -1
    assert tk(4, 4096, 0) == 0                     # nothing asked: nothing enqueued
