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
