"""ctypes declarations of include/dflash.h.

Loads the in-tree libdflash.so. There is no fallback: if the library is not
built, importing the binding fails with the reason.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash.so")

MAX_TAPS = 8
MAX_LAYERS = 64
BLOCK = 16
MAX_TOPK = 16

OK = 0
E_INVALID_ARG = -1
E_TAPS_RANGE = -2
E_TAPS_REPEATED = -3
E_CAUSAL = -4
E_SHAPE = -5
E_CAPACITY = -6
E_WORKSPACE = -7
E_CUDA = -8
E_TIMEOUT = -9
E_DEVICE_FAULT = -10
E_UNSUPPORTED = -11

STATUS_BAD_TOKEN = 1
STATUS_TIMEOUT = 2
STATUS_BAD_DRAFT = 4

LAYER_FULL = 0
LAYER_SLIDING = 1
VARIANT_V1 = 1
VARIANT_2 = 2
VERIFY_GREEDY = 0
VERIFY_SAMPLE = 1
FUSE_INJECT_KV = 1


class Config(C.Structure):
    _fields_ = [
        ("variant", C.c_int32),
        ("hidden", C.c_int32),
        ("n_taps", C.c_int32),
        ("tap_layers", C.c_int32 * MAX_TAPS),
        ("target_layers", C.c_int32),
        ("n_layers", C.c_int32),
        ("n_q_heads", C.c_int32),
        ("n_kv_heads", C.c_int32),
        ("head_dim", C.c_int32),
        ("ffn", C.c_int32),
        ("vocab", C.c_int32),
        ("block", C.c_int32),
        ("mask_token", C.c_int32),
        ("causal", C.c_int32),
        ("sliding_window", C.c_int32),
        ("layer_kind", C.c_int32 * MAX_LAYERS),
        ("rope_theta", C.c_float),
        ("rms_eps", C.c_float),
        ("conv_groups", C.c_int32),
    ]


class LayerWeights(C.Structure):
    _fields_ = [
        (n, C.c_void_p)
        for n in (
            "input_norm",
            "q_proj",
            "k_proj",
            "v_proj",
            "o_proj",
            "q_norm",
            "k_norm",
            "post_norm",
            "gate_proj",
            "up_proj",
            "down_proj",
        )
    ]


class Weights(C.Structure):
    _fields_ = [
        ("fc", C.c_void_p),
        ("hidden_norm", C.c_void_p),
        ("norm", C.c_void_p),
        ("embed", C.c_void_p),
        ("layers", C.POINTER(LayerWeights)),
        ("conv_norm", C.c_void_p),
        ("conv_proj", C.c_void_p),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libdflash.so is not built ({LIB_PATH}); run __graft_entry__.build() "
            "or python block_diffusion_speculative_tap_gb300/build.py"
        )
    lib = C.CDLL(LIB_PATH)
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    P = C.POINTER

    def fn(name, res, *args):
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = list(args)

    fn("dflash_strerror", C.c_char_p, C.c_int)
    fn("dflash_launch_count", i64)
    fn("dflash_config_validate", C.c_int, P(Config))
    fn("dflash_kind", C.c_char_p, P(Config))
    fn("dflash_tap_row_bytes", i64, P(Config))
    fn("dflash_fused_row_bytes", i64, P(Config))
    fn("dflash_create", C.c_int, P(Config), P(Weights), P(vp))
    fn("dflash_destroy", C.c_int, vp)
    fn("dflash_state_bytes", C.c_int, vp, C.c_int, C.c_int, P(sz))
    fn("dflash_state_init", C.c_int, vp, vp, sz, C.c_int, C.c_int, vp, P(vp))
    fn("dflash_state_free", C.c_int, vp)
    fn("dflash_state_length", C.c_int, vp, C.c_int, P(i64))
    fn("dflash_state_truncate", C.c_int, vp, vp, C.c_int, i64, vp, sz, vp)
    fn("dflash_device_status", C.c_int, vp, vp, P(i32))
    fn("dflash_state_wait_probe", C.c_int, vp, C.c_int64, vp)
    fn("dflash_state_ring", C.c_int, vp, P(vp))
    fn("dflash_state_cache", C.c_int, vp, C.c_int, P(vp), P(vp), P(C.c_int))
    fn("dflash_fuse_workspace_bytes", C.c_int, vp, C.c_int, P(sz))
    fn("dflash_fuse_taps", C.c_int, vp, vp, P(vp), i64, C.c_int, P(i32), P(i64), P(i32), C.c_int, vp, sz, vp)
    fn("dflash_draft_workspace_bytes", C.c_int, vp, vp, C.c_int, C.c_int, P(sz))
    fn("dflash_draft_block", C.c_int, vp, vp, C.c_int, C.c_int, vp, vp, vp, vp, C.c_int, vp, sz, vp)
    fn("dflash_draft_stages", C.c_int, vp, vp, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp, sz, vp)
    fn("dflash_draft_head", C.c_int, vp, vp, C.c_int, vp, vp, vp, vp, C.c_int, vp, sz, vp)
    fn("dflash_topk", C.c_int, vp, C.c_int, C.c_int, C.c_int, C.c_float, vp, vp, vp, vp, vp)
    fn("dflash_draft_stop", C.c_int, vp, C.c_int, C.c_int, C.c_float, C.c_float, vp, vp, vp)
    fn("dflash_draft_conv", C.c_int, vp, vp, C.c_int, vp, vp, sz, vp)
    fn("dflash_select_path_workspace_bytes", C.c_int, C.c_int, C.c_int, C.c_int, P(sz))
    fn("dflash_tree_size", C.c_int, C.c_int, vp, C.c_int, P(C.c_int))
    fn("dflash_tree_build", C.c_int, C.c_int, C.c_int, vp, C.c_int, vp, vp, vp, vp, vp, vp, vp)
    fn("dflash_tree_verify_workspace_bytes", C.c_int, C.c_int, C.c_int, P(sz))
    fn("dflash_tree_verify", C.c_int, C.c_int, C.c_int, vp, C.c_int, vp, vp, vp, vp, vp, vp, sz, vp)
    fn("dflash_select_path", C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp, vp, vp, vp, vp, vp, vp, sz,
       vp)
    fn("dflash_verify_workspace_bytes", C.c_int, C.c_int, C.c_int, C.c_int, P(sz))
    fn("dflash_verify", C.c_int, C.c_int, C.c_int, C.c_int, vp, C.c_int, vp, vp, vp, C.c_float, vp, vp, vp, sz, vp)
    fn("dflash_verify_sample_noalloc", C.c_int, C.c_int, C.c_int, vp, C.c_int, vp, vp, vp, C.c_float, vp, vp, vp)
    fn("dflash_trace_enable", C.c_int, C.c_int)
    fn("dflash_trace_count", C.c_int)
    fn("dflash_trace_get", C.c_int, C.c_int, P(C.c_char_p), P(C.c_float), P(C.c_double), P(C.c_double))
    return lib


lib = _load()

EXPORTED = [
    "dflash_strerror",
    "dflash_launch_count",
    "dflash_config_validate",
    "dflash_kind",
    "dflash_tap_row_bytes",
    "dflash_fused_row_bytes",
    "dflash_create",
    "dflash_destroy",
    "dflash_state_bytes",
    "dflash_state_init",
    "dflash_state_free",
    "dflash_state_length",
    "dflash_state_truncate",
    "dflash_device_status",
    "dflash_state_wait_probe",
    "dflash_state_ring",
    "dflash_state_cache",
    "dflash_fuse_workspace_bytes",
    "dflash_fuse_taps",
    "dflash_draft_workspace_bytes",
    "dflash_draft_block",
    "dflash_draft_stages",
    "dflash_draft_head",
    "dflash_topk",
    "dflash_draft_stop",
    "dflash_draft_conv",
    "dflash_select_path_workspace_bytes",
    "dflash_select_path",
    "dflash_tree_size",
    "dflash_tree_build",
    "dflash_tree_verify_workspace_bytes",
    "dflash_tree_verify",
    "dflash_verify_workspace_bytes",
    "dflash_verify",
    "dflash_verify_sample_noalloc",
    "dflash_trace_enable",
    "dflash_trace_count",
    "dflash_trace_get",
]


class DFlashError(RuntimeError):
    def __init__(self, code, where=""):
        self.code = code
        msg = lib.dflash_strerror(code).decode()
        super().__init__(f"{where}: {msg} ({code})" if where else f"{msg} ({code})")


def check(rc, where=""):
    if rc != OK:
        raise DFlashError(rc, where)
    return rc


def make_config(model: dict) -> Config:
    c = Config()
    c.variant = model.get("variant", VARIANT_V1)
    c.hidden = model["hidden"]
    c.n_taps = model["n_taps"]
    taps = list(model.get("tap_layers", []))[:MAX_TAPS]
    for i, t in enumerate(taps):
        c.tap_layers[i] = t
    c.target_layers = model["target_layers"]
    c.n_layers = model["n_layers"]
    c.n_q_heads = model["n_q_heads"]
    c.n_kv_heads = model["n_kv_heads"]
    c.head_dim = model["head_dim"]
    c.ffn = model["ffn"]
    c.vocab = model["vocab"]
    c.block = model.get("block", BLOCK)
    c.mask_token = model["mask_token"]
    c.causal = model.get("causal", 0)
    c.sliding_window = model.get("sliding_window", 0)
    kinds = list(model.get("layer_kinds", []))[:MAX_LAYERS]
    for i, k in enumerate(kinds):
        c.layer_kind[i] = k
    c.rope_theta = model.get("rope_theta", 1.0e6)
    c.rms_eps = model.get("rms_eps", 1.0e-6)
    c.conv_groups = model.get("conv_groups", 0)
    return c
