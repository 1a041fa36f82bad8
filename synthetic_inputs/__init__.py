"""Seeded synthetic inputs for the DFlash drafting hot path.

This module is shared by the tests, the bench and the oracle's callers. It
holds workload shapes and random-number draws only: none of the method's
arithmetic (no norms, projections, attention, sampling or verification) lives
here. Random numbers the method consumes (uniforms for sampling) are drawn
here and passed to both the oracle and the CUDA path as inputs.

Everything is drawn with torch's seeded generators and rounded to bf16 by
torch, so a given (seed, shape) pair yields the same tensor on every call.

Workload presets follow the five drafter configurations of the hot path:
a tiny drafter, a 9B-shaped DFlash v1 drafter at batch 1, the same drafter
over a 32k fused-row ring, a 32-stream serving round, and a drafter with the
DFlash2 geometry (5 taps of hidden 5120). Weight statistics: projections
N(0, 0.02); norm gains 1 + N(0, 0.02) so that a gain-indexing mistake is
visible; tap planes N(0, 1).
"""
from __future__ import annotations

import copy

import torch

FULL = 0
SLIDING = 1

VARIANT_V1 = 1
VARIANT_2 = 2

BLOCK = 16


def _preset_9b():
    return dict(
        variant=VARIANT_V1,
        hidden=4096,
        n_taps=8,
        # eight taps of a 32-layer target, evenly spread from shallow to deep
        tap_layers=[1, 5, 9, 13, 17, 21, 25, 29],
        target_layers=32,
        n_layers=6,
        n_q_heads=32,
        n_kv_heads=8,
        head_dim=128,
        ffn=12288,
        vocab=151936,
        block=BLOCK,
        mask_token=151935,
        causal=0,
        sliding_window=2048,
        layer_kinds=[SLIDING] * 5 + [FULL],
        rope_theta=1.0e6,
        rms_eps=1.0e-6,
    )


def presets():
    """Return the five workload presets as {name: dict}.

    Each preset holds the drafter configuration (``model``) and the workload
    around it: streams, context lengths, ring capacity, top-k and the verify
    mode with its logit distribution.
    """
    tiny = dict(
        model=dict(
            variant=VARIANT_V1,
            hidden=256,
            n_taps=5,
            tap_layers=[1, 3, 5, 7, 9],
            target_layers=12,
            n_layers=2,
            n_q_heads=8,
            n_kv_heads=4,
            head_dim=32,
            ffn=768,
            vocab=4096,
            block=BLOCK,
            mask_token=4095,
            causal=0,
            sliding_window=2048,
            layer_kinds=[FULL, FULL],
            rope_theta=1.0e6,
            rms_eps=1.0e-6,
        ),
        streams=1,
        context=[128],
        ring=256,
        topk=4,
        verify="greedy",
        target_logit_std=1.0,
        seed=1234,
    )
    nine_b = dict(
        model=_preset_9b(),
        streams=1,
        context=[4096],
        ring=8192,
        topk=8,
        verify="greedy",
        target_logit_std=1.0,
        seed=1235,
    )
    long32k = dict(
        model=_preset_9b(),
        streams=1,
        context=[32768 - 1024],
        ring=32768,
        topk=8,
        verify="greedy",
        target_logit_std=1.0,
        seed=1236,
    )
    serve32 = dict(
        model=_preset_9b(),
        streams=32,
        context=None,  # drawn: uniform in [1024, 16384]
        context_range=(1024, 16384),
        ring=16384 + 1024,
        topk=8,
        verify="greedy",
        target_logit_std=2.0,
        planted_accept=True,
        seed=1237,
    )
    d2geom = dict(
        model=dict(
            variant=VARIANT_V1,
            hidden=5120,
            n_taps=5,
            tap_layers=[5, 19, 33, 47, 61],
            target_layers=64,
            n_layers=5,
            n_q_heads=40,
            n_kv_heads=8,
            head_dim=128,
            ffn=17408,
            vocab=151936,
            block=BLOCK,
            mask_token=151935,
            causal=0,
            sliding_window=2048,
            layer_kinds=[FULL] * 5,
            rope_theta=1.0e6,
            rms_eps=1.0e-6,
        ),
        streams=8,
        context=[8192] * 8,
        ring=8192 + 1024,
        topk=8,
        verify="sample",
        temperature=1.0,
        target_logit_std=1.0,
        seed=1238,
    )
    return {
        "tiny": tiny,
        "9b": nine_b,
        "long32k": long32k,
        "serve32": serve32,
        "dflash2geom": d2geom,
    }


def preset(name):
    p = copy.deepcopy(presets()[name])
    if p["context"] is None:
        lo, hi = p["context_range"]
        g = torch.Generator().manual_seed(p["seed"] + 17)
        p["context"] = torch.randint(lo, hi + 1, (p["streams"],), generator=g).tolist()
    return p


def shrink(model, **over):
    """A copy of a drafter config with some fields replaced (small test shapes)."""
    m = copy.deepcopy(model)
    m.update(over)
    if "layer_kinds" not in over:
        m["layer_kinds"] = (m["layer_kinds"] * m["n_layers"])[: m["n_layers"]]
    if "n_taps" in over and "tap_layers" not in over:
        m["tap_layers"] = list(range(1, 2 * m["n_taps"], 2))
        m["target_layers"] = max(m["target_layers"], 2 * m["n_taps"])
    if "vocab" in over and "mask_token" not in over:
        m["mask_token"] = m["vocab"] - 1
    return m


# ----------------------------------------------------------------------------
# random draws


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal_bf16(shape, std, mean, g, device):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def weight_names(model):
    """Tensor names of a drafter: eleven per layer plus fc, hidden_norm, norm.

    The embedding / LM head is the target's and is not counted.
    """
    per_layer = [
        "input_layernorm",
        "q_proj",
        "k_proj",
        "v_proj",
        "o_proj",
        "q_norm",
        "k_norm",
        "post_attention_layernorm",
        "gate_proj",
        "up_proj",
        "down_proj",
    ]
    names = ["fc", "hidden_norm", "norm"]
    for l in range(model["n_layers"]):
        names += [f"layers.{l}.{n}" for n in per_layer]
    return names


def make_weights(model, seed, device="cpu", std=0.02):
    """Draw a drafter's weights (bf16). Returns a dict of tensors.

    Layout (row-major, [out_features, in_features] for projections):
      fc [H, N*H], hidden_norm [H], norm [H], embed [V, H] (shared LM head),
      layers[l]: input_layernorm [H], q_proj [nq*d, H], k_proj [nkv*d, H],
      v_proj [nkv*d, H], o_proj [H, nq*d], q_norm [d], k_norm [d],
      post_attention_layernorm [H], gate_proj [F, H], up_proj [F, H],
      down_proj [H, F].
    """
    H = model["hidden"]
    N = model["n_taps"]
    d = model["head_dim"]
    nq = model["n_q_heads"]
    nkv = model["n_kv_heads"]
    F = model["ffn"]
    V = model["vocab"]
    g = _gen(seed, device)

    def proj(o, i):
        return _normal_bf16((o, i), std, 0.0, g, device)

    def gain(n):
        return _normal_bf16((n,), std, 1.0, g, device)

    w = {
        "fc": proj(H, N * H),
        "hidden_norm": gain(H),
        "norm": gain(H),
        "embed": proj(V, H),
        "layers": [],
    }
    for _ in range(model["n_layers"]):
        w["layers"].append(
            {
                "input_layernorm": gain(H),
                "q_proj": proj(nq * d, H),
                "k_proj": proj(nkv * d, H),
                "v_proj": proj(nkv * d, H),
                "o_proj": proj(H, nq * d),
                "q_norm": gain(d),
                "k_norm": gain(d),
                "post_attention_layernorm": gain(H),
                "gate_proj": proj(F, H),
                "up_proj": proj(F, H),
                "down_proj": proj(H, F),
            }
        )
    if model.get("conv_groups", 0):
        # DFlash2's two-tap dynamic convolution: its norm gain and the
        # projection to two tap logits per channel group
        w["conv_norm"] = gain(H)
        w["conv_proj"] = proj(2 * model["conv_groups"], H)
    return w


def make_taps(model, rows, seed, device="cpu"):
    """N tap planes, each [rows, H] bf16 drawn from N(0, 1)."""
    g = _gen(seed, device)
    return [
        _normal_bf16((rows, model["hidden"]), 1.0, 0.0, g, device)
        for _ in range(model["n_taps"])
    ]


def make_logits(shape, std, seed, device="cpu"):
    """Logit rows N(0, std^2) rounded to bf16."""
    return _normal_bf16(tuple(shape), std, 0.0, _gen(seed, device), device)


def make_uniforms(shape, seed, device="cpu"):
    """Uniform numbers in [0, 1) (fp32)."""
    return torch.rand(tuple(shape), generator=_gen(seed, device), device=device, dtype=torch.float32)


def make_token_ids(shape, vocab, seed, device="cpu", exclude=None):
    """Uniform token ids in [0, vocab); ``exclude`` (e.g. the mask token) is remapped to 0."""
    t = torch.randint(0, vocab, tuple(shape), generator=_gen(seed, device), device=device, dtype=torch.int64)
    if exclude is not None:
        t = torch.where(t == exclude, torch.zeros_like(t), t)
    return t.to(torch.int32)


def make_accept_lengths(streams, seed):
    """Planted accept lengths L in {0, ..., 16} (16 and 15 both mean a full block)."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randint(0, BLOCK + 1, (streams,), generator=g).tolist()


def plant_accepts(target_logits, draft_ids, lengths):
    """Rewrite target logit rows so greedy verification accepts a planted prefix.

    target_logits: [S, 16, V] bf16 (modified in place); draft_ids: [S, 15] int.
    For stream s with planted length L: rows i < min(L, 15) get
    logit[d_{i+1}] = rowmax + 1 (the draft token becomes the unique argmax);
    for L <= 14, row L gets logit[d_{L+1}] = rowmax - 1 if the draft token was
    the argmax there, so the first mismatch happens at row L.
    This is input construction for a seeded workload, not verification.
    """
    S = target_logits.shape[0]
    ids = draft_ids.to(torch.int64).cpu()
    for s in range(S):
        L = int(lengths[s])
        for i in range(min(L, BLOCK - 1)):
            row = target_logits[s, i]
            row[ids[s, i]] = (row.float().max() + 1.0).to(row.dtype)
        if L <= BLOCK - 2:
            row = target_logits[s, L]
            x = ids[s, L]
            if int(torch.argmax(row.float())) == int(x):
                row[x] = (row.float().max() - 1.0).to(row.dtype)
    return target_logits


def make_codebooks(vocab, rank, seed, std=0.1, device="cpu"):
    """A selector's pair codebooks U, W: two [vocab, rank] bf16 draws from
    N(0, std^2) (synthetic: the pages publish only the rank)."""
    g = _gen(seed, device)
    return _normal_bf16((vocab, rank), std, 0.0, g, device), _normal_bf16((vocab, rank), std, 0.0, g, device)


def anchor_ids(streams, vocab, mask_token, seed, device="cpu"):
    return make_token_ids((streams,), vocab, seed, device, exclude=mask_token)


def n_params(model):
    H, N, d = model["hidden"], model["n_taps"], model["head_dim"]
    nq, nkv, F = model["n_q_heads"], model["n_kv_heads"], model["ffn"]
    per_layer = 2 * H + 2 * d + nq * d * H * 2 + 2 * nkv * d * H + 3 * F * H
    return N * H * H + 2 * H + model["vocab"] * H + model["n_layers"] * per_layer
