"""Conditioning of the drafted function itself (oracle only, CPU).

The drafter rounds its activations to bf16 between operators. An error of
the size of fp32 accumulation over a few thousand terms (2^-20 relative),
added to the residual after every layer, flips a growing share of those
roundings layer after layer, so two correct fp32 implementations of the same
method drift apart with depth. This test
measures that drift on a six-layer drafter with the workloads' weight
statistics: it is why six-layer logits are checked stage by stage against
the stated tolerance, and end to end against an envelope taken from the
oracle's own arithmetic run in float32 (pinned below).
"""
import numpy as np

import oracle as O
import synthetic_inputs as SI


def _drift(L):
    m = dict(
        variant=1, hidden=1024, n_taps=2, tap_layers=[3, 9], target_layers=16, n_layers=L, n_q_heads=8,
        n_kv_heads=2, head_dim=128, ffn=3072, vocab=2048, block=16, mask_token=2047, causal=0,
        sliding_window=64, layer_kinds=[O.FULL] * L, rope_theta=1.0e6, rms_eps=1.0e-6,
    )
    w = O.weights_to_f64(SI.make_weights(m, 42))
    ref = O.OracleStreams(m, w, 1)
    ref.append(0, [O.to_f64(t) for t in SI.make_taps(m, 48, 43)])
    C = ref.length(0)
    X = O.block_embed(m, w, 7)
    Xp = X.copy()
    rng = np.random.default_rng(0)
    for l in range(L):
        X = O.draft_layer(m, w, l, X, ref.k[0][l], ref.v[0][l], C)
        Xp = O.draft_layer(m, w, l, Xp, ref.k[0][l], ref.v[0][l], C)
        Xp = Xp * (1.0 + 2.0 ** -20 * rng.standard_normal(Xp.shape))
    a, b = O.draft_head(m, w, X), O.draft_head(m, w, Xp)
    return np.abs(a - b).mean(), np.abs(a).mean()


def test_fp32_sized_errors_are_amplified_with_depth():
    d1, s1 = _drift(1)
    d2, s2 = _drift(2)
    d6, s6 = _drift(6)
    # 2^-20 (about 1e-6) of noise a layer ends up as ~0.5% of the logits
    assert d6 / s6 > 1e-3
    # and it grows with depth
    assert d1 < d2 < d6 and d6 > 1.5 * d2


def _pair(L, seed=42):
    m = dict(
        variant=1, hidden=1024, n_taps=2, tap_layers=[3, 9], target_layers=16, n_layers=L, n_q_heads=8,
        n_kv_heads=2, head_dim=128, ffn=3072, vocab=2048, block=16, mask_token=2047, causal=0,
        sliding_window=64, layer_kinds=[O.FULL] * L, rope_theta=1.0e6, rms_eps=1.0e-6,
    )
    w = O.weights_to_f64(SI.make_weights(m, seed))
    taps = [O.to_f64(t) for t in SI.make_taps(m, 48, seed + 1)]
    ref = O.OracleStreams(m, w, 1)
    ref.append(0, taps)
    o64, X64 = ref.draft(0, 7)
    with O.arithmetic(np.float32):
        r32 = O.OracleStreams(m, O.weights_as(w, np.float32), 1)
        r32.append(0, taps)
        o32, X32 = r32.draft(0, 7)
        kinds = {r32.fused[0].dtype, r32.k[0][0].dtype, X32.dtype, o32.dtype}
    return o64, o32, X64, kinds


def test_float32_arithmetic_mode():
    """The end-to-end envelope of the GPU parity tests comes from the
    oracle's own arithmetic run in float32. That run computes in float32
    (every stored array is float32 inside the block, float64 again after
    it), it is the same method (at one layer it matches the float64 run
    within the stated tolerance, where a dropped term or a wrong rounding
    point would be far outside it), and its distance from the float64 run
    grows with depth (so the envelope measures the drift, not zero)."""
    o64, o32, X64, kinds = _pair(1)
    assert kinds == {np.dtype(np.float32)}
    assert X64.dtype == np.float64 and o64.dtype == np.float64
    err = np.abs(o32 - o64)
    assert np.all(err <= 2e-2 + 1e-2 * np.abs(o64))
    assert err.max() > 0  # not secretly float64
    d1 = err.mean()
    o64, o32, _, _ = _pair(6)
    d6 = np.abs(o32 - o64).mean()
    assert d6 > 2 * d1
