"""Pins for the oracle: checks against what the pages and the mathematics fix.

None of these compares the oracle with itself. Each test uses a closed form,
a value printed on the pages, a library routine for a special case, brute
force on tiny inputs, or an invariant that a plausible mistake breaks.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import synthetic_inputs as SI

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tiny_model(**over):
    m = SI.presets()["tiny"]["model"]
    m.update(over)
    return m


def _weights64(model, seed=7):
    return O.weights_to_f64(SI.make_weights(model, seed))


# ----------------------------------------------------------------------------
# bf16 rounding: against torch's float32 -> bfloat16 converter (RNE)


def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    # random magnitudes across the exponent range, both signs
    mant = rng.uniform(1.0, 2.0, 200000)
    ex = rng.integers(-140, 127, 200000)
    x = (mant * np.exp2(ex) * rng.choice([-1.0, 1.0], 200000)).astype(np.float32)
    # exact ties: a bf16 value plus half of its spacing (representable in fp32)
    base = torch.randn(20000).to(torch.bfloat16).float().numpy()
    _, e = np.frexp(base.astype(np.float64))
    ties = (base.astype(np.float64) + np.sign(base) * np.exp2(e - 9)).astype(np.float32)
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 1e-45, 3.0e38, -3.0e38])])
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = O.round_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_bf16_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to the even 1.0
    assert O.round_bf16(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 lies halfway between 1+2^-7 and 1+2^-6: ties to 1 + 2^-6
    assert O.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert O.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7


# ----------------------------------------------------------------------------
# RMSNorm and RoPE closed forms


def test_rms_norm_constant_vector_closed_form():
    for c, eps in [(3.0, 1e-6), (0.5, 0.25), (-2.0, 4.0)]:
        x = np.full((3, 10), c)
        g = np.arange(1, 11, dtype=np.float64)
        got = O.rms_norm(x, g, eps)
        assert np.allclose(got, c / math.sqrt(c * c + eps) * g, rtol=1e-14, atol=0)


def test_rms_norm_uses_mean_not_sum():
    x = np.array([[3.0, 4.0]])  # mean square 12.5
    got = O.rms_norm(x, np.ones(2), 0.0)
    assert np.allclose(got, x / math.sqrt(12.5))


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).normal(size=(5, 3, 32))
    assert np.array_equal(O.rope(x, np.zeros((5, 1)), 1e6), x)


def test_rope_rotate_half_closed_form():
    theta = 100.0
    p = 7.0
    e = np.eye(4)
    out = O.rope(e, np.full(4, p), theta)
    w1 = theta ** -0.5
    assert np.allclose(out[0], [math.cos(p), 0, math.sin(p), 0])
    assert np.allclose(out[1], [0, math.cos(p * w1), 0, math.sin(p * w1)])
    assert np.allclose(out[2], [-math.sin(p), 0, math.cos(p), 0])
    assert np.allclose(out[3], [0, -math.sin(p * w1), 0, math.cos(p * w1)])


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(2)
    q, k = rng.normal(size=64), rng.normal(size=64)
    s1 = O.rope(q, 100, 1e4) @ O.rope(k, 37, 1e4)
    s2 = O.rope(q, 1063, 1e4) @ O.rope(k, 1000, 1e4)
    assert abs(s1 - s2) < 1e-9
    assert abs(np.linalg.norm(O.rope(q, 12345, 1e6)) - np.linalg.norm(q)) < 1e-12


# ----------------------------------------------------------------------------
# attention


def _attention_brute(q, k, v):
    nq, d = q.shape[1], q.shape[2]
    grp = nq // k.shape[1]
    out = np.zeros_like(q)
    for r in range(q.shape[0]):
        for h in range(nq):
            g = h // grp
            sc = [sum(q[r, h, i] * k[j, g, i] for i in range(d)) / math.sqrt(d) for j in range(k.shape[0])]
            m = max(sc)
            wts = [math.exp(s - m) for s in sc]
            tot = sum(wts)
            for i in range(d):
                out[r, h, i] = sum(wts[j] * v[j, g, i] for j in range(k.shape[0])) / tot
    return out


def test_attention_matches_brute_force():
    rng = np.random.default_rng(3)
    q = rng.normal(size=(16, 4, 8))
    k = rng.normal(size=(21, 2, 8))
    v = rng.normal(size=(21, 2, 8))
    assert np.allclose(O.block_attention(q, k, v), _attention_brute(q, k, v), rtol=1e-12, atol=1e-12)


def test_attention_equal_scores_average_values_per_group():
    rng = np.random.default_rng(4)
    q = np.zeros((16, 6, 8))  # all scores zero -> uniform weights
    k = rng.normal(size=(9, 2, 8))
    v = rng.normal(size=(9, 2, 8))
    out = O.block_attention(q, k, v)
    for h in range(6):
        assert np.allclose(out[:, h, :], v[:, h // 3, :].mean(axis=0))


def test_attention_is_not_causal():
    # the last key is strongly preferred by every row, the first row included
    q = np.ones((16, 1, 4)) * 5.0
    k = np.zeros((20, 1, 4))
    k[-1] = 10.0
    v = np.zeros((20, 1, 4))
    v[-1] = 1.0
    out = O.block_attention(q, k, v)
    assert np.all(out[0, 0] > 0.999)


def test_visible_positions_enumerated():
    assert list(O.visible_positions(O.SLIDING, 10, 4)) == [6, 7, 8, 9]
    assert list(O.visible_positions(O.SLIDING, 3, 4)) == [0, 1, 2]
    assert list(O.visible_positions(O.FULL, 10, 4)) == list(range(10))
    assert list(O.visible_positions(O.SLIDING, 0, 4)) == []


# ----------------------------------------------------------------------------
# tap fusion


def test_fusion_single_tap_identity_fc_is_rmsnorm():
    rng = np.random.default_rng(5)
    plane = O.round_bf16(rng.normal(size=(7, 16)))
    got = O.fuse_taps([plane], np.eye(16), np.ones(16), 1e-6)
    want = O.round_bf16(plane / np.sqrt((plane ** 2).mean(axis=1, keepdims=True) + 1e-6))
    assert np.array_equal(got, want)


def test_fusion_concatenates_tap_zero_first():
    rng = np.random.default_rng(6)
    a = O.round_bf16(rng.normal(size=(3, 8)))
    b = O.round_bf16(rng.normal(size=(3, 8)))
    pick0 = np.concatenate([np.eye(8), np.zeros((8, 8))], axis=1)
    pick1 = np.concatenate([np.zeros((8, 8)), np.eye(8)], axis=1)
    g = np.ones(8)
    assert np.array_equal(O.fuse_taps([a, b], pick0, g, 0.0), O.fuse_taps([a], np.eye(8), g, 0.0))
    assert np.array_equal(O.fuse_taps([a, b], pick1, g, 0.0), O.fuse_taps([b], np.eye(8), g, 0.0))


def test_fused_rows_are_bf16():
    m = _tiny_model()
    w = _weights64(m)
    planes = [O.to_f64(p) for p in SI.make_taps(m, 5, 3)]
    f = O.fuse_taps(planes, w["fc"], w["hidden_norm"], m["rms_eps"])
    assert np.array_equal(O.round_bf16(f), f)


# ----------------------------------------------------------------------------
# the block forward: structure pinned by special cases


def test_block_with_zero_output_projections_reduces_to_lm_head_of_mask_embedding():
    """With o_proj = down_proj = 0 both residual adds contribute nothing, so
    the residual stays the embedding and every mask row's logits are the LM
    head applied to the normed mask-token embedding."""
    m = _tiny_model(n_layers=1, layer_kinds=[O.FULL])
    w = _weights64(m)
    for lw in w["layers"]:
        lw["o_proj"][:] = 0.0
        lw["down_proj"][:] = 0.0
    C = 5
    ctx_k = [np.zeros((C, m["n_kv_heads"], m["head_dim"]))]
    ctx_v = [np.zeros((C, m["n_kv_heads"], m["head_dim"]))]
    logits, X = O.draft_block(m, w, ctx_k, ctx_v, C, anchor=17)
    e = w["embed"][m["mask_token"]]
    z = O.round_bf16(e / np.sqrt((e ** 2).mean() + m["rms_eps"]) * w["norm"])
    want = O.round_bf16(w["embed"] @ z)
    assert logits.shape == (15, m["vocab"])
    for r in range(15):
        assert np.array_equal(logits[r], want)
    assert np.array_equal(X[0], w["embed"][17])


def test_block_attention_with_zero_queries_averages_the_window():
    """q_proj = 0 makes every score zero, so the attention output of each
    head is the mean of the values its kv head sees: the sliding window's
    context rows (positions >= C - W) plus the sixteen block rows."""
    m = _tiny_model(n_layers=1, layer_kinds=[O.SLIDING], sliding_window=5)
    w = _weights64(m)
    lw = w["layers"][0]
    lw["q_proj"][:] = 0.0
    lw["down_proj"][:] = 0.0
    nkv, d, nq, H = m["n_kv_heads"], m["head_dim"], m["n_q_heads"], m["hidden"]
    C = 12
    rng = np.random.default_rng(9)
    ctx_k = [O.round_bf16(rng.normal(size=(C, nkv, d)))]
    ctx_v = [O.round_bf16(rng.normal(size=(C, nkv, d)))]
    anchor = 33
    _, X = O.draft_block(m, w, ctx_k, ctx_v, C, anchor)
    tokens = [anchor] + [m["mask_token"]] * 15
    X0 = w["embed"][tokens]
    h = O.round_bf16(X0 / np.sqrt((X0 ** 2).mean(axis=1, keepdims=True) + m["rms_eps"]) * lw["input_layernorm"])
    vb = O.round_bf16(h @ lw["v_proj"].T).reshape(16, nkv, d)
    grp = nq // nkv

    def expect(first):
        vis = np.concatenate([ctx_v[0][first:], vb], axis=0)
        mean = vis.mean(axis=0)  # [nkv, d]
        att = np.stack([mean[hh // grp] for hh in range(nq)]).reshape(nq * d)
        return X0 + O.round_bf16(att)[None, :] @ lw["o_proj"].T

    # 5 window rows + 16 block rows; a bf16 flip of the averaged value moves
    # X by a few 1e-5 at most, a wrong window by far more
    err = np.abs(X - expect(C - 5)).max()
    assert err < 1e-4
    assert np.abs(X - expect(0)).max() > 20 * max(err, 1e-6)
    assert np.abs(X - expect(C - 4)).max() > 20 * max(err, 1e-6)


def test_sliding_window_wider_than_context_equals_full():
    m_full = _tiny_model(layer_kinds=[O.FULL, O.FULL])
    m_slide = _tiny_model(layer_kinds=[O.SLIDING, O.SLIDING], sliding_window=64)
    w = _weights64(m_full)
    rng = np.random.default_rng(10)
    C = 40
    ks = [O.round_bf16(rng.normal(size=(C, 4, 32))) for _ in range(2)]
    vs = [O.round_bf16(rng.normal(size=(C, 4, 32))) for _ in range(2)]
    a, _ = O.draft_block(m_full, w, ks, vs, C, 5)
    b, _ = O.draft_block(m_slide, w, ks, vs, C, 5)
    assert np.array_equal(a, b)
    m_narrow = _tiny_model(layer_kinds=[O.SLIDING, O.SLIDING], sliding_window=8)
    c, _ = O.draft_block(m_narrow, w, ks, vs, C, 5)
    assert not np.array_equal(a, c)


def test_context_order_does_not_matter():
    """Non-causal attention over the context: permuting the context rows
    (each keeps its own RoPE'd key) leaves the block's output unchanged."""
    m = _tiny_model()
    w = _weights64(m)
    rng = np.random.default_rng(11)
    C = 30
    ks = [O.round_bf16(rng.normal(size=(C, 4, 32))) for _ in range(2)]
    vs = [O.round_bf16(rng.normal(size=(C, 4, 32))) for _ in range(2)]
    perm = rng.permutation(C)
    _, Xa = O.draft_block(m, w, ks, vs, C, 5)
    _, Xb = O.draft_block(m, w, [k[perm] for k in ks], [v[perm] for v in vs], C, 5)
    assert np.allclose(Xa, Xb, rtol=1e-10, atol=1e-12)


def test_streams_chunked_append_and_truncate_equal_fresh():
    m = _tiny_model()
    w = _weights64(m)
    planes = [O.to_f64(p) for p in SI.make_taps(m, 40, 21)]
    one = O.OracleStreams(m, w, 1)
    one.append(0, planes)
    two = O.OracleStreams(m, w, 1)
    two.append(0, [p[:25] for p in planes])
    two.append(0, [p[25:] for p in planes])
    assert np.array_equal(one.fused[0], two.fused[0])
    for l in range(m["n_layers"]):
        assert np.array_equal(one.k[0][l], two.k[0][l])
        assert np.array_equal(one.v[0][l], two.v[0][l])
    two.truncate(0, 10)
    two.append(0, [p[10:] for p in planes])
    la, _ = one.draft(0, 9)
    lb, _ = two.draft(0, 9)
    assert np.array_equal(la, lb)


# ----------------------------------------------------------------------------
# candidates and verification


def test_topk_matches_sorted_tuples_with_ties():
    rng = np.random.default_rng(12)
    row = rng.integers(-3, 4, size=300).astype(np.float64)
    ids, vals = O.topk(row, 9)
    want = sorted(range(300), key=lambda i: (-row[i], i))[:9]
    assert list(ids) == want
    assert list(vals) == [row[i] for i in want]


def test_greedy_golden_cases():
    with open(os.path.join(GOLDEN, "greedy_verify_cases.json")) as f:
        spec = json.load(f)
    for case in spec["cases"]:
        V = case["vocab"]
        tl = np.zeros((16, V))
        for i, pk in enumerate(case["peaks"]):
            for j in pk:
                tl[i, j] = 2.0
        a, toks = O.greedy_verify(case["draft"], tl)
        assert a == case["expect_a"], case["name"]
        assert toks == case["expect_tokens"], case["name"]


def test_greedy_invariants_random():
    rng = np.random.default_rng(13)
    for _ in range(200):
        V = 5
        tl = rng.normal(size=(16, V))
        d = rng.integers(0, V, 15)
        a, toks = O.greedy_verify(d, tl)
        assert 0 <= a <= 15
        assert toks[a] == int(np.argmax(tl[a]))
        assert all(toks[i] == d[i] == int(np.argmax(tl[i])) for i in range(a))
        assert all(t == -1 for t in toks[a + 1:])


def test_inverse_cdf_midpoint_grid_reproduces_weights():
    wts = np.array([0.0, 3.0, 1.0, 0.0, 4.0])
    n = 8000
    counts = np.zeros(5)
    for k in range(n):
        j, _ = O.inverse_cdf(wts, (k + 0.5) / n)
        counts[j] += 1
    assert np.allclose(counts / n, wts / wts.sum(), atol=1.0 / n)
    assert O.inverse_cdf(wts, 0.0)[0] == 1  # zero-weight entries are never drawn


def test_sampling_rule_output_distribution_is_target():
    """The first committed token's distribution equals p (losslessness).

    Exact decomposition of the rule: the draft x ~ q is accepted with
    probability min(1, p(x)/q(x)); otherwise the residual draw follows
    max(p - q, 0) normalised. Acceptance and residual frequencies are
    measured from the oracle on midpoint grids of the uniforms; combined,
    they must give p within the grids' resolution."""
    V = 6
    T = 1.0
    rng = np.random.default_rng(14)
    tl = rng.normal(size=(16, V)) * 1.5
    dl = rng.normal(size=(15, V)) * 1.5
    p = np.exp(tl[0] - tl[0].max())
    p /= p.sum()
    q = np.exp(dl[0] - dl[0].max())
    q /= q.sum()
    n = 2000
    grid = (np.arange(n) + 0.5) / n
    acc = np.zeros(V)
    for x in range(V):
        d = np.full(15, x)
        d[1:] = 0
        hits = 0
        for u in grid:
            uni = np.zeros((16, 2))
            uni[0, 0] = u
            uni[1:, 0] = 0.999999  # later positions do not matter here
            a, toks, _ = O.sampling_verify(d, tl, dl, uni, T)
            hits += a >= 1
        acc[x] = hits / n
    assert np.allclose(acc, np.minimum(1.0, p / q), atol=1.5 / n)
    # residual draw: force a rejection at position 0 with a draft x where q > p
    x = int(np.argmax(q - p))
    res = np.zeros(V)
    for u in grid:
        uni = np.full((16, 2), 0.5)
        uni[0, 0] = 1.0 - 1e-12
        uni[0, 1] = u
        a, toks, _ = O.sampling_verify(np.full(15, x), tl, dl, uni, T)
        assert a == 0
        res[toks[0]] += 1
    res /= n
    r = np.maximum(p - q, 0)
    assert np.allclose(res, r / r.sum(), atol=1.5 / n)
    out = q * acc + (q * (1 - acc)).sum() * res
    assert np.allclose(out, p, atol=4.0 / n)


def test_sampling_rule_chi_square():
    """Draw d_1 ~ q and run the rule many times; the first committed token
    must follow p (chi-square at 1e-3 significance)."""
    from scipy.stats import chisquare

    V = 5
    rng = np.random.default_rng(15)
    tl = rng.normal(size=(16, V))
    dl = rng.normal(size=(15, V))
    p = np.exp(tl[0] - tl[0].max())
    p /= p.sum()
    n = 20000
    counts = np.zeros(V)
    for _ in range(n):
        ud = rng.random(15)
        d, _ = O.sample_rows(dl, 1.0, ud)
        a, toks, _ = O.sampling_verify(d, tl, dl, rng.random((16, 2)), 1.0)
        counts[toks[0]] += 1
    stat = chisquare(counts, p * n)
    assert stat.pvalue > 1e-3


def test_sampling_all_accepted_draws_bonus_from_last_row():
    V = 4
    tl = np.zeros((16, V))
    dl = np.zeros((15, V))  # p == q everywhere: every test accepts
    tl[15] = [0.0, 0.0, 50.0, 0.0]
    d = np.arange(15) % V
    a, toks, _ = O.sampling_verify(d, tl, dl, np.full((16, 2), 0.5), 1.0)
    assert a == 15 and toks[:15] == list(d) and toks[15] == 2


def test_temperature_scales_logits():
    row = np.array([0.0, 1.0, 2.0])
    assert np.allclose(O.softmax_t(row, 2.0), O.softmax_t(row / 2.0, 1.0))
    assert O.softmax_t(row, 0.01)[2] > 0.999


# ----------------------------------------------------------------------------
# constants, inventory and refusals printed on the pages


def test_page_constants():
    with open(os.path.join(GOLDEN, "page_constants.json")) as f:
        c = json.load(f)
    H = c["hidden_9b"]
    assert O.fused_row_bytes(H) == c["fused_row_bytes_at_4096"]
    assert O.raw_plane_bytes(c["taps_v1"], H) == c["raw_tap_bytes_at_4096_eight_taps"]
    assert O.tap_row_bytes(1, c["taps_v1"], H) == c["tap_row_bytes_v1_eight_taps_factor"] * H * 2
    assert O.tap_row_bytes(2, c["taps_dflash2"], H) == O.raw_plane_bytes(5, H)
    assert O.drafter_tensor_count(c["layers_9b_drafter"]) == c["tensor_names_9b_drafter"]
    assert O.BLOCK == c["block"] and O.BLOCK - 1 == c["mask_rows"]
    assert O.kind_name(1) == c["kind_v1"] and O.kind_name(2) == c["kind_dflash2"]
    m = SI.presets()["9b"]["model"]
    assert len(SI.weight_names(m)) == c["tensor_names_9b_drafter"]
    assert m["n_taps"] == c["taps_v1"]
    d2 = SI.presets()["dflash2geom"]["model"]
    assert d2["tap_layers"] == c["dflash2_tap_layers"]
    assert d2["sliding_window"] == c["dflash2_sliding_window"]


def test_refusals():
    m = SI.presets()["9b"]["model"]
    assert O.validate_config(m) is None
    bad = dict(m, tap_layers=[1, 5, 9, 13, 17, 21, 25, 32])
    assert O.validate_config(bad) == "taps past the target"
    bad = dict(m, tap_layers=[1, 5, 9, 13, 17, 21, 25, 25])
    assert O.validate_config(bad) == "taps repeated"
    bad = dict(m, causal=1)
    assert O.validate_config(bad) == "causal"
    for name in SI.presets():
        assert O.validate_config(SI.presets()[name]["model"]) is None


# ---------------------------------------------------------------- min-p stop
def test_draft_confidence_closed_forms():
    """Confidence = top-1 softmax probability (Strata #3457 "Problem and
    result", reading in the oracle): equal logits give 1/V; one logit a over
    V-1 logits b give 1 / (1 + (V-1) e^((b-a)/T)); two tied maxima split it."""
    V = 1000
    c = O.draft_confidence(np.zeros((1, V)), 1.0)
    assert abs(c[0] - 1.0 / V) < 1e-15
    V, a, b, T = 100, 2.0, 0.5, 0.7
    row = np.full(V, b)
    row[37] = a
    want = 1.0 / (1.0 + (V - 1) * np.exp((b - a) / T))
    got = O.draft_confidence(row[None, :], T)[0]
    assert abs(got - want) < 1e-14 * want
    row[80] = a  # two maxima
    want2 = 1.0 / (2.0 + (V - 2) * np.exp((b - a) / T))
    assert abs(O.draft_confidence(row[None, :], T)[0] - want2) < 1e-14 * want2
    # a hotter softmax is less confident, a colder one more
    rng = np.random.default_rng(3)
    rows = rng.normal(size=(5, 50))
    c1, c2, c3 = (O.draft_confidence(rows, t) for t in (0.5, 1.0, 2.0))
    assert np.all(c1 > c2) and np.all(c2 > c3)


def test_draft_stop_rule():
    """The draft stops at the first position whose confidence is below min-p
    (equality keeps drafting); the length is in [0, 15]."""
    conf = np.full((4, 15), 0.9)
    conf[1, 2] = 0.6
    conf[1, 5] = 0.1  # after the stop: irrelevant
    conf[2, 0] = 0.69
    conf[3, :] = 0.7
    conf[3, 14] = 0.2
    assert O.draft_stop(conf, 0.7).tolist() == [15, 2, 0, 14]
    assert O.draft_stop(conf, 0.0).tolist() == [15, 15, 15, 15]
    assert O.draft_stop(conf, 1.0).tolist() == [0, 0, 0, 0]


# ----------------------------------------------------------------------------
# helpers of the layer: SiLU, arg-max, the context K/V


def test_silu_closed_forms():
    # silu(x) = x * sigmoid(x): zero at 0, sigmoid(1) and -sigmoid(-1) at +-1,
    # silu(x) - silu(-x) = x, and x for large x
    assert O.silu(np.float64(0.0)) == 0.0
    assert abs(O.silu(np.float64(1.0)) - 0.7310585786300049) < 1e-15
    assert abs(O.silu(np.float64(-1.0)) + 0.2689414213699951) < 1e-15
    x = np.linspace(-20, 20, 81)
    assert np.allclose(O.silu(x) - O.silu(-x), x, rtol=0, atol=1e-12)
    assert abs(O.silu(np.float64(40.0)) - 40.0) < 1e-12


def test_argmax_lowest_takes_the_first_of_ties():
    assert O.argmax_lowest([1.0, 3.0, 3.0, 2.0]) == 1
    assert O.argmax_lowest([5.0] * 7) == 0
    assert O.argmax_lowest([-4.0, -1.0, -2.0, -1.0]) == 1
    assert O.argmax_lowest([float("-inf"), 0.0]) == 1


def test_context_kv_properties():
    """K/V of context rows: V does not depend on the position; RoPE is a
    rotation, so each key head keeps its length (k_norm with unit gain makes
    that length sqrt(d) at every position), and a key pair's dot product
    depends only on the distance between the two positions."""
    m = _tiny_model()
    w = _weights64(m, seed=11)
    layer = dict(w["layers"][0])
    d, nkv = m["head_dim"], m["n_kv_heads"]
    layer["k_norm"] = np.ones(d)
    rng = np.random.default_rng(3)
    fused = O.round_bf16(rng.standard_normal((2, m["hidden"])))
    rows = np.concatenate([fused, fused])  # the same two rows at two position pairs
    k, v = O.context_kv(rows, [0, 5, 37, 42], layer, m)
    assert np.array_equal(v[:2], v[2:])
    # head lengths: sqrt(d) up to the bf16 rounding of the stored keys
    assert np.allclose(np.linalg.norm(k, axis=-1), math.sqrt(d), rtol=2 ** -7, atol=0)
    # relative positions: (0, 5) and (37, 42) are both 5 apart
    dots_a = np.einsum("hd,hd->h", k[0], k[1])
    dots_b = np.einsum("hd,hd->h", k[2], k[3])
    assert np.allclose(dots_a, dots_b, rtol=0, atol=d * 2 ** -6)
    # and a different distance gives different dots (the rotation is not the identity)
    k2, _ = O.context_kv(rows[:2], [0, 9], layer, m)
    assert not np.allclose(np.einsum("hd,hd->h", k2[0], k2[1]), dots_a, rtol=0, atol=d * 2 ** -6)
    assert k.shape == (4, nkv, d)


def test_layer_halves_add_to_the_residual():
    """Each half of a layer adds its branch to the residual (two residual adds
    a layer): with a zero output projection the half returns X unchanged, and
    the added branch does not depend on X's scale (an RMSNorm input: X and 3X
    give the same branch up to the bf16 rounding of the norm's output)."""
    m = _tiny_model()
    w = _weights64(m, seed=13)
    rng = np.random.default_rng(5)
    X = rng.standard_normal((O.BLOCK, m["hidden"]))
    C = 9
    nkv, d = m["n_kv_heads"], m["head_dim"]
    ck = O.round_bf16(rng.standard_normal((C, nkv, d)))
    cv = O.round_bf16(rng.standard_normal((C, nkv, d)))
    wz = {**w, "layers": [dict(L) for L in w["layers"]]}
    wz["layers"][0]["o_proj"] = np.zeros_like(w["layers"][0]["o_proj"])
    wz["layers"][0]["down_proj"] = np.zeros_like(w["layers"][0]["down_proj"])
    assert np.array_equal(O.attention_half(m, wz, 0, X, ck, cv, C), X)
    assert np.array_equal(O.mlp_half(m, wz, 0, X), X)
    a1 = O.attention_half(m, w, 0, X, ck, cv, C) - X
    a3 = O.attention_half(m, w, 0, 3 * X, ck, cv, C) - 3 * X
    assert np.allclose(a1, a3, rtol=0, atol=1e-6 + 2 ** -6 * np.abs(a1).max())
    g1 = O.mlp_half(m, w, 0, X) - X
    g3 = O.mlp_half(m, w, 0, 3 * X) - 3 * X
    assert np.allclose(g1, g3, rtol=0, atol=1e-6 + 2 ** -6 * np.abs(g1).max())


# ---------------------------------------------------------------- candidate-path selector
def _codebooks(case):
    V, r = case["vocab"], case["rank"]
    U = np.zeros((V, r))
    W = np.zeros((V, r))
    for k, v in case["U"].items():
        U[int(k)] = v
    for k, v in case["W"].items():
        W[int(k)] = v
    return U, W


def test_selector_golden_cases():
    with open(os.path.join(GOLDEN, "selector_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        U, W = _codebooks(c)
        ranks, ids, score, margin = O.select_path(c["cand_ids"], c["cand_vals"], U, W)
        want = -np.inf if c["score"] == "-inf" else c["score"]
        assert ranks == c["ranks"] and ids == c["ids"], c["name"]
        assert score == want and margin == c["margin"], (c["name"], score, margin)


def test_selector_brute_force():
    """Every path enumerated on small cases: the chosen path has the highest
    score, and the margin is the gap to the best other path."""
    rng = np.random.default_rng(5)
    for P in (1, 2, 3, 4):
        for k in (1, 2, 3, 4):
            V, r = 20, 5
            ids = np.stack([rng.choice(V, size=k, replace=False) for _ in range(P)])
            vals = rng.standard_normal((P, k))
            U, W = rng.standard_normal((V, r)), rng.standard_normal((V, r))
            scores = {}
            for path in itertools.product(range(k), repeat=P):
                e = sum(U[ids[i, path[i]]] @ W[ids[i + 1, path[i + 1]]] for i in range(P - 1))
                scores[path] = sum(vals[i, path[i]] for i in range(P)) + e
            order = sorted(scores, key=lambda p: -scores[p])
            ranks, got, score, margin = O.select_path(ids, vals, U, W)
            assert tuple(ranks) == order[0] and got == [int(ids[i, a]) for i, a in enumerate(ranks)]
            assert abs(score - scores[order[0]]) < 1e-12
            assert abs(O.path_score(ranks, ids, vals, U, W) - score) < 1e-12
            if len(order) > 1:
                assert abs(margin - (scores[order[0]] - scores[order[1]])) < 1e-12


def test_selector_rank0_is_per_position_top1():
    """TensorFold #1851 item 1: with no codebooks (rank 0) the edge term is
    zero, so the path is each position's highest candidate (the lowest
    index among equal ones)."""
    rng = np.random.default_rng(6)
    ids = rng.integers(0, 100, size=(15, 16))
    vals = np.round(rng.standard_normal((15, 16)) * 4) / 4  # many exact ties
    ranks, got, score, _ = O.select_path(ids, vals, np.zeros((100, 0)), np.zeros((100, 0)))
    assert ranks == [int(np.argmax(v)) for v in vals]
    assert score == sum(v.max() for v in vals)
    assert np.all(O.selector_edges(ids, np.zeros((100, 0)), np.zeros((100, 0))) == 0)


# ---------------------------------------------------------------- tree drafting and verification
def _tree_logits(case, N, V):
    rows = np.zeros((N, V))
    for n, t in enumerate(case["argmax"]):
        rows[n][t] = 1.0
    for n, t in case.get("tie_with", []):
        rows[n][t] = 1.0
    return rows


def test_tree_golden_cases():
    with open(os.path.join(GOLDEN, "tree_verify_cases.json")) as f:
        g = json.load(f)
    t = g["tree"]
    tokens, parents, depths = O.tree_nodes(t["anchor"], t["topk_ids"], t["widths"])
    assert (tokens, parents, depths) == (t["tokens"], t["parents"], t["depths"])
    mask = O.tree_mask(parents)
    assert np.nonzero(mask[len(tokens) - 1])[0].tolist() == t["ancestors_of_last"]
    for c in g["cases"]:
        a, out, node = O.tree_greedy_verify(tokens, parents, _tree_logits(c, len(tokens), t["vocab"]))
        assert (a, out, node) == (c["accept"], c["tokens"], c["node"]), c["name"]


def test_tree_structure():
    """Node count 1 + sum_j prod_{i<=j} b_i; breadth-first order (depths
    non-decreasing, a parent before its children, a node's children
    contiguous and in candidate order); the mask row of a node has its
    depth + 1 entries and contains its parent's."""
    rng = np.random.default_rng(3)
    for widths in ([1] * 15, [4, 2, 2, 1, 1], [16], [3, 3, 3, 3], [2] * 7):
        topk = rng.integers(0, 1000, size=(15, 16))
        tokens, parents, depths = O.tree_nodes(11, topk, widths)
        assert len(tokens) == 1 + sum(int(np.prod(widths[: j + 1])) for j in range(len(widths)))
        assert depths == sorted(depths) and all(parents[n] < n for n in range(1, len(tokens)))
        mask = O.tree_mask(parents)
        for n in range(1, len(tokens)):
            assert mask[n].sum() == depths[n] + 1 and np.all(mask[n] >= mask[parents[n]])
            kids = [c for c in range(len(tokens)) if parents[c] == parents[n]]
            assert kids == list(range(kids[0], kids[0] + len(kids)))
            assert tokens[n] == topk[depths[n] - 1][kids.index(n)]


def test_single_branch_tree_is_greedy_verify():
    """A tree with one candidate at every depth is the drafted chain itself;
    its verification must equal the chain's greedy verification (node j's
    target row is the chain's row j)."""
    rng = np.random.default_rng(4)
    V = 50
    for trial in range(200):
        topk = rng.integers(0, V, size=(15, 4))
        tl = rng.standard_normal((16, V))
        L = int(rng.integers(0, 17))
        for i in range(min(L, 15)):  # plant a prefix of accepts
            tl[i][topk[i][0]] = tl[i].max() + 1.0
        tokens, parents, _ = O.tree_nodes(3, topk, [1] * 15)
        a, out, node = O.tree_greedy_verify(tokens, parents, tl)
        ga, gout = O.greedy_verify(topk[:, 0], tl)
        assert (a, out) == (ga, gout) and node == a


# ---------------------------------------------------------------- DFlash2 two-tap dynamic convolution
def _conv_model(H=256, G=4):
    return dict(hidden=H, conv_groups=G, rms_eps=1e-6)


def test_block_conv_zero_projection_averages_adjacent_rows():
    """conv_proj = 0: every tap logit is 0, so both taps weigh 1/2. With
    constant rows X_i = c_i (|c_i| = 2) and a unit gain the normed rows are
    exactly sign(c_i) (bf16 rounds 1 - 1e-7 to 1), so
    X'_i = c_i + (sign(c_{i-1}) + sign(c_i)) / 2 with nothing before row 0."""
    m = _conv_model()
    c = np.array([2.0, -2.0, -2.0, 2.0] * 4)
    X = np.repeat(c[:, None], m["hidden"], axis=1)
    w = {"conv_norm": np.ones(m["hidden"]), "conv_proj": np.zeros((2 * m["conv_groups"], m["hidden"]))}
    out = O.block_conv(m, w, X)
    sg = np.sign(c)
    want = c + 0.5 * (np.concatenate([[0.0], sg[:-1]]) + sg)
    assert np.array_equal(out, np.repeat(want[:, None], m["hidden"], axis=1))


def test_block_conv_tap_order():
    """Tap 0 reads the previous row, tap 1 the row itself: a projection that
    makes tap 0 dominate adds the previous row's normed values (row 0 gets
    nothing), one that makes tap 1 dominate adds the row's own."""
    m = _conv_model()
    H, G = m["hidden"], m["conv_groups"]
    rng = np.random.default_rng(1)
    X = np.abs(rng.standard_normal((16, H))) + 1.0  # positive rows: positive normed values
    g = np.ones(H)
    h = O.round_bf16(O.rms_norm(X, g, 1e-6))
    for tap in (0, 1):
        P = np.zeros((2 * G, H))
        P[tap::2] = 1.0  # logit of `tap` = sum of the row's normed values (> 200), the other 0
        out = O.block_conv(m, {"conv_norm": g, "conv_proj": P}, X)
        add = np.concatenate([np.zeros((1, H)), h[:-1]]) if tap == 0 else h
        assert np.allclose(out, X + add, rtol=0, atol=1e-12)


def test_block_conv_locality_and_groups():
    """Row j reaches only rows j and j + 1; a projection that only feeds
    group 0's logits leaves every other group at the even average."""
    m = _conv_model(H=512, G=8)
    H, G = 512, 8
    rng = np.random.default_rng(2)
    X = rng.standard_normal((16, H))
    w = {"conv_norm": 1 + 0.02 * rng.standard_normal(H), "conv_proj": 0.05 * rng.standard_normal((2 * G, H))}
    out = O.block_conv(m, w, X)
    for j in (0, 7, 15):
        X2 = X.copy()
        X2[j] += rng.standard_normal(H)
        out2 = O.block_conv(m, w, X2)
        moved = [i for i in range(16) if not np.array_equal(out[i], out2[i])]
        assert moved == [i for i in (j, j + 1) if i < 16]
    P = np.zeros((2 * G, H))
    P[0:2] = rng.standard_normal((2, H))  # group 0's two taps only
    out = O.block_conv(m, {"conv_norm": w["conv_norm"], "conv_proj": P}, X)
    h = O.round_bf16(O.rms_norm(X, w["conv_norm"], 1e-6))
    prev = np.concatenate([np.zeros((1, H)), h[:-1]])
    gs = H // G
    assert np.allclose(out[:, gs:], X[:, gs:] + 0.5 * (prev[:, gs:] + h[:, gs:]), rtol=0, atol=1e-12)
    assert not np.allclose(out[:, :gs], X[:, :gs] + 0.5 * (prev[:, :gs] + h[:, :gs]))


def test_conv_drafter_block_and_config():
    """A DFlash2-layout drafter with the convolution runs it after the last
    layer (one more residual in the stage list, equal to block_conv of the
    one before); a v1 config with a convolution is refused (the v1 layout
    has no conv tensor, TensorFold #1851 item 1), and so are group counts
    that do not split the hidden width into multiples of 16."""
    m = SI.shrink(SI.presets()["tiny"]["model"], variant=2, conv_groups=4)
    w = O.weights_to_f64(SI.make_weights(m, 5))
    ref = O.OracleStreams(m, w, 1)
    ref.append(0, [O.to_f64(t) for t in SI.make_taps(m, 20, 6)])
    logits, Xs = ref.draft(0, 3, keep_residuals=True)
    assert len(Xs) == 2 * m["n_layers"] + 2
    assert np.array_equal(Xs[-1], O.block_conv(m, w, Xs[-2]))
    assert np.array_equal(logits, O.draft_head(m, w, Xs[-1]))
    assert O.validate_config(m) is None
    assert O.validate_config(dict(m, variant=1)) is not None
    assert O.validate_config(dict(m, conv_groups=3)) is not None  # 256 / 3
    assert O.validate_config(dict(m, conv_groups=32)) is not None  # groups of 8 channels
