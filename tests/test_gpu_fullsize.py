"""Full-size parity on the four large workloads, in the launch shapes the bench
times. The oracle computes sampled outputs one by one: sampled fused rows and
K/V rows of a fill, and the full draft of sampled streams (it fuses only
those streams' contexts). The end-to-end drafts are compared element by
element within the envelope the oracle's own float32 run gives (parity_util);
every stage within the stated tolerance. Everything else is checked by
properties that hold at any size (top-k consistent with the logits, planted
acceptance lengths, valid sampling outcomes).
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic_inputs as SI
from parity_util import assert_close, check_topk_consistent, compare_draft, f64, oracle_stream, staged_parity

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def D():
    import block_diffusion_speculative_tap_gb300 as D

    return D


def sampled_rows(n, k, seed, tile=256):
    """k seeded rows of an n-row fill, plus the first and last rows and the
    rows on both sides of the first, middle and last row-tile boundaries of
    the wide fc GEMM (256 rows a tile)."""
    rng = np.random.default_rng(seed)
    idx = set(rng.choice(n, size=min(k, n), replace=False).tolist())
    idx |= {0, n - 1}
    for b in {tile, (n // 2 // tile) * tile, ((n - 1) // tile) * tile}:
        if 0 < b < n:
            idx |= {b - 1, b}
    return np.array(sorted(idx))


def check_rows(st, m, w64, taps_host, s, base, rows):
    """Fused rows and K/V cache rows of positions base + rows (oracle on those rows only)."""
    planes = [p[rows] for p in taps_host]
    fused = O.fuse_taps(planes, w64["fc"], w64["hidden_norm"], m["rms_eps"])
    ring = st.ring_view()[s, base + rows].cpu().float().numpy()
    assert_close(ring, fused, "sampled fused rows")
    pos = base + rows
    for l, lw in enumerate(w64["layers"]):
        K, V, cap = st.cache_view(l)
        k, v = O.context_kv(fused, pos, lw, m)
        if m["layer_kinds"][l] == SI.SLIDING:
            keep = pos >= st.length(s) - cap
            slots = pos[keep] % cap
            k, v = k[keep], v[keep]
        else:
            slots = pos
        if len(slots) == 0:
            continue
        kg = K[s][:, slots].permute(1, 0, 2).cpu().float().numpy()
        vg = V[s][:, slots].permute(1, 0, 2).cpu().float().numpy()
        assert_close(kg, k, f"K rows layer {l}")
        assert_close(vg, v, f"V rows layer {l}")


@pytest.fixture(scope="module")
def nine_b(D):
    P = SI.preset("9b")
    m = P["model"]
    w = SI.make_weights(m, P["seed"], device="cuda")
    dr = D.Drafter(m, w)
    w64 = O.weights_to_f64(w)
    yield P, m, w, dr, (w64, O.weights_as(w64, np.float32))
    dr.close()


def test_9b_batch1_decode_round(D, nine_b):
    P, m, w, dr, (w64, w32) = nine_b
    C0 = P["context"][0]
    st = dr.new_state(1, P["ring"])
    ctx = SI.make_taps(m, C0 + 16, P["seed"] + 1, device="cuda")
    st.fuse_taps([t[:C0] for t in ctx], [(0, 0, C0)])  # prompt fill (4096 rows)
    st.fuse_taps([t[C0:] for t in ctx], [(0, C0, 16)])  # the round's 16 committed rows
    host = [f64(t) for t in ctx]
    check_rows(st, m, w64, [h[:C0] for h in host], 0, 0, sampled_rows(C0, 40, 1))
    check_rows(st, m, w64, [h[C0:] for h in host], 0, C0, np.arange(16))
    anchor = SI.anchor_ids(1, m["vocab"], m["mask_token"], P["seed"] + 2, device="cuda")
    logits, ids, vals = st.draft(anchor, k=P["topk"])
    check_topk_consistent(logits, ids, vals)
    ref = oracle_stream(m, w64, host, w32)
    o32 = ref.draft32(0, int(anchor[0]))
    ol = staged_parity(st, ref, 0, m, 0, int(anchor[0]), P["topk"])
    compare_draft(logits.cpu().float().numpy(), ids.cpu().numpy(), ol, o32, P["topk"])
    # verification on the drafted top-1 ids: planted acceptance is recovered
    tl = SI.make_logits((1, 16, m["vocab"]), P["target_logit_std"], P["seed"] + 3)
    L = 9
    SI.plant_accepts(tl, ids[:, 0].reshape(1, 15).cpu(), [L])
    a, toks = D.verify_greedy(ids, tl.cuda())
    assert int(a[0]) == L
    assert toks[0, :L].tolist() == ids[:L, 0].tolist()
    assert int(toks[0, L]) == int(torch.argmax(tl[0, L].float()))
    rc, bits = st.status()
    assert rc == 0 and bits == 0


def test_long32k_append_and_windowed_draft(D, nine_b):
    P0, m, w, dr, (w64, w32) = nine_b
    P = SI.preset("long32k")
    C0 = P["context"][0]
    st = dr.new_state(1, P["ring"])
    ctx = SI.make_taps(m, C0 + 16, P["seed"] + 1, device="cuda")
    st.fuse_taps([t[:C0] for t in ctx], [(0, 0, C0)])
    st.fuse_taps([t[C0:] for t in ctx], [(0, C0, 16)])
    host = [f64(t) for t in ctx]
    check_rows(st, m, w64, [h[:C0] for h in host], 0, 0, sampled_rows(C0, 24, 2))
    check_rows(st, m, w64, [h[C0:] for h in host], 0, C0, np.arange(16))
    anchor = SI.anchor_ids(1, m["vocab"], m["mask_token"], P["seed"] + 2, device="cuda")
    logits, ids, vals = st.draft(anchor, k=P["topk"])
    check_topk_consistent(logits, ids, vals)
    ref = oracle_stream(m, w64, host, w32)
    o32 = ref.draft32(0, int(anchor[0]))
    ol = staged_parity(st, ref, 0, m, 0, int(anchor[0]), P["topk"])
    compare_draft(logits.cpu().float().numpy(), ids.cpu().numpy(), ol, o32, P["topk"])
    rc, bits = st.status()
    assert rc == 0 and bits == 0


def test_serve32_shared_round(D, nine_b):
    P0, m, w, dr, (w64, w32) = nine_b
    P = SI.preset("serve32")
    ctx = P["context"]
    S = len(ctx)
    st = dr.new_state(S, P["ring"])
    taps = SI.make_taps(m, sum(ctx), P["seed"] + 1, device="cuda")
    offs = np.concatenate([[0], np.cumsum(ctx)])
    st.fuse_taps(taps, [(s, 0, ctx[s]) for s in range(S)])
    anchors = SI.anchor_ids(S, m["vocab"], m["mask_token"], P["seed"] + 2, device="cuda")
    logits, ids, vals = st.draft(anchors, k=P["topk"])
    check_topk_consistent(logits, ids, vals)
    lg = logits.cpu().float().numpy().reshape(S, 15, -1)
    idn = ids.cpu().numpy().reshape(S, 15, -1)
    # concurrent == solo. Up to four streams a call (the split-K fixed by
    # the weights) a stream's draft is bit-identical to its solo draft; a
    # 32-stream round runs the throughput GEMM configuration, another fp32
    # summation order, so there the stream drafted inside the round and the
    # same stream drafted alone each meet the end-to-end envelope against the
    # oracle.
    solo, _, _ = st.draft(anchors[5:6].contiguous(), s_begin=5, k=P["topk"])
    four, _, _ = st.draft(anchors[4:8].contiguous(), s_begin=4, k=P["topk"])
    assert torch.equal(solo, four[15:30])
    s_min = int(np.argmin(ctx))
    solo_lg, solo_ids, _ = st.draft(anchors[s_min : s_min + 1].contiguous(), s_begin=s_min, k=P["topk"])
    solo_lg, solo_ids = solo_lg.cpu().float().numpy(), solo_ids.cpu().numpy()
    for s in sorted({s_min, int(np.argmax(ctx))}):
        host = [f64(t[offs[s] : offs[s + 1]]) for t in taps]
        ref = oracle_stream(m, w64, host, w32)
        o32 = ref.draft32(0, int(anchors[s]))
        ol = staged_parity(st, ref, 0, m, s, int(anchors[s]), P["topk"])
        compare_draft(lg[s], idn[s], ol, o32, P["topk"])
        if s == s_min:
            compare_draft(solo_lg, solo_ids, ol, o32, P["topk"])
    # greedy verification of every stream against planted target logits
    tl = SI.make_logits((S, 16, m["vocab"]), P["target_logit_std"], P["seed"] + 3)
    lengths = SI.make_accept_lengths(S, P["seed"] + 4)
    SI.plant_accepts(tl, ids[:, 0].reshape(S, 15).cpu(), lengths)
    a, toks = D.verify_greedy(ids, tl.cuda())
    assert a.cpu().tolist() == [min(L, 15) for L in lengths]
    rc, bits = st.status()
    assert rc == 0 and bits == 0


def test_dflash2_geometry_sampling_round(D):
    P = SI.preset("dflash2geom")
    m = P["model"]
    w = SI.make_weights(m, P["seed"], device="cuda")
    dr = D.Drafter(m, w)
    ctx = P["context"]
    S = len(ctx)
    st = dr.new_state(S, P["ring"])
    taps = SI.make_taps(m, sum(ctx), P["seed"] + 1, device="cuda")
    offs = np.concatenate([[0], np.cumsum(ctx)])
    st.fuse_taps(taps, [(s, 0, ctx[s]) for s in range(S)])
    anchors = SI.anchor_ids(S, m["vocab"], m["mask_token"], P["seed"] + 2, device="cuda")
    logits, ids, vals = st.draft(anchors, k=P["topk"])
    check_topk_consistent(logits, ids, vals)
    w64 = O.weights_to_f64(w)
    lg = logits.cpu().float().numpy().reshape(S, 15, -1)
    idn = ids.cpu().numpy().reshape(S, 15, -1)
    # drafted tokens sampled from the drafter's rows, then sampling verification
    T = P["temperature"]
    ud = SI.make_uniforms((S * 15,), P["seed"] + 3, device="cuda")
    _, _, draft = D.topk(logits, 0, temperature=T, uniforms=ud)
    tl = SI.make_logits((S, 16, m["vocab"]), P["target_logit_std"], P["seed"] + 4, device="cuda")
    u = SI.make_uniforms((S, 16, 2), P["seed"] + 5, device="cuda")
    a, toks = D.verify_sample(draft.view(S, 15), tl, logits.view(S, 15, -1), u, T)
    a, toks, dd = a.cpu().tolist(), toks.cpu().tolist(), draft.view(S, 15).cpu().tolist()
    for s in range(S):
        assert 0 <= a[s] <= 15
        assert toks[s][: a[s]] == dd[s][: a[s]]
        assert 0 <= toks[s][a[s]] < m["vocab"]
        assert all(t == -1 for t in toks[s][a[s] + 1 :])
    rc, bits = st.status()
    assert rc == 0 and bits == 0
    s = S - 1
    host = [f64(t[offs[s] : offs[s + 1]]) for t in taps]
    ref = oracle_stream(m, w64, host)
    o32 = ref.draft32(0, int(anchors[s]))
    ol = staged_parity(st, ref, 0, m, s, int(anchors[s]), P["topk"])
    compare_draft(lg[s], idn[s], ol, o32, P["topk"])
    dr.close()
