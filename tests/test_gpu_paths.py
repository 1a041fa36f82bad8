"""GPU parity of the rows after the draft's top-k: the DFlash2 candidate-path
selector (dflash_select_path) against the oracle's max-sum recursion.

Path ids and candidate indices must equal the oracle's bit for bit, except
where the oracle's own margin (its best path's score minus the best score of
any other path) is within the GPU's fp32 error bound: there both paths are
correct to that precision, and the GPU's path is checked to be a valid path
whose oracle score is within the bound of the best. The bound is derived in
`fp32_bound` below.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
import synthetic_inputs as SI

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U32 = 2.0 ** -24  # fp32 unit roundoff


@pytest.fixture(scope="module")
def D():
    import block_diffusion_speculative_tap_gb300 as D

    return D


def fp32_bound(ids, vals, U, W):
    """Worst-case difference between the GPU's fp32 path score and the exact
    one. An edge is a sequential fp32 sum of r exact bf16 products, within
    r * u * sum_j |U_j W_j| of exact; a path sums 2P - 1 terms in fp32, within
    2P * u * (sum of their magnitudes). Doubled for the two paths a decision
    compares, and doubled again as a safety factor."""
    P, k = ids.shape
    V, r = U.shape
    valid = (ids >= 0) & (ids < V)
    safe = np.where(valid, ids, 0)
    Ua = np.abs(U[safe]) * valid[..., None]
    Wa = np.abs(W[safe]) * valid[..., None]
    eabs = np.einsum("iar,ibr->iab", Ua[:-1], Wa[1:]).max() if P > 1 and r > 0 else 0.0
    nabs = np.abs(np.where(valid, vals, 0.0)).max()
    edge_err = r * U32 * eabs
    sum_err = 2 * P * U32 * (P * nabs + (P - 1) * eabs)
    return 4.0 * ((P - 1) * edge_err + sum_err) + 1e-30


def check_paths(D, ids, vals, U, W, P):
    """Run the GPU selector on [S, P, k] candidates and compare each stream
    with the oracle. Returns (exact, exempt) stream counts."""
    S, _, k = ids.shape
    gi = torch.from_numpy(ids.astype(np.int32)).cuda()
    gv = torch.from_numpy(vals.astype(np.float32)).cuda()
    gU = U if isinstance(U, torch.Tensor) else torch.from_numpy(U).to(torch.bfloat16)
    gW = W if isinstance(W, torch.Tensor) else torch.from_numpy(W).to(torch.bfloat16)
    pid, prk, psc = D.select_path(gi, gv, gU.cuda().contiguous(), gW.cuda().contiguous(), positions=P)
    pid, prk, psc = pid.cpu().numpy(), prk.cpu().numpy(), psc.cpu().numpy()
    U64, W64 = O.to_f64(gU), O.to_f64(gW)
    exact = exempt = 0
    for s in range(S):
        v64 = vals[s].astype(np.float32).astype(np.float64)
        ranks, oid, score, margin = O.select_path(ids[s], v64, U64, W64)
        if score == -np.inf:
            assert list(pid[s]) == [-1] * P and list(prk[s]) == [-1] * P and psc[s] == -np.inf
            exact += 1
            continue
        B = fp32_bound(ids[s], v64, U64, W64)
        assert abs(float(psc[s]) - score) <= B / 2, (s, psc[s], score, B)
        if margin > B:
            assert list(prk[s]) == ranks and list(pid[s]) == oid, (s, list(prk[s]), ranks, margin)
            exact += 1
        else:
            # a near-tie: any path within the bound of the best is correct
            assert all(0 <= a < k for a in prk[s]) and list(pid[s]) == [int(ids[s, i, a]) for i, a in enumerate(prk[s])]
            assert O.path_score(list(prk[s]), ids[s], v64, U64, W64) >= score - B
            exempt += 1
    return exact, exempt


def test_selector_golden_cases_on_gpu(D):
    with open(os.path.join(GOLDEN, "selector_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        V, r = c["vocab"], c["rank"]
        r8 = max(8, (r + 7) // 8 * 8)  # the kernel reads whole 16-byte pieces: pad with zero columns
        U = np.zeros((V, r8))
        W = np.zeros((V, r8))
        for key, v in c["U"].items():
            U[int(key), : len(v)] = v
        for key, v in c["W"].items():
            W[int(key), : len(v)] = v
        ids = np.asarray(c["cand_ids"])[None]
        vals = np.asarray(c["cand_vals"])[None]
        P = ids.shape[1]
        gi = torch.from_numpy(ids.astype(np.int32)).cuda()
        gv = torch.from_numpy(vals.astype(np.float32)).cuda()
        gU = torch.from_numpy(U).to(torch.bfloat16).cuda()
        gW = torch.from_numpy(W).to(torch.bfloat16).cuda()
        pid, prk, psc = D.select_path(gi, gv, gU, gW, positions=P)
        want = -np.inf if c["score"] == "-inf" else c["score"]
        assert pid[0].tolist() == c["ids"] and prk[0].tolist() == c["ranks"], c["name"]
        assert float(psc[0]) == want, c["name"]


@pytest.mark.parametrize("P,k,r", [(1, 4, 8), (2, 1, 8), (7, 3, 0), (15, 16, 256), (16, 5, 40), (15, 8, 512)])
def test_selector_matches_oracle(D, P, k, r):
    """Seeded candidates (some ids outside the vocabulary), node scores and
    codebooks over every shape limit: one to sixteen positions, one to
    sixteen candidates, rank 0 to 512."""
    S, V = 6, 1000
    rng = np.random.default_rng(1000 * P + 10 * k + r)
    ids = rng.integers(0, V, size=(S, P, k))
    ids[rng.random((S, P, k)) < 0.03] = -5  # not candidates
    ids[0, 0, 0] = V + 7
    vals = rng.standard_normal((S, P, k)).astype(np.float32)
    U, W = SI.make_codebooks(V, r, 77 + r)
    exact, exempt = check_paths(D, ids, vals, U, W, P)
    print(f"P={P} k={k} r={r}: {exact} streams exact, {exempt} near-ties")
    assert exact >= S - 2


def test_selector_rank0_is_top1_on_gpu(D):
    """With rank 0 (no codebooks) the path is each position's first highest
    candidate: the draft's top-1 when the candidates are its sorted top-k."""
    S, P, k, V = 4, 15, 16, 500
    rng = np.random.default_rng(9)
    ids = rng.integers(0, V, size=(S, P, k))
    vals = (np.round(rng.standard_normal((S, P, k)) * 2) / 2).astype(np.float32)  # exact ties
    gi = torch.from_numpy(ids.astype(np.int32)).cuda()
    gv = torch.from_numpy(vals).cuda()
    empty = torch.zeros(V, 0, dtype=torch.bfloat16, device="cuda")
    pid, prk, _ = D.select_path(gi, gv, empty, empty, positions=P)
    assert prk.cpu().numpy().tolist() == np.argmax(vals, axis=2).tolist()


def test_selector_full_size_round(D):
    """32 streams x 15 positions, top-16 candidates of N(0, 2) logits over a
    151936-token vocabulary (dflash_topk on the GPU), rank-256 codebooks of
    the same vocabulary: every stream against the oracle."""
    S, P, k, V, r = 32, 15, 16, 151936, 256
    logits = SI.make_logits((S * P, V), 2.0, 4242, device="cuda")
    ids, vals, _ = D.topk(logits, k)
    U, W = SI.make_codebooks(V, r, 4243, device="cuda")
    exact, exempt = check_paths(D, ids.view(S, P, k).cpu().numpy(), vals.view(S, P, k).cpu().numpy(), U, W, P)
    print(f"full size: {exact} streams exact, {exempt} near-ties")
    # bf16 logits near the top of N(0, 2) tie exactly (spacing 1/16 at 8), so
    # some streams have another path within the fp32 bound; those are checked
    # for validity and near-optimality above
    assert exact >= S // 2


def test_selector_refusals(D):
    from block_diffusion_speculative_tap_gb300 import _abi as A
    import ctypes as C

    nb = C.c_size_t()
    assert A.lib.dflash_select_path_workspace_bytes(2, 15, 16, C.byref(nb)) == 0 and nb.value == 2 * 14 * 256 * 4
    assert A.lib.dflash_select_path_workspace_bytes(2, 17, 16, C.byref(nb)) == -1
    assert A.lib.dflash_select_path_workspace_bytes(2, 15, 17, C.byref(nb)) == -1
    gi = torch.zeros(2, 15, 4, dtype=torch.int32, device="cuda")
    gv = torch.zeros(2, 15, 4, dtype=torch.float32, device="cuda")
    U = torch.zeros(16, 12, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(D.DFlashError) as e:  # rank not a multiple of 8
        D.select_path(gi, gv, U, U, positions=15)
    assert e.value.code == -1
    out = torch.zeros(2, 15, dtype=torch.int32, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    rc = A.lib.dflash_select_path(2, 15, 4, 16, 8, C.c_void_p(gi.data_ptr()), C.c_void_p(gv.data_ptr()),
                                  C.c_void_p(U.data_ptr()), C.c_void_p(U.data_ptr()), C.c_void_p(out.data_ptr()),
                                  None, None, C.c_void_p(small.data_ptr()), 16, None)
    assert rc == -7  # workspace too small


# ---------------------------------------------------------------- tree drafting and verification
def _plant_tree_path(tl, tokens, parents, rng):
    """Make the target follow a random root-to-leaf path for a random number
    of steps: at each node on it, the next node's token becomes the row's
    unique maximum (input construction, not verification)."""
    N = len(tokens)
    children = [[] for _ in range(N)]
    for n, p in enumerate(parents):
        if p >= 0:
            children[p].append(n)
    cur = 0
    steps = int(rng.integers(0, 17))
    for _ in range(steps):
        if not children[cur]:
            break
        nxt = children[cur][int(rng.integers(0, len(children[cur])))]
        row = tl[cur]
        row[tokens[nxt]] = (row.float().max() + 1.0).to(row.dtype)
        cur = nxt


def check_trees(D, anchors, topk_ids, widths, tl):
    """GPU tree build and verification against the oracle, every stream
    (integer outputs: bit-exact)."""
    S = anchors.numel()
    tokens, parents, depths, mask = D.tree_build(anchors, topk_ids, widths)
    a, out, node = D.tree_verify(tokens, tl, widths)
    tok, par, dep = tokens.cpu().numpy(), parents.cpu().numpy(), depths.cpu().numpy()
    msk = mask.cpu().numpy().view(np.uint32)
    a, out, node = a.cpu().numpy(), out.cpu().numpy(), node.cpu().numpy()
    ids = topk_ids.cpu().numpy().reshape(S, 15, -1)
    N = tok.shape[1]
    for s in range(S):
        t, p, d = O.tree_nodes(int(anchors[s]), ids[s], widths)
        assert tok[s].tolist() == t and par[s].tolist() == p and dep[s].tolist() == d, s
        om = O.tree_mask(p)
        bits = np.unpackbits(msk[s].view(np.uint8), bitorder="little").reshape(N, -1)[:, :N].astype(bool)
        assert np.array_equal(bits, om), s
        rows = tl[s].float().cpu().numpy()
        oa, oout, onode = O.tree_greedy_verify(t, p, rows)
        assert (int(a[s]), out[s].tolist(), int(node[s])) == (oa, oout, onode), (s, a[s], oa)
    return a


def test_tree_golden_case_on_gpu(D):
    with open(os.path.join(GOLDEN, "tree_verify_cases.json")) as f:
        g = json.load(f)
    t = g["tree"]
    topk = np.zeros((15, 3), dtype=np.int32)
    topk[:3] = t["topk_ids"]
    anchors = torch.tensor([t["anchor"]], dtype=torch.int32, device="cuda")
    gt = torch.from_numpy(topk).cuda()
    tokens, parents, depths, mask = D.tree_build(anchors, gt, t["widths"])
    assert tokens[0].tolist() == t["tokens"] and parents[0].tolist() == t["parents"] and depths[0].tolist() == t["depths"]
    last = mask[0, -1].cpu().numpy().view(np.uint32)
    assert [n for n in range(len(t["tokens"])) if last[n // 32] >> (n % 32) & 1] == t["ancestors_of_last"]
    N, V = len(t["tokens"]), t["vocab"]
    for c in g["cases"]:
        rows = torch.zeros(1, N, V, dtype=torch.bfloat16)
        for n, tk in enumerate(c["argmax"]):
            rows[0, n, tk] = 1.0
        for n, tk in c.get("tie_with", []):
            rows[0, n, tk] = 1.0
        a, out, node = D.tree_verify(tokens, rows.cuda(), t["widths"])
        assert (int(a[0]), out[0].tolist(), int(node[0])) == (c["accept"], c["tokens"], c["node"]), c["name"]


@pytest.mark.parametrize("widths", [[1] * 15, [4, 2, 2, 1, 1], [16], [3, 3, 3, 3], [2] * 7, [5, 3, 1, 1, 1, 1, 1, 1]])
def test_tree_matches_oracle(D, widths):
    S, V, k = 6, 2048, 16
    rng = np.random.default_rng(sum(widths) * 7 + len(widths))
    logits = SI.make_logits((S * 15, V), 1.0, 600 + len(widths), device="cuda")
    topk_ids, _, _ = D.topk(logits, k)
    anchors = SI.anchor_ids(S, V, V - 1, 601, device="cuda")
    N = D.tree_size(widths, k)
    tl = SI.make_logits((S, N, V), 1.0, 602 + N)
    t64 = topk_ids.cpu().numpy().reshape(S, 15, k)
    for s in range(S):
        t, p, _ = O.tree_nodes(int(anchors[s]), t64[s], widths)
        _plant_tree_path(tl[s], t, p, rng)
    a = check_trees(D, anchors, topk_ids, widths, tl.cuda())
    print(f"widths {widths}: {N} nodes, accept lengths {a.tolist()}")


def test_single_branch_tree_equals_chain_verify(D):
    """All widths 1: the tree is the drafted chain, and its verification on
    the GPU equals dflash_verify(GREEDY) on the chain's target rows."""
    S, V = 16, 4096
    logits = SI.make_logits((S * 15, V), 1.0, 700, device="cuda")
    topk_ids, _, _ = D.topk(logits, 4)
    anchors = SI.anchor_ids(S, V, V - 1, 701, device="cuda")
    tl = SI.make_logits((S, 16, V), 1.0, 702)
    SI.plant_accepts(tl, topk_ids[:, 0].reshape(S, 15).cpu(), SI.make_accept_lengths(S, 703))
    tl = tl.cuda()
    tokens, _, _, _ = D.tree_build(anchors, topk_ids, [1] * 15, want_mask=False)
    a, out, _ = D.tree_verify(tokens, tl, [1] * 15)
    ga, gout = D.verify_greedy(topk_ids, tl)
    assert torch.equal(a, ga) and torch.equal(out, gout)


def test_tree_full_size_round(D):
    """32 streams, vocabulary 151936, a 93-node tree a stream (widths 4, 2,
    2, 1, 1, 1, 1) from the top-8 of N(0, 2) draft logits; the target's
    logits for every node with a planted path: every stream against the
    oracle."""
    S, V, k, widths = 32, 151936, 8, [4, 2, 2, 1, 1, 1, 1]
    rng = np.random.default_rng(77)
    logits = SI.make_logits((S * 15, V), 2.0, 800, device="cuda")
    topk_ids, _, _ = D.topk(logits, k)
    anchors = SI.anchor_ids(S, V, V - 1, 801, device="cuda")
    N = D.tree_size(widths, k)
    assert N == 93
    tl = SI.make_logits((S, N, V), 2.0, 802)
    t64 = topk_ids.cpu().numpy().reshape(S, 15, k)
    for s in range(S):
        t, p, _ = O.tree_nodes(int(anchors[s]), t64[s], widths)
        _plant_tree_path(tl[s], t, p, rng)
    a = check_trees(D, anchors, topk_ids, widths, tl.cuda())
    assert a.max() > 0


def test_tree_refusals(D):
    from block_diffusion_speculative_tap_gb300 import _abi as A
    import ctypes as C

    n = C.c_int()
    w = (C.c_int32 * 3)(4, 2, 9)
    assert A.lib.dflash_tree_size(3, w, 8, C.byref(n)) == -1  # a width above k
    w = (C.c_int32 * 3)(4, 2, 8)
    assert A.lib.dflash_tree_size(3, w, 8, C.byref(n)) == 0 and n.value == 1 + 4 + 8 + 64
    big = (C.c_int32 * 4)(16, 16, 16, 1)
    assert A.lib.dflash_tree_size(4, big, 16, C.byref(n)) == -1  # more than 1024 nodes
    assert A.lib.dflash_tree_size(0, w, 8, C.byref(n)) == -1
    assert A.lib.dflash_tree_size(16, (C.c_int32 * 16)(*([1] * 16)), 8, C.byref(n)) == -1


def test_dflash2_style_round(D):
    """The rows chained as a DFlash2-style round on six streams of a
    three-layer drafter with the two-tap convolution: fill, a top-16 draft
    (end to end within the oracle's envelope), the selector's path through
    the GPU's own candidates, greedy verification of that path against
    planted target logits, and a tree from the same draft verified against
    its own target rows; every integer output against the oracle on the
    same inputs."""
    from parity_util import OraclePair, compare_draft

    m = SI.shrink(SI.presets()["tiny"]["model"], variant=2, conv_groups=4, n_layers=3, layer_kinds=[1, 1, 0],
                  sliding_window=64)
    w = SI.make_weights(m, 951, device="cuda")
    dr = D.Drafter(m, w)
    ctx = [40, 100, 7, 200, 64, 1]
    S, V, k = len(ctx), m["vocab"], 16
    st = dr.new_state(S, 512)
    ref = OraclePair(m, O.weights_to_f64(w), S)
    taps = SI.make_taps(m, sum(ctx), 952, device="cuda")
    segs, r0 = [], 0
    for s, c in enumerate(ctx):
        segs.append((s, 0, c))
        ref.append(s, [O.to_f64(t[r0 : r0 + c]) for t in taps])
        r0 += c
    st.fuse_taps(taps, segs)
    anchors = SI.anchor_ids(S, V, m["mask_token"], 953, device="cuda")
    logits, ids, vals = st.draft(anchors, k=k)
    rc, bits = st.status()
    assert rc == 0 and bits == 0
    lg = logits.cpu().float().numpy().reshape(S, 15, V)
    idn = ids.cpu().numpy().reshape(S, 15, k)
    for s in range(S):
        ol, _ = ref.draft(s, int(anchors[s]))
        compare_draft(lg[s], idn[s], ol, ref.draft32(s, int(anchors[s])), k, require_checked=False)
    # the selector on the draft's own top-16
    U, W = SI.make_codebooks(V, 64, 954)
    exact, exempt = check_paths(D, idn, vals.cpu().numpy().reshape(S, 15, k), U, W, 15)
    assert exact >= S - 1
    pid, _, _ = D.select_path(ids.view(S, 15, k).contiguous(), vals.view(S, 15, k).contiguous(), U.cuda(), W.cuda())
    # greedy verification of the chosen path
    tl = SI.make_logits((S, 16, V), 1.0, 955)
    SI.plant_accepts(tl, pid.cpu(), SI.make_accept_lengths(S, 956))
    a, toks = D.verify_greedy(pid.contiguous(), tl.cuda())
    for s in range(S):
        oa, ot = O.greedy_verify(pid[s].cpu().tolist(), O.to_f64(tl[s]))
        assert int(a[s]) == oa and toks[s].cpu().tolist() == ot
    # a tree from the same draft
    widths = [4, 2, 1, 1]
    N = D.tree_size(widths, k)
    tt = SI.make_logits((S, N, V), 1.0, 957)
    rng = np.random.default_rng(958)
    for s in range(S):
        t, p, _ = O.tree_nodes(int(anchors[s]), idn[s], widths)
        _plant_tree_path(tt[s], t, p, rng)
    check_trees(D, anchors, ids, widths, tt.cuda())
