"""GPU parity of top-k, sampling draws and verification against the oracle.

Inputs are seeded synthetic logits fed to both sides. Ids, accept lengths and
tokens are compared bit for bit; a sampling decision is exempt only when the
oracle's float64 margin to the other outcome is below 1e-5 of the total, and
such cases are counted and checked for validity instead.

The 1e-5 bound is the kernel's fp32 error budget: each weight exp((x-m)/T)
is the SFU's base-2 exponential of one fused multiply-add, x*log2(e)/T -
m*log2(e)/T, with relative error <= 2^-22 plus |x-m|/T * 2^-23 from rounding
the argument (<= 4e-6 for |x-m|/T <= 30), and the running sums add
<= 8 + 5 + 37 + 16 + 8 fp32 roundings along any path (lane, warp scan,
warp-slice steps, warps, the eight slices of a verification row's cluster),
about 5e-6 of the total; probabilities divide two such sums.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
import synthetic_inputs as SI
from parity_util import f64

pytestmark = pytest.mark.gpu

MARGIN = 1e-5


@pytest.fixture(scope="module")
def D():
    import block_diffusion_speculative_tap_gb300 as D

    return D


def _tie_heavy(rows, V, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(-4, 5, (rows, V), generator=g).float() * 0.5
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("rows", [37, 130])  # a cluster a row / a CTA a row
@pytest.mark.parametrize("V,k", [(4096, 4), (151936, 8), (5000, 16), (136, 3), (151936, 1)])
def test_topk_matches_oracle(D, V, k, rows):
    lg = SI.make_logits((rows, V), 1.0, seed=V + k)
    lg[5:9] = _tie_heavy(4, V, 3)  # rows full of exact ties
    ids, vals, _ = D.topk(lg.cuda(), k)
    ids, vals = ids.cpu().numpy(), vals.cpu().numpy()
    ref = f64(lg)
    for r in range(rows):
        oi, ov = O.topk(ref[r], k)
        assert list(ids[r]) == list(oi), r
        assert np.array_equal(vals[r].astype(np.float64), ov), r


def test_topk_empty_and_zero_k(D):
    lg = SI.make_logits((0, 4096), 1.0, seed=1).cuda()
    ids, vals, _ = D.topk(lg, 4)
    assert ids.shape == (0, 4)
    lg = SI.make_logits((3, 4096), 1.0, seed=1).cuda()
    ids, vals, s = D.topk(lg, 0, uniforms=torch.rand(3, device="cuda"))
    assert s.shape == (3,)


@pytest.mark.parametrize("T,V,std", [(1.0, 151936, 3.0), (0.7, 151936, 3.0), (1.0, 4096, 2.0)])
def test_sampling_draws_match_oracle(D, T, V, std):
    rows = 64
    lg = SI.make_logits((rows, V), std, seed=11)
    u = SI.make_uniforms((rows,), seed=12)
    _, _, s = D.topk(lg.cuda(), 0, temperature=T, uniforms=u.cuda())
    s = s.cpu().numpy()
    ref_ids, margins = O.sample_rows(f64(lg), T, f64(u))
    clear = margins > MARGIN
    assert clear.sum() >= rows // 4, clear.sum()
    assert np.array_equal(s[clear], ref_ids[clear])
    # a near-tie draw must still sit within the error budget of u on the CDF
    uu = f64(u)
    for r in np.nonzero(~clear)[0]:
        p = O.softmax_t(f64(lg[r]), T)
        c = np.cumsum(p)
        j = int(s[r])
        lo = c[j - 1] if j > 0 else 0.0
        assert p[j] > 0 and lo - 2 * MARGIN <= uu[r] <= c[j] + 2 * MARGIN, r


def test_greedy_golden_fixtures(D):
    with open(os.path.join(os.path.dirname(__file__), "golden", "greedy_verify_cases.json")) as f:
        cases = json.load(f)["cases"]
    S = len(cases)
    V = cases[0]["vocab"]
    tl = torch.zeros(S, 16, V)
    draft = torch.zeros(S, 15, dtype=torch.int32)
    for s, c in enumerate(cases):
        for i, pk in enumerate(c["peaks"]):
            for j in pk:
                tl[s, i, j] = 2.0
        draft[s] = torch.tensor(c["draft"])
    a, toks = D.verify_greedy(draft.cuda(), tl.to(torch.bfloat16).cuda())
    a, toks = a.cpu().tolist(), toks.cpu().tolist()
    for s, c in enumerate(cases):
        assert a[s] == c["expect_a"], c["name"]
        assert toks[s] == c["expect_tokens"], c["name"]


@pytest.mark.parametrize("S,V,std", [(32, 151936, 2.0), (5, 4096, 1.0)])
def test_greedy_planted_matches_oracle(D, S, V, std):
    tl = SI.make_logits((S, 16, V), std, seed=21)
    draft = SI.make_token_ids((S, 15), V, seed=22)
    lengths = SI.make_accept_lengths(S, seed=23)
    SI.plant_accepts(tl, draft, lengths)
    a, toks = D.verify_greedy(draft.cuda(), tl.cuda())
    a, toks = a.cpu().tolist(), toks.cpu().tolist()
    ref = f64(tl)
    for s in range(S):
        oa, ot = O.greedy_verify(draft[s].tolist(), ref[s])
        assert a[s] == oa == min(lengths[s], 15)
        assert toks[s] == ot


def test_greedy_out_of_range_draft_never_accepted(D):
    V = 4096
    tl = torch.zeros(1, 16, V)
    tl[0, :, 7] = 1.0
    draft = torch.full((1, 15), 7, dtype=torch.int32)
    draft[0, 3] = V + 5
    a, toks = D.verify_greedy(draft.cuda(), tl.to(torch.bfloat16).cuda())
    assert a.item() == 3 and toks[0, 3].item() == 7


def _sampling_inputs(S, V, seed, noise, std):
    tl = SI.make_logits((S, 16, V), std, seed)
    dl = (tl[:, :15].float() + noise * SI.make_logits((S, 15, V), 1.0, seed + 1).float()).to(torch.bfloat16)
    # drafted tokens: drawn from the drafter's rows (input construction)
    g = torch.Generator().manual_seed(seed + 2)
    probs = torch.softmax(dl.float(), dim=-1).view(-1, V)
    draft = torch.multinomial(probs, 1, generator=g).view(S, 15).to(torch.int32)
    u = SI.make_uniforms((S, 16, 2), seed + 3)
    return tl, dl, draft, u


@pytest.mark.parametrize(
    "S,V,noise,T,std",
    [
        (8, 151936, 0.3, 1.0, 3.0),
        (16, 4096, 1.0, 1.0, 2.0),
        (16, 4096, 0.5, 0.6, 2.0),
        # 17 and 3 groups of 8 values over a row's 8 cluster slices: uneven and empty slices
        (16, 136, 1.0, 1.0, 2.0),
        (16, 24, 1.0, 0.8, 1.0),
    ],
)
def test_sampling_verify_matches_oracle(D, S, V, noise, T, std):
    tl, dl, draft, u = _sampling_inputs(S, V, 31 + S, noise, std)
    a, toks = D.verify_sample(draft.cuda(), tl.cuda(), dl.cuda(), u.cuda(), T)
    a, toks = a.cpu().tolist(), toks.cpu().tolist()
    tr, dr, ur = f64(tl), f64(dl), f64(u)
    checked = 0
    for s in range(S):
        oa, ot, margins = O.sampling_verify(draft[s].tolist(), tr[s], dr[s], ur[s], T)
        if min(margins) <= MARGIN:
            # near tie somewhere in the chain: the result must still be valid
            assert 0 <= a[s] <= 15
            assert toks[s][: a[s]] == draft[s].tolist()[: a[s]]
            assert 0 <= toks[s][a[s]] < V and all(t == -1 for t in toks[s][a[s] + 1 :])
            continue
        checked += 1
        assert a[s] == oa, s
        assert toks[s] == ot, s
    assert checked >= max(2, S // 4), checked


@pytest.mark.parametrize("V", [8, 136, 4096, 151936])
def test_sampling_verify_zero_residual_draws_target(D, V):
    """A rejection whose draft distribution equals the target's leaves an
    all-zero residual max(p - q, 0): the token is then drawn from the
    target's distribution (the oracle's fallback). Identical target and draft
    rows accept every in-vocabulary draft (u * q < p with q = p); an id
    outside the vocabulary is rejected, at positions 0, 7 and 14."""
    S = 3
    tl = SI.make_logits((S, 16, V), 2.0, seed=900 + V)
    dl = tl[:, :15].clone()
    draft = SI.make_token_ids((S, 15), V, seed=901 + V)
    rej = [0, 7, 14]
    for s in range(S):
        draft[s, rej[s]] = V + 3
    u = SI.make_uniforms((S, 16, 2), seed=902 + V)
    a, toks = D.verify_sample(draft.cuda(), tl.cuda(), dl.cuda(), u.cuda(), 1.0)
    a, toks = a.cpu().tolist(), toks.cpu().tolist()
    for s in range(S):
        i = rej[s]
        assert a[s] == i, (s, a[s])
        assert toks[s][:i] == draft[s].tolist()[:i]
        assert all(t == -1 for t in toks[s][i + 1 :])
        p = O.softmax_t(f64(tl[s, i]), 1.0)
        j, m = O.inverse_cdf(p, float(u[s, i, 1]))
        if m > MARGIN:
            assert toks[s][i] == j, (s, toks[s][i], j)
        else:
            c = np.cumsum(p)
            t = toks[s][i]
            lo = c[t - 1] if t > 0 else 0.0
            assert p[t] > 0 and lo - 2 * MARGIN <= float(u[s, i, 1]) <= c[t] + 2 * MARGIN


def test_sampling_verify_distribution_is_target(D):
    """Many single-position trials: the first committed token follows p
    (chi-square), the lossless property of the sampling rule."""
    from scipy.stats import chisquare

    V, n = 8, 4096
    tl1 = torch.tensor([[0.5, 1.0, -1.0, 2.0, 0.0, -0.5, 1.5, 0.25]])
    dl1 = torch.tensor([[1.0, 0.0, 0.5, 1.0, 1.0, -1.0, 0.0, 2.0]])
    tl = tl1.to(torch.bfloat16).expand(n, V).reshape(n, 1, V).expand(n, 16, V).contiguous()
    dl = dl1.to(torch.bfloat16).expand(n, V).reshape(n, 1, V).expand(n, 15, V).contiguous()
    q = torch.softmax(dl1.to(torch.bfloat16).float(), -1)[0]
    g = torch.Generator().manual_seed(5)
    draft = torch.multinomial(q.expand(n, V), 15, replacement=True, generator=g).to(torch.int32)
    u = torch.rand(n, 16, 2, generator=g)
    a, toks = D.verify_sample(draft.cuda(), tl.cuda(), dl.cuda(), u.cuda(), 1.0)
    first = toks[:, 0].cpu().numpy()
    p = torch.softmax(tl1.to(torch.bfloat16).double(), -1)[0].numpy()
    counts = np.bincount(first, minlength=V)
    assert chisquare(counts, p * n).pvalue > 1e-3



# ---------------------------------------------------------------- min-p stop
@pytest.mark.parametrize("S,V,T", [(1, 151936, 1.0), (3, 4096, 0.7), (2, 136, 2.0)])
def test_draft_stop_vs_oracle(S, V, T):
    """Confidence (top-1 softmax probability) within 1e-4 relative of the
    oracle on the same bf16 logits; stop lengths exact, except where an
    oracle confidence sits within that tolerance of min-p (counted)."""
    import block_diffusion_speculative_tap_gb300 as D

    g = torch.Generator().manual_seed(4100 + V)
    # peaked rows so that confidences spread over (0, 1)
    logits = torch.randn(S * 15, V, generator=g) * 2.0
    hot = torch.randint(0, V, (S * 15,), generator=g)
    lift = torch.rand(S * 15, generator=g) * 14.0
    logits[torch.arange(S * 15), hot] += lift
    logits = logits.to(torch.bfloat16)
    conf_ref = O.draft_confidence(logits.float().numpy().astype(np.float64), T)
    min_p = float(np.median(conf_ref))
    conf, lens = D.draft_stop(logits.cuda(), min_p, temperature=T)
    conf = conf.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(conf - conf_ref) <= 1e-4 * conf_ref), np.max(np.abs(conf - conf_ref) / conf_ref)
    want = O.draft_stop(conf_ref.reshape(S, 15), min_p)
    got = lens.cpu().numpy()
    near = 0
    for s in range(S):
        row = conf_ref.reshape(S, 15)[s]
        # the rule's decision at each inspected row must be clear of the tolerance
        n_clear = True
        for i in range(min(int(want[s]) + 1, 15)):
            if abs(row[i] - min_p) <= 1e-4 * row[i]:
                n_clear = False
        if n_clear:
            assert got[s] == want[s], (s, got[s], want[s])
        else:
            near += 1
    assert near < S or S == 1


def test_draft_stop_rejects_bad_arguments():
    import block_diffusion_speculative_tap_gb300 as D

    x = torch.zeros(15, 136, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(D.DFlashError):
        D.draft_stop(x, 1.5)
    with pytest.raises(D.DFlashError):
        D.draft_stop(x, 0.5, temperature=0.0)
    conf, lens = D.draft_stop(x, 0.5)
    torch.cuda.synchronize()
    assert abs(float(conf[0]) - 1.0 / 136) < 1e-6 and int(lens[0]) == 0
