"""Pins for the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own arithmetic: the oracle is called as a
black box (its decisions integrated exactly over the uniforms by bisection),
and the result is compared with the *goal* of the method -- sampling from the
target -- or with closed forms, library routines and worked examples printed
on the pages:

* exact enumeration: the emitted-token sequence is distributed exactly as
  autoregressive sampling from p, for arbitrary q ("the output distribution is
  the same as sampling from the target model alone, for any approximation
  model" -- Leviathan et al. explainer; "Why it's exact" -- Kadimisetty notes);
* acceptance probability = sum_x min(p, q) = 1 - TVD(p, q) (DistillSpec Sec. 3
  definition of beta and Sec. 4 "TVD as proxy for the acceptance rate");
* P(exactly i accepted) = alpha^i - alpha^(i+1), P(all gamma) = alpha^gamma
  (CS Drafting summary App. C.1);
* greedy = longest prefix agreeing with argmax p, plus the target argmax
  (Kadimisetty notes, "Greedy vs sampling") -- against numpy.argmax;
* gamma = 0 reduces to an inverse-CDF draw from p_1 -- against
  numpy.cumsum + numpy.searchsorted;
* q = p always accepts (Kadimisetty notes step 3: p >= q is always accepted);
* lse against scipy.special.logsumexp;
* 1 <= emitted <= gamma + 1 (Leviathan et al. explainer);
* worked examples printed on the pages (tests/golden/worked_examples.json).
"""
import itertools
import json
import math
import os
from collections import defaultdict

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "worked_examples.json")))


def bf16_bits(a):
    """Round float32 values to bf16 (round-to-nearest-even) and return the bits."""
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def as_f64(rows):
    rows = np.asarray(rows)
    if rows.dtype == np.uint16:
        return (rows.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return rows.astype(np.float64)


def probs(row, T):
    return softmax(as_f64(row) / T)


# --------------------------------------------------------------------------
# exact integration of the oracle's decisions over its uniforms

def _bisect(pred, iters=62):
    """pred(0) False, pred(1) True, monotone: returns inf{x: pred(x)}."""
    lo, hi = 0.0, 1.0
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if pred(mid):
            hi = mid
        else:
            lo = mid
    return hi


def accept_threshold(call, i, gamma):
    """P(position i is accepted | positions < i accepted) = sup{r: accepted}."""
    r = [0.0] * gamma

    def rejected(rv):
        r[i] = rv
        n, _ = call.run(r, 0.5)
        return n == i

    if not rejected(1.0):
        return 1.0
    return _bisect(rejected)


def draw_distribution(call, j, gamma, V):
    """Distribution of the final token given n = j, integrating u over [0,1)."""
    r = [0.0] * gamma
    if j < gamma:
        r[j] = 1.0

    def tok(u):
        n, toks = call.run(r, u)
        assert n == j
        return toks[j]

    last = 1.0 - 2.0**-53
    bounds = [0.0]
    for k in range(1, V):
        if tok(0.0) >= k:
            bounds.append(0.0)
        elif tok(last) < k:
            bounds.append(1.0)
        else:
            bounds.append(_bisect(lambda u: tok(u) >= k))
    bounds.append(1.0)
    return np.diff(np.array(bounds))


def step_distribution(oracle_mod, p_rows_of, q_rows_of, prefix, gamma, V, T, enc, lib=None):
    """Exact distribution of the block a verify step emits after `prefix`."""
    out = defaultdict(float)
    for x in itertools.product(range(V), repeat=gamma):
        qprob = 1.0
        for i in range(gamma):
            qprob *= probs(enc(q_rows_of(prefix + list(x[:i]))), T)[x[i]]
        if qprob == 0.0:
            continue
        p_rows = np.stack([enc(p_rows_of(prefix + list(x[:i]))) for i in range(gamma + 1)])
        q_rows = (np.stack([enc(q_rows_of(prefix + list(x[:i]))) for i in range(gamma)])
                  if gamma else None)
        call = oracle_mod.SeqCaller(p_rows, q_rows, list(x), T, lib=lib)
        theta = [accept_threshold(call, i, gamma) for i in range(gamma)]
        reach = 1.0
        for j in range(gamma + 1):
            pj = reach * ((1.0 - theta[j]) if j < gamma else 1.0)
            if pj > 0.0:
                dist = draw_distribution(call, j, gamma, V)
                for k in range(V):
                    if dist[k] > 0.0:
                        out[tuple(x[:j]) + (k,)] += qprob * pj * dist[k]
            if j < gamma:
                reach *= theta[j]
    return out


def toy_table(tag, V, scale, neg_inf=False):
    def rows_of(prefix):
        rng = np.random.default_rng([tag, len(prefix)] + [t + 1 for t in prefix])
        l = (scale * rng.standard_normal(V)).astype(np.float32)
        if neg_inf and rng.random() < 0.5:
            l[rng.integers(V)] = -np.inf
        return l
    return rows_of


def sequence_distribution(oracle_mod, p_of, q_of, V, gamma, L, T, enc, lib=None):
    memo = {}
    dist = defaultdict(float)

    def expand(prefix, prob):
        if len(prefix) >= L:
            dist[tuple(prefix[:L])] += prob
            return
        key = tuple(prefix)
        if key not in memo:
            memo[key] = step_distribution(oracle_mod, p_of, q_of, list(prefix), gamma, V, T, enc,
                                          lib=lib)
        for block, pb in memo[key].items():
            expand(list(prefix) + list(block), prob * pb)

    expand([], 1.0)
    return dist


def target_sequence_distribution(p_of, V, L, T, enc):
    out = {}
    for y in itertools.product(range(V), repeat=L):
        pr = 1.0
        for j in range(L):
            pr *= probs(enc(p_of(list(y[:j]))), T)[y[j]]
        out[y] = pr
    return out


ENCODERS = {"fp32": lambda a: np.asarray(a, np.float32), "bf16": bf16_bits}


@pytest.mark.parametrize("V,gamma,L,T,dtype,q_kind", [
    (3, 2, 3, 1.0, "fp32", "unrelated"),
    (2, 3, 4, 0.7, "fp32", "noisy"),
    (3, 2, 3, 0.7, "bf16", "noisy_neginf"),
    (4, 1, 2, 1.3, "fp32", "unrelated"),
])
def test_exact_enumeration_output_is_target_distribution(oracle_mod, V, gamma, L, T, dtype,
                                                         q_kind):
    enc = ENCODERS[dtype]
    p_of = toy_table(11, V, 1.5, neg_inf=q_kind.endswith("neginf"))
    if q_kind == "unrelated":
        q_of = toy_table(23, V, 2.0)
    else:
        noise = toy_table(37, V, 0.8)

        def q_of(prefix):
            return p_of(prefix) + noise(prefix) if not q_kind.endswith("neginf") else \
                np.where(np.isfinite(p_of(prefix)), p_of(prefix) + noise(prefix), 0.0)
    got = sequence_distribution(oracle_mod, p_of, q_of, V, gamma, L, T, enc)
    want = target_sequence_distribution(p_of, V, L, T, enc)
    assert abs(sum(got.values()) - 1.0) < 1e-12
    err = max(abs(got.get(y, 0.0) - want[y]) for y in want)
    assert err < 1e-12, err


def test_single_position_acceptance_is_sum_of_min(oracle_mod):
    rng = np.random.default_rng(3)
    for V, T in [(5, 1.0), (6, 0.6), (8, 1.7)]:
        lp = (1.3 * rng.standard_normal(V)).astype(np.float32)
        lq = (1.3 * rng.standard_normal(V)).astype(np.float32)
        pp, qq = probs(lp, T), probs(lq, T)
        acc = 0.0
        for x in range(V):
            call = oracle_mod.SeqCaller(np.stack([lp, lp]), lq[None, :], [x], T)
            acc += qq[x] * accept_threshold(call, 0, 1)
        beta = np.minimum(pp, qq).sum()
        assert abs(acc - beta) < 1e-13
        assert abs(acc - (1.0 - 0.5 * np.abs(pp - qq).sum())) < 1e-13


def test_accept_count_law_iid(oracle_mod):
    """Identical rows at every position: P(n = i) = a^i (1 - a), P(n = g) = a^g."""
    rng = np.random.default_rng(9)
    V, gamma, T = 4, 3, 1.0
    lp = (1.2 * rng.standard_normal(V)).astype(np.float32)
    lq = (1.2 * rng.standard_normal(V)).astype(np.float32)
    pp, qq = probs(lp, T), probs(lq, T)
    alpha = np.minimum(pp, qq).sum()
    pn = np.zeros(gamma + 1)
    for x in itertools.product(range(V), repeat=gamma):
        call = oracle_mod.SeqCaller(np.stack([lp] * (gamma + 1)), np.stack([lq] * gamma),
                                    list(x), T)
        th = [accept_threshold(call, i, gamma) for i in range(gamma)]
        w = np.prod([qq[t] for t in x])
        reach = 1.0
        for j in range(gamma):
            pn[j] += w * reach * (1 - th[j])
            reach *= th[j]
        pn[gamma] += w * reach
    law = [alpha**i - alpha**(i + 1) for i in range(gamma)] + [alpha**gamma]
    np.testing.assert_allclose(pn, law, rtol=0, atol=1e-13)
    # and the expected emitted count matches the oracle's closed form
    assert abs((pn * np.arange(1, gamma + 2)).sum()
               - oracle_mod.block_efficiency(alpha, gamma)) < 1e-12


def test_expected_emitted_non_iid_matches_enumeration(oracle_mod):
    rng = np.random.default_rng(13)
    V, gamma, T = 3, 3, 0.9
    lps = (1.1 * rng.standard_normal((gamma + 1, V))).astype(np.float32)
    lqs = (1.1 * rng.standard_normal((gamma, V))).astype(np.float32)
    beta = [np.minimum(probs(lps[i], T), probs(lqs[i], T)).sum() for i in range(gamma)]
    e = 0.0
    for x in itertools.product(range(V), repeat=gamma):
        call = oracle_mod.SeqCaller(lps, lqs, list(x), T)
        th = [accept_threshold(call, i, gamma) for i in range(gamma)]
        w = np.prod([probs(lqs[i], T)[x[i]] for i in range(gamma)])
        reach = 1.0
        for j in range(gamma + 1):
            pj = reach * ((1 - th[j]) if j < gamma else 1.0)
            e += w * pj * (j + 1)
            if j < gamma:
                reach *= th[j]
    assert abs(e - oracle_mod.expected_emitted(beta)) < 1e-12


def test_golden_rule_of_thumb_and_geometric_series(oracle_mod):
    g = GOLDEN["rule_of_thumb_block_efficiency"]
    tau = oracle_mod.block_efficiency(g["alpha"], g["k"])
    assert abs(tau - g["tokens_per_pass"]) <= 0.5
    assert abs(tau - sum(g["alpha"]**i for i in range(g["k"] + 1))) < 1e-12
    assert oracle_mod.block_efficiency(1.0, 5) == 6.0
    for a in GOLDEN["accept_count_law"]["alphas"]:
        law = [a**i - a**(i + 1) for i in range(7)] + [a**7]
        assert abs(sum(law) - 1.0) < 1e-12


def test_golden_disco_figure_1(oracle_mod):
    """SL = 5: t1..t3 accepted, t4 rejected -> 3 drafts + 1 corrected token."""
    g = GOLDEN["disco_figure_1"]
    rng = np.random.default_rng(21)
    V, gamma, T = 7, g["gamma"], 1.0
    p = (rng.standard_normal((gamma + 1, V))).astype(np.float32)
    q = p[:gamma].copy()
    x = [int(np.argmax(q[i])) for i in range(gamma)]
    p[3, x[3]] = -np.inf          # the target gives t4 no mass: always rejected
    q[4] += rng.standard_normal(V).astype(np.float32)
    for seed in range(50):
        r = [oracle_mod.accept_uniform(seed, 0, i + 1) for i in range(gamma)]
        res = oracle_mod.verify_seq_u(p, q, x, T, r, oracle_mod.draw_uniform(seed, 0, 4))
        assert res["n"] == g["accepted"]
        emitted = res["tokens"][res["tokens"] >= 0]
        assert len(emitted) == g["emitted"]
        assert list(emitted[:3]) == x[:3] and emitted[3] != x[3]


def test_q_equal_p_accepts_everything(oracle_mod):
    rng = np.random.default_rng(4)
    for dtype in ["fp32", "bf16"]:
        enc = ENCODERS[dtype]
        p = enc(rng.standard_normal((6, 50)) * 3)
        x = rng.integers(0, 50, 5)
        for s in range(20):
            r = [oracle_mod.accept_uniform(s, 0, i + 1) for i in range(5)]
            res = oracle_mod.verify_seq_u(p, p[:5], x, 0.8, r, 0.3)
            assert res["n"] == 5 and list(res["tokens"][:5]) == list(x)


def test_gamma_zero_is_inverse_cdf_of_p(oracle_mod):
    rng = np.random.default_rng(8)
    for V, T, dtype in [(1000, 1.0, "fp32"), (777, 0.7, "bf16"), (5, 2.0, "fp32")]:
        enc = ENCODERS[dtype]
        row = enc(rng.standard_normal(V) * 2.5)
        c = np.cumsum(probs(row, T))
        checked = 0
        for u in rng.random(300):
            res = oracle_mod.verify_seq_u(row[None, :], None, [], T, [], float(u))
            assert res["n"] == 0
            want = int(np.searchsorted(c, u * c[-1], side="right"))
            if res["draw_margin"] > 1e-9:
                assert res["tokens"][0] == want
                checked += 1
            assert res["tokens"][1:].tolist() == []
        assert checked > 250


def test_zero_mass_tokens_are_never_emitted(oracle_mod):
    rng = np.random.default_rng(12)
    V = 9
    p = rng.standard_normal((3, V)).astype(np.float32)
    p[:, [2, 5]] = -np.inf
    q = rng.standard_normal((2, V)).astype(np.float32)
    x = [0, 1]
    for s in range(300):
        r = [oracle_mod.accept_uniform(s, 0, i + 1) for i in range(2)]
        res = oracle_mod.verify_seq_u(p, q, x, 1.0, r, oracle_mod.draw_uniform(s, 0, 1))
        n = res["n"]
        assert res["tokens"][n] not in (2, 5)


def test_lse_matches_scipy(oracle_mod):
    rng = np.random.default_rng(2)
    for V, T in [(1, 1.0), (17, 0.3), (32000, 0.8), (5000, 2.0)]:
        row = (rng.standard_normal(V) * 4).astype(np.float32)
        want = logsumexp(row.astype(np.float64) / T)
        assert abs(oracle_mod.row_lse(row, T) - want) <= 1e-13 * max(1.0, abs(want))
    row = np.array([-np.inf, 0.5, -np.inf], np.float32)
    assert abs(oracle_mod.row_lse(row, 0.5) - 1.0) < 1e-15
    assert oracle_mod.row_lse(np.array([-np.inf, -np.inf], np.float32), 1.0) is None
    assert oracle_mod.row_lse(np.array([0.0, np.nan], np.float32), 1.0) is None
    assert oracle_mod.row_lse(np.array([0.0, np.inf], np.float32), 1.0) is None


def test_acceptance_margins_are_distance_to_p_over_q(oracle_mod):
    rng = np.random.default_rng(17)
    V, gamma, T = 30, 4, 0.9
    p = (2 * rng.standard_normal((gamma + 1, V))).astype(np.float32)
    q = (2 * rng.standard_normal((gamma, V))).astype(np.float32)
    x = rng.integers(0, V, gamma)
    r = [0.0, 0.0, 0.0, 0.0]
    res = oracle_mod.verify_seq_u(p, q, x, T, r, 0.5)
    assert res["n"] == gamma
    for i in range(gamma):
        ratio = probs(p[i], T)[x[i]] / probs(q[i], T)[x[i]]
        assert abs(res["acc_margin"][i] - ratio) < 1e-12 * max(1.0, ratio)


def _greedy_closed_form(p_rows, x):
    a = [int(np.argmax(as_f64(r))) for r in p_rows]
    n = 0
    while n < len(x) and x[n] == a[n]:
        n += 1
    return n, a[:n + 1]


def test_greedy_is_argmax_decoding(oracle_mod):
    rng = np.random.default_rng(6)
    for trial in range(200):
        V = int(rng.integers(1, 40))
        gamma = int(rng.integers(0, 6))
        dtype = "bf16" if trial % 2 else "fp32"
        raw = np.round(rng.standard_normal((gamma + 1, V)) * 2, 1 if trial % 3 else 0)
        rows = ENCODERS[dtype](raw)                      # coarse values: many ties
        a = [int(np.argmax(as_f64(r))) for r in rows]
        x = [a[i] if rng.random() < 0.6 else int(rng.integers(V)) for i in range(gamma)]
        res = oracle_mod.verify_greedy_seq(rows, x)
        n, toks = _greedy_closed_form(rows, x)
        assert res["n"] == n
        assert list(res["tokens"][:n + 1]) == toks
        assert all(t == -1 for t in res["tokens"][n + 1:])


def test_batch_invariants_and_bad_inputs(oracle_mod):
    rng = np.random.default_rng(10)
    B, gm, V, T = 40, 6, 300, 0.8
    g = rng.integers(0, gm + 1, B).astype(np.int32)
    p_off = np.cumsum(g + 1) - (g + 1)
    q_off = np.cumsum(g) - g
    tgt = (2 * rng.standard_normal((int((g + 1).sum()), V))).astype(np.float32)
    dft = (2 * rng.standard_normal((max(int(g.sum()), 1), V))).astype(np.float32)
    toks = rng.integers(0, V, (B, gm)).astype(np.int32)
    # bad inputs in three sequences
    g_bad = g.copy()
    g_bad[3] = gm + 1
    toks[5, 0] = V if g[5] > 0 else toks[5, 0]
    tgt[p_off[7], 11] = np.nan
    for T_run in (T, 0.0):
        res = oracle_mod.verify_batch(tgt, dft if T_run > 0 else None, p_off, q_off, toks, g_bad,
                                      T_run, seed=1234)
        assert res["rc"] == oracle_mod.ERR_INPUT
        for b in range(B):
            n = res["n"][b]
            bad = b == 3 or (b == 5 and g[5] > 0) or b == 7
            if bad:
                assert n == -1 and (res["tokens"][b] == -1).all()
                continue
            assert 0 <= n <= g[b]                       # 1 <= emitted <= gamma + 1
            assert list(res["tokens"][b][:n]) == list(toks[b][:n])
            assert 0 <= res["tokens"][b][n] < V
            assert (res["tokens"][b][n + 1:] == -1).all()


def test_batch_seq_ids_reproduce_subsets(oracle_mod):
    rng = np.random.default_rng(14)
    B, gm, V, T = 12, 3, 64, 1.0
    g = np.full(B, gm, np.int32)
    tgt = (2 * rng.standard_normal((B * (gm + 1), V))).astype(np.float32)
    dft = (2 * rng.standard_normal((B * gm, V))).astype(np.float32)
    toks = rng.integers(0, V, (B, gm)).astype(np.int32)
    p_off = np.arange(B) * (gm + 1)
    q_off = np.arange(B) * gm
    full = oracle_mod.verify_batch(tgt, dft, p_off, q_off, toks, g, T, seed=77)
    sub = [2, 9, 10]
    rows_p = np.concatenate([np.arange(p_off[b], p_off[b] + gm + 1) for b in sub])
    rows_q = np.concatenate([np.arange(q_off[b], q_off[b] + gm) for b in sub])
    part = oracle_mod.verify_batch(tgt[rows_p], dft[rows_q], np.arange(3) * (gm + 1),
                                   np.arange(3) * gm, toks[sub], g[sub], T, seed=77,
                                   seq_ids=sub)
    assert (part["n"] == full["n"][sub]).all()
    assert (part["tokens"] == full["tokens"][sub]).all()


def test_monte_carlo_first_token_is_p1_and_acceptance_is_beta(oracle_mod):
    """Seeded (Philox) path: the first emitted token ~ p_1 for any q."""
    from scipy import stats
    rng = np.random.default_rng(31)
    V, gamma, T, B = 6, 2, 1.0, 200_000
    p = (1.0 * rng.standard_normal((gamma + 1, V))).astype(np.float32)
    q = (1.0 * rng.standard_normal((gamma, V))).astype(np.float32)
    qq = probs(q[0], T)
    # each sequence draws its own draft tokens from q (the drafter), shares rows
    x = np.stack([rng.choice(V, B, p=probs(q[i], T)) for i in range(gamma)], 1).astype(np.int32)
    res = oracle_mod.verify_batch(p, q, np.zeros(B, np.int64), np.zeros(B, np.int64), x,
                                  np.full(B, gamma, np.int32), T, seed=2024)
    assert res["rc"] == 0
    first = res["tokens"][:, 0]
    counts = np.bincount(first, minlength=V)
    pp = probs(p[0], T)
    assert stats.chisquare(counts, B * pp).pvalue > 1e-4
    beta = np.minimum(pp, qq).sum()
    acc = (res["n"] >= 1).mean()
    assert abs(acc - beta) < 5 * math.sqrt(beta * (1 - beta) / B)


# --------------------------------------------------------------------------
# planted mistakes: copies of the oracle source with one plausible error each
# must FAIL the enumeration pin (the mistakes live only in temporary builds)

MUTANTS = {
    "residual_sign": ("p * fmax(0.0, -expm1(log_q - log_p))", "p * fmax(0.0, -expm1(log_p - log_q))"),
    "ratio_inverted": ("double ratio = exp(lenient_log(log_p, len_kind, eps) - log_q);",
                       "double ratio = exp(log_q - lenient_log(log_p, len_kind, eps));"),
    "temperature_only_on_p": ("double log_q = logit_at(qr, dtype, x[i]) / T - lse_q[i];",
                              "double log_q = logit_at(qr, dtype, x[i]) - lse_q[i];"),
    "residual_row_off_by_one": ("const void *q_row = (n < gamma) ? row_ptr(q_rows, n, row_stride, dtype) : NULL;",
                                "const void *q_row = (n < gamma) ? row_ptr(q_rows, n > 0 ? n - 1 : 0, row_stride, dtype) : NULL;"),
    "bonus_from_first_row": ("const void *p_row = row_ptr(p_rows, n, row_stride, dtype);",
                             "const void *p_row = row_ptr(p_rows, n < gamma ? n : 0, row_stride, dtype);"),
    "cdf_offset": ("if (c_k > t) { k = v; break; }\n    }\n    if (k < 0) {\n        /* t at or past",
                   "if (c_k > t) { k = v > 0 ? v - 1 : v; break; }\n    }\n    if (k < 0) {\n        /* t at or past"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_enumeration_pin_catches_planted_mistakes(oracle_mod, tmp_path, name):
    import subprocess
    src_path = os.path.join(os.path.dirname(oracle_mod.__file__), "specverify_oracle.c")
    src = open(src_path).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o",
                    str(so), str(mpath), "-lm", "-lpthread"], check=True)
    lib = oracle_mod.load_variant(str(so))
    V, gamma, L, T = 3, 2, 3, 0.7
    p_of = toy_table(11, V, 1.5)
    noise = toy_table(37, V, 0.8)

    def q_of(prefix):
        return p_of(prefix) + noise(prefix)
    enc = ENCODERS["fp32"]
    got = sequence_distribution(oracle_mod, p_of, q_of, V, gamma, L, T, enc, lib=lib)
    want = target_sequence_distribution(p_of, V, L, T, enc)
    err = max(abs(got.get(y, 0.0) - want[y]) for y in want)
    assert err > 1e-4, (name, err)


def _margin_by_cumsum(w, u):
    """The draw of the inverse CDF over weights w (token order) at t = u R,
    and its margin min(t - C_{k-1}, C_k - t) / R, from numpy's cumulative
    sum."""
    c = np.cumsum(w)
    R = c[-1]
    t = u * R
    k = int(np.searchsorted(c, t, side="right"))
    lo = c[k - 1] if k > 0 else 0.0
    return k, min(t - lo, c[k] - t) / R


def test_draw_margin_bonus_draw_matches_cumsum(oracle_mod):
    # gamma = 0: the final token is drawn from p_1 itself
    rng = np.random.default_rng(21)
    for V, T, dtype in [(64, 1.0, "fp32"), (300, 0.7, "bf16"), (7, 1.5, "fp32")]:
        row = ENCODERS[dtype](rng.standard_normal(V) * 2.0)
        w = probs(row, T)
        for u in rng.random(200):
            res = oracle_mod.verify_seq_u(row[None, :], None, [], T, [], float(u))
            k, m = _margin_by_cumsum(w, float(u))
            assert res["tokens"][0] == k
            assert res["draw_margin"] == pytest.approx(m, rel=1e-9, abs=1e-13)


def test_draw_margin_residual_draw_matches_cumsum(oracle_mod):
    # a rejection at position 1 (ratio below one half, uniform 0.75): the
    # final token comes from max(0, p_1 - q_1)
    rng = np.random.default_rng(22)
    V, T = 40, 0.9
    checked = 0
    for trial in range(200):
        p = rng.standard_normal((2, V)).astype(np.float32) * 2.0
        q = rng.standard_normal((1, V)).astype(np.float32) * 2.0
        pp, qq = probs(p[0], T), probs(q[0], T)
        ratio = pp / np.maximum(qq, 1e-300)
        x = int(np.argmin(ratio))
        if ratio[x] >= 0.5:
            continue
        u = float(rng.random())
        res = oracle_mod.verify_seq_u(p, q, [x], T, [0.75], u)
        assert res["n"] == 0
        k, m = _margin_by_cumsum(np.maximum(0.0, pp - qq), u)
        assert res["tokens"][0] == k
        assert res["draw_margin"] == pytest.approx(m, rel=1e-8, abs=1e-12)
        checked += 1
    assert checked > 150
