"""Pins for the oracle's restricted-sampling verify (per-sequence temperature,
top-k and top-p: the serving variants of "Speculative Decoding and
Distillation" (Kadimisetty notes), "Greedy vs sampling"), against what the
pages and the mathematics fix. The oracle is called as a black box.

* Exact enumeration: with drafts drawn from the restricted draft
  distribution q', the emitted sequence is distributed exactly as
  autoregressive sampling from the restricted target p' -- the exactness of
  speculative sampling (Leviathan et al. explainer; Kadimisetty notes "Why
  it's exact") holds for any pair of distributions.
* top-k = 1 is greedy decoding: the restricted verify equals the greedy
  oracle (itself pinned against numpy.argmax) for any draft tokens.
* No restriction (k = V, p = 1) equals the lossless verify.
* The restricted distribution of a row against numpy: a stable sort, a
  cumulative sum, the cut at p and the renormalisation.
* Per-sequence temperatures equal single-temperature runs of the subsets.
* Planted mistakes in copies of the oracle source must fail these pins.
"""
import itertools
import os
import subprocess
from collections import defaultdict

import numpy as np
import pytest
from scipy.special import softmax

from test_oracle_pins import ENCODERS, accept_threshold, as_f64, draw_distribution, toy_table


def numpy_restricted(row, T, k, p):
    """The restricted distribution written out with numpy."""
    l = as_f64(row)
    V = l.shape[0]
    order = np.argsort(-l, kind="stable")[:min(k, V)]
    w = np.exp(l[order] / T - l[order[0]] / T)
    c = np.cumsum(w) / w.sum()
    m = int(np.searchsorted(c, p, side="left")) + 1   # first prefix reaching p
    m = min(m, len(order))
    out = np.zeros(V)
    out[order[:m]] = w[:m] / w[:m].sum()
    return out


@pytest.mark.parametrize("V,T,k,p,dtype", [(50, 1.0, 5, 1.0, "fp32"), (50, 0.7, 10, 0.8, "fp32"),
                                           (300, 1.3, 32, 0.9, "bf16"), (7, 1.0, 7, 0.5, "fp32"),
                                           (9, 0.5, 1, 1.0, "bf16"), (40, 1.0, 40, 0.999, "fp32")])
def test_restricted_row_against_numpy(oracle_mod, V, T, k, p, dtype):
    rng = np.random.default_rng(V + k)
    for trial in range(20):
        row = ENCODERS[dtype](2.0 * rng.standard_normal(V))
        rc, prob = oracle_mod.restricted_row(row, T, k, p)
        assert rc == 0
        np.testing.assert_allclose(prob, numpy_restricted(row, T, k, p), rtol=1e-12, atol=1e-15)
    # ties (a few distinct values): lower index first
    row = ENCODERS[dtype](rng.integers(0, 3, V).astype(np.float64))
    rc, prob = oracle_mod.restricted_row(row, T, k, p)
    np.testing.assert_allclose(prob, numpy_restricted(row, T, k, p), rtol=1e-12, atol=1e-15)


def restricted_step(oracle_mod, p_of, q_of, prefix, gamma, V, T, k, pp, enc):
    """Exact distribution of the block a restricted verify step emits after
    `prefix`, with draft tokens drawn from the restricted q'."""
    out = defaultdict(float)
    for x in itertools.product(range(V), repeat=gamma):
        qprob = 1.0
        for i in range(gamma):
            qprob *= oracle_mod.restricted_row(enc(q_of(prefix + list(x[:i]))), T, k, pp)[1][x[i]]
        if qprob == 0.0:
            continue
        p_rows = np.stack([enc(p_of(prefix + list(x[:i]))) for i in range(gamma + 1)])
        q_rows = np.stack([enc(q_of(prefix + list(x[:i]))) for i in range(gamma)])
        call = oracle_mod.RestrictedSeqCaller(p_rows, q_rows, list(x), T, k, pp)
        theta = [accept_threshold(call, i, gamma) for i in range(gamma)]
        reach = 1.0
        for j in range(gamma + 1):
            pj = reach * ((1.0 - theta[j]) if j < gamma else 1.0)
            if pj > 0.0:
                dist = draw_distribution(call, j, gamma, V)
                for t in range(V):
                    if dist[t] > 0.0:
                        out[tuple(x[:j]) + (t,)] += qprob * pj * dist[t]
            if j < gamma:
                reach *= theta[j]
    return out


@pytest.mark.parametrize("V,gamma,L,T,k,pp,dtype", [(4, 2, 3, 1.0, 3, 1.0, "fp32"),
                                                    (5, 1, 2, 0.8, 4, 0.7, "fp32"),
                                                    (4, 2, 3, 1.2, 2, 0.9, "bf16")])
def test_restricted_enumeration_output_is_restricted_target(oracle_mod, V, gamma, L, T, k, pp,
                                                            dtype):
    enc = ENCODERS[dtype]
    p_of = toy_table(5, V, 1.5)
    q_of = toy_table(6, V, 1.5)
    memo = {}
    got = defaultdict(float)

    def expand(prefix, prob):
        if len(prefix) >= L:
            got[tuple(prefix[:L])] += prob
            return
        key = tuple(prefix)
        if key not in memo:
            memo[key] = restricted_step(oracle_mod, p_of, q_of, list(prefix), gamma, V, T, k, pp,
                                        enc)
        for block, pb in memo[key].items():
            expand(list(prefix) + list(block), prob * pb)

    expand([], 1.0)
    want = {}
    for y in itertools.product(range(V), repeat=L):
        pr = 1.0
        for j in range(L):
            pr *= numpy_restricted(enc(p_of(list(y[:j]))), T, k, pp)[y[j]]
        want[y] = pr
    assert abs(sum(got.values()) - 1.0) < 1e-12
    err = max(abs(got.get(y, 0.0) - want[y]) for y in want)
    assert err < 1e-12, err


def _random_batch(rng, B, gm, V, dtype="bf16", scale=2.0):
    g = rng.integers(0, gm + 1, B).astype(np.int32)
    tgt = ENCODERS[dtype](scale * rng.standard_normal((int((g + 1).sum()), V)))
    dft = ENCODERS[dtype](scale * rng.standard_normal((max(int(g.sum()), 1), V)))
    p_off = (np.cumsum(g + 1) - (g + 1)).astype(np.int64)
    q_off = (np.cumsum(g) - g).astype(np.int64)
    return g, tgt, dft, p_off, q_off


def test_top1_is_greedy_decoding(oracle_mod):
    rng = np.random.default_rng(81)
    B, gm, V = 60, 5, 400
    g, tgt, dft, p_off, q_off = _random_batch(rng, B, gm, V)
    x = rng.integers(0, V, (B, gm)).astype(np.int32)
    # many drafts agree with the target argmax, so that long prefixes occur
    for b in range(B):
        for i in range(g[b]):
            if rng.random() < 0.7:
                x[b, i] = int(np.argmax(as_f64(tgt[p_off[b] + i])))
    res = oracle_mod.verify_batch_restricted(tgt, dft, p_off, q_off, x, g, 0.8, 1, seed=3)
    greedy = oracle_mod.verify_batch(tgt, None, p_off, None, x, g, 0.0)
    assert res["rc"] == 0
    np.testing.assert_array_equal(res["n"], greedy["n"])
    np.testing.assert_array_equal(res["tokens"], greedy["tokens"])
    assert (res["n"] > 0).any()


def test_no_restriction_equals_lossless_verify(oracle_mod):
    rng = np.random.default_rng(83)
    B, gm, V, T = 50, 4, 300, 0.9
    g, tgt, dft, p_off, q_off = _random_batch(rng, B, gm, V, dtype="fp32")
    x = rng.integers(0, V, (B, gm)).astype(np.int32)
    for seed in range(4):
        res = oracle_mod.verify_batch_restricted(tgt, dft, p_off, q_off, x, g, T, V, 1.0,
                                                 seed=seed)
        ref = oracle_mod.verify_batch(tgt, dft, p_off, q_off, x, g, T, seed=seed)
        np.testing.assert_array_equal(res["n"], ref["n"])
        np.testing.assert_array_equal(res["tokens"], ref["tokens"])


def test_per_sequence_parameters_match_single_runs(oracle_mod):
    rng = np.random.default_rng(85)
    B, gm, V = 30, 4, 200
    g, tgt, dft, p_off, q_off = _random_batch(rng, B, gm, V)
    x = rng.integers(0, V, (B, gm)).astype(np.int32)
    T = rng.choice([0.5, 0.9, 1.4], B)
    k = rng.choice([1, 4, 16, 32], B).astype(np.int32)
    pp = rng.choice([0.6, 0.95, 1.0], B)
    res = oracle_mod.verify_batch_restricted(tgt, dft, p_off, q_off, x, g, T, k, pp, seed=7)
    assert res["rc"] == 0
    for b in range(B):
        one = oracle_mod.verify_batch_restricted(
            tgt[p_off[b]:p_off[b] + g[b] + 1], dft[q_off[b]:q_off[b] + max(g[b], 1)], [0], [0],
            x[b:b + 1], g[b:b + 1], T[b], k[b], pp[b], seed=7, seq_ids=[b])
        assert one["n"][0] == res["n"][b]
        np.testing.assert_array_equal(one["tokens"][0], res["tokens"][b])
        # the final token has positive restricted target probability
        n = res["n"][b]
        prob = numpy_restricted(tgt[p_off[b] + n], T[b], k[b], pp[b])
        assert prob[res["tokens"][b][n]] > 0.0


def test_restricted_rejects_bad_parameters(oracle_mod):
    rng = np.random.default_rng(87)
    g, tgt, dft, p_off, q_off = _random_batch(rng, 4, 2, 50)
    x = rng.integers(0, 50, (4, 2)).astype(np.int32)
    res = oracle_mod.verify_batch_restricted(tgt, dft, p_off, q_off, x, g, [1.0, 0.0, 1.0, 1.0],
                                             [4, 4, 0, 4], [1.0, 1.0, 1.0, 1.5], seed=1)
    assert res["n"][0] >= 0 and list(res["n"][1:]) == [-1, -1, -1]


MUTANTS = {
    "residual_not_p_minus_q": ("                w[v] = fmax(0.0, pp[v] - qq[v]);\n                R += w[v];\n            }\n            if (!(R > 0.0))  /* zero residual mass through rounding: draw from p' */",
                               "                w[v] = fmax(0.0, pp[v]);\n                R += w[v];\n            }\n            if (!(R > 0.0))  /* zero residual mass through rounding: draw from p' */"),
    "ratio_inverted": ("        double ratio = qv > 0.0 ? pv / qv : (pv > 0.0 ? INFINITY : 0.0);",
                       "        double ratio = pv > 0.0 ? qv / pv : (qv > 0.0 ? INFINITY : 0.0);"),
    "topk_ties_to_higher_index": ("        while (at > 0 && l > logit_at(row, dtype, idx[at - 1])) {\n            idx[at] = idx[at - 1];\n            --at;\n        }\n        idx[at] = v;\n        if (kept < k) ++kept;\n    }\n    double l0",
                                  "        while (at > 0 && l >= logit_at(row, dtype, idx[at - 1])) {\n            idx[at] = idx[at - 1];\n            --at;\n        }\n        idx[at] = v;\n        if (kept < k) ++kept;\n    }\n    double l0"),
    "top_p_not_renormalised": ("    for (int32_t j = 0; j < m; ++j) prob[idx[j]] = w[j] / z;",
                               "    for (int32_t j = 0; j < m; ++j) prob[idx[j]] = w[j] / total;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_restricted_pins_catch_planted_mistakes(oracle_mod, tmp_path, monkeypatch, name):
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "specverify_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o",
                    str(so), str(mpath), "-lm", "-lpthread"], check=True)
    monkeypatch.setattr(oracle_mod, "_lib", oracle_mod.load_variant(str(so)))
    failed = False
    try:
        if name in ("topk_ties_to_higher_index", "top_p_not_renormalised"):
            test_restricted_row_against_numpy(oracle_mod, 50, 0.7, 10, 0.8, "fp32")
            test_restricted_row_against_numpy(oracle_mod, 300, 1.3, 32, 0.9, "bf16")
        else:
            test_restricted_enumeration_output_is_restricted_target(oracle_mod, 4, 2, 3, 1.0, 3,
                                                                    1.0, "fp32")
    except AssertionError:
        failed = True
    assert failed, name
