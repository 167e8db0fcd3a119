"""Pins for the oracle's lossy accept test, acceptance statistics and draft
features (the ranked next rows of the verify path), checked against what the
pages and the mathematics fix. The oracle is called as a black box.

* Lenience ("DistillSpec" Sec. 4 "DistillSpec with lossy SD"; App. A.3
  Algorithm A.1, the rejection threshold f(p_i(y), eps) / q_i(y) and the
  unchanged residual norm(max(0, p - q))): eps = 1 reproduces the lossless
  outputs bit for bit; the accept decisions integrated over the uniform give
  acceptance sum_x q(x) min(1, f(p(x), eps) / q(x)) for each f; the law of the
  emitted token follows Algorithm A.1 with the residual of p - q; the page's
  worked example (f_sq, eps = 0.1: a hundred times more likely to be
  accepted); acceptance grows as eps falls.
* beta = sum min(p, q) and TVD ("DistillSpec" Sec. 3 and Sec. 4): beta equals
  the acceptance of the oracle's own accept test integrated over its
  uniform; TVD against scipy's L1 distance; the special cases q = p and
  disjoint supports; the expected emitted count against a Monte Carlo run of
  the seeded verify.
* Draft features ("DISCO" Sec. 3 Eq. 2 and App. D.1): entropy against
  scipy.stats.entropy and closed forms; top-k against numpy's stable sort,
  ties to the lower index.
* Planted mistakes in copies of the oracle source must fail these pins.
"""
import json
import os
import subprocess

import numpy as np
import pytest
from scipy.spatial.distance import cityblock
from scipy.special import softmax
from scipy.stats import entropy as scipy_entropy

from test_oracle_pins import (ENCODERS, accept_threshold, as_f64, bf16_bits,
                              draw_distribution, probs)

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "worked_examples.json")))

# The lenience functions as the page defines them, on probabilities.
F = {
    "lin": lambda p, e: p / e,
    "sq": lambda p, e: p / e**2,
    "exp": lambda p, e: p**e,
}


def _rows(rng, V, scale=1.5, n=2, dtype="fp32"):
    return ENCODERS[dtype](scale * rng.standard_normal((n, V)))


# --------------------------------------------------------------------------
# lenience

@pytest.mark.parametrize("kind", ["lin", "sq", "exp"])
def test_lenience_eps_one_is_lossless_bit_for_bit(oracle_mod, kind):
    rng = np.random.default_rng(41)
    B, gm, V, T = 40, 4, 300, 0.8
    g = rng.integers(0, gm + 1, B).astype(np.int32)
    tgt = ENCODERS["bf16"](2.0 * rng.standard_normal((int((g + 1).sum()), V)))
    dft = ENCODERS["bf16"](2.0 * rng.standard_normal((max(int(g.sum()), 1), V)))
    p_off = (np.cumsum(g + 1) - (g + 1)).astype(np.int64)
    q_off = (np.cumsum(g) - g).astype(np.int64)
    x = rng.integers(0, V, (B, gm)).astype(np.int32)
    base = oracle_mod.verify_batch(tgt, dft, p_off, q_off, x, g, T, seed=5)
    got = oracle_mod.verify_batch(tgt, dft, p_off, q_off, x, g, T, seed=5, lenience=kind,
                                  eps=1.0)
    assert base["rc"] == got["rc"] == 0
    for key in ("n", "tokens", "acc_margin", "draw_margin"):
        np.testing.assert_array_equal(base[key], got[key])


@pytest.mark.parametrize("kind,eps", [("lin", 0.5), ("sq", 0.6), ("exp", 0.3), ("lin", 0.05),
                                      ("sq", 0.2), ("exp", 0.8)])
def test_lenient_acceptance_is_expected_min(oracle_mod, kind, eps):
    """One position: the accept decisions integrated over r give
    sum_x q(x) min(1, f(p(x), eps) / q(x))."""
    rng = np.random.default_rng(43)
    for V, T, dtype in [(5, 1.0, "fp32"), (7, 0.7, "bf16")]:
        lp, lq = _rows(rng, V, dtype=dtype)
        pp, qq = probs(lp, T), probs(lq, T)
        acc = 0.0
        for x in range(V):
            call = oracle_mod.SeqCaller(np.stack([lp, lp]), lq[None, :], [x], T,
                                        lenience=kind, eps=eps)
            acc += qq[x] * accept_threshold(call, 0, 1)
        want = float(np.sum(qq * np.minimum(1.0, F[kind](pp, eps) / qq)))
        assert abs(acc - want) < 1e-12, (kind, eps, acc, want)


@pytest.mark.parametrize("kind,eps", [("lin", 0.5), ("sq", 0.7), ("exp", 0.4)])
def test_lenient_emitted_token_law(oracle_mod, kind, eps):
    """Algorithm A.1 with lenience, one position: the emitted token is x with
    probability q(x) a(x), a = min(1, f(p, eps)/q), and otherwise drawn from
    norm(max(0, p - q)) -- the residual does not depend on the lenience."""
    rng = np.random.default_rng(47)
    V, T = 5, 0.9
    for trial in range(3):
        lp2 = _rows(rng, V, n=2)
        lq = _rows(rng, V, n=1)[0]
        pp, qq = probs(lp2[0], T), probs(lq, T)
        a = np.minimum(1.0, F[kind](pp, eps) / qq)
        res = np.maximum(0.0, pp - qq)
        want = qq * a + (1.0 - np.sum(qq * a)) * res / res.sum()
        got = np.zeros(V)
        for x in range(V):
            call = oracle_mod.SeqCaller(lp2, lq[None, :], [x], T, lenience=kind, eps=eps)
            th = accept_threshold(call, 0, 1)
            got[x] += qq[x] * th
            if th < 1.0:      # rejected for some r: then the residual draw
                got += qq[x] * (1.0 - th) * draw_distribution(call, 0, 1, V)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_golden_f_sq_hundred_times_more_likely(oracle_mod):
    g = GOLDEN["lenience_f_sq_example"]
    rng = np.random.default_rng(53)
    V, T = 6, 1.0
    lp = rng.standard_normal(V).astype(np.float32)
    lq = lp.copy()
    x = 2
    lp[x] -= 8.0            # p(x)/q(x) ~ e^-8: far below eps^2
    lq[x] += 0.0
    base = oracle_mod.SeqCaller(np.stack([lp, lp]), lq[None, :], [x], T)
    len_ = oracle_mod.SeqCaller(np.stack([lp, lp]), lq[None, :], [x], T, lenience=g["lenience"],
                                eps=g["eps"])
    a0 = accept_threshold(base, 0, 1)
    a1 = accept_threshold(len_, 0, 1)
    assert a1 < 1.0
    assert abs(a1 / a0 - g["acceptance_factor"]) < 1e-9 * g["acceptance_factor"]


def test_acceptance_grows_as_eps_falls(oracle_mod):
    """f is decreasing in eps (the page's definition), so acceptance is too."""
    rng = np.random.default_rng(59)
    V, T = 6, 1.0
    lp, lq = _rows(rng, V)
    qq = probs(lq, T)
    for kind in ("lin", "sq", "exp"):
        prev = -1.0
        for eps in (1.0, 0.8, 0.5, 0.2, 0.05):
            acc = sum(qq[x] * accept_threshold(oracle_mod.SeqCaller(
                np.stack([lp, lp]), lq[None, :], [x], T, lenience=kind, eps=eps), 0, 1)
                for x in range(V))
            assert acc >= prev - 1e-15
            prev = acc


def test_lenience_rejects_eps_outside_0_1(oracle_mod):
    p = np.zeros((2, 4), np.float32)
    q = np.zeros((1, 4), np.float32)
    x = np.zeros((1, 1), np.int32)
    for kind, eps in [("lin", 0.0), ("sq", -0.5), ("exp", 1.5), ("lin", float("nan"))]:
        res = oracle_mod.verify_batch(p, q, [0], [0], x, [1], 1.0, lenience=kind, eps=eps)
        assert res["rc"] == oracle_mod.ERR_ARG


# --------------------------------------------------------------------------
# beta and TVD

def test_beta_is_the_enumerated_acceptance(oracle_mod):
    """beta from the pair statistics equals the acceptance of the oracle's
    accept test, integrated over its uniform and averaged over x ~ q."""
    rng = np.random.default_rng(61)
    for V, T, dtype in [(5, 1.0, "fp32"), (8, 0.6, "bf16"), (4, 1.7, "fp32")]:
        lp, lq = _rows(rng, V, dtype=dtype)
        qq = probs(lq, T)
        acc = sum(qq[x] * accept_threshold(oracle_mod.SeqCaller(
            np.stack([lp, lp]), lq[None, :], [x], T), 0, 1) for x in range(V))
        rc, beta, tvd = oracle_mod.pair_stats(lp, lq, T)
        assert rc == 0
        assert abs(beta - acc) < 1e-13
        # TVD against scipy's L1 distance of the two distributions
        assert abs(tvd - 0.5 * cityblock(probs(lp, T), qq)) < 1e-13
        assert abs(beta + tvd - 1.0) < 1e-13


def test_beta_special_cases(oracle_mod):
    rng = np.random.default_rng(67)
    row = ENCODERS["bf16"](3.0 * rng.standard_normal(1000))
    rc, beta, tvd = oracle_mod.pair_stats(row, row, 0.7)
    assert rc == 0 and abs(beta - 1.0) < 1e-13 and abs(tvd) < 1e-13
    a = np.full(10, -np.inf, np.float32)
    b = np.full(10, -np.inf, np.float32)
    a[:5] = rng.standard_normal(5)
    b[5:] = rng.standard_normal(5)
    rc, beta, tvd = oracle_mod.pair_stats(a, b, 1.0)
    assert rc == 0 and beta == 0.0 and abs(tvd - 1.0) < 1e-15
    bad = np.zeros(10, np.float32)
    bad[3] = np.nan
    assert oracle_mod.pair_stats(bad, a, 1.0)[0] == oracle_mod.ERR_INPUT


def test_pair_stats_batch_layout_and_expected_emitted(oracle_mod):
    """Batch layout (NaN past gamma_b) and E[emitted] = 1 + sum_k prod_{i<=k} beta_i
    against a Monte Carlo run of the seeded verify on shared rows."""
    rng = np.random.default_rng(71)
    V, gm, T, B = 12, 3, 1.0, 60_000
    p = _rows(rng, V, scale=1.0, n=gm + 1)
    q = _rows(rng, V, scale=1.0, n=gm)
    g = np.full(B, gm, np.int32)
    g[:3] = [0, 1, 2]
    zeros = np.zeros(B, np.int64)
    st = oracle_mod.pair_stats_batch(p, q, zeros, zeros, g, T)
    assert st["rc"] == 0
    assert np.isnan(st["beta"][0]).all() and np.isnan(st["beta"][1][1:]).all()
    for i in range(gm):
        rc, b_i, t_i = oracle_mod.pair_stats(p[i], q[i], T)
        assert st["beta"][5][i] == b_i and st["tvd"][5][i] == t_i
    x = np.stack([rng.choice(V, B, p=probs(q[i], T)) for i in range(gm)], 1).astype(np.int32)
    res = oracle_mod.verify_batch(p, q, zeros, zeros, x, g, T, seed=77)
    emitted = (res["n"][3:] + 1).astype(np.float64)
    want = oracle_mod.expected_emitted(st["beta"][5])
    assert abs(emitted.mean() - want) < 5 * emitted.std() / np.sqrt(len(emitted))


# --------------------------------------------------------------------------
# draft features

def test_entropy_and_topk_against_scipy_and_numpy(oracle_mod):
    rng = np.random.default_rng(73)
    for V, T, dtype, k in [(50, 1.0, "fp32", 5), (1000, 0.7, "bf16", 10), (7, 1.3, "fp32", 7),
                           (3000, 1.0, "bf16", 16)]:
        row = ENCODERS[dtype](2.0 * rng.standard_normal(V))
        rc, h, prob, idx = oracle_mod.row_features(row, T, k)
        assert rc == 0
        q = softmax(as_f64(row) / T)
        assert abs(h - scipy_entropy(q)) < 1e-12 * max(1.0, h)
        order = np.argsort(-as_f64(row), kind="stable")[:k]
        np.testing.assert_array_equal(idx, order)
        np.testing.assert_allclose(prob, q[order], rtol=1e-13, atol=0)


def test_entropy_closed_forms_and_ties(oracle_mod):
    V = 64
    rc, h, prob, idx = oracle_mod.row_features(np.zeros(V, np.float32), 1.0, 4)
    assert rc == 0 and abs(h - np.log(V)) < 1e-13
    np.testing.assert_array_equal(idx, [0, 1, 2, 3])          # ties: lower index first
    np.testing.assert_allclose(prob, 1.0 / V, rtol=1e-14)
    one = np.full(V, -np.inf, np.float32)
    one[17] = 3.0
    rc, h, prob, idx = oracle_mod.row_features(one, 0.5, 3)
    assert rc == 0 and h == 0.0 and idx[0] == 17 and prob[0] == 1.0
    two = np.full(V, -np.inf, np.float32)
    two[5], two[9] = 0.0, np.log(3.0)
    rc, h, prob, idx = oracle_mod.row_features(two, 1.0, 2)
    w = np.exp(np.float64(two[9]))          # 3, up to the float32 rounding of log 3
    a = w / (1.0 + w)
    assert abs(h - (-a * np.log(a) - (1 - a) * np.log(1 - a))) < 1e-13
    np.testing.assert_array_equal(idx, [9, 5])
    # k beyond V: padded
    rc, h, prob, idx = oracle_mod.row_features(np.zeros(3, np.float32), 1.0, 5)
    np.testing.assert_array_equal(idx, [0, 1, 2, -1, -1])
    assert prob[3] == 0.0


def test_features_batch_matches_rows(oracle_mod):
    rng = np.random.default_rng(79)
    rows = bf16_bits(rng.standard_normal((9, 700)) * 2.5)
    out = oracle_mod.row_features_batch(rows, 0.8, 6)
    assert out["rc"] == 0
    for r in range(9):
        rc, h, prob, idx = oracle_mod.row_features(rows[r], 0.8, 6)
        assert out["entropy"][r] == h
        np.testing.assert_array_equal(out["topk_idx"][r], idx)
        np.testing.assert_array_equal(out["topk_prob"][r], prob)


# --------------------------------------------------------------------------
# planted mistakes

MUTANTS = {
    "lenience_on_q": ("double ratio = exp(lenient_log(log_p, len_kind, eps) - log_q);",
                      "double ratio = exp(log_p - lenient_log(log_q, len_kind, eps));"),
    "f_sq_single_power": ("case ORACLE_LENIENCE_SQ: return log_p - 2.0 * log(eps);",
                          "case ORACLE_LENIENCE_SQ: return log_p - log(eps);"),
    "f_exp_as_product": ("case ORACLE_LENIENCE_EXP: return eps * log_p;",
                         "case ORACLE_LENIENCE_EXP: return log_p + log(eps);"),
    "tvd_without_half": ("*tvd_out = 0.5 * nsum_get(&d);", "*tvd_out = nsum_get(&d);"),
    "beta_max_not_min": ("nsum_add(&b, fmin(p, q));", "nsum_add(&b, fmax(p, q));"),
    "entropy_without_lse": ("double log_q = l / T - lse;", "double log_q = l / T;"),
    "topk_ties_to_higher_index": ("while (at > 0 && l > logit_at(row, dtype, topk_idx[at - 1])) {",
                                  "while (at > 0 && l >= logit_at(row, dtype, topk_idx[at - 1])) {"),
}


def _mutant(oracle_mod, tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "specverify_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o",
                    str(so), str(mpath), "-lm", "-lpthread"], check=True)
    return oracle_mod.load_variant(str(so))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(oracle_mod, tmp_path, monkeypatch, name):
    lib = _mutant(oracle_mod, tmp_path, name)
    monkeypatch.setattr(oracle_mod, "_lib", lib)
    failed = False
    tests = {
        "lenience_on_q": lambda: test_lenient_acceptance_is_expected_min(oracle_mod, "sq", 0.6),
        "f_sq_single_power": lambda: test_lenient_acceptance_is_expected_min(oracle_mod, "sq",
                                                                             0.6),
        "f_exp_as_product": lambda: test_lenient_acceptance_is_expected_min(oracle_mod, "exp",
                                                                            0.3),
        "tvd_without_half": lambda: test_beta_is_the_enumerated_acceptance(oracle_mod),
        "beta_max_not_min": lambda: test_beta_is_the_enumerated_acceptance(oracle_mod),
        "entropy_without_lse": lambda: test_entropy_and_topk_against_scipy_and_numpy(oracle_mod),
        "topk_ties_to_higher_index": lambda: test_entropy_closed_forms_and_ties(oracle_mod),
    }
    try:
        tests[name]()
    except AssertionError:
        failed = True
    assert failed, name
