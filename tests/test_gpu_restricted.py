"""Parity of the restricted sampling verify with the CPU oracle, through the C ABI.

"Speculative Decoding and Distillation" (Kadimisetty notes), "Greedy vs
sampling": temperature, top-k and top-p restrict the target and the draft
distributions alike and the accept / residual rule runs on the restricted
ones. Per sequence a temperature, a top-k (1..32) and a top-p; the drafts
are sampled from the restricted draft distribution (as a drafter using the
same sampling settings would), with a few replaced by arbitrary tokens so
that the q'(x) = 0 conventions (ratio +inf or 0) are exercised.

Decision rule as in the lossless parity tests: accepted counts and tokens
bit-exact except at decisions inside the flag bands (accept |r - ratio| <
1e-5, draw point within 1e-5 / V of a CDF boundary); the flagged decisions
count toward the run's flag budget. The kernel builds the restricted
distributions in double precision from the same logits, so flags are rare.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import compare, record
from speculative_decoding_token_gb300 import workload

pytestmark = pytest.mark.gpu

BITS = {"bad_gamma": 1, "bad_row": 2, "bad_token": 4, "bad_logit": 8, "timeout": 16,
        "bad_param": 32}
# Informational bits. A zero-mass residual is not only a rounding event here:
# a draft token outside both kept sets has ratio 0 and is rejected, and when
# the two restricted rows are equal the residual max(0, p' - q') is zero
# everywhere, so the token is drawn from p' (the oracle does the same).
INFORMATIONAL = (1 << 8) | (1 << 9)


@pytest.fixture(scope="module")
def svm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_token_gb300 as sv
    sv.build()
    sv.load()
    oracle.build()
    return sv


def _params(B, rng, k_max=32):
    T = rng.choice(np.array([0.5, 0.7, 1.0, 1.3], np.float32), B)
    k = rng.integers(1, k_max + 1, B).astype(np.int32)
    p = rng.uniform(0.3, 1.0, B).astype(np.float32)
    p[rng.random(B) < 0.3] = 1.0
    return T, k, p


def _restricted_drafts(host, T, k, p, rng, frac_any=0.05):
    """Draft tokens drawn from the restricted draft rows (oracle's definition);
    a fraction replaced by uniform tokens."""
    g = host["gamma"]
    q_off = host["q_row_off"]
    V = host["draft"].shape[1]
    toks = np.array(host["draft_tokens"], copy=True)
    for b in range(len(g)):
        for i in range(int(g[b])):
            if rng.random() < frac_any:
                toks[b, i] = rng.integers(0, V)
                continue
            rc, prob = oracle.restricted_row(host["draft"][q_off[b] + i], float(T[b]),
                                             int(k[b]), float(p[b]))
            assert rc == 0
            idx = np.nonzero(prob)[0]
            toks[b, i] = rng.choice(idx, p=prob[idx] / prob[idx].sum())
    return toks


def _run(svm, h, batch, toks, T, k, p, seed):
    dev = batch.target.device
    n, out = h.verify_restricted(batch.target, batch.draft, batch.p_row_off, batch.q_row_off,
                                 torch.from_numpy(toks).to(dev), batch.gamma,
                                 torch.from_numpy(T).to(dev), torch.from_numpy(k).to(dev),
                                 None if p is None else torch.from_numpy(p).to(dev), seed)
    return n.cpu().numpy(), out.cpu().numpy()


def _oracle(host, toks, T, k, p, seed):
    ora = oracle.verify_batch_restricted(host["target"], host["draft"], host["p_row_off"],
                                         host["q_row_off"], toks, host["gamma"],
                                         T.astype(np.float64), k,
                                         None if p is None else p.astype(np.float64), seed=seed)
    ora["gamma"] = host["gamma"]
    ora["seqs"] = np.arange(len(host["gamma"]))
    return ora


def _properties(batch, toks, n, out):
    g = batch.gamma.cpu().numpy()
    for b in range(batch.B):
        assert 0 <= n[b] <= g[b]
        assert (out[b, :n[b]] == toks[b, :n[b]]).all()
        assert 0 <= out[b, n[b]] < batch.V
        assert (out[b, n[b] + 1:] == -1).all()


CASES = {
    # label: (config, overrides, data seed, verify seeds)
    "b256_g1to10_v152064_bf16": (3, dict(), 1301, (11, 12)),
    "b64_g8_v128256_bf16": (2, dict(), 1302, (21,)),
    "b8_g5_v32000_bf16": (1, dict(), 1303, (31, 32, 33)),
    "b16_g4_v32000_fp32": (0, dict(B=16), 1304, (41, 42)),
    "b24_g0to6_v1001_fp32": (0, dict(B=24, V=1001, gamma=(0, 6)), 1305, (51,)),
    "b32_g0to3_v7_bf16": (1, dict(B=32, V=7, gamma=(0, 3)), 1306, (61,)),
}


@pytest.mark.parametrize("label", sorted(CASES))
def test_restricted_parity(svm, label):
    cfg, over, ds, seeds = CASES[label]
    batch = workload.make_batch(cfg, device="cuda", seed=ds, **over)
    if batch.V % 8:
        # a ragged vocabulary: rows padded to a 16-byte stride
        pad = (batch.V + 7) // 8 * 8
        for name in ("target", "draft"):
            t = getattr(batch, name)
            full = torch.zeros(t.shape[0], pad, dtype=t.dtype, device=t.device)
            full[:, :batch.V] = t
            setattr(batch, name, full[:, :batch.V])
    rng = np.random.default_rng(ds)
    T, k, p = _params(batch.B, rng)
    host = workload.to_host_arrays(batch)
    toks = _restricted_drafts(host, T, k, p, rng)
    h = svm.SpecVerify(batch.B, max(batch.gamma_max, 1), batch.V)
    for seed in seeds:
        n, out = _run(svm, h, batch, toks, T, k, p, seed)
        _properties(batch, toks, n, out)
        ora = _oracle(host, toks, T, k, p, seed)
        assert ora["rc"] == 0
        st = compare(n, out, ora, batch.V)
        assert not st["hard"], st["hard"][:5]
        record(f"restricted {label}", st)
    assert h.device_status() & ~INFORMATIONAL == 0
    h.close()


def test_restricted_special_parameters(svm):
    """top-k 1 (greedy on both sides), top-p None, top-k above V, temperature
    extremes; the same batch run twice in a row (the kernel leaves its
    counters zero for the next call)."""
    batch = workload.make_batch(1, device="cuda", seed=1310, B=16, gamma=(0, 6))
    host = workload.to_host_arrays(batch)
    rng = np.random.default_rng(1310)
    B = batch.B
    T = np.where(np.arange(B) % 3 == 0, np.float32(0.05), np.float32(4.0)).astype(np.float32)
    k = np.where(np.arange(B) % 2 == 0, 1, 32).astype(np.int32)
    toks = _restricted_drafts(host, T, k, np.ones(B, np.float32), rng)
    h = svm.SpecVerify(B, batch.gamma_max, batch.V)
    ora = _oracle(host, toks, T, k, None, 77)
    assert ora["rc"] == 0
    for _ in range(2):
        n, out = _run(svm, h, batch, toks, T, k, None, 77)
        st = compare(n, out, ora, batch.V)
        assert not st["hard"], st["hard"][:5]
        record("restricted special parameters", st)
    assert h.device_status() & ~INFORMATIONAL == 0
    # top-1: the restricted target is one-hot on the argmax, the final token
    # is that argmax whenever every draft was accepted
    tgt = batch.target.float().cpu().numpy()
    p_off = host["p_row_off"]
    for b in range(B):
        if k[b] == 1 and n[b] == host["gamma"][b]:
            assert out[b, n[b]] == int(np.argmax(tgt[p_off[b] + n[b]]))
    h.close()


def test_restricted_tiny_vocabulary_and_ties(svm):
    """V = 1 and V = 5 with top-k 32 (k clipped to V); rows with many equal
    logits, where top-k keeps the lower token indices."""
    for V, dt in ((1, torch.float32), (5, torch.bfloat16), (300, torch.bfloat16)):
        B, gm = 6, 3
        g = torch.Generator().manual_seed(V)
        tgt = torch.randint(-3, 3, (B * (gm + 1), V), generator=g).float().to(dt)
        dft = torch.randint(-3, 3, (B * gm, V), generator=g).float().to(dt)
        stride = (V + 7) // 8 * 8
        tp = torch.zeros(tgt.shape[0], stride, dtype=dt)
        tp[:, :V] = tgt
        dp = torch.zeros(dft.shape[0], stride, dtype=dt)
        dp[:, :V] = dft
        gamma = torch.tensor([0, 1, 2, 3, 3, 2], dtype=torch.int32)
        p_off = torch.arange(B, dtype=torch.int64) * (gm + 1)
        q_off = torch.arange(B, dtype=torch.int64) * gm
        toks = torch.randint(0, V, (B, gm), generator=g, dtype=torch.int32)
        T = np.full(B, 0.9, np.float32)
        k = np.array([32, 1, 2, 3, 32, 8], np.int32)
        p = np.array([1.0, 0.5, 0.9, 0.2, 0.99, 1.0], np.float32)
        h = svm.SpecVerify(B, gm, V)
        tpd, dpd = tp.cuda()[:, :V], dp.cuda()[:, :V]
        n, out = h.verify_restricted(tpd, dpd, p_off.cuda(), q_off.cuda(), toks.cuda(),
                                     gamma.cuda(), torch.from_numpy(T).cuda(),
                                     torch.from_numpy(k).cuda(), torch.from_numpy(p).cuda(), 5)
        n, out = n.cpu().numpy(), out.cpu().numpy()
        host_t = workload.to_numpy_logits(tgt)
        host_d = workload.to_numpy_logits(dft)
        ora = oracle.verify_batch_restricted(host_t, host_d, p_off.numpy(), q_off.numpy(),
                                             toks.numpy(), gamma.numpy(), T.astype(np.float64),
                                             k, p.astype(np.float64), seed=5)
        assert ora["rc"] == 0
        ora["gamma"] = gamma.numpy()
        ora["seqs"] = np.arange(B)
        st = compare(n, out, ora, V)
        assert not st["hard"], (V, st["hard"][:5])
        record("restricted tiny V and ties", st)
        assert h.device_status() & ~INFORMATIONAL == 0
        h.close()


def test_restricted_bad_inputs(svm):
    """Bad parameters, tokens, gamma and logits fail their own sequence only,
    with the matching status bits; a NaN after the first rejection is still
    found (every row is read)."""
    batch = workload.make_batch(0, device="cuda", seed=1320, B=10, V=4096, gamma=4)
    host = workload.to_host_arrays(batch)
    rng = np.random.default_rng(1320)
    T, k, p = _params(batch.B, rng)
    toks = _restricted_drafts(host, T, k, p, rng, frac_any=0.0)
    T[1] = 0.0                      # bad temperature
    k[2] = 0                        # bad top-k
    k[3] = 33
    p[4] = 0.0                      # bad top-p
    toks[5, 1] = batch.V            # bad token
    gamma = batch.gamma.clone()
    gamma[6] = batch.gamma_max + 1  # bad gamma
    tgt = batch.target.clone()
    tgt[int(host["p_row_off"][7]) + 4, 17] = float("nan")   # the bonus row of sequence 7
    dft = batch.draft.clone()
    dft[int(host["q_row_off"][8]) + 3, 5] = float("inf")
    h = svm.SpecVerify(batch.B, batch.gamma_max + 1, batch.V)
    dev = batch.target.device
    n, out = h.verify_restricted(tgt, dft, batch.p_row_off, batch.q_row_off,
                                 torch.from_numpy(toks).to(dev), gamma.to(dev),
                                 torch.from_numpy(T).to(dev), torch.from_numpy(k).to(dev),
                                 torch.from_numpy(p).to(dev), 9)
    n, out = n.cpu().numpy(), out.cpu().numpy()
    st = h.device_status() & ~INFORMATIONAL
    assert st == BITS["bad_param"] | BITS["bad_token"] | BITS["bad_gamma"] | BITS["bad_logit"]
    for b in range(1, 9):
        assert n[b] == -1 and (out[b] == -1).all(), b
    # the good sequences agree with the oracle
    host2 = dict(host)
    host2["target"] = workload.to_numpy_logits(tgt)
    host2["draft"] = workload.to_numpy_logits(dft)
    host2["gamma"] = gamma.cpu().numpy()
    ora = oracle.verify_batch_restricted(host2["target"], host2["draft"], host2["p_row_off"],
                                         host2["q_row_off"], toks, host2["gamma"],
                                         T.astype(np.float64), k, p.astype(np.float64), seed=9)
    # (top-k 33 is outside the library's range 1..32 only: the oracle takes any k >= 1)
    assert (ora["n"][[1, 2, 4, 5, 6, 7, 8]] == -1).all()
    for b in (0, 9):
        assert n[b] == ora["n"][b] and (out[b] == ora["tokens"][b]).all()
    # host-checked arguments launch nothing
    with pytest.raises(svm.SpecVerifyError):
        h.verify_restricted(tgt, dft, batch.p_row_off, batch.q_row_off,
                            torch.from_numpy(toks).to(dev), gamma.to(dev), None,
                            torch.from_numpy(k).to(dev), None, 9)
    h.close()
