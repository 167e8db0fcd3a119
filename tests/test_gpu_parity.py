"""Parity of the CUDA verify step with the CPU oracle, through the C ABI.

Small shapes (every sequence checked, several tiles per row and a ragged
tail), the five synthetic workloads at full size (sampled sequences checked
one by one, properties checked for all), greedy mode bit-exact, and the
edge cases: gamma = 0, B = 0, ragged vocabulary tails, shared rows, q = p,
invalid inputs, determinism and host buffers.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import (FLAG_BUDGET, FLAG_LOG, LSE_RTOL, compare, flag_report, lse_buffers,
                         lse_errors, oracle_temperature, record, run_oracle)
from speculative_decoding_token_gb300 import workload

pytestmark = pytest.mark.gpu

# status bits that report how a draw was computed, not an error: the draw's
# exact slow path and the zero-mass fallback both give the oracle's token
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


def _check(st):
    """No mismatch outside the flag bands; the flag budget itself is checked
    over the whole run (test_flag_budget_over_the_run)."""
    assert not st["hard"], st
    assert st["flagged_mismatches"] <= st["flagged"]


def _verify(svm, batch, seed, greedy=False, with_lse=True):
    h = svm.SpecVerify(batch.B, max(batch.gamma_max, 1), batch.V)
    p_lse, q_lse = lse_buffers(batch)
    n, toks = h.verify_batch(batch, seed=seed, greedy=greedy,
                             p_lse=None if greedy or not with_lse else p_lse,
                             q_lse=None if greedy or not with_lse else q_lse)
    torch.cuda.synchronize()
    status = h.device_status()
    h.close()
    return n.cpu().numpy(), toks.cpu().numpy(), p_lse, q_lse, status


SMALL = [
    # config, overrides, data seeds
    (0, dict(), range(6)),
    (1, dict(), range(3)),
    (2, dict(B=6), range(2)),
    (3, dict(B=20), range(2)),
    (4, dict(B=6), range(2)),
]


@pytest.mark.parametrize("cfg,over,seeds", SMALL, ids=[f"cfg{c[0]}" for c in SMALL])
def test_sampling_parity_small(svm, cfg, over, seeds):
    for ds in seeds:
        batch = workload.make_batch(cfg, device="cuda", seed=1000 * cfg + ds, **over)
        seed = 77 + ds
        n, toks, p_lse, q_lse, status = _verify(svm, batch, seed)
        assert status == 0
        ora = run_oracle(batch, seed)
        assert ora["rc"] == 0
        st = compare(n, toks, ora, batch.V)
        _check(st)
        record(f"{workload.CONFIGS[cfg]['name']} small B, every row + lse", st)
        assert lse_errors(batch, ora, p_lse, q_lse) <= LSE_RTOL
        # the same uniforms on the needed-rows path (no logsumexp outputs)
        n2, toks2, _, _, status2 = _verify(svm, batch, seed, with_lse=False)
        assert status2 == 0
        st2 = compare(n2, toks2, ora, batch.V)
        _check(st2)
        record(f"{workload.CONFIGS[cfg]['name']} small B, needed rows", st2)


@pytest.mark.parametrize("cfg,over", [(1, dict()), (4, dict(B=6)), (3, dict(B=12))])
def test_greedy_parity_small(svm, cfg, over):
    batch = workload.make_batch(cfg, device="cuda", **over)
    # make most drafts agree with the target argmax so that long prefixes occur
    am = batch.draft_tokens.clone()
    g = batch.gamma.cpu().tolist()
    p_off = batch.p_row_off.cpu().tolist()
    for b in range(batch.B):
        for i in range(g[b]):
            am[b, i] = batch.target[p_off[b] + i].float().argmax().to(torch.int32)
    keep = torch.rand(batch.B, batch.gamma_max, device="cuda") < 0.8
    batch.draft_tokens = torch.where(keep, am, batch.draft_tokens).contiguous()
    n, toks, _, _, status = _verify(svm, batch, 0, greedy=True)
    assert status == 0
    ora = run_oracle(batch, 0, greedy=True)
    st = compare(n, toks, ora, batch.V, greedy=True)
    assert not st["hard"], st
    assert (n > 0).any()


# Full-size parity, in the benchmark's launch configuration. Every sequence
# is compared with the oracle, on the path the benchmark times (no logsumexp
# outputs: rows after a sequence's first rejection are skipped, tickets are
# dealt or claimed as at full size) and on the every-row path (logsumexp
# outputs, checked at 1e-5 relative). Several input batches (data seeds) and
# uniforms (verify seeds) per workload, so that the decisions summed over the
# run are many enough for the flag budget to mean something.
FULL = {
    # config: (data seeds, verify seeds per batch)
    1: ((1, 11, 21, 31, 41, 51, 61, 71), (4242, 4243, 4244)),
    2: ((2, 12), (4244, 4245, 4246)),
    3: ((3, 4), (4245, 4246, 4247, 1_000_003, 2_000_006)),
    4: ((4,), (4246, 4247, 4248, 4249, 4250, 4251)),
}


def _properties(batch, n, toks):
    g = batch.gamma.cpu().numpy()
    x = batch.draft_tokens.cpu().numpy()
    assert ((n >= 0) & (n <= g)).all()
    for b in range(batch.B):
        assert (toks[b][:n[b]] == x[b][:n[b]]).all()
        assert 0 <= toks[b][n[b]] < batch.V
        assert (toks[b][n[b] + 1:] == -1).all()


@pytest.mark.parametrize("cfg", sorted(FULL))
def test_full_size_parity_every_sequence(svm, cfg):
    data_seeds, verify_seeds = FULL[cfg]
    name = workload.CONFIGS[cfg]["name"]
    greedy_too = workload.CONFIGS[cfg].get("greedy", False)
    for ds in data_seeds:
        batch = workload.make_batch(cfg, device="cuda", seed=ds)
        h = svm.SpecVerify(batch.B, max(batch.gamma_max, 1), batch.V)
        host = workload.to_host_arrays(batch)
        T = oracle_temperature(batch.T)
        for seed in verify_seeds:
            ora = oracle.verify_batch(host["target"], host["draft"], host["p_row_off"],
                                      host["q_row_off"], host["draft_tokens"], host["gamma"], T,
                                      seed=seed)
            assert ora["rc"] == 0
            ora["gamma"] = host["gamma"]
            ora["seqs"] = np.arange(batch.B)
            # the benchmark's path: no logsumexp outputs
            n, toks = h.verify_batch(batch, seed=seed)
            n, toks = n.cpu().numpy(), toks.cpu().numpy()
            _properties(batch, n, toks)
            st = compare(n, toks, ora, batch.V)
            _check(st)
            record(f"{name} needed rows", st)
            # every row read, logsumexp outputs
            p_lse, q_lse = lse_buffers(batch)
            n2, toks2 = h.verify_batch(batch, seed=seed, p_lse=p_lse, q_lse=q_lse)
            n2, toks2 = n2.cpu().numpy(), toks2.cpu().numpy()
            st2 = compare(n2, toks2, ora, batch.V)
            _check(st2)
            record(f"{name} every row + lse", st2)
            assert lse_errors(batch, ora, p_lse, q_lse) <= LSE_RTOL
        if greedy_too:
            ng, tg = h.verify_batch(batch, greedy=True)
            orag = oracle.verify_batch(host["target"], None, host["p_row_off"], None,
                                       host["draft_tokens"], host["gamma"], 0.0)
            assert (ng.cpu().numpy() == orag["n"]).all()
            assert (tg.cpu().numpy() == orag["tokens"]).all()
        assert h.device_status() == 0
        h.close()
        del batch, host


def test_single_sequence_200_rounds(svm):
    """The batch-1 workload as specified: 200 rounds, fresh rows and seed + round
    each round, both paths, every decision compared with the oracle."""
    cfg = 0
    name = workload.CONFIGS[cfg]["name"]
    h = svm.SpecVerify(1, 4, 32000)
    for rnd in range(workload.CONFIGS[cfg]["rounds"]):
        batch = workload.make_batch(cfg, device="cuda", seed=rnd)
        seed = rnd
        host = workload.to_host_arrays(batch)
        ora = oracle.verify_batch(host["target"], host["draft"], host["p_row_off"],
                                  host["q_row_off"], host["draft_tokens"], host["gamma"],
                                  oracle_temperature(batch.T), seed=seed)
        ora["gamma"] = host["gamma"]
        ora["seqs"] = np.arange(1)
        n, toks = h.verify_batch(batch, seed=seed)
        st = compare(n.cpu().numpy(), toks.cpu().numpy(), ora, batch.V)
        _check(st)
        record(f"{name} needed rows", st)
        p_lse, q_lse = lse_buffers(batch)
        n2, toks2 = h.verify_batch(batch, seed=seed, p_lse=p_lse, q_lse=q_lse)
        st2 = compare(n2.cpu().numpy(), toks2.cpu().numpy(), ora, batch.V)
        _check(st2)
        record(f"{name} every row + lse", st2)
        assert lse_errors(batch, ora, p_lse, q_lse) <= LSE_RTOL
    assert h.device_status() == 0
    h.close()


def _manual_batch(V, dtype, rows_p, rows_q, stride=None, device="cuda", seed=0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    stride = stride or V
    tdt = {"fp32": torch.float32, "bf16": torch.bfloat16}[dtype]
    tp = (2.0 * torch.randn(rows_p, stride, generator=g)).to(tdt)
    tq = (2.0 * torch.randn(max(rows_q, 1), stride, generator=g)).to(tdt)
    return tp.to(device), tq.to(device)


# V = 300007 has more draw chunks than a warp's ring holds: its finalize takes
# the general (double-precision) path, the others the staged fast path.
@pytest.mark.parametrize("V,stride,dtype", [(50257, 50264, "bf16"), (1001, 1004, "fp32"),
                                            (5, 8, "fp32"), (3, 8, "bf16"), (32769, 32776, "bf16"),
                                            (8193, 8196, "fp32"), (300007, 300008, "bf16")])
def test_ragged_vocab_and_padded_stride(svm, V, stride, dtype):
    B, gm = 7, 4
    gam = torch.tensor([0, 1, 2, 3, 4, 4, 2], dtype=torch.int32)
    p_off = torch.cumsum(gam.long() + 1, 0) - (gam.long() + 1)
    q_off = torch.cumsum(gam.long(), 0) - gam.long()
    full_p, full_q = _manual_batch(V, dtype, int((gam + 1).sum()), int(gam.sum()), stride)
    tgt = full_p[:, :V]
    dft = full_q[:, :V]
    x = torch.randint(0, V, (B, gm), dtype=torch.int32)
    d_p_off, d_q_off, d_x, d_gam = p_off.cuda(), q_off.cuda(), x.cuda(), gam.cuda()
    h = svm.SpecVerify(B, gm, V)
    for seed in range(5):
        n, toks = h.verify(tgt, dft, d_p_off, d_q_off, d_x, d_gam, 0.9, seed)
        torch.cuda.synchronize()
        ora = oracle.verify_batch(workload.to_numpy_logits(tgt), workload.to_numpy_logits(dft),
                                  p_off.numpy(), q_off.numpy(), x.numpy(), gam.numpy(),
                                  oracle_temperature(0.9), seed=seed)
        ora["gamma"] = gam.numpy()
        ora["seqs"] = np.arange(B)
        st = compare(n.cpu().numpy(), toks.cpu().numpy(), ora, V)
        assert not st["hard"], (seed, st)
        ng, tg = h.verify(tgt, None, d_p_off, None, d_x, d_gam, 0.0, 0, greedy=True)
        orag = oracle.verify_batch(workload.to_numpy_logits(tgt), None, p_off.numpy(), None,
                                   x.numpy(), gam.numpy(), 0.0)
        assert (ng.cpu().numpy() == orag["n"]).all()
        assert (tg.cpu().numpy() == orag["tokens"]).all()
    assert h.device_status() == 0
    h.close()


def test_empty_batch_and_gamma_zero(svm):
    h = svm.SpecVerify(4, 3, 1000)
    tgt = torch.randn(4, 1000, device="cuda")
    empty_i32 = torch.zeros(0, dtype=torch.int32, device="cuda")
    empty_i64 = torch.zeros(0, dtype=torch.int64, device="cuda")
    n, toks = h.verify(tgt, tgt, empty_i64, empty_i64,
                       torch.zeros(0, 3, dtype=torch.int32, device="cuda"), empty_i32, 1.0, 0)
    assert n.numel() == 0
    gam = torch.zeros(4, dtype=torch.int32, device="cuda")
    off = torch.arange(4, dtype=torch.int64, device="cuda")
    x = torch.zeros(4, 3, dtype=torch.int32, device="cuda")
    for seed in range(10):
        n, toks = h.verify(tgt, tgt, off, off, x, gam, 1.0, seed)
        ora = oracle.verify_batch(tgt.cpu().numpy(), tgt.cpu().numpy(), off.cpu().numpy(),
                                  off.cpu().numpy(), x.cpu().numpy(), gam.cpu().numpy(), 1.0,
                                  seed=seed)
        ora["gamma"] = gam.cpu().numpy()
        ora["seqs"] = np.arange(4)
        st = compare(n.cpu().numpy(), toks.cpu().numpy(), ora, 1000)
        assert not st["hard"]
        assert (n.cpu() == 0).all()
    h.close()


def test_shared_rows_and_q_equal_p(svm):
    V, B, gm = 4096, 64, 6
    tgt = (3 * torch.randn(gm + 1, V, device="cuda")).to(torch.bfloat16)
    dft = tgt[:gm].clone()
    x = torch.randint(0, V, (B, gm), dtype=torch.int32, device="cuda")
    zeros = torch.zeros(B, dtype=torch.int64, device="cuda")
    gam = torch.full((B,), gm, dtype=torch.int32, device="cuda")
    h = svm.SpecVerify(B, gm, V)
    n, toks = h.verify(tgt, dft, zeros, zeros, x, gam, 0.6, 5)
    assert (n.cpu() == gm).all()                      # q = p: every draft accepted
    assert (toks[:, :gm] == x).all()
    ora = oracle.verify_batch(workload.to_numpy_logits(tgt), workload.to_numpy_logits(dft),
                              zeros.cpu().numpy(), zeros.cpu().numpy(), x.cpu().numpy(),
                              gam.cpu().numpy(), oracle_temperature(0.6), seed=5)
    ora["gamma"] = gam.cpu().numpy()
    ora["seqs"] = np.arange(B)
    assert not compare(n.cpu().numpy(), toks.cpu().numpy(), ora, V)["hard"]
    h.close()


def _invalid_batch(nan_row_of_4):
    V, B, gm = 3000, 8, 3
    g = torch.Generator().manual_seed(0)
    gam = torch.full((B,), gm, dtype=torch.int32)
    tgt = torch.randn(B * (gm + 1), V, generator=g)
    dft = torch.randn(B * gm, V, generator=g)
    p_off = torch.arange(B, dtype=torch.int64) * (gm + 1)
    q_off = torch.arange(B, dtype=torch.int64) * gm
    x = torch.randint(0, V, (B, gm), dtype=torch.int32, generator=g)
    gam[1] = gm + 1                    # bad gamma
    x[2, 1] = V                        # bad token
    p_off[3] = B * (gm + 1) - 1        # rows past the end of the buffer
    tgt[4 * (gm + 1) + nan_row_of_4, 17] = float("nan")
    dft[5 * gm + 0, :] = float("-inf")  # a row of all -inf
    tgt[6 * (gm + 1) + 0, 5] = float("inf")
    return V, B, gm, tgt, dft, p_off, q_off, x, gam


@pytest.mark.parametrize("with_lse", [False, True])
def test_invalid_inputs_flag_only_their_sequence(svm, with_lse):
    # with logsumexp outputs every row is read, so a bad logit anywhere flags
    # its sequence; without them the bad rows here lie at position 1, which
    # every verify reads
    V, B, gm, tgt, dft, p_off, q_off, x, gam = _invalid_batch(2 if with_lse else 0)
    h = svm.SpecVerify(B, gm, V)
    dev = [t.cuda() for t in (tgt, dft, p_off, q_off, x, gam)]
    kw = {}
    if with_lse:
        kw = dict(p_lse=torch.empty(B * (gm + 1), device="cuda"),
                  q_lse=torch.empty(B * gm, device="cuda"))
    n, toks = h.verify(*dev, 1.0, 3, **kw)
    status = h.device_status()
    n = n.cpu().numpy()
    assert list(n[1:7]) == [-1] * 6
    assert (toks.cpu().numpy()[1:7] == -1).all()
    assert n[0] >= 0 and n[7] >= 0
    for bit in ("bad_gamma", "bad_token", "bad_row", "bad_logit"):
        assert status & svm.STATUS_BITS[bit], (bit, status)
    assert h.device_status() == 0      # read clears
    ora = oracle.verify_batch(tgt.numpy(), dft.numpy(), p_off.numpy(), q_off.numpy(), x.numpy(),
                              gam.numpy(), 1.0, seed=3)
    assert list(ora["n"]) == list(n)
    # greedy: NaN target logit flags the sequence too
    ng, _ = h.verify(dev[0], None, dev[2], None, dev[4], dev[5], 0.0, 0, greedy=True)
    assert ng.cpu().numpy()[4] == -1
    h.close()


def test_rows_after_first_rejection_are_not_read(svm):
    # Sequence 0 rejects at position 1 for sure (q_1 puts all its mass on x_1,
    # p_1 almost none), so rows 2.. are never needed: a NaN there leaves the
    # result valid -- equal to the oracle on the NaN-free rows -- unless
    # logsumexp outputs ask for every row.
    V, B, gm = 4096, 2, 3
    g = torch.Generator().manual_seed(1)
    tgt = torch.randn(B * (gm + 1), V, generator=g)
    dft = torch.randn(B * gm, V, generator=g)
    x = torch.randint(0, V, (B, gm), dtype=torch.int32, generator=g)
    tgt[0, x[0, 0]] = -40.0
    dft[0, x[0, 0]] = 40.0
    clean = tgt.clone()
    tgt[2, 7] = float("nan")           # p_3 of sequence 0
    gam = torch.full((B,), gm, dtype=torch.int32)
    p_off = torch.arange(B, dtype=torch.int64) * (gm + 1)
    q_off = torch.arange(B, dtype=torch.int64) * gm
    h = svm.SpecVerify(B, gm, V)
    dev = [t.cuda() for t in (tgt, dft, p_off, q_off, x, gam)]
    n, toks = h.verify(*dev, 1.0, 21)
    assert h.device_status() == 0
    ora = oracle.verify_batch(clean.numpy(), dft.numpy(), p_off.numpy(), q_off.numpy(), x.numpy(),
                              gam.numpy(), 1.0, seed=21)
    assert int(ora["n"][0]) == 0
    ora["gamma"] = gam.numpy()
    ora["seqs"] = np.arange(B)
    assert not compare(n.cpu().numpy(), toks.cpu().numpy(), ora, V)["hard"]
    n2, _ = h.verify(*dev, 1.0, 21, p_lse=torch.empty(B * (gm + 1), device="cuda"),
                     q_lse=torch.empty(B * gm, device="cuda"))
    assert int(n2.cpu()[0]) == -1
    assert h.device_status() & svm.STATUS_BITS["bad_logit"]
    h.close()


def test_deterministic_and_host_buffers(svm):
    batch = workload.make_batch(3, device="cuda", B=10, seed=9)
    h = svm.SpecVerify(batch.B, batch.gamma_max, batch.V)
    a = [t.cpu().clone() for t in h.verify_batch(batch, seed=11)]
    b = [t.cpu().clone() for t in h.verify_batch(batch, seed=11)]
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        c = [t.cpu().clone() for t in h.verify_batch(batch, seed=11, stream=s)]
    assert all(torch.equal(x, y) for x, y in zip(a, c))
    hb = [t.cpu() for t in (batch.target, batch.draft, batch.p_row_off, batch.q_row_off,
                             batch.draft_tokens, batch.gamma)]
    d = h.verify(*hb, batch.T, 11)
    assert not d[0].is_cuda
    assert all(torch.equal(x, y) for x, y in zip(a, d))
    h.close()


def test_first_token_distribution_is_p1(svm):
    """Whole sampling path, statistically: the first emitted token ~ p_1."""
    from scipy import stats
    V, gm, B, T = 48, 2, 100_000, 0.9
    g = torch.Generator(device="cpu").manual_seed(3)
    tgt = (1.2 * torch.randn(gm + 1, V, generator=g)).cuda()
    dft = (1.2 * torch.randn(gm, V, generator=g)).cuda()
    qprob = torch.softmax(dft / T, dim=1)
    x = torch.stack([torch.multinomial(qprob[i], B, replacement=True) for i in range(gm)],
                    1).to(torch.int32)
    zeros = torch.zeros(B, dtype=torch.int64, device="cuda")
    gam = torch.full((B,), gm, dtype=torch.int32, device="cuda")
    h = svm.SpecVerify(B, gm, V)
    n, toks = h.verify(tgt, dft, zeros, zeros, x.contiguous(), gam, T, 123)
    first = toks[:, 0].cpu().numpy()
    counts = np.bincount(first, minlength=V)
    p1 = torch.softmax(tgt[0].double() / T, 0).cpu().numpy()
    assert stats.chisquare(counts, B * p1).pvalue > 1e-4
    beta = np.minimum(p1, torch.softmax(dft[0].double() / T, 0).cpu().numpy()).sum()
    acc = (n.cpu().numpy() >= 1).mean()
    assert abs(acc - beta) < 5 * np.sqrt(beta * (1 - beta) / B)
    h.close()


def test_timing_api(svm):
    # B = 16: the fused kernel (smaller batches take the cluster kernel, below)
    batch = workload.make_batch(1, device="cuda", B=16)
    h = svm.SpecVerify(batch.B, batch.gamma_max, batch.V)
    h.set_timing(True)
    for s in range(3):
        h.verify_batch(batch, seed=s)
    ms, launches = h.get_timing(svm.KERNEL_FUSED, reset=False)
    assert launches == 3 and ms > 0
    assert h.get_timing(svm.KERNEL_PLAN)[1] == 0  # planned inside the fused kernel
    assert h.get_timing(svm.KERNEL_DRAW)[1] == 0  # the draw runs inside the fused kernel
    assert h.get_timing(svm.KERNEL_ROWSTATS)[1] == 0
    ms2, l2 = h.get_timing(svm.KERNEL_FUSED, reset=True)
    assert l2 == 3 and ms2 == ms
    assert h.get_timing(svm.KERNEL_FUSED)[1] == 0
    h.verify_batch(batch, seed=9, greedy=True)
    assert h.get_timing(svm.KERNEL_ROWSTATS)[1] == 1
    assert h.get_timing(svm.KERNEL_ACCEPT)[1] == 1
    assert h.get_timing(svm.KERNEL_FUSED)[1] == 0
    assert h.get_timing(svm.KERNEL_SMALL)[1] == 0
    h.get_timing(svm.KERNEL_FUSED, reset=True)
    # a batch of 8 (gamma <= 16, a few MB of logits): one cluster kernel per call
    small = workload.make_batch(1, device="cuda")
    for s in range(2):
        h.verify_batch(small, seed=s)
    assert h.get_timing(svm.KERNEL_SMALL)[1] == 2
    assert h.get_timing(svm.KERNEL_FUSED)[1] == 0
    h.close()


# Lossy accept test (DistillSpec Sec. 4; Algorithm A.1's threshold
# f(p, eps) / q): every workload at small B and the benchmark workload at full
# size, on both paths, each lenience function; eps = 1 equals the lossless call.
LOSSY = [(0, dict(), "lin", 0.5), (1, dict(), "sq", 0.7), (2, dict(B=8), "exp", 0.4),
         (3, dict(B=24), "sq", 0.3), (4, dict(B=8), "lin", 0.2), (3, dict(), "exp", 0.6),
         (3, dict(), "lin", 0.9)]


@pytest.mark.parametrize("cfg,over,kind,eps", LOSSY,
                         ids=[f"cfg{c}-{k}-{e}" + ("-full" if not o else "")
                              for c, o, k, e in LOSSY])
def test_lossy_parity(svm, cfg, over, kind, eps):
    batch = workload.make_batch(cfg, device="cuda", seed=300 + cfg, **over)
    h = svm.SpecVerify(batch.B, max(batch.gamma_max, 1), batch.V)
    name = workload.CONFIGS[cfg]["name"]
    for seed in (11, 12):
        ora = run_oracle(batch, seed, lenience=kind, eps=eps)
        assert ora["rc"] == 0
        n, toks = h.verify_batch(batch, seed=seed, lenience=kind, eps=eps)
        st = compare(n.cpu().numpy(), toks.cpu().numpy(), ora, batch.V)
        _check(st)
        record(f"{name} lossy {kind}, needed rows", st)
        p_lse, q_lse = lse_buffers(batch)
        n2, toks2 = h.verify_batch(batch, seed=seed, lenience=kind, eps=eps, p_lse=p_lse,
                                   q_lse=q_lse)
        st2 = compare(n2.cpu().numpy(), toks2.cpu().numpy(), ora, batch.V)
        _check(st2)
        record(f"{name} lossy {kind}, every row + lse", st2)
    # f(p, eps) >= p, so with the same uniforms every sequence accepts at
    # least as many drafts as under the lossless test; eps = 1 is lossless
    lossy = h.verify_batch(batch, seed=11, lenience=kind, eps=eps)[0].cpu()
    ref = h.verify_batch(batch, seed=11)
    assert (lossy >= ref[0].cpu()).all()
    one = h.verify_batch(batch, seed=11, lenience=kind, eps=1.0)
    assert torch.equal(one[0], ref[0]) and torch.equal(one[1], ref[1])
    assert h.device_status() & ~INFORMATIONAL == 0
    h.close()


def test_lossy_rejects_bad_eps(svm):
    batch = workload.make_batch(1, device="cuda")
    h = svm.SpecVerify(batch.B, batch.gamma_max, batch.V)
    for kind, eps in (("lin", 0.0), ("sq", 1.5), ("exp", -0.1), ("lin", float("nan"))):
        with pytest.raises(svm.SpecVerifyError) as err:
            h.verify_batch(batch, seed=1, lenience=kind, eps=eps)
        assert err.value.rc == svm.ERR_INVALID_ARG
    h.close()


def test_wait_limit_times_out_cleanly_and_the_next_call_is_exact(svm):
    """A wait on another warp that runs out sets the timeout status bit and the
    kernel returns (no trap, no hang); the handle stays usable and the next
    call, with the default limit, matches the oracle."""
    batch = workload.make_batch(2, device="cuda", B=8, seed=5)
    h = svm.SpecVerify(batch.B, batch.gamma_max, batch.V)
    h.set_wait_limit(1)   # 1 ns: the first poll that finds no work gives up
    n, toks = h.verify_batch(batch, seed=3)
    torch.cuda.synchronize()
    status = h.device_status()
    assert status & svm.STATUS_BITS["timeout"], status
    g = batch.gamma.cpu().numpy()
    n = n.cpu().numpy()
    toks = toks.cpu().numpy()
    assert ((n == -1) | ((n >= 0) & (n <= g))).all()
    assert (toks[n == -1] == -1).all()
    h.set_wait_limit(0)   # back to the default bound
    n2, toks2 = h.verify_batch(batch, seed=3)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    ora = run_oracle(batch, 3)
    _check(compare(n2.cpu().numpy(), toks2.cpu().numpy(), ora, batch.V))
    h.close()


def test_flag_budget_over_the_run(svm):
    """Flagged decisions (inside the rounding bands) are fewer than 1e-4 of
    all decisions compared in this run."""
    if not FLAG_LOG:
        pytest.skip("no comparison ran in this session")
    dec = sum(e["decisions"] for e in FLAG_LOG.values())
    flagged = sum(e["flagged"] for e in FLAG_LOG.values())
    assert flagged < FLAG_BUDGET * dec, "\n".join(flag_report())
