"""The small-batch sampling and greedy kernels (one thread-block cluster per
sequence) against the oracle, through the C ABI.

Batches of at most 8 sequences with gamma_max <= 16 whose row slices fit a
CTA's shared memory take this kernel instead of the fused one; both compute
the step of "DistillSpec" Sec. 3 / App. A.3 Algorithm A.1. Decision rule as in
the other parity tests (bit-exact outside the R11/R12 bands). Cases at the
kernel's limits: 8 sequences, gamma up to 16, vocabularies with a ragged tail
(the last CTA's slice), fp32 and bf16, every lenience, gamma = 0, bad logits in
rows the result needs and in rows it does not (ignored without logsumexp
outputs, as the large-batch kernel does), and the logsumexp outputs.
"""
import numpy as np
import pytest
import torch

import oracle

from parity_util import compare, lse_buffers, lse_errors, record, run_oracle, LSE_RTOL
from speculative_decoding_token_gb300 import workload

pytestmark = pytest.mark.gpu

INFORMATIONAL = (1 << 8) | (1 << 9)


@pytest.fixture(scope="module")
def svm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_token_gb300 as sv
    import oracle
    sv.build()
    sv.load()
    oracle.build()
    return sv


def _padded(batch):
    if batch.V % 8:
        pad = (batch.V + 7) // 8 * 8
        for name in ("target", "draft"):
            t = getattr(batch, name)
            full = torch.zeros(t.shape[0], pad, dtype=t.dtype, device=t.device)
            full[:, :batch.V] = t
            setattr(batch, name, full[:, :batch.V])
    return batch


CASES = {
    # label: (config, overrides, verify seeds)
    "b8_g0to16_v20000_bf16": (1, dict(B=8, V=20000, gamma=(0, 16)), (1, 2, 3)),
    "b8_g0to16_v20003_bf16": (1, dict(B=8, V=20003, gamma=(0, 16)), (4, 5)),
    "b7_g0to16_v1001_fp32": (0, dict(B=7, V=1001, gamma=(0, 16)), (6, 7)),
    "b3_g5_v9999_fp32": (0, dict(B=3, V=9999, gamma=5), (8, 9)),
    "b8_g5_v32000_bf16": (1, dict(), (10, 11)),
}


@pytest.mark.parametrize("label", sorted(CASES))
def test_small_kernel_parity(svm, label):
    cfg, over, seeds = CASES[label]
    batch = _padded(workload.make_batch(cfg, device="cuda", seed=700 + len(label), **over))
    h = svm.SpecVerify(batch.B, max(batch.gamma_max, 1), batch.V)
    h.set_timing(True)
    for seed in seeds:
        for lse in (False, True):
            p_lse, q_lse = lse_buffers(batch)
            n, toks = h.verify_batch(batch, seed=seed, p_lse=p_lse if lse else None,
                                     q_lse=q_lse if lse else None)
            ora = run_oracle(batch, seed)
            assert ora["rc"] == 0
            st = compare(n.cpu().numpy(), toks.cpu().numpy(), ora, batch.V)
            assert not st["hard"], st["hard"][:5]
            record(f"small kernel {label}", st)
            if lse:
                assert lse_errors(batch, ora, p_lse, q_lse) <= LSE_RTOL
    assert h.get_timing(svm.KERNEL_SMALL)[1] == 2 * len(seeds)
    assert h.get_timing(svm.KERNEL_FUSED)[1] == 0
    assert h.device_status() & ~INFORMATIONAL == 0
    h.close()


@pytest.mark.parametrize("kind,eps", [("lin", 0.5), ("sq", 0.7), ("exp", 0.4)])
def test_small_kernel_lenience(svm, kind, eps):
    batch = _padded(workload.make_batch(1, device="cuda", seed=740, B=8, V=20000,
                                        gamma=(0, 16)))
    h = svm.SpecVerify(batch.B, batch.gamma_max, batch.V)
    for seed in (21, 22):
        n, toks = h.verify_batch(batch, seed=seed, lenience=kind, eps=eps)
        ora = run_oracle(batch, seed, lenience=kind, eps=float(np.float32(eps)))
        assert ora["rc"] == 0
        st = compare(n.cpu().numpy(), toks.cpu().numpy(), ora, batch.V)
        assert not st["hard"], st["hard"][:5]
        record(f"small kernel lossy {kind}", st)
    assert h.device_status() & ~INFORMATIONAL == 0
    h.close()


def test_small_kernel_bad_rows(svm):
    """A NaN in a row the result needs fails its sequence; after the first
    rejection it is ignored without logsumexp outputs and fails the sequence
    with them (every row is then validated). Other sequences are unaffected."""
    batch = workload.make_batch(1, device="cuda", seed=750, B=6, V=20000, gamma=6)
    seed = 31
    n0, _ = svm.SpecVerify(batch.B, batch.gamma_max, batch.V).verify_batch(batch, seed=seed)
    n0 = n0.cpu().numpy()
    # a sequence that rejects early: poison its last target row (after the rejection)
    early = [b for b in range(batch.B) if n0[b] <= 2]
    assert early, n0
    b_late = early[0]
    tgt = batch.target.clone()
    p_off = batch.p_row_off.cpu().numpy()
    tgt[int(p_off[b_late]) + batch.gamma_max, 11] = float("nan")
    # another sequence: poison its first target row (always needed)
    b_first = next(b for b in range(batch.B) if b != b_late)
    tgt[int(p_off[b_first]), 7] = float("nan")
    bad = workload.Batch(**{**batch.__dict__, "target": tgt})
    h = svm.SpecVerify(batch.B, batch.gamma_max, batch.V)
    n, toks = h.verify_batch(bad, seed=seed)
    n, toks = n.cpu().numpy(), toks.cpu().numpy()
    assert n[b_first] == -1 and (toks[b_first] == -1).all()
    assert n[b_late] == n0[b_late]
    for b in range(batch.B):
        if b not in (b_first,):
            assert n[b] == n0[b]
    assert h.device_status() & ~INFORMATIONAL == 8  # BAD_LOGIT
    p_lse, q_lse = lse_buffers(bad)
    n2, _ = h.verify_batch(bad, seed=seed, p_lse=p_lse, q_lse=q_lse)
    n2 = n2.cpu().numpy()
    assert n2[b_late] == -1 and n2[b_first] == -1
    h.close()


GREEDY_CASES = {
    # label: (config, overrides)
    "b8_g0to16_v20003_bf16": (1, dict(B=8, V=20003, gamma=(0, 16))),
    "b8_g5_v32000_bf16": (1, dict()),
    "b6_g7_v256000_fp32": (4, dict(B=6)),
    "b3_g4_v1001_fp32": (0, dict(B=3, V=1001, gamma=4)),
}


@pytest.mark.parametrize("label", sorted(GREEDY_CASES))
def test_small_greedy_parity(svm, label):
    """The greedy step of a small batch (one cluster per sequence) is bit-exact
    with the oracle: drafts mostly equal to the target argmax (long prefixes),
    ragged vocabularies, gamma from 0 to 16, bf16 and fp32."""
    cfg, over = GREEDY_CASES[label]
    batch = _padded(workload.make_batch(cfg, device="cuda", seed=760 + len(label), **over))
    am = batch.draft_tokens.clone()
    g = batch.gamma.cpu().tolist()
    p_off = batch.p_row_off.cpu().tolist()
    for b in range(batch.B):
        for i in range(g[b]):
            am[b, i] = batch.target[p_off[b] + i].float().argmax().to(torch.int32)
    gen = torch.Generator(device="cpu").manual_seed(761)
    keep = (torch.rand(batch.B, batch.gamma_max, generator=gen) < 0.8).to("cuda")
    batch.draft_tokens = torch.where(keep, am, batch.draft_tokens).contiguous()
    h = svm.SpecVerify(batch.B, max(batch.gamma_max, 1), batch.V)
    h.set_timing(True)
    n, toks = h.verify_batch(batch, greedy=True)
    ora = run_oracle(batch, 0, greedy=True)
    assert ora["rc"] == 0
    st = compare(n.cpu().numpy(), toks.cpu().numpy(), ora, batch.V, greedy=True)
    assert not st["hard"], st["hard"][:5]
    assert (n.cpu().numpy() > 0).any()
    assert h.get_timing(svm.KERNEL_SMALL)[1] == 1
    assert h.get_timing(svm.KERNEL_ROWSTATS)[1] == 0
    assert h.device_status() == 0
    h.close()


def test_small_greedy_ties_and_bad_rows(svm):
    """Ties go to the lower index across the cluster's column slices; an all
    -inf row has argmax 0; a NaN in a row the scan reads fails only its
    sequence; bad gamma, offsets and tokens are reported as on the other path."""
    B, gm, V = 6, 4, 3000
    g = torch.Generator().manual_seed(5)
    tgt = torch.randint(0, 3, (B * (gm + 1), V), generator=g).float()
    tgt[0, :] = float("-inf")                  # sequence 0, row 1: argmax 0
    tgt[5 + 2, 2999] = 50.0                    # sequence 1, row 3: the last column
    tgt[5 + 2, 1] = 50.0                       # ... tied with column 1: 1 wins
    tgt[10 + 1, 7] = float("nan")              # sequence 2, row 2
    p_off = torch.arange(B, dtype=torch.int64) * (gm + 1)
    gam = torch.tensor([4, 4, 4, 4, 2, 3], dtype=torch.int32)
    x = torch.zeros(B, gm, dtype=torch.int32)
    for b in range(B):
        for i in range(gm):
            x[b, i] = int(torch.argmax(tgt[p_off[b] + i]))
    x[3, 1] = V + 5                            # a bad token
    p_off[4] = B * (gm + 1) - 1                # rows past the end
    gam[5] = gm + 3                            # a bad gamma
    dev = [t.cuda() for t in (tgt, p_off, x, gam)]
    h = svm.SpecVerify(B, gm, V)
    n, toks = h.verify(dev[0], None, dev[1], None, dev[2], dev[3], 0.0, 0, greedy=True)
    n, toks = n.cpu().numpy(), toks.cpu().numpy()
    ora = oracle.verify_batch(tgt.numpy(), None, p_off.numpy(), None, x.numpy(), gam.numpy(), 0.0)
    assert list(n) == list(ora["n"])
    assert (toks == ora["tokens"]).all()
    status = h.device_status()
    for bit in ("bad_gamma", "bad_token", "bad_row", "bad_logit"):
        assert status & svm.STATUS_BITS[bit], (bit, status)
    assert n[0] >= 0 and n[1] >= 0 and (n[2:] == -1).all()
    h.close()
