"""Parity of the per-row diagnostics with the CPU oracle, through the C ABI.

* Acceptance statistics ("DistillSpec" Sec. 3 beta = sum min(p, q); Sec. 4
  TVD): beta and TVD of every position of the workloads, against the
  oracle's double-precision sums. Tolerance 1e-5 absolute on each (both lie
  in [0, 1]): the kernel's fp32 terms carry about 2e-6 relative error (the
  exponent rounding of l log2(e)/T - log2 S), so the sums are good to a few
  1e-6.
* Draft features ("DISCO" Sec. 3 Eq. 2, App. D.1): entropy within 1e-5
  relative (floor 1 on |H|, the logsumexp rule), top-k probabilities within
  1e-5 relative, top-k token indices bit-exact (an ordering of the raw
  logits with ties to the lower index), on Zipf-shaped, near-one-hot and
  tie-heavy rows, fp32 and bf16, ragged vocabularies.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import oracle_temperature
from speculative_decoding_token_gb300 import workload

pytestmark = pytest.mark.gpu

STAT_ATOL = 1e-5
ENT_RTOL = 1e-5
PROB_RTOL = 1e-5


@pytest.fixture(scope="module")
def svm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_token_gb300 as sv
    sv.build()
    sv.load()
    oracle.build()
    return sv


@pytest.mark.parametrize("cfg,over", [(1, dict()), (2, dict(B=16)), (3, dict()),
                                      (4, dict(B=24)), (0, dict(B=3, V=1001))],
                         ids=["cfg1", "cfg2-B16", "cfg3-full", "cfg4-B24", "cfg0-V1001"])
def test_acceptance_stats_parity(svm, cfg, over):
    batch = workload.make_batch(cfg, device="cuda", seed=900 + cfg, **over)
    if batch.V % 8:
        # a ragged vocabulary: rows padded to a 16-byte stride
        pad = (batch.V + 7) // 8 * 8
        for name in ("target", "draft"):
            t = getattr(batch, name)
            full = torch.zeros(t.shape[0], pad, dtype=t.dtype, device=t.device)
            full[:, :batch.V] = t
            setattr(batch, name, full[:, :batch.V])
    h = svm.SpecVerify(batch.B, max(batch.gamma_max, 1), batch.V)
    beta, tvd = h.acceptance_stats(batch)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    a = workload.to_host_arrays(batch)
    ora = oracle.pair_stats_batch(a["target"], a["draft"], a["p_row_off"], a["q_row_off"],
                                  a["gamma"], oracle_temperature(batch.T))
    assert ora["rc"] == 0
    gb, gt = beta.cpu().numpy().astype(np.float64), tvd.cpu().numpy().astype(np.float64)
    ob, ot = ora["beta"], ora["tvd"]
    gm = batch.gamma_max
    assert gb.shape == ob.shape == (batch.B, gm)
    assert (np.isnan(gb) == np.isnan(ob)).all()
    m = ~np.isnan(ob)
    assert np.abs(gb[m] - ob[m]).max() <= STAT_ATOL
    assert np.abs(gt[m] - ot[m]).max() <= STAT_ATOL
    h.close()


def test_acceptance_stats_special_cases(svm):
    V, B, gm = 5000, 3, 2
    g = torch.Generator().manual_seed(2)
    tgt = torch.randn(B * (gm + 1), V, generator=g)
    dft = torch.randn(B * gm, V, generator=g)
    dft[0] = tgt[0]                                   # q = p at (0, 1): beta 1, TVD 0
    dft[2, :2500] = float("-inf")                     # disjoint supports at (1, 1)
    tgt[3, 2500:] = float("-inf")
    tgt[6 + 1, 17] = float("nan")                     # bad row at (2, 2)
    gam = torch.full((B,), gm, dtype=torch.int32)
    p_off = torch.arange(B, dtype=torch.int64) * (gm + 1)
    q_off = torch.arange(B, dtype=torch.int64) * gm
    x = torch.zeros(B, gm, dtype=torch.int32)
    batch = workload.Batch(tgt.cuda(), dft.cuda(), p_off.cuda(), q_off.cuda(), x.cuda(),
                           gam.cuda(), 1.0, "fp32", gm)
    h = svm.SpecVerify(B, gm, V)
    beta, tvd = h.acceptance_stats(batch)
    beta, tvd = beta.cpu().numpy(), tvd.cpu().numpy()
    assert abs(beta[0, 0] - 1.0) < 1e-5 and abs(tvd[0, 0]) < 1e-6
    assert beta[1, 0] == 0.0 and abs(tvd[1, 0] - 1.0) < 1e-5
    assert np.isnan(beta[2, 1]) and np.isnan(tvd[2, 1]) and not np.isnan(beta[2, 0])
    assert h.device_status() & svm.STATUS_BITS["bad_logit"]
    h.close()


def _feature_rows(kind, device="cuda"):
    g = torch.Generator(device="cpu").manual_seed(7)
    if kind == "cfg1-draft":
        return workload.make_batch(1, device=device, seed=71).draft
    if kind == "cfg3-draft":
        return workload.make_batch(3, device=device, seed=73, B=48).draft
    if kind == "cfg4-target":   # fp32, 10 % near-one-hot rows
        return workload.make_batch(4, device=device, seed=74, B=12).target
    if kind == "ties-bf16":     # a few distinct values: many ties at the top
        return torch.randint(0, 6, (37, 20000), generator=g).to(torch.bfloat16).to(device)
    if kind == "ragged-fp32":   # V not a multiple of the vector width, padded stride
        full = (3 * torch.randn(9, 1004, generator=g)).to(device)
        return full[:, :1001]
    if kind in ("masked-bf16", "masked-fp32"):   # -inf logits (a masked vocabulary)
        rows = 3 * torch.randn(8, 12000, generator=g)
        rows[0, :6000] = float("-inf")
        rows[1, ::3] = float("-inf")
        rows[2, 3:] = float("-inf")                  # three tokens left
        rows[3, torch.randperm(12000, generator=g)[:9000]] = float("-inf")
        dt = torch.bfloat16 if kind == "masked-bf16" else torch.float32
        return rows.to(dt).to(device)
    raise KeyError(kind)


@pytest.mark.parametrize("kind,T,k", [("cfg1-draft", 0.8, 10), ("cfg3-draft", 0.7, 32),
                                      ("cfg4-target", 1.0, 8), ("ties-bf16", 1.0, 16),
                                      ("ragged-fp32", 0.6, 5), ("cfg1-draft", 1.3, 1),
                                      ("masked-bf16", 0.7, 12), ("masked-fp32", 1.0, 4),
                                      ("masked-bf16", 0.3, 3)])
def test_row_features_parity(svm, kind, T, k):
    rows = _feature_rows(kind)
    h = svm.SpecVerify(1, 1, rows.shape[1])
    ent, prob, idx = h.row_features(rows, T, k)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    host = workload.to_numpy_logits(rows)
    ora = oracle.row_features_batch(host, oracle_temperature(T), k)
    assert ora["rc"] == 0
    ge = ent.cpu().numpy().astype(np.float64)
    assert (np.abs(ge - ora["entropy"]) <= ENT_RTOL * np.maximum(1.0, np.abs(ora["entropy"]))).all()
    np.testing.assert_array_equal(idx.cpu().numpy(), ora["topk_idx"])
    gp = prob.cpu().numpy().astype(np.float64)
    assert (np.abs(gp - ora["topk_prob"]) <= PROB_RTOL * ora["topk_prob"] + 1e-12).all()
    h.close()


def test_row_features_bad_rows_and_k_past_v(svm):
    rows = torch.randn(4, 3000, device="cuda")
    rows[1, 5] = float("nan")
    rows[2, :] = float("-inf")
    rows[3, 7] = float("inf")
    h = svm.SpecVerify(1, 1, 3000)
    ent, prob, idx = h.row_features(rows, 1.0, 4)
    ent, prob, idx = ent.cpu().numpy(), prob.cpu().numpy(), idx.cpu().numpy()
    assert not np.isnan(ent[0]) and np.isnan(ent[1:]).all()
    assert (idx[1:] == -1).all() and np.isnan(prob[1:]).all()
    assert h.device_status() & svm.STATUS_BITS["bad_logit"]
    small = torch.randn(2, 4, device="cuda")[:, :3]      # V = 3, rows 16 bytes apart
    ent, prob, idx = h.row_features(small, 1.0, 5)
    assert (idx.cpu().numpy()[:, 3:] == -1).all() and (prob.cpu().numpy()[:, 3:] == 0).all()
    h.close()
