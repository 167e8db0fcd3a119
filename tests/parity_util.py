"""Comparison of the CUDA verify step with the CPU oracle.

Decision rule (the tolerance of the verify step's specification): accepted
counts and emitted tokens must be bit-exact, except at decisions whose margin
is below a band -- an accept test with |r - p/q| < 1e-5, or a final draw whose
point t lies within 1e-5 / V of a CDF boundary, measured in units of the
total mass (the gap is read in units of the mean token mass 1/V; a literal
absolute 1e-5 would flag most draws at V >= 1e5). Flagged decisions are
counted; any mismatch outside the bands fails.
"""
import numpy as np
import torch

import oracle
from speculative_decoding_token_gb300 import workload

ACC_BAND = 1e-5
DRAW_BAND_UNITS = 1e-5     # times 1/V
LSE_RTOL = 1e-5
# The budget of the verify step's specification: flagged decisions must be
# fewer than this fraction of all decisions, summed over a run.
FLAG_BUDGET = 1e-4

# Decisions and flags of every GPU-vs-oracle comparison of the session, per
# workload label: the full-size parity tests add to it, a final test checks
# the summed budget and the terminal summary prints the rates.
FLAG_LOG = {}


def record(label, st):
    """Add the counts of one comparison to the session's flag log."""
    e = FLAG_LOG.setdefault(label, dict(comparisons=0, decisions=0, flagged=0,
                                        flagged_literal=0, mismatches=0,
                                        flagged_mismatches=0))
    e["comparisons"] += 1
    for k in ("decisions", "flagged", "flagged_literal", "mismatches", "flagged_mismatches"):
        e[k] += int(st[k])


def flag_report():
    """Lines of a per-workload table of flag rates (both readings of the draw band)."""
    lines = []
    tot = dict(decisions=0, flagged=0, flagged_literal=0, mismatches=0)
    for label in sorted(FLAG_LOG):
        e = FLAG_LOG[label]
        for k in tot:
            tot[k] += e[k]
        d = max(e["decisions"], 1)
        lines.append(f"{label:44s} comparisons {e['comparisons']:5d} decisions {e['decisions']:7d} "
                     f"flagged {e['flagged']:3d} ({e['flagged'] / d:.2e}) literal-band flagged "
                     f"{e['flagged_literal']:6d} ({e['flagged_literal'] / d:.2e}) mismatches "
                     f"{e['mismatches']} (all flagged: {e['flagged_mismatches']})")
    if FLAG_LOG:
        d = max(tot["decisions"], 1)
        lines.append(f"{'total':44s} decisions {tot['decisions']:7d} flagged {tot['flagged']} "
                     f"({tot['flagged'] / d:.2e}; budget < {FLAG_BUDGET:g}) literal-band flagged "
                     f"{tot['flagged_literal']} ({tot['flagged_literal'] / d:.2e}) mismatches "
                     f"{tot['mismatches']}")
    return lines


def oracle_temperature(T):
    """The library receives T as a float; the oracle must see the same value."""
    return float(np.float32(T))


def run_oracle(batch, seed, greedy=False, seqs=None, lenience="none", eps=1.0):
    a = workload.to_host_arrays(batch, seqs)
    T = 0.0 if greedy else oracle_temperature(batch.T)
    res = oracle.verify_batch(a["target"], None if greedy else a["draft"], a["p_row_off"],
                              a["q_row_off"], a["draft_tokens"], a["gamma"], T, seed=seed,
                              seq_ids=a["seq_ids"], lenience=lenience,
                              eps=float(np.float32(eps)))
    res["gamma"] = a["gamma"]
    res["seqs"] = a["seq_ids"] if a["seq_ids"] is not None else np.arange(len(a["gamma"]))
    return res


def compare(gpu_n, gpu_tok, ora, V, greedy=False):
    """Per-sequence comparison; returns counts and the list of hard mismatches."""
    gpu_n = np.asarray(gpu_n)
    gpu_tok = np.asarray(gpu_tok)
    st = dict(sequences=len(gpu_n), decisions=0, flagged=0, flagged_literal=0, mismatches=0,
              flagged_mismatches=0, hard=[])
    band = DRAW_BAND_UNITS / V
    for j, b in enumerate(ora["seqs"]):
        on, gn = int(ora["n"][j]), int(gpu_n[j])
        g = int(ora["gamma"][j])
        if on < 0 or gn < 0:
            if on != gn or not (gpu_tok[j] == -1).all():
                st["hard"].append((int(b), "validity", on, gn))
            continue
        if greedy:
            st["decisions"] += min(on + 1, g) + 1
            if on != gn or not np.array_equal(ora["tokens"][j], gpu_tok[j]):
                st["mismatches"] += 1
                st["hard"].append((int(b), "greedy", on, gn))
            continue
        k = min(on + 1, g)
        m = ora["acc_margin"][j][:k]
        st["decisions"] += k + 1
        st["flagged"] += int((m < ACC_BAND).sum())
        dm = float(ora["draw_margin"][j])
        st["flagged"] += int(dm < band)
        st["flagged_literal"] += int((m < ACC_BAND).sum()) + int(dm < 1e-5)
        if gn != on:
            st["mismatches"] += 1
            i = min(gn, on)
            if i < g and ora["acc_margin"][j][i] < ACC_BAND:
                st["flagged_mismatches"] += 1
            else:
                st["hard"].append((int(b), "accept", on, gn, float(ora["acc_margin"][j][i])
                                   if i < g else None))
        elif not np.array_equal(ora["tokens"][j], gpu_tok[j]):
            st["mismatches"] += 1
            if dm < band:
                st["flagged_mismatches"] += 1
            else:
                st["hard"].append((int(b), "draw", int(ora["tokens"][j][on]),
                                   int(gpu_tok[j][on]), dm))
    return st


def lse_errors(batch, ora, p_lse, q_lse):
    """Largest relative lse error over the rows of the compared sequences."""
    p_lse = p_lse.detach().cpu().numpy().astype(np.float64)
    q_lse = q_lse.detach().cpu().numpy().astype(np.float64)
    p_off = batch.p_row_off.cpu().numpy()
    q_off = batch.q_row_off.cpu().numpy()
    worst = 0.0
    for j, b in enumerate(ora["seqs"]):
        if ora["n"][j] < 0:
            continue
        g = int(ora["gamma"][j])
        for i in range(g + 1):
            want = ora["lse_p"][j][i]
            got = p_lse[p_off[b] + i]
            worst = max(worst, abs(got - want) / max(1.0, abs(want)))
        for i in range(g):
            want = ora["lse_q"][j][i]
            got = q_lse[q_off[b] + i]
            worst = max(worst, abs(got - want) / max(1.0, abs(want)))
    return worst


def lse_buffers(batch):
    dev = batch.target.device
    return (torch.full((batch.target.shape[0],), float("nan"), device=dev),
            torch.full((max(batch.draft.shape[0], 1),), float("nan"), device=dev))
