"""Seeded synthetic inputs for the verify step: logit rows, draft tokens, ragged gamma.

This module only *generates* inputs; it holds none of the verify step's
arithmetic. Both the CUDA library's tests/benchmark and the CPU oracle consume
the tensors it returns (the oracle through the numpy views of
``to_host_arrays``).

The rows stand in for the outputs of a target model and a draft model (no
weights or datasets are needed: the verify step only ever sees logit rows).
Recipe, per target row: ``l_v = -s * ln(rank_v) + N(0, sigma_j)`` with ``rank``
a fresh random permutation of 1..V. A draft row is its target row plus
``N(0, sigma_d)`` noise; both are then rounded to the logit dtype. Draft tokens
are drawn from ``softmax(draft_row / T)`` of the *rounded* draft row, i.e. from
the same draft distribution the verifier sees -- this sampling is the drafter's
job, not the verifier's. Optionally a fraction of target rows is made
near-one-hot (the top logit raised to 20 above the runner-up) before the draft
rows are derived from them.

Layout (sequence-major, packed ragged): sequence b owns target rows
``p_row_off[b] .. p_row_off[b] + gamma[b]`` and draft rows
``q_row_off[b] .. q_row_off[b] + gamma[b] - 1``; ``draft_tokens`` is
``[B, gamma_max]`` with unused slots set to 0.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

# The five synthetic workloads (vocabulary sizes: the 32k T5 tokenizer and the
# 128256 / 152064 / 256000 vocabularies of current target models).
CONFIGS = {
    0: dict(name="b1_g4_v32000_fp32_t1.0", B=1, gamma=4, V=32000, dtype="fp32", T=1.0,
            s=1.1, sigma_j=0.5, sigma_d=1.0, seed=0, rounds=200),
    1: dict(name="b8_g5_v32000_bf16_t0.8", B=8, gamma=5, V=32000, dtype="bf16", T=0.8,
            s=1.1, sigma_j=0.5, sigma_d=0.7, seed=1, greedy=True),
    2: dict(name="b64_g8_v128256_bf16_t1.0", B=64, gamma=8, V=128256, dtype="bf16", T=1.0,
            s=1.0, sigma_j=0.5, sigma_d=1.0, seed=2),
    3: dict(name="b256_g1to10_v152064_bf16_t0.7", B=256, gamma=(1, 10), V=152064,
            dtype="bf16", T=0.7, s=1.2, sigma_j=0.5, sigma_d=(0.3, 2.0), seed=3),
    4: dict(name="b512_g7_v256000_fp32_t1.0", B=512, gamma=7, V=256000, dtype="fp32", T=1.0,
            s=0.9, sigma_j=1.0, sigma_d=0.5, seed=4, one_hot_frac=0.1, greedy=True),
}

TORCH_DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class Batch:
    target: torch.Tensor          # [target_rows, V] fp32 or bf16
    draft: torch.Tensor           # [draft_rows, V] same dtype
    p_row_off: torch.Tensor       # [B] int64
    q_row_off: torch.Tensor       # [B] int64
    draft_tokens: torch.Tensor    # [B, gamma_max] int32
    gamma: torch.Tensor           # [B] int32
    T: float
    dtype: str
    gamma_max: int
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.gamma.shape[0])

    @property
    def V(self) -> int:
        return int(self.target.shape[1])

    def logit_bytes(self, greedy: bool = False) -> int:
        """Bytes of logits one verify call reads once: every target row, plus
        every draft row when sampling."""
        esz = self.target.element_size()
        g = self.gamma.to(torch.int64)
        rows = int((g + 1).sum()) + (0 if greedy else int(g.sum()))
        return rows * self.V * esz

    def draft_token_count(self) -> int:
        return int(self.gamma.to(torch.int64).sum())


def _rows_zipf(gen, rows, V, s, sigma_j, device, chunk):
    base = -s * torch.log(torch.arange(1, V + 1, device=device, dtype=torch.float32))
    out = torch.empty(rows, V, device=device, dtype=torch.float32)
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        u = torch.rand(r1 - r0, V, generator=gen, device=device)
        perm = torch.argsort(u, dim=1)
        del u
        blk = torch.empty(r1 - r0, V, device=device, dtype=torch.float32)
        blk.scatter_(1, perm, base.expand(r1 - r0, V))
        del perm
        blk += sigma_j * torch.randn(r1 - r0, V, generator=gen, device=device)
        out[r0:r1] = blk
    return out


def make_batch(cfg, device="cpu", *, B=None, V=None, gamma=None, seed=None,
               chunk_rows=256) -> Batch:
    """Build one synthetic batch for config `cfg` (a dict or a CONFIGS key).

    B, V, gamma and seed override the config (tests use smaller shapes with
    the same value distributions). gamma may be an int or an (lo, hi) range
    for a ragged batch (uniform per sequence, inclusive).
    """
    if not isinstance(cfg, dict):
        cfg = CONFIGS[int(cfg)]
    B = int(cfg["B"] if B is None else B)
    V = int(cfg["V"] if V is None else V)
    gspec = cfg["gamma"] if gamma is None else gamma
    seed = int(cfg["seed"] if seed is None else seed)
    T = float(cfg["T"])
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)

    if isinstance(gspec, (tuple, list)):
        lo, hi = int(gspec[0]), int(gspec[1])
        g = torch.randint(lo, hi + 1, (B,), generator=gen, device=dev)
        gamma_max = hi
    else:
        g = torch.full((B,), int(gspec), device=dev, dtype=torch.int64)
        gamma_max = int(gspec)
    g = g.to(torch.int64)

    sd = cfg["sigma_d"]
    if isinstance(sd, (tuple, list)):
        sigma_d = sd[0] + (sd[1] - sd[0]) * torch.rand(B, generator=gen, device=dev)
    else:
        sigma_d = torch.full((B,), float(sd), device=dev)

    p_cnt = g + 1
    p_off = torch.cumsum(p_cnt, 0) - p_cnt
    q_off = torch.cumsum(g, 0) - g
    P = int(p_cnt.sum())
    Q = int(g.sum())

    target32 = _rows_zipf(gen, P, V, float(cfg["s"]), float(cfg["sigma_j"]), dev, chunk_rows)
    frac = float(cfg.get("one_hot_frac", 0.0))
    if frac > 0.0:
        pick = torch.rand(P, generator=gen, device=dev) < frac
        idx = torch.nonzero(pick).flatten()
        for r0 in range(0, idx.numel(), chunk_rows):
            rows = idx[r0:r0 + chunk_rows]
            blk = target32[rows]
            top2 = torch.topk(blk, 2, dim=1)
            k = top2.indices[:, 0]
            blk[torch.arange(blk.shape[0], device=dev), k] = top2.values[:, 1] + 20.0
            target32[rows] = blk

    tdt = TORCH_DTYPES[cfg["dtype"]]
    # draft rows: target row (b, i) + per-sequence noise, for i = 1..gamma_b
    seq_of_q = torch.repeat_interleave(torch.arange(B, device=dev), g)
    pos_of_q = torch.arange(Q, device=dev) - q_off[seq_of_q]
    src_rows = p_off[seq_of_q] + pos_of_q
    draft = torch.empty(Q, V, device=dev, dtype=tdt)
    tokens_flat = torch.empty(Q, device=dev, dtype=torch.int64)
    for r0 in range(0, Q, chunk_rows):
        r1 = min(Q, r0 + chunk_rows)
        noise = torch.randn(r1 - r0, V, generator=gen, device=dev)
        blk = (target32[src_rows[r0:r1]] + noise * sigma_d[seq_of_q[r0:r1]].unsqueeze(1)).to(tdt)
        draft[r0:r1] = blk
        probs = torch.softmax(blk.to(torch.float32) / T, dim=1)
        tokens_flat[r0:r1] = torch.multinomial(probs, 1, generator=gen).flatten()
    target = target32.to(tdt)
    del target32

    draft_tokens = torch.zeros(B, max(gamma_max, 1), device=dev, dtype=torch.int32)
    if Q > 0:
        draft_tokens[seq_of_q, pos_of_q] = tokens_flat.to(torch.int32)
    draft_tokens = draft_tokens[:, :gamma_max].contiguous()
    meta = dict(cfg)
    meta.update(B=B, V=V, seed=seed, gamma_spec=gspec)
    return Batch(target=target.contiguous(), draft=draft.contiguous(),
                 p_row_off=p_off.contiguous(), q_row_off=q_off.contiguous(),
                 draft_tokens=draft_tokens, gamma=g.to(torch.int32).contiguous(), T=T,
                 dtype=cfg["dtype"], gamma_max=gamma_max, meta=meta)


def to_numpy_logits(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of logit rows: float32, or uint16 bit patterns for bf16."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_host_arrays(batch: Batch, seqs=None) -> dict:
    """Host copies of a batch (or of the sequences `seqs` of it, repacked),
    in the argument order of the oracle's batch call. `seq_ids` keeps the
    original sequence indices so that counter-based uniforms line up."""
    if seqs is None:
        return dict(target=to_numpy_logits(batch.target), draft=to_numpy_logits(batch.draft),
                    p_row_off=batch.p_row_off.cpu().numpy(),
                    q_row_off=batch.q_row_off.cpu().numpy(),
                    draft_tokens=batch.draft_tokens.cpu().numpy(),
                    gamma=batch.gamma.cpu().numpy(), seq_ids=None)
    seqs = [int(s) for s in seqs]
    g = batch.gamma.cpu().numpy()
    p_off = batch.p_row_off.cpu().numpy()
    q_off = batch.q_row_off.cpu().numpy()
    p_rows, q_rows, np_off, nq_off = [], [], [], []
    pc = qc = 0
    for b in seqs:
        np_off.append(pc)
        nq_off.append(qc)
        p_rows.extend(range(p_off[b], p_off[b] + g[b] + 1))
        q_rows.extend(range(q_off[b], q_off[b] + g[b]))
        pc += g[b] + 1
        qc += g[b]
    dev = batch.target.device
    tgt = to_numpy_logits(batch.target[torch.tensor(p_rows, device=dev, dtype=torch.long)])
    if q_rows:
        dft = to_numpy_logits(batch.draft[torch.tensor(q_rows, device=dev, dtype=torch.long)])
    else:
        dft = tgt[:1]
    return dict(target=tgt, draft=dft, p_row_off=np.array(np_off, np.int64),
                q_row_off=np.array(nq_off, np.int64),
                draft_tokens=batch.draft_tokens.cpu().numpy()[seqs],
                gamma=g[seqs].astype(np.int32), seq_ids=np.array(seqs, np.int32))
