"""TEST INFRASTRUCTURE: the CPU oracle of the speculative-sampling verify step.

A plain double-precision C implementation (``specverify_oracle.c``) with its
own Philox4x32-10, loaded through ctypes. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package; the library under ``speculative_decoding_token_gb300`` never
does, and the oracle never calls the library.

Logit rows are passed as numpy arrays: ``float32`` for fp32 logits, or
``uint16`` holding the raw bf16 bit patterns for bf16 logits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specverify_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_ARG = -1
ERR_INPUT = -4

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_f64p = ctypes.POINTER(ctypes.c_double)
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build/liboracle.so``.

    ``-ffp-contract=off`` keeps every double operation separately rounded, so
    the oracle gives the same results on x86-64 and aarch64 hosts.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
        lib.oracle_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_u24.argtypes = [ctypes.c_uint32]
        lib.oracle_u24.restype = ctypes.c_double
        lib.oracle_u52.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
        lib.oracle_u52.restype = ctypes.c_double
        lib.oracle_accept_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
        lib.oracle_accept_uniform.restype = ctypes.c_double
        lib.oracle_draw_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
        lib.oracle_draw_uniform.restype = ctypes.c_double
        lib.oracle_row_lse.argtypes = [_vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_double, _f64p]
        lib.oracle_row_lse.restype = ctypes.c_int
        lib.oracle_row_argmax.argtypes = [_vp, ctypes.c_int32, ctypes.c_int64, _i64p]
        lib.oracle_row_argmax.restype = ctypes.c_int
        lib.oracle_verify_seq_u.argtypes = [
            _vp, _vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _i32p,
            ctypes.c_double, _f64p, ctypes.c_double, _i32p, _i32p, _f64p, _f64p, _f64p, _f64p,
            _i32p]
        lib.oracle_verify_seq_u.restype = ctypes.c_int
        lib.oracle_verify_greedy_seq.argtypes = [
            _vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _i32p, _i32p,
            _i32p]
        lib.oracle_verify_greedy_seq.restype = ctypes.c_int
        lib.oracle_verify_seq_u_lenient.argtypes = [
            _vp, _vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _i32p,
            ctypes.c_double, ctypes.c_int32, ctypes.c_double, _f64p, ctypes.c_double, _i32p,
            _i32p, _f64p, _f64p]
        lib.oracle_verify_seq_u_lenient.restype = ctypes.c_int
        lib.oracle_verify_batch_lenient.argtypes = [
            _vp, _vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, _i32p, _i32p, _i32p,
            ctypes.c_double, ctypes.c_int32, ctypes.c_double, ctypes.c_uint64, _i32p, _i32p,
            _f64p, _f64p, _f64p, _f64p, _i32p, ctypes.c_int32]
        lib.oracle_verify_batch_lenient.restype = ctypes.c_int
        lib.oracle_pair_stats.argtypes = [_vp, _vp, ctypes.c_int32, ctypes.c_int64,
                                          ctypes.c_double, _f64p, _f64p]
        lib.oracle_pair_stats.restype = ctypes.c_int
        lib.oracle_row_features.argtypes = [_vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_double,
                                            ctypes.c_int32, _f64p, _f64p, _i64p]
        lib.oracle_row_features.restype = ctypes.c_int
        lib.oracle_pair_stats_batch.argtypes = [
            _vp, _vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, _i32p,
            ctypes.c_double, _f64p, _f64p, ctypes.c_int32]
        lib.oracle_pair_stats_batch.restype = ctypes.c_int
        lib.oracle_row_features_batch.argtypes = [
            _vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_double,
            ctypes.c_int32, _f64p, _f64p, _i64p, ctypes.c_int32]
        lib.oracle_row_features_batch.restype = ctypes.c_int
        lib.oracle_verify_batch_restricted.argtypes = [
            _vp, _vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, _i32p, _i32p, _i32p,
            _f64p, _i32p, _f64p, ctypes.c_uint64, _i32p, _i32p, _f64p, _f64p, ctypes.c_int32]
        lib.oracle_verify_batch_restricted.restype = ctypes.c_int
        lib.oracle_verify_seq_restricted_u.argtypes = [
            _vp, _vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _i32p,
            ctypes.c_double, ctypes.c_int32, ctypes.c_double, _f64p, ctypes.c_double, _i32p,
            _i32p]
        lib.oracle_verify_seq_restricted_u.restype = ctypes.c_int
        lib.oracle_restricted_row.argtypes = [_vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_double,
                                              ctypes.c_int32, ctypes.c_double, _f64p]
        lib.oracle_restricted_row.restype = ctypes.c_int
        lib.oracle_verify_batch.argtypes = [
            _vp, _vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, _i32p, _i32p, _i32p,
            ctypes.c_double, ctypes.c_uint64, _i32p, _i32p, _f64p, _f64p, _f64p, _f64p, _i32p,
            ctypes.c_int32]
        lib.oracle_verify_batch.restype = ctypes.c_int
        lib.oracle_block_efficiency.argtypes = [ctypes.c_double, ctypes.c_int32]
        lib.oracle_block_efficiency.restype = ctypes.c_double
        lib.oracle_expected_emitted.argtypes = [_f64p, ctypes.c_int32]
        lib.oracle_expected_emitted.restype = ctypes.c_double
        return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
        return _lib


def load_variant(path: str):
    """Load another build of the oracle source (the mutation tests compile
    copies with a planted mistake to show that the pins catch it)."""
    return _configure(ctypes.CDLL(path))


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    raise TypeError("logits must be float32 or uint16 (raw bf16 bits)")


def philox4x32_10(ctr, key):
    """Philox4x32-10 block function: 4 counter words, 2 key words -> 4 words."""
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c, ctypes.c_uint32), _ptr(k, ctypes.c_uint32),
                                 _ptr(out, ctypes.c_uint32))
    return tuple(int(v) for v in out)


def u24(x: int) -> float:
    return _load().oracle_u24(x)


def u52(x0: int, x1: int) -> float:
    return _load().oracle_u52(x0, x1)


def accept_uniform(seed: int, b: int, i: int) -> float:
    return _load().oracle_accept_uniform(seed, b, i)


def draw_uniform(seed: int, b: int, i: int) -> float:
    return _load().oracle_draw_uniform(seed, b, i)


def row_lse(row: np.ndarray, T: float):
    """Natural-log logsumexp of row/T; None for a bad row (NaN, +inf, all -inf)."""
    row = np.ascontiguousarray(row)
    out = ctypes.c_double()
    rc = _load().oracle_row_lse(row.ctypes.data, _dtype_code(row), row.shape[-1], T,
                                ctypes.byref(out))
    return out.value if rc == OK else None


def row_argmax(row: np.ndarray):
    row = np.ascontiguousarray(row)
    out = ctypes.c_int64()
    rc = _load().oracle_row_argmax(row.ctypes.data, _dtype_code(row), row.shape[-1],
                                   ctypes.byref(out))
    return out.value if rc == OK else None


def verify_seq_u(p_rows: np.ndarray, q_rows: np.ndarray, x, T: float, r, u: float) -> dict:
    """One verify step with explicit uniforms.

    p_rows: [gamma+1, V], q_rows: [gamma, V] (same dtype), x: gamma draft
    tokens, r: gamma accept-test uniforms, u: the final-draw uniform.
    """
    p_rows = np.ascontiguousarray(p_rows)
    gamma = p_rows.shape[0] - 1
    V = p_rows.shape[1]
    q_rows = np.ascontiguousarray(q_rows if gamma > 0 else p_rows[:1])
    x = np.ascontiguousarray(np.asarray(x, dtype=np.int32).reshape(-1))
    r = np.ascontiguousarray(np.asarray(r, dtype=np.float64).reshape(-1))
    if gamma == 0:
        x = np.zeros(1, np.int32)
        r = np.zeros(1, np.float64)
    n = ctypes.c_int32()
    toks = np.full(gamma + 1, -1, np.int32)
    lp = np.zeros(gamma + 1)
    lq = np.zeros(max(gamma, 1))
    am = np.full(max(gamma, 1), np.nan)
    dm = ctypes.c_double(np.nan)
    fb = ctypes.c_int32(0)
    rc = _load().oracle_verify_seq_u(
        p_rows.ctypes.data, q_rows.ctypes.data, V, _dtype_code(p_rows), V, gamma,
        _ptr(x, ctypes.c_int32), T, _ptr(r, ctypes.c_double), u, ctypes.byref(n),
        _ptr(toks, ctypes.c_int32), _ptr(lp, ctypes.c_double), _ptr(lq, ctypes.c_double),
        _ptr(am, ctypes.c_double), ctypes.byref(dm), ctypes.byref(fb))
    return {"rc": rc, "n": n.value, "tokens": toks, "lse_p": lp, "lse_q": lq[:gamma],
            "acc_margin": am[:gamma], "draw_margin": dm.value, "fallback": fb.value}


def verify_greedy_seq(p_rows: np.ndarray, x) -> dict:
    p_rows = np.ascontiguousarray(p_rows)
    gamma = p_rows.shape[0] - 1
    V = p_rows.shape[1]
    x = np.ascontiguousarray(np.asarray(x, dtype=np.int32).reshape(-1))
    if gamma == 0:
        x = np.zeros(1, np.int32)
    n = ctypes.c_int32()
    toks = np.full(gamma + 1, -1, np.int32)
    rc = _load().oracle_verify_greedy_seq(p_rows.ctypes.data, V, _dtype_code(p_rows), V, gamma,
                                          _ptr(x, ctypes.c_int32), ctypes.byref(n),
                                          _ptr(toks, ctypes.c_int32))
    return {"rc": rc, "n": n.value, "tokens": toks}


LENIENCE = {"none": 0, "lin": 1, "sq": 2, "exp": 3}


def verify_batch(target: np.ndarray, draft, p_row_off, q_row_off, draft_tokens, gamma,
                 T: float, seed: int = 0, seq_ids=None, nthreads: int | None = None,
                 lenience: str = "none", eps: float = 1.0) -> dict:
    """Batch verify in the library's ragged layout (see specverify_oracle.c).

    target: [target_rows, row_stride], draft: [draft_rows, row_stride] or None
    (greedy), draft_tokens: [B, gamma_max] int32, gamma: [B]. ``T <= 0``
    selects the greedy verify. ``lenience`` ("none", "lin", "sq", "exp") and
    ``eps`` select the lossy accept test f(p, eps) / q. Returns numpy arrays n [B], tokens
    [B, gamma_max+1], lse_p [B, gamma_max+1], lse_q [B, gamma_max],
    acc_margin [B, gamma_max], draw_margin [B], fallback [B] and the code rc.
    """
    target = np.ascontiguousarray(target)
    code = _dtype_code(target)
    stride = target.shape[1]
    gamma = np.ascontiguousarray(np.asarray(gamma, dtype=np.int32).reshape(-1))
    B = gamma.shape[0]
    draft_tokens = np.ascontiguousarray(np.asarray(draft_tokens, dtype=np.int32).reshape(B, -1))
    gm = draft_tokens.shape[1]
    p_off = np.ascontiguousarray(np.asarray(p_row_off, dtype=np.int64).reshape(-1))
    q_off = np.ascontiguousarray(np.asarray(q_row_off if q_row_off is not None else np.zeros(B),
                                            dtype=np.int64).reshape(-1))
    if draft is None:
        draft = target[:1]
    draft = np.ascontiguousarray(draft)
    if draft.dtype != target.dtype or draft.shape[1] != stride:
        raise ValueError("draft and target logits must share dtype and row stride")
    sid = None if seq_ids is None else np.ascontiguousarray(np.asarray(seq_ids, np.int32))
    n = np.full(B, -1, np.int32)
    toks = np.full((B, gm + 1), -1, np.int32)
    lp = np.full((B, gm + 1), np.nan)
    lq = np.full((B, max(gm, 1)), np.nan)
    am = np.full((B, max(gm, 1)), np.nan)
    dm = np.full(B, np.nan)
    fb = np.zeros(B, np.int32)
    dt_buf = draft_tokens if gm > 0 else np.zeros((B, 1), np.int32)
    if nthreads is None:
        nthreads = max(1, min(os.cpu_count() or 1, 64))
    rc = _load().oracle_verify_batch_lenient(
        target.ctypes.data, draft.ctypes.data, stride, code, stride, target.shape[0],
        draft.shape[0], B, gm, _ptr(p_off, ctypes.c_int64), _ptr(q_off, ctypes.c_int64),
        _ptr(dt_buf, ctypes.c_int32), _ptr(gamma, ctypes.c_int32),
        None if sid is None else _ptr(sid, ctypes.c_int32), T, LENIENCE[lenience], float(eps),
        seed,
        _ptr(n, ctypes.c_int32), _ptr(toks, ctypes.c_int32), _ptr(lp, ctypes.c_double),
        _ptr(lq, ctypes.c_double), _ptr(am, ctypes.c_double), _ptr(dm, ctypes.c_double),
        _ptr(fb, ctypes.c_int32), nthreads)
    return {"rc": rc, "n": n, "tokens": toks, "lse_p": lp, "lse_q": lq[:, :gm],
            "acc_margin": am[:, :gm], "draw_margin": dm, "fallback": fb}


def pair_stats(p_row: np.ndarray, q_row: np.ndarray, T: float):
    """(beta, TVD) of one position: sum min(p, q) and 1/2 sum |p - q|."""
    p_row = np.ascontiguousarray(p_row)
    q_row = np.ascontiguousarray(q_row)
    b, d = ctypes.c_double(), ctypes.c_double()
    rc = _load().oracle_pair_stats(p_row.ctypes.data, q_row.ctypes.data, _dtype_code(p_row),
                                   p_row.shape[-1], T, ctypes.byref(b), ctypes.byref(d))
    return rc, b.value, d.value


def row_features(row: np.ndarray, T: float, k: int):
    """(rc, entropy, top-k probabilities, top-k token indices) of softmax(row / T)."""
    row = np.ascontiguousarray(row)
    h = ctypes.c_double()
    prob = np.zeros(max(k, 1), np.float64)
    idx = np.zeros(max(k, 1), np.int64)
    rc = _load().oracle_row_features(row.ctypes.data, _dtype_code(row), row.shape[-1], T, k,
                                     ctypes.byref(h), _ptr(prob, ctypes.c_double),
                                     _ptr(idx, ctypes.c_int64))
    return rc, h.value, prob[:k], idx[:k]


def pair_stats_batch(target: np.ndarray, draft: np.ndarray, p_row_off, q_row_off, gamma,
                     T: float, nthreads: int | None = None) -> dict:
    """beta and TVD of positions 1..gamma_b of every sequence ([B, gamma_max], NaN past
    gamma_b), in the batch layout of verify_batch."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    gamma = np.ascontiguousarray(np.asarray(gamma, dtype=np.int32).reshape(-1))
    B = gamma.shape[0]
    gm = int(gamma.max()) if B else 0
    p_off = np.ascontiguousarray(np.asarray(p_row_off, dtype=np.int64).reshape(-1))
    q_off = np.ascontiguousarray(np.asarray(q_row_off, dtype=np.int64).reshape(-1))
    beta = np.full((B, max(gm, 1)), np.nan)
    tvd = np.full((B, max(gm, 1)), np.nan)
    if nthreads is None:
        nthreads = max(1, min(os.cpu_count() or 1, 64))
    rc = _load().oracle_pair_stats_batch(
        target.ctypes.data, draft.ctypes.data, target.shape[1], _dtype_code(target),
        target.shape[1], target.shape[0], draft.shape[0], B, gm, _ptr(p_off, ctypes.c_int64),
        _ptr(q_off, ctypes.c_int64), _ptr(gamma, ctypes.c_int32), T,
        _ptr(beta, ctypes.c_double), _ptr(tvd, ctypes.c_double), nthreads)
    return {"rc": rc, "beta": beta[:, :gm], "tvd": tvd[:, :gm]}


def row_features_batch(rows: np.ndarray, T: float, k: int, V: int | None = None,
                       nthreads: int | None = None) -> dict:
    """Entropy and top-k of softmax(row / T) for every row of ``rows``."""
    rows = np.ascontiguousarray(rows)
    n = rows.shape[0]
    V = rows.shape[1] if V is None else V
    ent = np.full(n, np.nan)
    prob = np.zeros((n, max(k, 1)), np.float64)
    idx = np.zeros((n, max(k, 1)), np.int64)
    if nthreads is None:
        nthreads = max(1, min(os.cpu_count() or 1, 64))
    rc = _load().oracle_row_features_batch(
        rows.ctypes.data, rows.shape[1], _dtype_code(rows), V, n, T, k,
        _ptr(ent, ctypes.c_double), _ptr(prob, ctypes.c_double), _ptr(idx, ctypes.c_int64),
        nthreads)
    return {"rc": rc, "entropy": ent, "topk_prob": prob[:, :k], "topk_idx": idx[:, :k]}


def restricted_row(row: np.ndarray, T: float, topk: int, topp: float = 1.0):
    """(rc, probabilities [V]) of the top-k / top-p restricted softmax(row / T)."""
    row = np.ascontiguousarray(row)
    prob = np.zeros(row.shape[-1], np.float64)
    rc = _load().oracle_restricted_row(row.ctypes.data, _dtype_code(row), row.shape[-1], T,
                                       int(topk), float(topp), _ptr(prob, ctypes.c_double))
    return rc, prob


def verify_batch_restricted(target: np.ndarray, draft: np.ndarray, p_row_off, q_row_off,
                            draft_tokens, gamma, T, topk, topp=None, seed: int = 0, seq_ids=None,
                            nthreads: int | None = None) -> dict:
    """Restricted-sampling verify: per-sequence temperature T [B], top-k topk [B]
    and top-p topp [B] (None: 1). Returns n, tokens, acc_margin, draw_margin, rc."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    gamma = np.ascontiguousarray(np.asarray(gamma, dtype=np.int32).reshape(-1))
    B = gamma.shape[0]
    draft_tokens = np.ascontiguousarray(np.asarray(draft_tokens, dtype=np.int32).reshape(B, -1))
    gm = draft_tokens.shape[1]
    p_off = np.ascontiguousarray(np.asarray(p_row_off, dtype=np.int64).reshape(-1))
    q_off = np.ascontiguousarray(np.asarray(q_row_off, dtype=np.int64).reshape(-1))
    Ts = np.ascontiguousarray(np.broadcast_to(np.asarray(T, np.float64), (B,)).copy())
    ks = np.ascontiguousarray(np.broadcast_to(np.asarray(topk, np.int32), (B,)).copy())
    ps = None if topp is None else np.ascontiguousarray(
        np.broadcast_to(np.asarray(topp, np.float64), (B,)).copy())
    sid = None if seq_ids is None else np.ascontiguousarray(np.asarray(seq_ids, np.int32))
    n = np.full(B, -1, np.int32)
    toks = np.full((B, gm + 1), -1, np.int32)
    am = np.full((B, max(gm, 1)), np.nan)
    dm = np.full(B, np.nan)
    dt_buf = draft_tokens if gm > 0 else np.zeros((B, 1), np.int32)
    if nthreads is None:
        nthreads = max(1, min(os.cpu_count() or 1, 64))
    rc = _load().oracle_verify_batch_restricted(
        target.ctypes.data, draft.ctypes.data, target.shape[1], _dtype_code(target),
        target.shape[1], target.shape[0], draft.shape[0], B, gm, _ptr(p_off, ctypes.c_int64),
        _ptr(q_off, ctypes.c_int64), _ptr(dt_buf, ctypes.c_int32), _ptr(gamma, ctypes.c_int32),
        None if sid is None else _ptr(sid, ctypes.c_int32), _ptr(Ts, ctypes.c_double),
        _ptr(ks, ctypes.c_int32), None if ps is None else _ptr(ps, ctypes.c_double), seed,
        _ptr(n, ctypes.c_int32), _ptr(toks, ctypes.c_int32), _ptr(am, ctypes.c_double),
        _ptr(dm, ctypes.c_double), nthreads)
    return {"rc": rc, "n": n, "tokens": toks, "acc_margin": am[:, :gm], "draw_margin": dm}


def block_efficiency(alpha: float, gamma: int) -> float:
    return _load().oracle_block_efficiency(alpha, gamma)


def expected_emitted(beta) -> float:
    b = np.ascontiguousarray(np.asarray(beta, dtype=np.float64).reshape(-1))
    return _load().oracle_expected_emitted(_ptr(b, ctypes.c_double), b.shape[0])


class RestrictedSeqCaller:
    """Repeated restricted-verify calls on fixed rows with explicit uniforms
    (for the exact-enumeration pins)."""

    def __init__(self, p_rows: np.ndarray, q_rows: np.ndarray, x, T: float, topk: int,
                 topp: float = 1.0):
        self.p = np.ascontiguousarray(p_rows)
        self.gamma = self.p.shape[0] - 1
        self.V = self.p.shape[1]
        self.q = np.ascontiguousarray(q_rows if self.gamma > 0 else self.p[:1])
        self.x = np.ascontiguousarray(np.asarray(x if self.gamma > 0 else [0], np.int32))
        self.T, self.k, self.pp = float(T), int(topk), float(topp)
        self.code = _dtype_code(self.p)
        self.r = np.zeros(max(self.gamma, 1), np.float64)
        self.toks = np.full(self.gamma + 1, -1, np.int32)
        self.n = ctypes.c_int32()

    def run(self, r, u: float):
        self.r[:self.gamma] = r
        rc = _load().oracle_verify_seq_restricted_u(
            self.p.ctypes.data, self.q.ctypes.data, self.V, self.code, self.V, self.gamma,
            _ptr(self.x, ctypes.c_int32), self.T, self.k, self.pp, _ptr(self.r, ctypes.c_double),
            u, ctypes.byref(self.n), _ptr(self.toks, ctypes.c_int32))
        if rc != OK:
            raise RuntimeError(f"oracle rc={rc}")
        return self.n.value, self.toks.copy()


class SeqCaller:
    """Repeated oracle calls on fixed rows with varying uniforms (buffers
    reused): the exact-enumeration pins call the oracle tens of thousands of
    times as a black box."""

    def __init__(self, p_rows: np.ndarray, q_rows: np.ndarray, x, T: float, lib=None,
                 lenience: str = "none", eps: float = 1.0):
        self.p = np.ascontiguousarray(p_rows)
        self.gamma = self.p.shape[0] - 1
        self.V = self.p.shape[1]
        self.q = np.ascontiguousarray(q_rows if self.gamma > 0 else self.p[:1])
        self.x = np.ascontiguousarray(np.asarray(x if self.gamma > 0 else [0], np.int32))
        self.T = float(T)
        self.code = _dtype_code(self.p)
        self.r = np.zeros(max(self.gamma, 1), np.float64)
        self.toks = np.full(self.gamma + 1, -1, np.int32)
        self.n = ctypes.c_int32()
        self._lib = lib if lib is not None else _load()
        self.kind = LENIENCE[lenience]
        self.eps = float(eps)

    def run(self, r, u: float):
        self.r[:self.gamma] = r
        if self.kind == 0:
            rc = self._lib.oracle_verify_seq_u(
                self.p.ctypes.data, self.q.ctypes.data, self.V, self.code, self.V, self.gamma,
                _ptr(self.x, ctypes.c_int32), self.T, _ptr(self.r, ctypes.c_double), u,
                ctypes.byref(self.n), _ptr(self.toks, ctypes.c_int32), None, None, None, None,
                None)
        else:
            rc = self._lib.oracle_verify_seq_u_lenient(
                self.p.ctypes.data, self.q.ctypes.data, self.V, self.code, self.V, self.gamma,
                _ptr(self.x, ctypes.c_int32), self.T, self.kind, self.eps,
                _ptr(self.r, ctypes.c_double), u, ctypes.byref(self.n),
                _ptr(self.toks, ctypes.c_int32), None, None)
        if rc != OK:
            raise RuntimeError(f"oracle rc={rc}")
        return self.n.value, self.toks.copy()
