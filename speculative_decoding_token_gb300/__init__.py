"""GB300 (sm_103a) speculative-sampling verify step.

This package is a thin ctypes binding of ``_build/libspecverify.so``, whose C
ABI is declared in ``include/specverify.h``. The binding only marshals
arguments (tensor pointers, sizes, the CUDA stream); every step of the verify
path -- temperature softmax statistics, the accept scan, the residual or bonus
draw and the greedy scan -- runs in the library's CUDA kernels. There is no
CPU fallback: without the built library every call raises.

The functions carry the C names (``specverify_create``, ``specverify_verify``,
...); :class:`SpecVerify` wraps them for torch tensors and also accepts host
tensors, copying them to the device and the results back (the end-to-end
path a caller with host buffers uses).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = ["SpecVerify", "SpecVerifyError", "build", "load", "specverify_create",
           "specverify_destroy", "specverify_verify", "specverify_verify_greedy",
           "specverify_verify_lossy", "LENIENCE", "specverify_verify_restricted",
           "specverify_verify_noalloc",
           "specverify_device_status", "specverify_status_string", "specverify_workspace_bytes",
           "specverify_set_timing", "specverify_get_timing", "specverify_set_wait_limit",
           "specverify_acceptance_stats", "specverify_row_features", "STATUS_BITS"]

OK = 0
ERR_INVALID_ARG = -1
ERR_CUDA = -2
ERR_OOM = -3
ERR_TOO_LARGE = -6
FP32 = 0
BF16 = 1

STATUS_BITS = {
    "bad_gamma": 1 << 0,
    "bad_row": 1 << 1,
    "bad_token": 1 << 2,
    "bad_logit": 1 << 3,
    "timeout": 1 << 4,
    "bad_param": 1 << 5,
    "draw_slow": 1 << 8,
    "draw_zero_mass": 1 << 9,
}

LENIENCE = {"none": 0, "lin": 1, "sq": 2, "exp": 3}

KERNEL_PLAN, KERNEL_ROWSTATS, KERNEL_DRAW, KERNEL_ACCEPT, KERNEL_FUSED = 0, 1, 2, 3, 4
KERNEL_RESTRICT_PLAN, KERNEL_RESTRICT_ROWS, KERNEL_RESTRICT_FINAL = 5, 6, 7
KERNEL_SMALL = 8

_lock = threading.Lock()
_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, rc: int, what: str):
        self.rc = rc
        super().__init__(f"{what}: {specverify_status_string(rc)} ({rc})")


class SpecverifyBatch(ctypes.Structure):
    """Mirror of ``specverify_batch`` (include/specverify.h)."""
    _fields_ = [("B", ctypes.c_int32), ("gamma_max", ctypes.c_int32), ("V", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("target_logits", ctypes.c_void_p),
                ("draft_logits", ctypes.c_void_p), ("row_stride", ctypes.c_int64),
                ("target_rows", ctypes.c_int64), ("draft_rows", ctypes.c_int64),
                ("p_row_off", ctypes.c_void_p), ("q_row_off", ctypes.c_void_p),
                ("draft_tokens", ctypes.c_void_p), ("gamma", ctypes.c_void_p)]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library for sm_103a (in-tree)."""
    return _build.build(force=force, verbose=verbose)


def load():
    """Load the built library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                f"CUDA library {_build.LIB} is missing: run "
                "speculative_decoding_token_gb300.build() (there is no CPU fallback)")
        lib = ctypes.CDLL(_build.LIB)
        vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        lib.specverify_create.argtypes = [ctypes.POINTER(vp), ctypes.c_int, i32, i32, i64]
        lib.specverify_destroy.argtypes = [vp]
        lib.specverify_verify.argtypes = [vp, ctypes.POINTER(SpecverifyBatch), ctypes.c_float,
                                          u64, vp, vp, vp, vp, vp]
        lib.specverify_verify_greedy.argtypes = [vp, ctypes.POINTER(SpecverifyBatch), vp, vp, vp]
        lib.specverify_verify_lossy.argtypes = [vp, ctypes.POINTER(SpecverifyBatch),
                                                ctypes.c_float, u64, i32, ctypes.c_float, vp, vp,
                                                vp, vp, vp]
        lib.specverify_verify_noalloc.argtypes = [ctypes.POINTER(SpecverifyBatch),
                                                  ctypes.c_float, u64, vp, vp, vp, vp, vp]
        lib.specverify_verify_restricted.argtypes = [vp, ctypes.POINTER(SpecverifyBatch), vp, vp,
                                                     vp, u64, vp, vp, vp]
        lib.specverify_device_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
        lib.specverify_status_string.argtypes = [ctypes.c_int]
        lib.specverify_status_string.restype = ctypes.c_char_p
        lib.specverify_workspace_bytes.argtypes = [vp, ctypes.POINTER(ctypes.c_size_t)]
        lib.specverify_set_timing.argtypes = [vp, ctypes.c_int]
        lib.specverify_get_timing.argtypes = [vp, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                              ctypes.POINTER(i64), ctypes.c_int]
        lib.specverify_set_wait_limit.argtypes = [vp, u64]
        lib.specverify_acceptance_stats.argtypes = [vp, ctypes.POINTER(SpecverifyBatch),
                                                    ctypes.c_float, vp, vp, vp]
        lib.specverify_row_features.argtypes = [vp, vp, i32, i64, i64, i64, ctypes.c_float, i32,
                                                vp, vp, vp, vp]
        for f in ("specverify_create", "specverify_destroy", "specverify_verify",
                  "specverify_verify_greedy", "specverify_verify_noalloc",
                  "specverify_verify_lossy", "specverify_verify_restricted",
                  "specverify_device_status",
                  "specverify_workspace_bytes", "specverify_set_timing",
                  "specverify_get_timing", "specverify_set_wait_limit",
                  "specverify_acceptance_stats", "specverify_row_features"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# C-named functions

def specverify_status_string(rc: int) -> str:
    return load().specverify_status_string(rc).decode()


def _check(rc: int, what: str):
    if rc != OK:
        raise SpecVerifyError(rc, what)


def specverify_create(device: int, max_batch: int, max_gamma: int, max_vocab: int):
    h = ctypes.c_void_p()
    _check(load().specverify_create(ctypes.byref(h), device, max_batch, max_gamma, max_vocab),
           "specverify_create")
    return h


def specverify_destroy(h) -> None:
    _check(load().specverify_destroy(h), "specverify_destroy")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_batch_struct(target, draft, p_row_off, q_row_off, draft_tokens, gamma) -> SpecverifyBatch:
    """Describe device tensors as a ``specverify_batch`` (no copies)."""
    import torch
    if target.dim() != 2 or target.stride(1) != 1:
        raise ValueError("target logits must be a 2-D tensor with unit column stride")
    dt = {torch.float32: FP32, torch.bfloat16: BF16}.get(target.dtype)
    if dt is None:
        raise ValueError("logits must be float32 or bfloat16")
    if draft is not None and draft.numel() > 0 and (
            draft.dtype != target.dtype or draft.stride(1) != 1 or
            draft.stride(0) != target.stride(0)):
        raise ValueError("draft logits must match the target's dtype and row stride")
    for name, t, want in (("p_row_off", p_row_off, torch.int64), ("gamma", gamma, torch.int32),
                          ("q_row_off", q_row_off, torch.int64),
                          ("draft_tokens", draft_tokens, torch.int32)):
        if t is not None and (t.dtype != want or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous {want} tensor")
    B = int(gamma.shape[0])
    gm = int(draft_tokens.shape[1]) if draft_tokens is not None and draft_tokens.dim() == 2 else 0
    return SpecverifyBatch(
        B=B, gamma_max=gm, V=int(target.shape[1]), dtype=dt,
        target_logits=target.data_ptr(),
        draft_logits=None if draft is None or draft.numel() == 0 else draft.data_ptr(),
        row_stride=int(target.stride(0)), target_rows=int(target.shape[0]),
        draft_rows=0 if draft is None else int(draft.shape[0]),
        p_row_off=p_row_off.data_ptr(),
        q_row_off=None if q_row_off is None else q_row_off.data_ptr(),
        draft_tokens=None if draft_tokens is None or draft_tokens.numel() == 0
        else draft_tokens.data_ptr(),
        gamma=gamma.data_ptr())


def specverify_verify(h, batch: SpecverifyBatch, temperature: float, seed: int, n_accepted,
                      out_tokens, p_lse=None, q_lse=None, stream=None) -> None:
    _check(load().specverify_verify(h, ctypes.byref(batch), float(temperature),
                                    int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(n_accepted),
                                    _ptr(out_tokens), _ptr(p_lse), _ptr(q_lse),
                                    _stream_handle(stream)), "specverify_verify")


def specverify_verify_lossy(h, batch: SpecverifyBatch, temperature: float, seed: int,
                            lenience: str, eps: float, n_accepted, out_tokens, p_lse=None,
                            q_lse=None, stream=None) -> None:
    _check(load().specverify_verify_lossy(h, ctypes.byref(batch), float(temperature),
                                          int(seed) & 0xFFFFFFFFFFFFFFFF, LENIENCE[lenience],
                                          float(eps), _ptr(n_accepted), _ptr(out_tokens),
                                          _ptr(p_lse), _ptr(q_lse), _stream_handle(stream)),
           "specverify_verify_lossy")


def specverify_verify_restricted(h, batch: SpecverifyBatch, temperature, top_k, top_p, seed: int,
                                 n_accepted, out_tokens, stream=None) -> None:
    """Restricted sampling verify: per-sequence temperature (float32 [B]),
    top-k (int32 [B], 1..32) and top-p (float32 [B] or None), device tensors."""
    _check(load().specverify_verify_restricted(h, ctypes.byref(batch), _ptr(temperature),
                                               _ptr(top_k), _ptr(top_p),
                                               int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(n_accepted),
                                               _ptr(out_tokens), _stream_handle(stream)),
           "specverify_verify_restricted")


def specverify_verify_greedy(h, batch: SpecverifyBatch, n_accepted, out_tokens,
                             stream=None) -> None:
    _check(load().specverify_verify_greedy(h, ctypes.byref(batch), _ptr(n_accepted),
                                           _ptr(out_tokens), _stream_handle(stream)),
           "specverify_verify_greedy")


def specverify_verify_noalloc(batch: SpecverifyBatch, temperature: float, seed: int, n_accepted,
                              out_tokens, p_lse=None, q_lse=None, stream=None) -> None:
    """Sampling verify without a handle and without any device allocation,
    for callers that may not call cudaMalloc (see include/specverify.h for the
    size limits and the shared-scratch rules)."""
    _check(load().specverify_verify_noalloc(ctypes.byref(batch), float(temperature),
                                            int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(n_accepted),
                                            _ptr(out_tokens), _ptr(p_lse), _ptr(q_lse),
                                            _stream_handle(stream)), "specverify_verify_noalloc")


def specverify_acceptance_stats(h, batch: SpecverifyBatch, temperature: float, beta, tvd,
                                stream=None) -> None:
    _check(load().specverify_acceptance_stats(h, ctypes.byref(batch), float(temperature),
                                              _ptr(beta), _ptr(tvd), _stream_handle(stream)),
           "specverify_acceptance_stats")


def specverify_row_features(h, rows, temperature: float, k: int, entropy, topk_prob, topk_idx,
                            V: int | None = None, stream=None) -> None:
    """Entropy and top-k of softmax(row / T) for every row of the 2-D device
    tensor ``rows`` (float32 or bfloat16, unit column stride)."""
    import torch
    dt = {torch.float32: FP32, torch.bfloat16: BF16}.get(rows.dtype)
    if dt is None or rows.dim() != 2 or rows.stride(1) != 1:
        raise ValueError("rows must be a 2-D float32 or bfloat16 tensor with unit column stride")
    _check(load().specverify_row_features(
        h, ctypes.c_void_p(rows.data_ptr()), dt, int(rows.shape[0]),
        int(rows.shape[1] if V is None else V), int(rows.stride(0)), float(temperature), int(k),
        _ptr(entropy), _ptr(topk_prob), _ptr(topk_idx), _stream_handle(stream)),
        "specverify_row_features")


def specverify_device_status(h, stream=None) -> int:
    v = ctypes.c_int32()
    _check(load().specverify_device_status(h, _stream_handle(stream), ctypes.byref(v)),
           "specverify_device_status")
    return v.value


def specverify_workspace_bytes(h) -> int:
    v = ctypes.c_size_t()
    _check(load().specverify_workspace_bytes(h, ctypes.byref(v)), "specverify_workspace_bytes")
    return v.value


def specverify_set_timing(h, enable: bool) -> None:
    _check(load().specverify_set_timing(h, 1 if enable else 0), "specverify_set_timing")


def specverify_set_wait_limit(h, ns: int) -> None:
    _check(load().specverify_set_wait_limit(h, int(ns)), "specverify_set_wait_limit")


def specverify_get_timing(h, kernel: int, reset: bool = False):
    ms = ctypes.c_double()
    n = ctypes.c_int64()
    _check(load().specverify_get_timing(h, kernel, ctypes.byref(ms), ctypes.byref(n),
                                        1 if reset else 0), "specverify_get_timing")
    return ms.value, n.value


# ---------------------------------------------------------------------------

class SpecVerify:
    """A handle on one CUDA device with workspace for batches up to the given sizes."""

    def __init__(self, max_batch: int, max_gamma: int, max_vocab: int, device: int | None = None):
        import torch
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.max_batch, self.max_gamma, self.max_vocab = max_batch, max_gamma, max_vocab
        self.h = specverify_create(self.device, max_batch, max_gamma, max_vocab)
        self._staging = {}

    def close(self):
        if getattr(self, "h", None) is not None:
            specverify_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _dev(self, t, key, stream=None):
        """Device copy of a host tensor into a reused staging buffer, made on
        `stream` (default: the current stream), so the verify call that runs
        there next sees it."""
        import torch
        if t is None or t.is_cuda:
            return t
        buf = self._staging.get(key)
        if buf is None or buf.dtype != t.dtype or buf.numel() < t.numel():
            buf = torch.empty(max(t.numel(), 1), dtype=t.dtype, device=f"cuda:{self.device}")
            self._staging[key] = buf
        out = buf[:t.numel()].view(t.shape)
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
            out.copy_(t, non_blocking=True)
        return out

    def verify(self, target, draft, p_row_off, q_row_off, draft_tokens, gamma, temperature,
               seed, *, greedy=False, p_lse=None, q_lse=None, stream=None, lenience="none",
               eps=1.0):
        """Run one verify step; returns (n_accepted [B], out_tokens [B, gamma_max+1]).

        Device tensors: results stay on the device, the call is asynchronous.
        Host tensors: inputs are copied in and results copied back (synchronous).
        """
        import torch
        host = not target.is_cuda
        target = self._dev(target, "target", stream)
        draft = None if greedy else self._dev(draft, "draft", stream)
        p_row_off = self._dev(p_row_off, "p_off", stream)
        q_row_off = None if greedy else self._dev(q_row_off, "q_off", stream)
        draft_tokens = self._dev(draft_tokens, "tokens", stream)
        gamma = self._dev(gamma, "gamma", stream)
        B = int(gamma.shape[0])
        gm = int(draft_tokens.shape[1]) if draft_tokens.dim() == 2 else 0
        n = torch.empty(B, dtype=torch.int32, device=target.device)
        toks = torch.empty(B, gm + 1, dtype=torch.int32, device=target.device)
        batch = make_batch_struct(target, draft, p_row_off, q_row_off, draft_tokens, gamma)
        if greedy:
            specverify_verify_greedy(self.h, batch, n, toks, stream=stream)
        elif lenience != "none":
            specverify_verify_lossy(self.h, batch, temperature, seed, lenience, eps, n, toks,
                                    p_lse, q_lse, stream=stream)
        else:
            specverify_verify(self.h, batch, temperature, seed, n, toks, p_lse, q_lse,
                              stream=stream)
        if host:
            if stream is not None:
                stream.synchronize()
            return n.cpu(), toks.cpu()
        return n, toks

    def verify_restricted(self, target, draft, p_row_off, q_row_off, draft_tokens, gamma,
                          temperature, top_k, top_p, seed, *, stream=None):
        """Restricted sampling verify (per-sequence temperature [B], top-k [B]
        in 1..32, top-p [B] or None); returns (n_accepted, out_tokens) like
        :meth:`verify`, host tensors in, host tensors out."""
        import torch
        host = not target.is_cuda
        target = self._dev(target, "target", stream)
        draft = self._dev(draft, "draft", stream)
        p_row_off = self._dev(p_row_off, "p_off", stream)
        q_row_off = self._dev(q_row_off, "q_off", stream)
        draft_tokens = self._dev(draft_tokens, "tokens", stream)
        gamma = self._dev(gamma, "gamma", stream)
        temperature = self._dev(temperature, "r_temp", stream)
        top_k = self._dev(top_k, "r_topk", stream)
        top_p = self._dev(top_p, "r_topp", stream)
        B = int(gamma.shape[0])
        gm = int(draft_tokens.shape[1]) if draft_tokens.dim() == 2 else 0
        n = torch.empty(B, dtype=torch.int32, device=target.device)
        toks = torch.empty(B, gm + 1, dtype=torch.int32, device=target.device)
        batch = make_batch_struct(target, draft, p_row_off, q_row_off, draft_tokens, gamma)
        specverify_verify_restricted(self.h, batch, temperature, top_k, top_p, seed, n, toks,
                                     stream=stream)
        if host:
            if stream is not None:
                stream.synchronize()
            return n.cpu(), toks.cpu()
        return n, toks

    def verify_batch(self, batch, seed=0, greedy=False, **kw):
        """Verify a :class:`workload.Batch`."""
        return self.verify(batch.target, batch.draft, batch.p_row_off, batch.q_row_off,
                           batch.draft_tokens, batch.gamma, batch.T, seed, greedy=greedy, **kw)

    def acceptance_stats(self, batch, temperature=None, stream=None):
        """beta and TVD [B, gamma_max] of a :class:`workload.Batch` (device tensors)."""
        import torch
        B, gm = batch.B, batch.gamma_max
        beta = torch.empty(B, max(gm, 1), dtype=torch.float32, device=batch.target.device)
        tvd = torch.empty_like(beta)
        st = make_batch_struct(batch.target, batch.draft, batch.p_row_off, batch.q_row_off,
                               batch.draft_tokens, batch.gamma)
        specverify_acceptance_stats(self.h, st, batch.T if temperature is None else temperature,
                                    beta, tvd, stream=stream)
        return beta[:, :gm], tvd[:, :gm]

    def row_features(self, rows, temperature, k, stream=None):
        """(entropy [n], top-k probabilities [n, k], top-k indices [n, k]) of device rows."""
        import torch
        n = int(rows.shape[0])
        ent = torch.empty(n, dtype=torch.float32, device=rows.device)
        prob = torch.empty(n, max(k, 1), dtype=torch.float32, device=rows.device)
        idx = torch.empty(n, max(k, 1), dtype=torch.int32, device=rows.device)
        specverify_row_features(self.h, rows, temperature, k, ent, prob, idx, stream=stream)
        return ent, prob[:, :k], idx[:, :k]

    def device_status(self, stream=None) -> int:
        return specverify_device_status(self.h, stream)

    def workspace_bytes(self) -> int:
        return specverify_workspace_bytes(self.h)

    def set_timing(self, enable: bool):
        specverify_set_timing(self.h, enable)

    def get_timing(self, kernel: int, reset: bool = False):
        return specverify_get_timing(self.h, kernel, reset)

    def set_wait_limit(self, ns: int):
        specverify_set_wait_limit(self.h, ns)
