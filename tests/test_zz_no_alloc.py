"""The no-allocation verify entry point, through the C ABI.

specverify_verify_noalloc serves callers that may not call cudaMalloc (a
serving process whose memory pool owns all free device memory, or a path
where an allocation's device-wide synchronisation is not acceptable). It runs
the same kernels as specverify_verify with their workspace in one fixed
device array shared by every call. These checks compare it with the handle
entry point on two calls in a row -- the second on a batch of another shape
and dtype, so stale scratch from the first call would show --, compare it with
the CPU oracle (including a batch at the limits of its scratch), and check
that oversized batches are refused. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import compare, lse_errors, run_oracle
from speculative_decoding_token_gb300 import workload

pytestmark = pytest.mark.gpu

LSE_RTOL = 1e-5


@pytest.fixture(scope="module")
def svm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_token_gb300 as sv
    sv.build()
    sv.load()
    oracle.build()
    return sv


def _lse_buffers(batch):
    return (torch.full((batch.target.shape[0],), float("nan"), device="cuda"),
            torch.full((max(batch.draft.shape[0], 1),), float("nan"), device="cuda"))


def _noalloc(svm, batch, seed):
    n = torch.full((batch.B,), -7, dtype=torch.int32, device="cuda")
    toks = torch.full((batch.B, batch.gamma_max + 1), -7, dtype=torch.int32, device="cuda")
    p_lse, q_lse = _lse_buffers(batch)
    st = svm.make_batch_struct(batch.target, batch.draft, batch.p_row_off, batch.q_row_off,
                               batch.draft_tokens, batch.gamma)
    svm.specverify_verify_noalloc(st, batch.T, seed, n, toks, p_lse, q_lse)
    torch.cuda.synchronize()
    return n.cpu(), toks.cpu(), p_lse.cpu(), q_lse.cpu()


def _with_handle(svm, batch, seed):
    h = svm.SpecVerify(batch.B, batch.gamma_max, batch.V)
    p_lse, q_lse = _lse_buffers(batch)
    n, toks = h.verify_batch(batch, seed=seed, p_lse=p_lse, q_lse=q_lse)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    h.close()
    return n.cpu(), toks.cpu(), p_lse.cpu(), q_lse.cpu()


def _lse_close(a, b):
    a, b = a.double().numpy(), b.double().numpy()
    same_nan = np.isnan(a) == np.isnan(b)
    ok = np.isnan(a) | (np.abs(a - b) <= LSE_RTOL * np.maximum(1.0, np.abs(b)))
    return bool(same_nan.all() and ok.all())


def test_noalloc_matches_handle_entry_point_on_two_calls(svm):
    first = workload.make_batch(1, device="cuda", seed=501)            # bf16, B=8, V=32000
    second = workload.make_batch(0, device="cuda", B=5, seed=502)      # fp32, B=5, V=32000
    for batch, seed in ((first, 9001), (second, 9002)):
        got = _noalloc(svm, batch, seed)
        want = _with_handle(svm, batch, seed)
        # same kernels and the same exp2 table: the decisions agree exactly
        assert torch.equal(got[0], want[0]), (got[0], want[0])
        assert torch.equal(got[1], want[1])
        assert _lse_close(got[2], want[2]) and _lse_close(got[3], want[3])
        g = batch.gamma.cpu()
        assert ((got[0] >= 0) & (got[0] <= g)).all()


def test_noalloc_refuses_batches_beyond_its_scratch(svm):
    batch = workload.make_batch(1, device="cuda", seed=503)
    n = torch.empty(batch.B, dtype=torch.int32, device="cuda")
    toks = torch.empty(batch.B, batch.gamma_max + 1, dtype=torch.int32, device="cuda")
    st = svm.make_batch_struct(batch.target, batch.draft, batch.p_row_off, batch.q_row_off,
                               batch.draft_tokens, batch.gamma)
    for field, value in (("B", 65), ("gamma_max", 17), ("V", 262145)):
        big = svm.SpecverifyBatch.from_buffer_copy(st)
        setattr(big, field, value)
        with pytest.raises(svm.SpecVerifyError) as err:
            svm.specverify_verify_noalloc(big, batch.T, 1, n, toks)
        assert err.value.rc == svm.ERR_TOO_LARGE


@pytest.mark.parametrize("cfg,over,seed", [
    (1, dict(), 7001),                                          # bf16, B=8, V=32000
    (0, dict(B=3), 7002),                                       # fp32
    # the limits of the fixed scratch: B = 64, gamma up to 16 (ragged, with
    # gamma = 0 sequences), V = 262144, bf16
    (3, dict(B=64, V=262144, gamma=(0, 16)), 7003),
])
def test_noalloc_matches_the_oracle(svm, cfg, over, seed):
    batch = workload.make_batch(cfg, device="cuda", seed=seed, **over)
    n, toks, p_lse, q_lse = _noalloc(svm, batch, seed)
    ora = run_oracle(batch, seed)
    assert ora["rc"] == 0
    st = compare(n.numpy(), toks.numpy(), ora, batch.V)
    assert not st["hard"], st
    assert lse_errors(batch, ora, p_lse, q_lse) <= LSE_RTOL
