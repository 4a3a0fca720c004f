"""Failure detection on the GPU without a fault: a kernel whose bounded
mbarrier wait runs out (nothing ever arrives) reports ERR_TIMEOUT through the
status word, returns, and leaves the context usable for the next launch."""

import time

import numpy as np
import pytest
import torch

from int8_hadamard_rotated_convrot_gb300 import convrot as cr

LIMIT_NS = 200_000_000  # 0.2 s


def _small_gemm(rng):
    X = torch.from_numpy(rng.standard_normal((130, 512)).astype(np.float32)).cuda()
    W = torch.from_numpy(rng.standard_normal((96, 512)).astype(np.float32)).cuda()
    px = cr.convrot_pack_activations(X, 64, cr.CODES_BF16)
    pw = cr.convrot_quantize_weights(W, 64, cr.CODES_BF16)
    return lambda st: cr.convrot_gemm_i32(px, pw, dev_status=st)


@pytest.mark.gpu
def test_wait_that_runs_out_reports_timeout_and_context_survives():
    rng = np.random.default_rng(7)
    gemm = _small_gemm(rng)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = gemm(st)
    torch.cuda.synchronize()

    t0 = time.perf_counter()
    cr.convrot_wait_check(st, LIMIT_NS, arrive=False)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(st.item()) == cr.ERR_TIMEOUT
    assert elapsed >= LIMIT_NS * 1e-9
    assert elapsed < 30.0

    # The same kernel with its barrier satisfied returns at once and leaves the status alone.
    st.zero_()
    t0 = time.perf_counter()
    cr.convrot_wait_check(st, LIMIT_NS, arrive=True)
    torch.cuda.synchronize()
    assert int(st.item()) == cr.OK
    assert time.perf_counter() - t0 < LIMIT_NS * 1e-9

    # The context is still usable: the GEMM gives the same integers and no status.
    after = gemm(st)
    torch.cuda.synchronize()
    assert int(st.item()) == cr.OK
    assert torch.equal(before, after)
