"""The allocation-free entry point, qgemm_run_noalloc, against qgemm_run.

qgemm_run_noalloc serves callers that cannot allocate device memory when
they run a projection (an engine whose allocator owns the GPU's memory, a
plugin with a fixed memory budget, code running while streams are being
captured): it needs no workspace and keeps the tcgen05 route's split-tile
partial sums in a scratch array inside the library instead.  Each case calls
it twice in a row through the C-ABI (the second call finds the first one's
leftovers in the shared array) and checks both results against qgemm_run's
output within the tolerance of the other parity tests, and against the
oracle.  This file is collected last on purpose: a failure here leaves every
other test already run.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_groupwise_gb300 import synth
from tests.tolerance import ELEM_ABS, ELEM_REL, assert_close

torch = pytest.importorskip("torch")
qg = pytest.importorskip("bit_weight_only_groupwise_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qg.qgemm_device_status(clear=True) == qg.QGEMM_OK


def host(Y):
    torch.cuda.synchronize()
    return Y.double().cpu().numpy()


@pytest.mark.parametrize("bits,N,K,T", [(4, 1000, 1024, 40), (5, 777, 2048, 300), (8, 2048, 512, 129),
                                        (4, 5120, 6144, 1024)])
def test_noalloc_matches_qgemm_run_twice_in_a_row(bits, N, K, T):
    p = synth.weights(50, N, K, bits)
    W = qg.GroupwiseWeights(bits, N, K, p["packed"], p["scales"], T_max=T)
    x = synth.activations(50, T, K, outliers=True)
    X = torch.from_numpy(x.view(np.int16)).cuda()
    ref = host(W.run(X))
    # a plan of its own, never bound: the weights come with the call
    st, plan = qg.qgemm_plan(N, K, bits, T)
    assert st == qg.QGEMM_OK
    try:
        cols = np.unique(np.concatenate([np.arange(0, T, 37), [T - 1]]))
        Yref, A = oracle.gemm_parent(p, x[cols])
        bound = 2 * (ELEM_REL * A + ELEM_ABS)
        for call in range(2):
            Y = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
            assert qg.qgemm_run_noalloc(plan, W.packed, X, T, Y) == qg.QGEMM_OK
            y = host(Y)
            # within the tolerance of the existing entry point's result ...
            assert np.all(np.isfinite(y)), f"call {call}"
            assert np.all(np.abs(y[cols] - ref[cols]) <= bound), f"call {call}"
            # ... and of the oracle
            assert_close(y[cols], Yref, A, f"noalloc call {call} int{bits} N={N} K={K} T={T}")
    finally:
        qg.qgemm_plan_destroy(plan)


def test_noalloc_rejects_what_its_scratch_cannot_hold():
    # 64 row blocks x 129 token tiles of 256 = 8,256 split-tile counters > 8,192
    N, K, T = 8192, 64, 256 * 128 + 1
    p = synth.weights(51, N, K, 4)
    W = qg.GroupwiseWeights(4, N, K, p["packed"], p["scales"], T_max=8)
    st, plan = qg.qgemm_plan(N, K, 4, T)
    assert st == qg.QGEMM_OK
    try:
        X = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda")
        Y = torch.empty((T, N), dtype=torch.float32, device="cuda")
        n0 = qg.qgemm_launch_count()
        assert qg.qgemm_run_noalloc(plan, W.packed, X, T, Y) == qg.QGEMM_ERR_WORKSPACE
        assert qg.qgemm_run_noalloc(plan, None, X, T, Y) == qg.QGEMM_ERR_INVALID_ARG
        assert qg.qgemm_run_noalloc(plan, W.packed, X, T + 1, Y) == qg.QGEMM_ERR_T_OUT_OF_DOMAIN
        assert qg.qgemm_launch_count() == n0
    finally:
        qg.qgemm_plan_destroy(plan)
