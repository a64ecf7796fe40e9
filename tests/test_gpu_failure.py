"""The timeout path of the kernels' bounded waits, on the GPU, without a fault.

Every wait inside the kernels is bounded: when one runs out, the kernel sets
the library's device status word to QGEMM_ERR_TIMEOUT and returns.  Here a
diagnostic kernel waits on a barrier that nothing completes (a flag nothing
sets); the test checks that the status word reports it, that reading and
clearing it work, and that the context still computes correct results.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_groupwise_gb300 import synth
from tests.tolerance import assert_close

torch = pytest.importorskip("torch")
qg = pytest.importorskip("bit_weight_only_groupwise_gb300")

pytestmark = pytest.mark.gpu


def test_wait_timeout_sets_the_status_and_leaves_the_context_usable():
    assert qg.qgemm_device_status(clear=True) == qg.QGEMM_OK
    try:
        n0 = qg.qgemm_launch_count()
        qg.check(qg.qgemm_selftest_timeout(), "selftest_timeout")
        assert qg.qgemm_launch_count() - n0 == 1
        assert qg.qgemm_device_status() == qg.QGEMM_ERR_TIMEOUT                # read, kept
        assert qg.qgemm_device_status(clear=True) == qg.QGEMM_ERR_TIMEOUT      # read, cleared
        assert qg.qgemm_device_status() == qg.QGEMM_OK
    finally:
        qg.qgemm_device_status(clear=True)
    # the context still runs both kinds of kernel correctly
    p = synth.weights(71, 512, 1024, 4)
    W = qg.GroupwiseWeights(4, 512, 1024, p["packed"], p["scales"], T_max=256)
    for T in (3, 256):
        x = synth.activations(71, T, 1024, outliers=True)
        Y = W.run(torch.from_numpy(x.view(np.int16)).cuda())
        torch.cuda.synchronize()
        Yref, A = oracle.gemm_parent(p, x)
        assert_close(Y.double().cpu().numpy(), Yref, A, f"after timeout T={T}")
    assert qg.qgemm_device_status() == qg.QGEMM_OK
