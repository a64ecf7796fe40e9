"""Dependent calls back to back under programmatic dependent launch.

A run's kernel may start while the previous kernel on the stream drains and
streams its packed weights before it waits for that kernel ("ninfer-3080
docs/performance.md", small-T kernels section: ramp-up and drain at kernel
boundaries, and programmatic dependent launch to hide the ramp).  X and Y
must still be ordered: here call A writes a bf16 Y that is call B's X, and B
writes the next round's input of A, for several rounds on one stream.  Each
link is compared with the oracle on the GPU's own input of that link, and
the same chain with reused (ping-pong) buffers, with and without the
programmatic launch, must reproduce the final outputs bitwise (every call is
bitwise repeatable for its plan and T, so any overlap of a read with a later
write would show).
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_groupwise_gb300 import synth
from tests.tolerance import assert_close

torch = pytest.importorskip("torch")
qg = pytest.importorskip("bit_weight_only_groupwise_gb300")

pytestmark = pytest.mark.gpu

K0, N1 = 1024, 2048        # A: N1 x K0 (int4); B: K0 x N1 (int5), so B's output is A's input
ROUNDS = 6


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qg.qgemm_device_status(clear=True) == qg.QGEMM_OK


@pytest.fixture(scope="module")
def pair():
    pa, pb = synth.weights(20, N1, K0, 4), synth.weights(21, K0, N1, 5)
    A = qg.GroupwiseWeights(4, N1, K0, pa["packed"], pa["scales"], T_max=64, out=qg.QGEMM_OUT_BF16)
    B = qg.GroupwiseWeights(5, K0, N1, pb["packed"], pb["scales"], T_max=64, out=qg.QGEMM_OUT_BF16)
    return pa, pb, A, B


def bits(t):
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def to_dev(x_bits):
    return torch.from_numpy(x_bits.view(np.int16).copy()).cuda().view(torch.bfloat16)


def bf16_to_f64(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def chain(A, B, x0, T, reuse, pdl):
    for W in (A, B):
        qg.check(qg.qgemm_plan_set_pdl(W.plan, pdl))
    s = torch.cuda.current_stream()
    if reuse:
        xs = [to_dev(x0), torch.empty((T, K0), dtype=torch.bfloat16, device="cuda")]
        y1 = torch.empty((T, N1), dtype=torch.bfloat16, device="cuda")
        for r in range(ROUNDS):
            A.run(xs[r % 2], y1, stream=s)
            B.run(y1, xs[(r + 1) % 2], stream=s)
        return bits(y1), bits(xs[ROUNDS % 2]), None
    xs = [to_dev(x0)] + [
        torch.empty((T, K0), dtype=torch.bfloat16, device="cuda") for _ in range(ROUNDS)]
    y1 = [torch.empty((T, N1), dtype=torch.bfloat16, device="cuda") for _ in range(ROUNDS)]
    for r in range(ROUNDS):
        A.run(xs[r], y1[r], stream=s)
        B.run(y1[r], xs[r + 1], stream=s)
    return bits(y1[-1]), bits(xs[-1]), ([bits(x) for x in xs], [bits(y) for y in y1])


@pytest.mark.parametrize("T", [1, 4, 13, 40])
def test_dependent_chain_matches_the_oracle_link_by_link(pair, T):
    pa, pb, A, B = pair
    x0 = synth.activations(22, T, K0, outliers=True)
    y_last, x_last, (xs, ys) = chain(A, B, x0, T, reuse=False, pdl=True)
    for r in range(ROUNDS):
        Yref, Aa = oracle.gemm_parent(pa, xs[r])
        assert_close(bf16_to_f64(ys[r]), Yref, Aa, f"A, round {r}, T={T}", bf16=True)
        Xref, Ab = oracle.gemm_parent(pb, ys[r])
        assert_close(bf16_to_f64(xs[r + 1]), Xref, Ab, f"B, round {r}, T={T}", bf16=True)
    # the same chain through reused buffers, with and without the programmatic launch
    for pdl in (True, False):
        y_r, x_r, _ = chain(A, B, x0, T, reuse=True, pdl=pdl)
        assert np.array_equal(y_r, y_last) and np.array_equal(x_r, x_last), f"pdl={pdl}"
    for W in (A, B):
        qg.check(qg.qgemm_plan_set_pdl(W.plan, True))
