"""GPU parity: the CUDA path through the C-ABI against the fp64 CPU oracle.

Every case draws seeded synthetic inputs, runs the library on the GPU and
compares element by element with the oracle on the same inputs (the
tolerance in tests/tolerance.py).  Wide workloads are compared on a seeded
subset of token columns: the oracle computes each column independently, so
a column subset of X gives exactly those columns of Y.

Bitwise checks cover what the method fixes exactly: basis activations make
every output a single product s*q (dequantisation exactness, nibble order,
the device pack permutation), identity weights return X, negated scales
negate Y, and repeated runs of one (plan, T) are bit-identical.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_groupwise_gb300 import synth
from tests.oracle_columns import gemm_columns, wide_columns
from tests.tolerance import assert_close

torch = pytest.importorskip("torch")
qg = pytest.importorskip("bit_weight_only_groupwise_gb300")

pytestmark = pytest.mark.gpu


def dev_x(x_bits):
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()


def y_host(Y):
    torch.cuda.synchronize()
    return Y.double().cpu().numpy()


def make_weights(parent, T_max):
    return qg.GroupwiseWeights(parent["bits"], parent["N"], parent["K"], parent["packed"], parent["scales"], T_max)


def check_against_oracle(parent, x, Y, cols=None, what=""):
    xs = x if cols is None else x[cols]
    Yref, A = gemm_columns(parent, xs)
    Yg = y_host(Y)
    if cols is not None:
        Yg = Yg[cols]
    return assert_close(Yg, Yref, A, what)


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qg.qgemm_device_status(clear=True) == qg.QGEMM_OK


# ------------------------------------------------------------ the named workloads

def test_tiny_gemv():
    w = synth.workload("tiny", 1)
    p = w["parents"][0]
    W = make_weights(p, T_max=1)
    Y = W.run(dev_x(w["x"]))
    check_against_oracle(p, w["x"], Y, what="tiny T=1")


@pytest.fixture(scope="module")
def decode_weights():
    p = synth.weights(0, 5120, 6144, 4)
    return p, make_weights(p, T_max=8)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8])
def test_decode_widths(decode_weights, T):
    p, W = decode_weights
    x = synth.activations(0, T, 6144, outliers=True)
    Y = W.run(dev_x(x))
    check_against_oracle(p, x, Y, what=f"decode T={T}")


@pytest.fixture(scope="module")
def batched_weights():
    p = synth.weights(0, 12288, 5120, 4)
    return p, make_weights(p, T_max=256)


@pytest.mark.parametrize("T", [16, 32, 64, 256])
def test_batched_widths(batched_weights, T):
    p, W = batched_weights
    x = synth.activations(0, T, 5120, outliers=True)
    Y = W.run(dev_x(x))
    check_against_oracle(p, x, Y, cols=wide_columns(T), what=f"batched T={T}")


@pytest.mark.parametrize("T", [4, 16, 64])
def test_multi_parent_shared_activation(T):
    wl = synth.workload("multi", T)
    ps = wl["parents"]
    Ws = [make_weights(p, T_max=64) for p in ps]
    X = dev_x(wl["x"])
    Ys = qg.run_multi(Ws, X)
    cols = wide_columns(T)
    for p, Y in zip(ps, Ys):
        check_against_oracle(p, wl["x"], Y, cols=cols, what=f"multi T={T} int{p['bits']}")
    # each parent alone: a different launch (its own split count), so the same
    # result within tolerance, and bitwise repeatable in itself
    for p, W, Y in zip(ps, Ws, Ys):
        Y1 = W.run(X)
        check_against_oracle(p, wl["x"], Y1, cols=cols, what=f"single T={T} int{p['bits']}")
        assert np.array_equal(y_host(W.run(X)), y_host(Y1))
    assert np.array_equal(y_host(qg.run_multi(Ws, X)[1]), y_host(Ys[1]))


@pytest.mark.parametrize("name,N,K", [("prefill_a", 7168, 5120), ("prefill_b", 5120, 6144)])
@pytest.mark.parametrize("T", [256, 1024, 4096])
def test_prefill_widths(name, N, K, T):
    p = synth.weights(0, N, K, 4)
    W = make_weights(p, T_max=T)
    x = synth.activations(0, T, K, outliers=True)
    Y = W.run(dev_x(x))
    check_against_oracle(p, x, Y, cols=wide_columns(T), what=f"{name} T={T}")


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("N", [1, 7, 129])
@pytest.mark.parametrize("T", [1, 9, 33])
def test_ragged_rows_and_widths(bits, N, T):
    K = 192
    p = synth.weights(7, N, K, bits)
    W = make_weights(p, T_max=64)
    x = synth.activations(7, T, K, outliers=True)
    # guard bands of NaN around Y catch stray writes
    buf = torch.full((T * N + 64,), float("nan"), dtype=torch.float32, device="cuda")
    Y = buf[32:32 + T * N].view(T, N)
    W.run(dev_x(x), Y)
    check_against_oracle(p, x, Y, what=f"ragged N={N} T={T} int{bits}")
    host = buf.cpu().numpy()
    assert np.isnan(host[:32]).all() and np.isnan(host[32 + T * N:]).all()


def test_single_group():
    p = synth.weights(3, 300, 64, 4)
    W = make_weights(p, T_max=4)
    x = synth.activations(3, 3, 64, outliers=False)
    check_against_oracle(p, x, W.run(dev_x(x)), what="K=64")


def test_domain_and_argument_errors():
    p = synth.weights(1, 128, 128, 4)
    W = make_weights(p, T_max=8)
    X = dev_x(synth.activations(1, 9, 128, outliers=False))
    Y = torch.empty((9, 128), dtype=torch.float32, device="cuda")
    n0 = qg.qgemm_launch_count()
    assert qg.qgemm_run(W.plan, X, 9, Y) == qg.QGEMM_ERR_T_OUT_OF_DOMAIN
    assert qg.qgemm_run(W.plan, X, 0, Y) == qg.QGEMM_OK                       # T = 0: no-op
    assert qg.qgemm_run(W.plan, X.data_ptr() + 2, 1, Y) == qg.QGEMM_ERR_ALIGNMENT
    assert qg.qgemm_run(W.plan, X, 1, Y.data_ptr() + 4) == qg.QGEMM_ERR_ALIGNMENT
    assert qg.qgemm_run(W.plan, None, 1, Y) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_launch_count() == n0                                       # nothing launched
    st, plan = qg.qgemm_plan(128, 100, qg.QGEMM_INT4, 8)
    assert st == qg.QGEMM_ERR_SHAPE
    st, plan = qg.qgemm_plan(128, 128, qg.QGEMM_INT4, 8)
    assert st == qg.QGEMM_OK
    assert qg.qgemm_run(plan, X, 1, Y) == qg.QGEMM_ERR_INVALID_ARG            # not bound
    assert qg.qgemm_plan_workspace_bytes(plan) == 0
    qg.qgemm_plan_destroy(plan)
    other = make_weights(synth.weights(1, 64, 256, 4), T_max=8)
    assert qg.qgemm_run_multi([W.plan, other.plan], X, 1, [Y, Y]) == qg.QGEMM_ERR_SHAPE


@pytest.mark.parametrize("T", [1, 8, 16, 32, 40, 300, 512])
def test_one_route_per_call(T):
    p = synth.weights(2, 256, 512, 4)
    W = make_weights(p, T_max=512)
    X = dev_x(synth.activations(2, T, 512, outliers=False))
    route = W.route(T)
    n0 = qg.qgemm_launch_count()
    W.run(X)
    launched = qg.qgemm_launch_count() - n0
    assert launched == 1, (route, launched)
    # 256 rows, 2 row blocks: the 128-token tile up to T = 511
    assert route == ("skinny8" if T <= 8 else "skinny16" if T <= 16 else "tcgen05_128x32" if T <= 32
                     else "tcgen05_128x64" if T <= 64 else "tcgen05_128x128" if T < 512 else "tcgen05_128x256")
    n0 = qg.qgemm_launch_count()
    qg.GroupwiseWeights(4, 256, 512, p["packed"], p["scales"], T_max=8)
    assert qg.qgemm_launch_count() - n0 == 2            # pack + its ordering kernel


# ------------------------------------------------------------ exact checks

@pytest.mark.parametrize("bits", [4, 5])
def test_basis_activations_give_exact_dequantised_weights(bits):
    N, K = 256, 512
    p = synth.weights(5, N, K, bits)
    ks = np.arange(0, K, 7)[:64]                                   # spans every group and lane
    T = len(ks)
    x = np.zeros((T, K), np.uint16)
    x[np.arange(T), ks] = 0x3F80                                   # bf16 1.0
    W = make_weights(p, T_max=64)
    Yg = y_host(W.run(dev_x(x)))
    Wd = oracle.dequant(bits, p["packed"], p["scales"], N, K)
    assert np.array_equal(Yg, Wd[:, ks].T)


def test_identity_weights_return_x():
    N = K = 128
    eye = np.eye(N, K, dtype=np.int8)
    ones = np.full((N, K // 64), 0x3C00, np.uint16)
    x = synth.activations(6, 5, K, outliers=True)
    W = qg.GroupwiseWeights(4, N, K, synth.pack_canonical(eye, 4), ones, T_max=8)
    Yg = y_host(W.run(dev_x(x)))
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(Yg, xv)


@pytest.mark.parametrize("T", [1, 4, 16, 64])
def test_negated_scales_and_repeatability(T):
    p = synth.weights(8, 1024, 1024, 5)
    q = dict(p, scales=p["scales"] ^ np.uint16(0x8000))
    W, Wn = make_weights(p, T_max=64), make_weights(q, T_max=64)
    X = dev_x(synth.activations(8, T, 1024, outliers=True))
    Y1, Y2, Yn = (y_host(W.run(X)), y_host(W.run(X)), y_host(Wn.run(X)))
    assert np.array_equal(Y1, Y2)
    assert np.array_equal(Yn, -Y1)


@pytest.mark.parametrize("bits,T", [(5, 32), (4, 64), (5, 8)])
def test_repeatable_when_the_stage_ring_wraps(bits, T):
    # 12288 rows x 5120 columns: each warp or CTA streams many more units than
    # its ring holds, so slot reuse must stay exact across the wraps
    p = synth.weights(10, 12288, 5120, bits)
    W = make_weights(p, T_max=64)
    x = synth.activations(10, T, 5120, outliers=True)
    X = dev_x(x)
    Y0 = y_host(W.run(X))
    for _ in range(12):
        assert np.array_equal(y_host(W.run(X)), Y0)
    Yref, A = oracle.gemm_parent(p, x[:4])
    assert_close(Y0[:4], Yref, A)


def test_column_independence_within_tolerance():
    p = synth.weights(9, 640, 1024, 4)
    W = make_weights(p, T_max=64)
    x = synth.activations(9, 40, 1024, outliers=True)
    Yall = y_host(W.run(dev_x(x)))
    for t in (0, 7, 39):
        Yt = y_host(W.run(dev_x(x[t:t + 1])))
        Yref, A = oracle.gemm_parent(p, x[t:t + 1])
        assert_close(Yt, Yref, A)
        assert np.all(np.abs(Yt[0] - Yall[t]) <= 2e-3 * A[0] + 2e-6)


@pytest.mark.parametrize("T", [4, 100])
def test_row_shards_reproduce_the_full_result(T):
    # the data-parallel split: each shard of rows packed and run on its own
    # gives exactly its columns of the unsharded result (rows are independent)
    from bit_weight_only_groupwise_gb300 import sharding
    N, K = 1000, 512
    p = synth.weights(12, N, K, 4)
    X = dev_x(synth.activations(12, T, K, outliers=True))
    full = y_host(make_weights(p, T_max=T).run(X))
    parts = []
    for rank in range(3):
        codes, scales, start, stop = sharding.shard_inputs(p["packed"], p["scales"], N, 3, rank)
        W = qg.GroupwiseWeights(4, stop - start, K, codes, scales, T_max=T)
        parts.append(y_host(W.run(X)))
    assert np.array_equal(np.concatenate(parts, axis=1), full)
