"""GPU parity of the fused outputs against the fp64 oracle.

Residual add (LinearAdd), the SwiGLU of a gate/up pair and bf16 output, on
every route (8-, 16- and 32-token small-T tiles, the tcgen05 tiles), both codecs,
ragged shapes, in place, with the argument errors of the extended entry
points.  Tolerances are in tests/tolerance.py: the residual add keeps the
GEMM's bound with |R| in the magnitude sum; SwiGLU propagates the gate and up
bounds through silu; bf16 adds half an ulp.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_groupwise_gb300 import synth
from tests.tolerance import assert_close, assert_close_swiglu

torch = pytest.importorskip("torch")
qg = pytest.importorskip("bit_weight_only_groupwise_gb300")

pytestmark = pytest.mark.gpu


def dev_x(x_bits):
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()


def host(Y):
    torch.cuda.synchronize()
    return Y.double().cpu().numpy()


def residual(seed, T, N):
    return np.random.default_rng(seed).normal(0.0, 8.0, (T, N)).astype(np.float32)


def weights(p, T_max, **kw):
    return qg.GroupwiseWeights(p["bits"], p["N"], p["K"], p["packed"], p["scales"], T_max, **kw)


def pair(gate, up, T_max, out=qg.QGEMM_OUT_F32):
    return qg.SwiGLUPair(gate["bits"], gate["N"], gate["K"], gate["packed"], gate["scales"], up["packed"],
                         up["scales"], T_max, out=out)


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qg.qgemm_device_status(clear=True) == qg.QGEMM_OK


WIDTHS = [1, 5, 8, 13, 16, 30, 77, 300]          # 8/16-token small-T tiles and the tcgen05 tiles
SKINNY32 = 2                                       # the 32-token small-T route, forced below


@pytest.mark.parametrize("T", WIDTHS)
@pytest.mark.parametrize("bits", [4, 5])
def test_residual_add(T, bits):
    N, K = 1000, 1024
    p = synth.weights(21, N, K, bits)
    W = weights(p, T_max=512, epilogue=qg.QGEMM_EPILOGUE_ADD)
    x = synth.activations(21, T, K, outliers=True)
    R = residual(21 + T, T, N)
    Y = W.run(dev_x(x), R=torch.from_numpy(R).cuda())
    Yref, A = oracle.linear_add(bits, p["packed"], p["scales"], x, R, N, K)
    assert_close(host(Y), Yref, A, f"add int{bits} T={T} ({W.route(T)})")


@pytest.mark.parametrize("T", [1, 16, 300])
def test_residual_add_in_place(T):
    N, K = 517, 512
    p = synth.weights(22, N, K, 4)
    W = weights(p, T_max=512, epilogue=qg.QGEMM_EPILOGUE_ADD)
    X = dev_x(synth.activations(22, T, K, outliers=True))
    R = torch.from_numpy(residual(22, T, N)).cuda()
    out_of_place = W.run(X, R=R)
    Y = R.clone()
    qg.check(qg.qgemm_run_ex(W.plan, X, T, Y, Y), "in place")
    torch.cuda.synchronize()
    assert torch.equal(Y, out_of_place)


@pytest.mark.parametrize("T", WIDTHS)
@pytest.mark.parametrize("bits,F,K", [(4, 1000, 1024), (5, 100, 512), (4, 8, 512), (4, 203, 2048)])
def test_swiglu_pair(T, bits, F, K):
    gate = synth.weights(23, F, K, bits, parent=0)
    up = synth.weights(23, F, K, bits, parent=1)
    P = pair(gate, up, T_max=512)
    x = synth.activations(23, T, K, outliers=True)
    Y = P.run(dev_x(x))
    assert tuple(Y.shape) == (T, F)
    out, g, u, Ag, Au = oracle.swiglu_pair(gate, up, x)
    assert_close_swiglu(host(Y), out, g, u, Ag, Au, f"swiglu int{bits} F={F} K={K} T={T} ({P.route(T)})")


@pytest.mark.parametrize("T", [1, 13, 30, 300])
def test_bf16_outputs(T):
    N, K = 640, 1024
    p = synth.weights(24, N, K, 4)
    x = synth.activations(24, T, K, outliers=True)
    X = dev_x(x)
    # plain
    Wb = weights(p, T_max=512, out=qg.QGEMM_OUT_BF16)
    Y = Wb.run(X)
    assert Y.dtype == torch.bfloat16
    Yref, A = oracle.gemm_parent(p, x)
    assert_close(host(Y), Yref, A, f"bf16 T={T}", bf16=True)
    # bitwise: the bf16 output is the fp32 output rounded to nearest even
    Yf = weights(p, T_max=512).run(X)
    assert torch.equal(Y, Yf.to(torch.bfloat16))
    # residual add
    R = residual(24, T, N)
    Wa = weights(p, T_max=512, epilogue=qg.QGEMM_EPILOGUE_ADD, out=qg.QGEMM_OUT_BF16)
    Ya = Wa.run(X, R=torch.from_numpy(R).cuda())
    Yref, A = oracle.linear_add(4, p["packed"], p["scales"], x, R, N, K)
    assert_close(host(Ya), Yref, A, f"bf16 add T={T}", bf16=True)
    # SwiGLU pair
    gate, up = synth.weights(25, 320, K, 4, parent=0), synth.weights(25, 320, K, 4, parent=1)
    Ys = pair(gate, up, T_max=512, out=qg.QGEMM_OUT_BF16).run(X)
    out, g, u, Ag, Au = oracle.swiglu_pair(gate, up, x)
    assert_close_swiglu(host(Ys), out, g, u, Ag, Au, f"bf16 swiglu T={T}", bf16=True)


@pytest.mark.parametrize("T", [1, 8, 16, 32, 40, 300])
def test_one_launch_and_repeatable(T):
    gate, up = synth.weights(26, 256, 512, 4, parent=0), synth.weights(26, 256, 512, 4, parent=1)
    P = pair(gate, up, T_max=512)
    X = dev_x(synth.activations(26, T, 512, outliers=False))
    n0 = qg.qgemm_launch_count()
    y0 = P.run(X).clone()
    assert qg.qgemm_launch_count() - n0 == 1
    for _ in range(3):
        assert torch.equal(P.run(X), y0)


def test_argument_errors():
    N, K, T = 128, 512, 4
    p = synth.weights(27, N, K, 4)
    X = dev_x(synth.activations(27, T, K, outliers=False))
    Y = torch.empty((T, N), dtype=torch.float32, device="cuda")
    R = torch.zeros((T, N), dtype=torch.float32, device="cuda")
    add = weights(p, T_max=8, epilogue=qg.QGEMM_EPILOGUE_ADD)
    plain = weights(p, T_max=8)
    n0 = qg.qgemm_launch_count()
    assert qg.qgemm_run_ex(add.plan, X, T, None, Y) == qg.QGEMM_ERR_INVALID_ARG      # ADD needs R
    assert qg.qgemm_run_ex(plain.plan, X, T, R, Y) == qg.QGEMM_ERR_INVALID_ARG      # STORE takes none
    assert qg.qgemm_run(add.plan, X, T, Y) == qg.QGEMM_ERR_INVALID_ARG             # plain entry point
    assert qg.qgemm_run_multi([add.plan], X, T, [Y]) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_run_ex(add.plan, X, T, R.data_ptr() + 4, Y) == qg.QGEMM_ERR_ALIGNMENT
    assert qg.qgemm_launch_count() == n0
    assert qg.qgemm_plan_set_epilogue(plain.plan, qg.QGEMM_EPILOGUE_ADD) == qg.QGEMM_ERR_INVALID_ARG  # bound
    st, h = qg.qgemm_plan(N, K, qg.QGEMM_INT4, 8)
    assert qg.qgemm_plan_set_epilogue(h, 7) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_plan_set_epilogue(h, qg.QGEMM_EPILOGUE_SWIGLU, 3) == qg.QGEMM_ERR_INVALID_ARG
    qg.qgemm_plan_destroy(h)
    assert qg.qgemm_pair_packed_bytes(0, K, qg.QGEMM_INT4) == 0
    assert qg.qgemm_pair_packed_bytes(9, K, qg.QGEMM_INT4) == qg.qgemm_packed_bytes(32, K, qg.QGEMM_INT4)
    # plain runs are unchanged by the extended path
    y1 = plain.run(X)
    qg.check(qg.qgemm_run_ex(plain.plan, X, T, None, Y), "run_ex plain")
    torch.cuda.synchronize()
    assert torch.equal(y1, Y)


@pytest.mark.parametrize("T", [17, 30])
def test_fused_outputs_on_the_32_token_small_t_tile(T):
    # the route table sends T = 17..32 to the tcgen05 route; the 32-token
    # small-T tile, forced, still serves the fused outputs
    N, K = 1000, 1024
    p = synth.weights(25, N, K, 5)
    x = synth.activations(25, T, K, outliers=True)
    W = weights(p, T_max=64, epilogue=qg.QGEMM_EPILOGUE_ADD)
    qg.check(qg.qgemm_plan_force_route(W.plan, SKINNY32), "force_route")
    assert W.route(T) == "skinny32"
    R = residual(25 + T, T, N)
    Y = W.run(dev_x(x), R=torch.from_numpy(R).cuda())
    Yref, A = oracle.linear_add(5, p["packed"], p["scales"], x, R, N, K)
    assert_close(host(Y), Yref, A, f"add skinny32 T={T}")
    gate, up = synth.weights(26, 203, K, 4, parent=0), synth.weights(26, 203, K, 4, parent=1)
    P = pair(gate, up, T_max=64, out=qg.QGEMM_OUT_BF16)
    qg.check(qg.qgemm_plan_force_route(P.plan, SKINNY32), "force_route")
    Ys = P.run(dev_x(x))
    out, g, u, Ag, Au = oracle.swiglu_pair(gate, up, x)
    assert_close_swiglu(host(Ys), out, g, u, Ag, Au, f"swiglu bf16 skinny32 T={T}", bf16=True)
