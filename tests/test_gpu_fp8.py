"""GPU parity of the FP8 (E4M3) weight codec against the fp64 oracle.

Checked on every route: the small-T token tiles of 8, 16 and 32 (the
straight-line kernel where K/64 is a multiple of 8, the ring kernel
otherwise; the 32-token tile forced, since the route table sends T = 17..32
to the tcgen05 route) and the tcgen05 tiles.  Every finite code decodes exactly (one-hot
activations return s * value bitwise, subnormal codes included, on both
kinds of route), parity at every width, ragged N, multi-parent launches
mixing FP8 with int4, and the fused outputs on FP8 weights.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_groupwise_gb300 import synth
from tests.tolerance import assert_close, assert_close_swiglu

torch = pytest.importorskip("torch")
qg = pytest.importorskip("bit_weight_only_groupwise_gb300")

pytestmark = pytest.mark.gpu

SKINNY32 = 2            # the 32-token small-T route, for qgemm_plan_force_route


def dev_x(x_bits):
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()


def host(Y):
    torch.cuda.synchronize()
    return Y.double().cpu().numpy()


def weights(p, T_max, **kw):
    return qg.GroupwiseWeights(p["bits"], p["N"], p["K"], p["packed"], p["scales"], T_max, **kw)


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qg.qgemm_device_status(clear=True) == qg.QGEMM_OK


@pytest.mark.parametrize("tw", [32, 128])
def test_every_code_decodes_exactly(tw):
    # row n holds the finite codes in a rotated order; X = one-hot columns, so
    # Y[t][n] = s[n][k/64] * value(code[n][k]) with k = column t: exact in fp32.
    # tw = 32 runs the 32-token small-T tile (forced), 128 the tcgen05 tile.
    N, K = 128, 512
    finite = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], np.uint8)        # 254 codes
    codes = np.stack([np.resize(np.roll(finite, 3 * n), K) for n in range(N)]).astype(np.uint8)
    scales = synth.group_scales(61, 1, N, K)
    p = {"bits": 8, "N": N, "K": K, "packed": codes, "scales": scales}
    W = weights(p, T_max=tw)
    if tw == 32:
        qg.check(qg.qgemm_plan_force_route(W.plan, SKINNY32), "force_route")
    ref_w = oracle.dequant(8, codes, scales, N, K)
    for k0 in range(0, K, tw):
        ks = np.arange(k0, k0 + tw)
        x = np.zeros((tw, K), np.uint16)
        x[np.arange(tw), ks] = 0x3F80                       # bf16 1.0
        Y = host(W.run(dev_x(x)))
        assert np.array_equal(Y, ref_w[:, ks].T), f"columns {k0}..{k0 + tw - 1} ({W.route(tw)})"


@pytest.mark.parametrize("T", [1, 3, 8, 13, 16, 24, 32, 33, 100, 300])
@pytest.mark.parametrize("N,K", [(5120, 6144), (1000, 1024), (130, 576), (300, 9216)])
@pytest.mark.parametrize("small_t_32", [False, True])
def test_parity(T, N, K, small_t_32):
    # K = 576 (9 groups) and 9216 (144 groups) take the ring kernel on the
    # small-T tiles; small_t_32 forces the 32-token small-T tile for T <= 32
    if small_t_32 and T > 32:
        pytest.skip("the 32-token tile covers T <= 32")
    p = synth.weights(62, N, K, 8)
    W = weights(p, T_max=512)
    if small_t_32:
        qg.check(qg.qgemm_plan_force_route(W.plan, SKINNY32), "force_route")
    x = synth.activations(62, T, K, outliers=True)
    Y = W.run(dev_x(x))
    Yref, A = oracle.gemm_parent(p, x)
    assert_close(host(Y), Yref, A, f"fp8 N={N} K={K} T={T} ({W.route(T)})")


@pytest.mark.parametrize("T", [2, 16])
def test_repeatable(T):
    p = synth.weights(63, 2432, 6144, 8)
    W = weights(p, T_max=32)
    X = dev_x(synth.activations(63, T, 6144, outliers=True))
    y0 = W.run(X).clone()
    for _ in range(3):
        assert torch.equal(W.run(X), y0)


@pytest.mark.parametrize("T", [4, 16, 64])
def test_multi_parent_with_int4(T):
    # every route serves both codecs in one launch (at T = 64 the tcgen05
    # route resolves the codec per tile)
    K = 5120
    pf = synth.weights(64, 4096, K, 8, parent=0)
    pi = synth.weights(64, 1024, K, 4, parent=1)
    ws = [weights(pf, T_max=64), weights(pi, T_max=64)]
    x = synth.activations(64, T, K, outliers=True)
    X = dev_x(x)
    n0 = qg.qgemm_launch_count()
    Ys = qg.run_multi(ws, X)
    assert qg.qgemm_launch_count() - n0 == 1
    for p, Y in zip((pf, pi), Ys):
        Yref, A = oracle.gemm_parent(p, x)
        assert_close(host(Y), Yref, A, f"multi int{p['bits']} T={T}")


@pytest.mark.parametrize("T", [1, 8, 30, 100])
def test_fused_outputs(T):
    K = 1024
    # residual add
    p = synth.weights(65, 700, K, 8)
    x = synth.activations(65, T, K, outliers=True)
    R = np.random.default_rng(T).normal(0, 4, (T, 700)).astype(np.float32)
    W = weights(p, T_max=128, epilogue=qg.QGEMM_EPILOGUE_ADD)
    Y = W.run(dev_x(x), R=torch.from_numpy(R).cuda())
    Yref, A = oracle.linear_add(8, p["packed"], p["scales"], x, R, 700, K)
    assert_close(host(Y), Yref, A, f"fp8 add T={T}")
    # SwiGLU pair
    gate, up = synth.weights(66, 203, K, 8, parent=0), synth.weights(66, 203, K, 8, parent=1)
    P = qg.SwiGLUPair(8, 203, K, gate["packed"], gate["scales"], up["packed"], up["scales"], T_max=128)
    Ys = P.run(dev_x(x))
    out, g, u, Ag, Au = oracle.swiglu_pair(gate, up, x)
    assert_close_swiglu(host(Ys), out, g, u, Ag, Au, f"fp8 swiglu T={T}")


def test_packed_size():
    assert qg.qgemm_packed_bytes(256, 512, qg.QGEMM_FP8) == 2 * (8192 + 256) * 8
