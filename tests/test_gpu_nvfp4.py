"""GPU parity of the NVFP4 weight codec against the fp64 oracle.

NVFP4 weights are E2M1 codes with an unsigned E4M3 scale per 16 columns and
an fp32 tensor scale.  A code times its block scale is exact in bf16, so the
kernels feed that product to the tensor cores and apply the tensor scale
where the other codecs apply their per-group scales.  Checked on every route
(the small-T tiles -- straight-line and ring kernels -- and the tcgen05
tiles): every code and a spread of block scales decode exactly (one-hot
activations return the dequantised weight bitwise), parity at every width
and on ragged shapes, repeatability, a multi-parent launch with int4, the
fused outputs, and the tensor scale.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_groupwise_gb300 import synth
from tests.tolerance import assert_close, assert_close_swiglu

torch = pytest.importorskip("torch")
qg = pytest.importorskip("bit_weight_only_groupwise_gb300")

pytestmark = pytest.mark.gpu

NVFP4 = synth.NVFP4
SKINNY32 = 2


def dev_x(x_bits):
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()


def host(Y):
    torch.cuda.synchronize()
    return Y.double().cpu().numpy()


def weights(p, T_max, **kw):
    return qg.GroupwiseWeights(NVFP4, p["N"], p["K"], p["packed"], p["scales"], T_max, tensor_scale=p["tscale"],
                               **kw)


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qg.qgemm_device_status(clear=True) == qg.QGEMM_OK


@pytest.mark.parametrize("tw,force", [(8, None), (32, SKINNY32), (128, None)])
def test_every_code_and_block_scale_decodes_exactly(tw, force):
    # row n holds the 16 E2M1 codes in a rotated order and a spread of UE4M3
    # block scales (subnormals, 1.0, the largest); X = one-hot columns, so
    # Y[t][n] = w[n][k] with k = column t, exact in fp32 (tensor scale 2^-3)
    N, K = 128, 512
    codes = np.stack([np.resize(np.roll(np.arange(16, dtype=np.uint8), n), K) for n in range(N)])
    finite = np.array([b for b in range(0x7F)], np.uint8)                    # every valid block scale
    bs = np.stack([np.resize(np.roll(finite, 5 * n), K // 16) for n in range(N)]).astype(np.uint8)
    p = {"bits": NVFP4, "N": N, "K": K, "codes": codes, "packed": synth.pack_nibbles(codes), "scales": bs,
         "tscale": 0.125}
    W = weights(p, T_max=tw)
    if force is not None:
        qg.check(qg.qgemm_plan_force_route(W.plan, force), "force_route")
    ref_w = oracle.dequant_nvfp4(p["packed"], bs, 0.125, N, K)
    for k0 in range(0, K, tw):
        ks = np.arange(k0, k0 + tw)
        x = np.zeros((tw, K), np.uint16)
        x[np.arange(tw), ks] = 0x3F80                                          # bf16 1.0
        Y = host(W.run(dev_x(x)))
        assert np.array_equal(Y, ref_w[:, ks].T), f"columns {k0}..{k0 + tw - 1} ({W.route(tw)})"


@pytest.mark.parametrize("T", [1, 3, 8, 13, 16, 24, 32, 33, 100, 300])
@pytest.mark.parametrize("N,K", [(5120, 6144), (1000, 1024), (130, 576)])
@pytest.mark.parametrize("small_t_32", [False, True])
def test_parity(T, N, K, small_t_32):
    # K = 576 (9 groups) takes the ring kernel on the small-T tiles
    if small_t_32 and T > 32:
        pytest.skip("the 32-token tile covers T <= 32")
    p = synth.weights(70, N, K, NVFP4)
    W = weights(p, T_max=512)
    if small_t_32:
        qg.check(qg.qgemm_plan_force_route(W.plan, SKINNY32), "force_route")
    x = synth.activations(70, T, K, outliers=True)
    Y = W.run(dev_x(x))
    Yref, A = oracle.gemm_parent(p, x)
    assert_close(host(Y), Yref, A, f"nvfp4 N={N} K={K} T={T} ({W.route(T)})")


@pytest.mark.parametrize("T", [2, 16, 64, 300])
def test_repeatable_and_tensor_scale(T):
    p = synth.weights(71, 2432, 6144, NVFP4)
    W = weights(p, T_max=512)
    X = dev_x(synth.activations(71, T, 6144, outliers=True))
    y0 = W.run(X).clone()
    for _ in range(3):
        assert torch.equal(W.run(X), y0)
    # doubling the tensor scale doubles every output exactly
    qg.check(qg.qgemm_plan_set_tensor_scale(W.plan, 2 * p["tscale"]), "set_tensor_scale")
    assert torch.equal(W.run(X), 2 * y0)


@pytest.mark.parametrize("T", [4, 16, 64])
def test_multi_parent_with_int4(T):
    K = 5120
    pn = synth.weights(72, 4096, K, NVFP4, parent=0)
    pi = synth.weights(72, 1024, K, 4, parent=1)
    ws = [weights(pn, T_max=64),
          qg.GroupwiseWeights(4, pi["N"], K, pi["packed"], pi["scales"], T_max=64)]
    x = synth.activations(72, T, K, outliers=True)
    n0 = qg.qgemm_launch_count()
    Ys = qg.run_multi(ws, dev_x(x))
    assert qg.qgemm_launch_count() - n0 == 1
    for p, Y in zip((pn, pi), Ys):
        Yref, A = oracle.gemm_parent(p, x)
        assert_close(host(Y), Yref, A, f"multi codec {p['bits']} T={T}")


def test_plan_rejects_a_tensor_scale_of_another_codec():
    st, plan = qg.qgemm_plan(256, 512, qg.QGEMM_INT4, 8)
    assert st == qg.QGEMM_OK
    try:
        assert qg.qgemm_plan_set_tensor_scale(plan, 2.0) == qg.QGEMM_ERR_INVALID_ARG
    finally:
        qg.qgemm_plan_destroy(plan)


@pytest.mark.parametrize("T", [1, 8, 30, 100])
def test_fused_outputs(T):
    K = 1024
    p = synth.weights(73, 700, K, NVFP4)
    x = synth.activations(73, T, K, outliers=True)
    # residual add: the oracle's plain result plus R (fp32, read exactly)
    R = np.random.default_rng(T).normal(0, 4, (T, 700)).astype(np.float32)
    W = weights(p, T_max=128, epilogue=qg.QGEMM_EPILOGUE_ADD)
    Y = W.run(dev_x(x), R=torch.from_numpy(R).cuda())
    Yp, A = oracle.gemm_parent(p, x)
    assert_close(host(Y), R.astype(np.float64) + Yp, A + np.abs(R.astype(np.float64)), f"nvfp4 add T={T}")
    # SwiGLU pair
    gate, up = synth.weights(74, 203, K, NVFP4, parent=0), synth.weights(74, 203, K, NVFP4, parent=1)
    P = qg.SwiGLUPair(NVFP4, 203, K, gate["packed"], gate["scales"], up["packed"], up["scales"], T_max=128,
                      tensor_scale=gate["tscale"])
    Ys = P.run(dev_x(x))
    out, g, u, Ag, Au = oracle.swiglu_pair(gate, up, x)
    assert_close_swiglu(host(Ys), out, g, u, Ag, Au, f"nvfp4 swiglu T={T}")
