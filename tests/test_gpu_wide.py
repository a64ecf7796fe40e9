"""The tcgen05 route's work split and tile widths, against the oracle.

The route cuts the (tile, group) units of a launch into one contiguous range
per CTA (stream-K), so a tile's 64-column groups may be summed by several
CTAs: the last one to finish adds the others' partial sums from the plan's
workspace in a fixed order.  These cases force many splits per tile, mix
codecs over one activation in one launch, and run every tile width (64,
128 and 256 tokens) on the same matrices; each result is compared element-wise with
the fp64 oracle and repeated runs must be bit-identical (the split tiles'
counters return to zero after every run).
"""
import numpy as np
import pytest

from bit_weight_only_groupwise_gb300 import synth
from tests.oracle_columns import gemm_columns, wide_columns
from tests.tolerance import assert_close

torch = pytest.importorskip("torch")
qg = pytest.importorskip("bit_weight_only_groupwise_gb300")

pytestmark = pytest.mark.gpu

SKINNY16, SKINNY32, WIDE128, WIDE256, WIDE64, WIDE32 = 1, 2, 3, 4, 5, 6


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert qg.qgemm_device_status(clear=True) == qg.QGEMM_OK


def dev_x(x_bits):
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()


def host(Y):
    torch.cuda.synchronize()
    return Y.double().cpu().numpy()


def weights(p, T_max, route=None):
    W = qg.GroupwiseWeights(p["bits"], p["N"], p["K"], p["packed"], p["scales"], T_max)
    if route is not None:
        qg.check(qg.qgemm_plan_force_route(W.plan, route), "force_route")
    return W


def check(p, x, Y, what, cols=None):
    cols = np.arange(x.shape[0]) if cols is None else cols
    Yref, A = gemm_columns(p, x[cols])
    assert_close(host(Y)[cols], Yref, A, what)


@pytest.mark.parametrize("N,K,T", [(256, 8192, 40), (130, 4096, 200), (1000, 1024, 129), (128, 64, 33)])
@pytest.mark.parametrize("route", [WIDE32, WIDE64, WIDE128, WIDE256])
def test_split_tiles_match_the_oracle(N, K, T, route):
    # few tiles and many groups: each tile is split over many CTAs
    p = synth.weights(40, N, K, 4)
    W = weights(p, T_max=256, route=route)
    x = synth.activations(40, T, K, outliers=True)
    X = dev_x(x)
    Y0 = W.run(X)
    check(p, x, Y0, f"N={N} K={K} T={T} {W.route(T)}")
    y0 = host(Y0)
    for _ in range(4):
        assert np.array_equal(host(W.run(X)), y0)


@pytest.mark.parametrize("T", [33, 64, 100, 256, 300])
def test_mixed_codecs_share_one_launch(T):
    K = 2048
    ps = [synth.weights(41, 640, K, 4, parent=0), synth.weights(41, 1500, K, 5, parent=1),
          synth.weights(41, 300, K, 8, parent=2)]
    Ws = [weights(p, T_max=512) for p in ps]
    x = synth.activations(41, T, K, outliers=True)
    X = dev_x(x)
    n0 = qg.qgemm_launch_count()
    Ys = qg.run_multi(Ws, X)
    assert qg.qgemm_launch_count() - n0 == 1
    for p, Y in zip(ps, Ys):
        check(p, x, Y, f"multi T={T} codec {p['bits']}", cols=wide_columns(T))
    again = qg.run_multi(Ws, X)
    for Y, Y1 in zip(Ys, again):
        assert torch.equal(Y, Y1)


@pytest.mark.parametrize("bits", [4, 5, 8])
def test_every_tile_width_agrees_with_the_oracle(bits):
    N, K, T = 777, 3072, 520
    p = synth.weights(42, N, K, bits)
    x = synth.activations(42, T, K, outliers=True)
    X = dev_x(x)
    cols = wide_columns(T)
    for route in (WIDE32, WIDE64, WIDE128, WIDE256):
        W = weights(p, T_max=T, route=route)
        check(p, x, W.run(X), f"int{bits} {W.route(T)}", cols=cols)


def test_forcing_a_wide_route_needs_its_workspace():
    p = synth.weights(43, 256, 512, 4)
    tiny = weights(p, T_max=16)
    assert qg.qgemm_plan_workspace_bytes(tiny.plan) == 0
    for route in (WIDE32, WIDE64, WIDE128):
        assert qg.qgemm_plan_force_route(tiny.plan, route) == qg.QGEMM_ERR_INVALID_ARG
    small = weights(p, T_max=32)
    assert qg.qgemm_plan_force_route(small.plan, WIDE128) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_plan_force_route(small.plan, WIDE64) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_plan_force_route(small.plan, WIDE32) == qg.QGEMM_OK
    mid = weights(p, T_max=128)
    assert qg.qgemm_plan_force_route(mid.plan, WIDE256) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_plan_force_route(mid.plan, WIDE128) == qg.QGEMM_OK
    assert qg.qgemm_plan_force_route(mid.plan, WIDE64) == qg.QGEMM_OK
    assert qg.qgemm_plan_force_route(mid.plan, -1) == qg.QGEMM_OK
    assert qg.qgemm_plan_force_route(mid.plan, 99) == qg.QGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("K", [6144, 576])
@pytest.mark.parametrize("T", [9, 17, 24, 32])
def test_forced_small_t_tiles(bits, K, T):
    # the table sends T > 16 to the tcgen05 route; the 16- and 32-token
    # small-T tiles (straight-line kernel at K = 6144, ring kernel at K = 576)
    # still serve every T they cover when forced
    p = synth.weights(44, 700, K, bits)
    x = synth.activations(44, T, K, outliers=True)
    X = dev_x(x)
    for route in (SKINNY16, SKINNY32):
        if route == SKINNY16 and T > 16:
            continue
        W = weights(p, T_max=64, route=route)
        assert W.route(T) == ("skinny16" if route == SKINNY16 else "skinny32")
        check(p, x, W.run(X), f"int{bits} K={K} T={T} {W.route(T)}")


@pytest.mark.parametrize("T_max", [17, 32, 64])
def test_table_route_within_a_narrow_domain(T_max):
    # a plan whose widths stop between 17 and 64 has the workspace of the
    # 32- and 64-token tcgen05 tiles the table picks for T = 17 .. 64
    N, K = 1000, 1024
    p = synth.weights(45, N, K, 4)
    W = weights(p, T_max=T_max)
    assert qg.qgemm_plan_workspace_bytes(W.plan) > 0
    for T in sorted(t for t in {17, 32, T_max} if t <= T_max):
        x = synth.activations(45 + T, T, K, outliers=True)
        assert W.route(T) == ("tcgen05_128x32" if T <= 32 else "tcgen05_128x64")
        check(p, x, W.run(dev_x(x)), f"T_max={T_max} T={T} {W.route(T)}")
