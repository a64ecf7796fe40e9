"""The Python binding rejects tensors of the wrong shape, dtype, layout or
device before anything reaches the C library: the C entry points see only
pointers, so a short X or Y would otherwise let a kernel read or write past
a buffer.  These checks run on the CPU; no library call is made."""
import pytest

torch = pytest.importorskip("torch")
qg = pytest.importorskip("bit_weight_only_groupwise_gb300")


def fake_weights(N=64, K=128, out=qg.QGEMM_OUT_F32, epilogue=qg.QGEMM_EPILOGUE_STORE, device="cpu"):
    # a holder without a plan: every check below must fire before the plan is used
    w = qg.GroupwiseWeights.__new__(qg.GroupwiseWeights)
    w.codec, w.N, w.K, w.T_max = qg.QGEMM_INT4, N, K, 16
    w.epilogue, w.out, w.plan = epilogue, out, None
    w.device = torch.device(device)
    return w


def raises_status(status, fn, *a, **kw):
    with pytest.raises(qg.QgemmError) as e:
        fn(*a, **kw)
    assert e.value.status == status, str(e.value)


@pytest.fixture(autouse=True)
def _no_library_calls(monkeypatch):
    # any call into the C library from here on is a failure
    def boom(*a, **kw):
        raise AssertionError("the binding called the C library before rejecting its arguments")
    for name in ("qgemm_run", "qgemm_run_ex", "qgemm_run_multi"):
        monkeypatch.setattr(qg, name, boom)
    monkeypatch.setattr(qg, "qgemm_status_string", lambda st: f"status {st}")


def test_x_with_the_wrong_k_is_rejected():
    w = fake_weights(K=128)
    raises_status(qg.QGEMM_ERR_SHAPE, w.run, torch.zeros((4, 64), dtype=torch.bfloat16))


def test_x_must_be_two_dimensional_bf16_and_contiguous():
    w = fake_weights(K=128)
    raises_status(qg.QGEMM_ERR_SHAPE, w.run, torch.zeros(128, dtype=torch.bfloat16))
    raises_status(qg.QGEMM_ERR_SHAPE, w.run, torch.zeros((4, 128), dtype=torch.float32))
    raises_status(qg.QGEMM_ERR_SHAPE, w.run, torch.zeros((128, 8), dtype=torch.bfloat16).t())


def test_outputs_and_residuals_must_match_the_plan():
    w = fake_weights(N=64, K=128)
    X = torch.zeros((4, 128), dtype=torch.int16)               # bf16 bit patterns are accepted
    raises_status(qg.QGEMM_ERR_SHAPE, w.run, X, torch.zeros((4, 63), dtype=torch.float32))
    raises_status(qg.QGEMM_ERR_SHAPE, w.run, X, torch.zeros((3, 64), dtype=torch.float32))
    raises_status(qg.QGEMM_ERR_SHAPE, w.run, X, torch.zeros((4, 64), dtype=torch.bfloat16))
    raises_status(qg.QGEMM_ERR_SHAPE, w.run, X, torch.zeros((64, 4), dtype=torch.float32).t())
    raises_status(qg.QGEMM_ERR_SHAPE, w.run, X, None, None, torch.zeros((4, 32), dtype=torch.float32))
    wb = fake_weights(N=64, K=128, out=qg.QGEMM_OUT_BF16)
    raises_status(qg.QGEMM_ERR_SHAPE, wb.run, X, torch.zeros((4, 64), dtype=torch.float32))


def test_tensors_on_another_device_are_rejected():
    w = fake_weights(device="cuda:0")
    raises_status(qg.QGEMM_ERR_INVALID_ARG, w.run, torch.zeros((4, 128), dtype=torch.bfloat16))


def test_run_multi_checks_every_parent_and_output():
    a, b = fake_weights(N=64, K=128), fake_weights(N=32, K=128)
    X = torch.zeros((2, 128), dtype=torch.bfloat16)
    raises_status(qg.QGEMM_ERR_SHAPE, qg.run_multi, [a, fake_weights(N=32, K=256)], X)
    raises_status(qg.QGEMM_ERR_SHAPE, qg.run_multi, [a, b], torch.zeros((2, 64), dtype=torch.bfloat16))
    raises_status(qg.QGEMM_ERR_SHAPE, qg.run_multi, [a, b], X,
                  [torch.zeros((2, 64)), torch.zeros((2, 64))])
    raises_status(qg.QGEMM_ERR_INVALID_ARG, qg.run_multi, [a, b], X, [torch.zeros((2, 64))])
    raises_status(qg.QGEMM_ERR_INVALID_ARG, qg.run_multi, [], X)
