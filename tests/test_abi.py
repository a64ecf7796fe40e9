"""The C-ABI library loads on the CPU and exports every symbol its header declares.

No compute call is made here (there is no GPU); calls that need a device
must report QGEMM_ERR_UNSUPPORTED instead of crashing.
"""
import os
import re
import shutil
import subprocess

import pytest

import bit_weight_only_groupwise_gb300 as qg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qgemm_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(qg.LIB_PATH):
        from bit_weight_only_groupwise_gb300 import build
        build.build()
    return qg.load()


def test_header_lists_the_boundary():
    names = declared_functions()
    for required in ("qgemm_pack_weights", "qgemm_plan", "qgemm_run", "qgemm_run_multi"):
        assert required in names
    assert names == sorted(qg.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_only_entry_points(lib):
    assert qg.qgemm_status_string(qg.QGEMM_OK) == "ok"
    assert "domain" in qg.qgemm_status_string(qg.QGEMM_ERR_T_OUT_OF_DOMAIN)
    # packed size: 128-row blocks x 64-column groups x unit bytes (4352 int4, 5376 int5)
    assert qg.qgemm_packed_bytes(256, 512, qg.QGEMM_INT4) == 2 * 8 * 4352
    assert qg.qgemm_packed_bytes(129, 64, qg.QGEMM_INT5) == 2 * 1 * 5376
    assert qg.qgemm_packed_bytes(5120, 6144, qg.QGEMM_INT4) == 40 * 96 * 4352
    for bad in ((0, 64, 4), (16, 100, 4), (16, 0, 4), (16, 64, 6)):
        assert qg.qgemm_packed_bytes(*bad) == 0
    # FP8 units: 8192 code bytes + 256 scale bytes
    assert qg.qgemm_packed_bytes(256, 512, qg.QGEMM_FP8) == 2 * 8 * 8448
    # a SwiGLU pair of F rows each packs as 16 * ceil(F / 8) rows
    assert qg.qgemm_pair_packed_bytes(8, 512, qg.QGEMM_INT4) == qg.qgemm_packed_bytes(16, 512, qg.QGEMM_INT4)
    assert qg.qgemm_pair_packed_bytes(17408, 5120, qg.QGEMM_INT4) == qg.qgemm_packed_bytes(34816, 5120, qg.QGEMM_INT4)
    assert qg.qgemm_pair_packed_bytes(203, 64, qg.QGEMM_FP8) == qg.qgemm_packed_bytes(416, 64, qg.QGEMM_FP8)
    for bad in ((0, 64, 4), (8, 100, 4), (8, 64, 7)):
        assert qg.qgemm_pair_packed_bytes(*bad) == 0
    assert qg.qgemm_route_name(-1) == "none"
    assert qg.qgemm_launch_count() >= 0


def test_argument_errors_before_any_device_work(lib):
    st, plan = qg.qgemm_plan(64, 100, qg.QGEMM_INT4, 8)
    assert st == qg.QGEMM_ERR_SHAPE and not plan
    st, plan = qg.qgemm_plan(64, 128, 7, 8)
    assert st == qg.QGEMM_ERR_INVALID_ARG
    st, plan = qg.qgemm_plan(64, 128, qg.QGEMM_INT4, 0)
    assert st == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_pack_weights(qg.QGEMM_INT4, 16, 64, None, None, None, 0) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_pack_weights(qg.QGEMM_INT4, 16, 96, 16, 16, 16, 0) == qg.QGEMM_ERR_SHAPE
    assert qg.qgemm_pack_weights(qg.QGEMM_INT4, 16, 64, 16, 16, 8, 0) == qg.QGEMM_ERR_ALIGNMENT
    assert qg.qgemm_run(None, 16, 1, 16, 0) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_run_multi([], 16, 1, [], 0) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_run_ex(None, 16, 1, None, 16, 0) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_plan_set_epilogue(None, qg.QGEMM_EPILOGUE_ADD) == qg.QGEMM_ERR_INVALID_ARG
    # the pair pack validates before launching anything
    assert qg.qgemm_pack_pair(qg.QGEMM_INT4, 8, 64, 16, 16, None, 16, 16, 0) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_pack_pair(qg.QGEMM_INT4, 0, 64, 16, 16, 16, 16, 16, 0) == qg.QGEMM_ERR_SHAPE
    assert qg.qgemm_pack_pair(qg.QGEMM_INT4, 8, 96, 16, 16, 16, 16, 16, 0) == qg.QGEMM_ERR_SHAPE
    assert qg.qgemm_pack_pair(qg.QGEMM_FP8, 8, 64, 16, 16, 16, 16, 8, 0) == qg.QGEMM_ERR_ALIGNMENT
    assert qg.qgemm_pack_pair(6, 8, 64, 16, 16, 16, 16, 16, 0) == qg.QGEMM_ERR_INVALID_ARG
    assert qg.qgemm_plan_destroy(None) == qg.QGEMM_OK


def test_plan_without_gpu_reports_unsupported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, plan = qg.qgemm_plan(256, 512, qg.QGEMM_INT4, 8)
    assert st == qg.QGEMM_ERR_UNSUPPORTED and not plan


def test_header_is_plain_c(lib, tmp_path):
    """A C99 program includes the header (-Wall -Werror), links every entry
    point against the library and runs the host-only calls."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    exe = str(tmp_path / "abi_check")
    libdir = os.path.dirname(qg.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", exe, "-L", libdir, "-lqgemm",
                    f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "abi ok", (out.returncode, out.stdout, out.stderr)
