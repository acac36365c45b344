"""The C ABI from plain C: ``abi_c_client.c`` compiles as strict C99 against
``include/ssm.h`` (no CUDA header, no C++), links against the built libssm.so
and runs on the host, without a GPU. It checks the host-only entry points and
the argument checks that precede any device work; its plan and sizes must
equal what the Python binding reports for the same problem."""
import os
import shutil
import subprocess

import pytest

from selective_state_space_119_b300 import build

build.build(quiet=True)
from selective_state_space_119_b300 import libssm as L  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIBDIR = os.path.dirname(L.LIB_PATH)


@pytest.fixture(scope="module")
def client_output(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    exe = str(tmp_path_factory.mktemp("abi") / "abi_c_client")
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "abi_c_client.c"),
                    "-L", LIBDIR, "-lssm", "-Wl,-rpath," + LIBDIR, "-o", exe],
                   check=True, capture_output=True, text=True, timeout=120)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    vals = {}
    for line in r.stdout.splitlines():
        for tok in line.split():
            k, _, v = tok.partition("=")
            if v:
                vals[k] = int(v)
    return vals


def test_c_client_checks_pass(client_output):
    assert client_output["failures"] == 0
    assert client_output["version"] == L.lib.ssm_version()


def test_c_client_plan_matches_binding(client_output):
    plan = L.ssm_scan_plan(4, 2048, 1536, 16, "bf16")
    for k in ("chunk_len", "nchunks", "channels_per_cta", "ctas", "kernels"):
        assert client_output[k] == plan[k], k


def test_c_client_sizes_match_binding(client_output):
    assert client_output["workspace_bytes"] == L.ssm_scan_workspace_bytes(4, 2048, 1536, 16, "bf16")
    assert client_output["workspace_bytes_bc_per_channel"] == L.ssm_scan_workspace_bytes(
        4, 2048, 1536, 16, "bf16", flags=L.SSM_FLAG_BC_PER_CHANNEL)
    assert client_output["checkpoint_bytes"] == 4 * (2048 // 8) * 1536 * 16 * 4
    assert client_output["bwd_workspace_bytes"] == L.ssm_scan_bwd_workspace_bytes(
        4, 2048, 1536, 16, "bf16")
