"""The product path has no CPU fallback: the binding refuses host tensors with
an error (it never computes on the CPU), and importing it without a built
libssm.so raises instead of degrading."""
import os
import shutil
import subprocess
import sys

import pytest

from selective_state_space_119_b300 import build

build.build(quiet=True)
from selective_state_space_119_b300 import libssm as L  # noqa: E402

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _host_inputs(b=1, l=8, d=16, n=16):
    x = torch.zeros(b, l, d)
    return x, x.clone(), -torch.ones(d, n), torch.zeros(b, l, n), torch.zeros(b, l, n)


def test_scan_refuses_host_tensors():
    x, delta, A, B, C = _host_inputs()
    with pytest.raises(ValueError, match="CUDA"):
        L.ssm_selective_scan_fwd(x, delta, A, B, C, workspace=torch.zeros(256, dtype=torch.uint8))


def test_every_entry_point_refuses_host_tensors():
    x, delta, A, B, C = _host_inputs()
    calls = [
        lambda: L.ssm_causal_conv1d_silu(x, torch.ones(16, 4)),
        lambda: L.ssm_state_update(torch.zeros(1, 16, 16), x[:, 0].contiguous(),
                                   delta[:, 0].contiguous(), A, B[:, 0].contiguous(),
                                   C[:, 0].contiguous()),
        lambda: L.ssm_selective_scan_fwd_ckpt(x, delta, A, B, C, out=torch.empty_like(x),
                                              final_state=torch.zeros(1, 16, 16),
                                              ckpt=torch.zeros(1, 1, 16, 16),
                                              workspace=torch.zeros(256, dtype=torch.uint8)),
        lambda: L.ssm_selective_scan_bwd(x, delta, A, B, C, torch.zeros(1, 1, 16, 16), x,
                                         workspace=torch.zeros(1 << 16, dtype=torch.uint8)),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="(?i)cuda"):   # the binding's or torch's own guard
            call()


def test_import_without_the_library_raises(tmp_path):
    pkg = tmp_path / "selective_state_space_119_b300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "selective_state_space_119_b300", "libssm.py"), pkg)
    (pkg / "__init__.py").write_text("")
    r = subprocess.run([sys.executable, "-c", "import selective_state_space_119_b300.libssm"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "not built" in r.stderr
