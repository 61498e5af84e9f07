"""The debug build (-DMUON_DEBUG): kernels range-check every table entry before using it.

* The debug library builds, runs the small GPU cases (every tile shape and launch mode,
  fp32 and split fp32, gather / scatter over 7 shards, the allocating and the
  allocation-free orthogonalization) with no check firing, and gives the same bits as
  the release library: the checks change no arithmetic.
* A table entry that is wrong is caught: muon_selftest_device_check runs the gather
  kernel on a chunk longer than its matrix (inside buffers sized so that nothing could
  fault anyway); the check records MUON_ERR_DEVICE_CHECK, the copy is skipped, and the
  context stays usable.  The release library refuses that self-test.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def debug_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from muon_optimizer_step_gb300.csrc import build
    return build.build(debug=True)


def _child(debug_lib, code, timeout=900):
    env = dict(os.environ, MUON_LIB=debug_lib)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stdout + r.stderr
    return r.stdout


def test_debug_build_matches_release_bit_for_bit(debug_lib, tmp_path):
    out = tmp_path / "debug.npz"
    _child(debug_lib, f"import sys; sys.argv = ['x', {str(out)!r}]; "
                      "import runpy; runpy.run_module('tests.debug_cases', run_name='__main__')")
    got = np.load(out)
    assert int(got["debug_build"][0]) == 1
    from tests import debug_cases
    want = debug_cases.run_cases()
    assert int(want["debug_build"][0]) == 0
    assert set(got.files) == set(want)
    for k in want:
        if k == "debug_build":
            continue
        assert np.array_equal(got[k], want[k]), k


def test_a_bad_table_entry_is_caught_and_the_context_survives(debug_lib):
    code = (
        "from muon_optimizer_step_gb300 import capi\n"
        "import torch\n"
        "assert capi.muon_debug_build()\n"
        "capi.muon_check()\n"
        "capi.muon_selftest_device_check()\n"
        "assert capi.muon_check_status() == capi.MUON_ERR_DEVICE_CHECK\n"
        "assert capi.muon_check_status() == capi.MUON_OK\n"
        "x = torch.ones(8, device='cuda') * 2\n"
        "assert float(x.sum()) == 16.0\n"
        "lay = capi.muon_layout_create([(40, 30)], 1, 1)\n"
        "ws = capi.workspace_tensor(lay)\n"
        "f = torch.randn(lay.full_numel, device='cuda')\n"
        "o = torch.zeros_like(f)\n"
        "capi.muon_orthogonalize_full(lay, ws, f, o, 5)\n"
        "capi.muon_check()\n"
        "assert float(o.abs().sum()) > 0\n"
        "print('ok')\n")
    assert "ok" in _child(debug_lib, code)
    from muon_optimizer_step_gb300 import capi
    assert not capi.muon_debug_build()
    with pytest.raises(capi.MuonError) as e:
        capi.muon_selftest_device_check()
    assert e.value.status == capi.MUON_ERR_UNSUPPORTED
