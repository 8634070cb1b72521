"""The checked build of the library (liblynx_checked.so: every kernel verifies
its index arithmetic where it addresses global memory, records a failed check
in lynx_device_errors bit 8 and clamps the index) on the hot path and its
widened rows.  Its outputs must equal the regular build's bit for bit, and no
check may fire.  The checked build runs in a child process (the binding picks
the library once per process, from LYNX_LIBRARY)."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_matches_and_no_check_fires(lynx_lib, cuda_dev, tmp_path):
    from split_stream_kv_gb300 import _build
    assert os.path.exists(_build.LIB_CHECKED), "the checked build is missing"
    path = tmp_path / "checked.npz"
    env = dict(os.environ, LYNX_LIBRARY="checked")
    r = subprocess.run([sys.executable, os.path.join(HERE, "_checked_cases.py"), str(path)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    checked = dict(np.load(path))
    assert bytes(checked["library"]).decode() == "liblynx_checked.so"
    assert int(checked["device_errors"][0]) == 0, "an index check fired"
    sys.path.insert(0, HERE)
    import _checked_cases
    plain = _checked_cases.run_cases()
    assert bytes(plain["library"]).decode() == "liblynx.so"
    names = sorted(k for k in plain if k not in ("library", "device_errors"))
    assert names == sorted(k for k in checked if k not in ("library", "device_errors"))
    for k in names:
        assert np.array_equal(plain[k], checked[k]), k
