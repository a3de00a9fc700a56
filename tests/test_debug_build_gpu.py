"""The bounds-checked build (-DTSK_DEBUG).

compute-sanitizer is not available on this GPU pool; in its place the
library has a build in which every computed global index and TMA coordinate
of the prefill, FP8, head-dimension-128 and decode kernels is checked
against the extent of its buffer before the access.  A failed check records
TSK_ERR_BOUNDS (-9) in the device status word and skips the access; the
kernel never traps.  These tests build it, run the small parity cases of
every entry point with it (status must stay 0, results must match the CPU
oracle), and make one check fire through a test hook that shrinks the
checked extent below the real one (every access it skips would have been
legal, so nothing faults)."""
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib(tmp_path_factory):
    from gqa_attention_prefill_gb300 import build
    build.build()
    return build.build(out=str(tmp_path_factory.mktemp("dbg") / "libtsk_mha_debug.so"),
                       defines=["TSK_DEBUG"])


def _run(debug_lib, args, timeout=1200):
    env = dict(os.environ, TSK_LIB_PATH=debug_lib, PYTHONPATH=ROOT)
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=timeout)


def test_small_parity_cases_with_every_check(debug_lib):
    r = _run(debug_lib, ["-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                         "tests/test_parity_gpu.py", "tests/test_parity_kvcache_gpu.py",
                         "tests/test_parity_paged_gpu.py", "tests/test_parity_decode_gpu.py",
                         "tests/test_parity_fp8_gpu.py", "tests/test_parity_d128_gpu.py",
                         "tests/test_parity_mha_gpu.py",
                         "-k", "not large_configs and not bench_config and not full_size "
                               "and not bench_configs and not window_config_full"])
    out = r.stdout + r.stderr
    assert r.returncode == 0, out[-4000:]
    assert " passed" in out


CHECK_FIRES = r'''
import numpy as np, torch
import inputgen, parity, gqa_attention_prefill_gb300 as pkg
pkg.load_library()
w = inputgen.make([300, 200], 8, 2, seed=43)
assert pkg.tsk_debug_shrink_extent(1) == 0
out, lse = parity.run_gpu(w, check_status=False)
st = pkg.tsk_get_device_status()
o = out.float().cpu().numpy()
print("status", st, "last row written", bool(np.isfinite(o[-1]).all()),
      "first rows written", bool(np.isfinite(o[:100]).all()))
assert st == -9, st
assert not np.isfinite(o[-1]).any() and np.isfinite(o[:100]).all()
assert pkg.tsk_debug_shrink_extent(0) == 0
print(parity.check_full(w, label="after the hook is cleared"))
'''


def test_a_failed_check_is_reported_and_skips_the_access(debug_lib):
    r = _run(debug_lib, ["-c", "import sys; sys.path.insert(0, 'tests')\n" + CHECK_FIRES])
    out = r.stdout + r.stderr
    assert r.returncode == 0, out[-4000:]
    assert "status -9" in out


def test_release_build_rejects_the_hook():
    import gqa_attention_prefill_gb300 as pkg
    from gqa_attention_prefill_gb300 import build
    build.build()
    pkg.load_library()
    assert pkg.tsk_debug_shrink_extent(1) == -2
