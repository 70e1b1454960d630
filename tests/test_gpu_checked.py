"""The bounds-checked build (build.py --checked, -DMGG_CHECKED) on a subset of the parity suite.

In that build every computed global index, tensor-map slot and TMEM column the kernels use is
tested against the call's extents before the access; a failure would record
MGG_ERR_DEVICE_BOUNDS in the workspace status word, which every parity test asserts to be 0.
The subset runs in a child process with MGG_LIB_VARIANT=checked, so the checked library is the
one loaded there; it covers both operations, single CTAs and pairs, both schedules, dense,
discrete and ragged operands, the register and TMA C paths, fp32 D with dbias and accumulate,
the half-width last column tiles of the wgrad, and the seeded random sweep of option
combinations."""
import os
import subprocess
import sys

import pytest

from moe_grouped_gemm_persistent_gb300.build import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SUBSET = " or ".join([
    "swiglu_dense", "geglu_value_fp32d_dbias", "discrete_n_geglu", "regpath_geglu_fp32d_dbias", "situglu",
    "k_n_fp32", "k_n_fp16_acc", "ragged_k_n_discrete", "out_blocked_acc", "many_experts", "m_n_blocked",
    "exact_ties", "narrow", "sweep",
])


# in range (value 5 < 10): status stays 0 and the guarded write happens; out of range (77 >= 10):
# MGG_ERR_DEVICE_BOUNDS, where 501, value 77, and the guarded write is skipped
BOUNDS_SNIPPET = """
import torch
from moe_grouped_gemm_persistent_gb300 import _lib
lib = _lib.load()
for v in (5, 77):
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    _lib.check(lib.mgg_test_bounds_check(st.data_ptr(), v, 10, None))
    torch.cuda.synchronize()
    print(*st.cpu().tolist())
"""


@pytest.mark.timeout(1800)
def test_parity_subset_under_the_bounds_checked_build():
    build(checked=True)
    env = dict(os.environ, MGG_LIB_VARIANT="checked")
    probe = subprocess.run([sys.executable, "-c", "from moe_grouped_gemm_persistent_gb300 import _lib;"
                            "print(_lib.load().mgg_test_build_flags())"], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip() == "1", probe.stderr[-2000:]
    # the check itself: an index outside its range is recorded (where 501, the value) and not used
    check = subprocess.run([sys.executable, "-c", BOUNDS_SNIPPET], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=300)
    assert check.returncode == 0 and check.stdout.split() == ["0", "0", "0", "1", "8", "501", "77", "0"], \
        (check.stdout, check.stderr[-2000:])
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-k", SUBSET,
                        "tests/test_gpu_parity.py", "tests/test_gpu_dsrelu.py", "tests/test_gpu_sweep.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1700)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail
