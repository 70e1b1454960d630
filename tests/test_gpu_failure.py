"""Failure paths the kernels already have, driven in the safe forms: a bounded wait that runs out
(the wait-timeout test hook: one CTA, or a cluster of two, waits on an mbarrier nothing arrives on,
with a limit of a few milliseconds, and returns with MGG_ERR_DEVICE_TIMEOUT), and the device-side
argument checks of every entry point, which must turn a call into no-ops with the outputs untouched.
No test here faults or hangs the GPU: every wait has a limit and every kernel returns."""
import re

import pytest
import torch

from moe_grouped_gemm_persistent_gb300 import _lib, api, synth
from moe_grouped_gemm_persistent_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    build()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("cluster", [0, 1])
def test_bounded_wait_times_out_and_reports(dev, cluster):
    lib = _lib.load()
    status = torch.full((4,), -1, dtype=torch.int32, device=dev)
    where = 42
    _lib.check(lib.mgg_test_wait_timeout(status.data_ptr(), 2_000_000, where, cluster, None))  # 2 ms
    st = lib.mgg_read_device_status(status.data_ptr(), None)
    assert st == _lib.MGG_ERR_DEVICE_TIMEOUT
    msg = lib.mgg_last_error().decode()
    assert re.search(r"where=42\b", msg), msg
    s = status.cpu().tolist()
    assert s[0] == _lib.MGG_ERR_DEVICE_TIMEOUT and s[1] == where and s[2] == 0
    assert s[3] == 7, s  # the wait failed, a later wait returned at once, the first record was kept
    # the context is still usable: an ordinary call afterwards succeeds
    spec, _ = synth.workload_specs("tiny")
    x = {k: v.to(dev) for k, v in synth.make_dglu_inputs(spec).items()}
    d_row = torch.empty(spec.M, 2 * spec.N, dtype=torch.bfloat16, device=dev)
    dprob = torch.zeros(spec.M, dtype=torch.float32, device=dev)
    ws = api.dglu_bwd(a=x["a"], b=x["b"], c=x["c"], padded_offsets=x["padded_offsets"], alpha=x["alpha"],
                      beta=x["beta"], prob=x["prob"], dprob=dprob, d_row=d_row)
    assert api.read_device_status(ws) == 0


def test_wait_timeout_hook_validates_arguments(dev):
    lib = _lib.load()
    status = torch.zeros(8, dtype=torch.int32, device=dev)
    assert lib.mgg_test_wait_timeout(status.data_ptr() + 4, 1000, 1, 0, None) == _lib.MGG_ERR_VALUE
    assert lib.mgg_test_wait_timeout(status.data_ptr(), 0, 1, 0, None) == _lib.MGG_ERR_VALUE
    assert lib.mgg_test_wait_timeout(status.data_ptr(), 10 ** 9, 1, 0, None) == _lib.MGG_ERR_VALUE
    assert lib.mgg_test_wait_timeout(status.data_ptr(), 1000, 1, 2, None) == _lib.MGG_ERR_VALUE


@pytest.mark.parametrize("cta", ["single", "pair"])
def test_wgrad_bad_offsets_leave_outputs_untouched(dev, cta):
    # the GEMM kernel reads the preparation kernel's verdict after its set-up (it may launch while
    # that kernel runs) and leaves at once, freeing its TMEM, in both CTA modes
    spec = synth.small_wgrad_spec("badoff", hidden=256)
    x = synth.make_wgrad_inputs(spec)
    out = torch.full((spec.L, spec.hidden, spec.inter), 3.0, dtype=torch.float32, device=dev)
    offs = torch.tensor([512, 512, 700, 1536], dtype=torch.int32, device=dev)  # 188 is not a multiple of 256
    ws = api.wgrad(a=x["a"].to(dev), b=x["b"].to(dev), offsets=offs, hidden=spec.hidden, inter=spec.inter, out=out,
                   cta=cta)
    assert api.read_device_status(ws) == _lib.MGG_ERR_DEVICE_OFFSETS
    assert (out == 3.0).all()
    # the next call on the same workspace runs normally
    good = torch.tensor([512, 512, 768, 1536], dtype=torch.int32, device=dev)
    ws = api.wgrad(a=x["a"].to(dev), b=x["b"].to(dev), offsets=good, hidden=spec.hidden, inter=spec.inter, out=out,
                   cta=cta, workspace=ws)
    assert api.read_device_status(ws) == 0
    assert not (out == 3.0).all()
