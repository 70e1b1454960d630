"""mgg_wgrad_noalloc: the grouped wgrad for callers that cannot allocate device memory.

Such callers (a plugin inside a host program that owns the whole device heap, or code that
must not trigger an allocation mid-run) cannot provide a workspace; this entry point keeps
its scratch in a fixed array inside the library instead.  The tests call it through the
C ABI several times in a row, with different problems so that each call runs on scratch left
behind by the one before, and compare every result with the CPU oracle and with the
workspace-based mgg_wgrad: two calls back to back; a third with accumulate_on_output and the
dynamic schedule, whose empty expert sits in a slot the previous call filled; one with the
documented maximum of 1024 experts, most of them empty; and one with bad offsets, which must
leave the outputs untouched (this entry point does not report the device check).  This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_persistent_gb300 import _lib, api, synth
from moe_grouped_gemm_persistent_gb300.build import build

from gpu_helpers import TOL, rel_fro, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    build()
    return torch.device("cuda", 0)


def _outputs(spec, dev, x=None):
    odt = synth.torch_dtype(spec.out_dtype)
    if spec.accumulate:
        return [x["out_old"][e].to(odt).clone() for e in range(spec.L)]
    return [torch.full((spec.hidden, spec.inter), float("nan"), dtype=odt, device=dev) for _ in range(spec.L)]


def _call(fn, spec, x, dev, outs, sched="dynamic"):
    kw = dict(out_ptrs=api.pointer_array(outs, dev), out_dtype=spec.out_dtype)
    fn(a=x["a"], b=x["b"], offsets=x["offsets"], hidden=spec.hidden, inter=spec.inter, a_major=spec.a_major,
       b_major=spec.b_major, input_order=spec.input_order, accumulate=spec.accumulate, sched=sched, **kw)
    torch.cuda.synchronize(dev)
    return torch.stack([o.cpu() for o in outs])


def _oracle(spec, x):
    old = None
    if spec.accumulate:
        old = to_np(x["out_old"].to(synth.torch_dtype(spec.out_dtype)).cpu())
    return oracle.wgrad(to_np(x["a"].cpu()), to_np(x["b"].cpu()), x["offsets"].cpu().numpy().astype(np.int64),
                        spec.hidden, spec.inter, a_major=spec.a_major, b_major=spec.b_major,
                        input_order=spec.input_order, accumulate=spec.accumulate, out_old=old)


def _inputs(spec, dev):
    y = synth.make_wgrad_inputs(spec)
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in y.items()}


def _check(spec, got, ref, what):
    assert not torch.isnan(got.float()).any(), what
    for e in range(spec.L):
        err = rel_fro(to_np(got[e]), ref[e])
        assert err <= TOL[spec.out_dtype], (what, e, err)
        if spec.counts[e] == 0 and not spec.accumulate:
            assert (got[e] == 0).all(), (what, e)


def test_noalloc_matches_workspace_entry_and_oracle_on_calls_in_a_row(dev):
    specs = [
        # tensor_ragged K-major A: per-expert tensor maps live in the fixed scratch
        synth.small_wgrad_spec("na1", counts=(512, 0, 256, 768), input_order="tensor_ragged"),
        # a different expert count, order and dtype for the second call
        synth.small_wgrad_spec("na2", L=3, counts=(256, 768, 256), hidden=256, inter=256, out_dtype="bf16",
                               a_major="m", b_major="k"),
    ]
    inputs = [_inputs(s, dev) for s in specs]
    refs = [_call(api.wgrad, s, x, dev, _outputs(s, dev)) for s, x in zip(specs, inputs)]
    for s, x, ref in zip(specs, inputs, refs):  # two no-alloc calls back to back
        got = _call(api.wgrad_noalloc, s, x, dev, _outputs(s, dev))
        for e in range(s.L):
            assert rel_fro(to_np(got[e]), to_np(ref[e])) <= TOL[s.out_dtype], (s.name, e)
        _check(s, got, _oracle(s, x), s.name)
    # third call: accumulate_on_output with the dynamic schedule (the scratch's tile counter and
    # active-expert count), ragged maps again, and expert 2 empty where the first call filled it
    s3 = synth.small_wgrad_spec("na3", counts=(256, 512, 0, 256), input_order="tensor_ragged", accumulate=True)
    x3 = _inputs(s3, dev)
    got = _call(api.wgrad_noalloc, s3, x3, dev, _outputs(s3, dev, x3), sched="dynamic")
    _check(s3, got, _oracle(s3, x3), s3.name)
    assert torch.equal(got[2], x3["out_old"][2].cpu()), "an empty expert under accumulate must stay untouched"
    want = _call(api.wgrad, s3, x3, dev, _outputs(s3, dev, x3), sched="dynamic")
    for e in range(s3.L):
        assert rel_fro(to_np(got[e]), to_np(want[e])) <= TOL["fp32"]


def test_noalloc_at_its_maximum_of_1024_experts(dev):
    """The fixed scratch holds the maps of 1024 experts: every one of them is written (empty experts
    as zeros) and each non-empty one matches the oracle."""
    L = 1024
    counts = np.zeros(L, dtype=np.int64)
    for e in (0, 3, 257, 511, 512, 700, 1000, 1023):
        counts[e] = 256
    spec = synth.WgradSpec("na_max", L=L, hidden=128, inter=128, counts=counts, input_order="tensor_ragged",
                           out_mode="discrete")
    x = _inputs(spec, dev)
    got = _call(api.wgrad_noalloc, spec, x, dev, _outputs(spec, dev))
    _check(spec, got, _oracle(spec, x), spec.name)


def test_noalloc_bad_offsets_leave_outputs_untouched(dev):
    spec = synth.small_wgrad_spec("na_bad", counts=(512, 0, 256, 768))
    x = _inputs(spec, dev)
    x["offsets"] = torch.tensor([512, 512, 700, 1536], dtype=torch.int32, device=dev)  # 188 tokens
    outs = [torch.full((spec.hidden, spec.inter), 5.0, dtype=torch.float32, device=dev) for _ in range(spec.L)]
    got = _call(api.wgrad_noalloc, spec, x, dev, outs)  # returns MGG_OK: the device check is not reported
    assert (got == 5.0).all()


def test_noalloc_rejects_more_experts_than_its_scratch(dev):
    lib = _lib.load()
    args = _lib.WgradArgs()
    args.hidden, args.inter, args.L, args.tokens_sum = 256, 128, 1025, 1025 * 256
    buf = torch.empty(1 << 16, dtype=torch.uint8, device=dev)
    args.a = args.b = args.offsets = args.out = buf.data_ptr()
    args.out_dtype = 2
    args.b_major = 1
    st = lib.mgg_wgrad_noalloc(args, None)
    assert st == _lib.MGG_ERR_VALUE
    assert "scratch" in lib.mgg_last_error().decode()
