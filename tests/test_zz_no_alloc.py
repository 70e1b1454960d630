"""mgg_wgrad_noalloc: the grouped wgrad for callers that cannot allocate device memory.

Such callers (a plugin inside a host program that owns the whole device heap, or code that
must not trigger an allocation mid-run) cannot provide a workspace; this entry point keeps
its scratch in a fixed array inside the library instead.  The test calls it through the
C ABI twice in a row, with different problems so that the second call runs on scratch left
behind by the first, and compares each result with the workspace-based mgg_wgrad.  This file
is collected last on purpose.
"""
import pytest
import torch

from moe_grouped_gemm_persistent_gb300 import _lib, api, synth
from moe_grouped_gemm_persistent_gb300.build import build

from gpu_helpers import TOL, rel_fro, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    build()
    return torch.device("cuda", 0)


def _outputs(spec, dev):
    odt = synth.torch_dtype(spec.out_dtype)
    return [torch.full((spec.hidden, spec.inter), float("nan"), dtype=odt, device=dev) for _ in range(spec.L)]


def _call(fn, spec, x, dev, outs):
    kw = dict(out_ptrs=api.pointer_array(outs, dev), out_dtype=spec.out_dtype)
    fn(a=x["a"], b=x["b"], offsets=x["offsets"], hidden=spec.hidden, inter=spec.inter, a_major=spec.a_major,
       b_major=spec.b_major, input_order=spec.input_order, accumulate=spec.accumulate, **kw)
    torch.cuda.synchronize(dev)
    return torch.stack([o.cpu() for o in outs])


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(dev):
    specs = [
        # tensor_ragged K-major A: per-expert tensor maps live in the fixed scratch
        synth.small_wgrad_spec("na1", counts=(512, 0, 256, 768), input_order="tensor_ragged"),
        # a different expert count, order and dtype for the second call
        synth.small_wgrad_spec("na2", L=3, counts=(256, 768, 256), hidden=256, inter=256, out_dtype="bf16",
                               a_major="m", b_major="k"),
    ]
    inputs = []
    for s in specs:
        y = synth.make_wgrad_inputs(s)
        inputs.append({k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in y.items()})
    refs = [_call(api.wgrad, s, x, dev, _outputs(s, dev)) for s, x in zip(specs, inputs)]
    for s, x, ref in zip(specs, inputs, refs):  # two no-alloc calls back to back
        got = _call(api.wgrad_noalloc, s, x, dev, _outputs(s, dev))
        assert not torch.isnan(got.float()).any()
        for e in range(s.L):
            assert rel_fro(to_np(got[e]), to_np(ref[e])) <= TOL[s.out_dtype], (s.name, e)


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
