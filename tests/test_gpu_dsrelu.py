"""GPU parity of the grouped GEMM + dsReLU backward (mgg_dsrelu_bwd) against the CPU oracle, and
of the per-expert amax and the D_col copy on both dgrad epilogues.

Tolerances as for the dGLU path (Frobenius-norm relative error: 1e-2 for 16-bit D_row, 2e-3 for
fp32 D_row and for dprob); amax is compared with 2e-3 relative error (it is a maximum of fp32
values before rounding); D_col must equal D_row bit for bit; the tile log must equal the oracle's
schedule exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_persistent_gb300 import api, synth
from moe_grouped_gemm_persistent_gb300.build import build

from gpu_helpers import TOL, TOL_DPROB, check_close, dglu_b_getter, rel_fro, tiles_from_log, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    build()
    return torch.device("cuda", 0)


def run_dsrelu_gpu(spec, x, dev, sched="dynamic", cta="auto", with_extras=True, dprob0=None):
    M, N, L = spec.M, spec.N, spec.L
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    keep = None
    if spec.b_mode == "dense":
        b_kw = dict(b=g["b"])
    else:
        keep = [t.to(dev) for t in x["b"]]
        b_kw = dict(b_ptrs=api.pointer_array(keep, dev), b_major=spec.b_major, N=N)
    dt = synth.torch_dtype(spec.d_dtype)
    d_row = torch.full((M, N), float("nan"), dtype=dt, device=dev)
    d_col = torch.full((M, N), float("nan"), dtype=dt, device=dev) if with_extras else None
    amax = torch.full((L,), -1.0, dtype=torch.float32, device=dev) if with_extras else None
    dprob = dprob0.to(dev).clone() if dprob0 is not None else torch.zeros(M, dtype=torch.float32, device=dev)
    log = torch.empty(4 * api.dglu_bwd_num_tiles(M, N), dtype=torch.int32, device=dev)
    ws = api.dsrelu_bwd(a=g["a"], c=g["c"], padded_offsets=g["padded_offsets"], alpha=g["alpha"], prob=g["prob"],
                        dprob=dprob, d_row=d_row, d_col=d_col, amax=amax, tile_log=log, sched=sched, cta=cta,
                        **b_kw)
    status = api.read_device_status(ws)
    torch.cuda.synchronize()
    del keep
    return dict(status=status, d_row=d_row.cpu(), d_col=None if d_col is None else d_col.cpu(), dprob=dprob.cpu(),
                amax=None if amax is None else amax.cpu(), tile_log=log.cpu())


def run_dsrelu_oracle(spec, x, dprob0=None):
    b_get = dglu_b_getter(spec, x["b"])
    return oracle.dsrelu_bwd(to_np(x["a"]), b_get, to_np(x["c"]), x["padded_offsets"].numpy(),
                             x["alpha"].numpy(), x["prob"].numpy(),
                             dprob_in=None if dprob0 is None else to_np(dprob0))


DSRELU_CASES = {
    "dense": dict(),
    "ktail_ntail": dict(K=328, N=160),           # N = 2 x 64 + 32: a half-filled last use
    "discrete_k": dict(b_mode="discrete", b_major="k"),
    "discrete_n_blocked": dict(b_mode="discrete", b_major="n", N=192),
    "discrete_n": dict(b_mode="discrete", b_major="n", N=96),
    "fp32d": dict(d_dtype="fp32"),
    "fp16": dict(c_dtype="fp16", d_dtype="fp16"),
    "wide": dict(N=544, K=192, counts=(512, 256)),
    "many_experts": dict(K=128, N=64, counts=(256, 0, 0, 512, 256, 0, 768, 256, 256, 0, 512)),
    "long_k": dict(K=4160, N=96, counts=(256, 0, 256)),
}


@pytest.mark.parametrize("cta", ["single", "pair"])
@pytest.mark.parametrize("case,sched", [(c, "dynamic") for c in DSRELU_CASES] + [("dense", "static"),
                                                                                   ("discrete_n", "static")])
def test_dsrelu_bwd_parity(dev, case, sched, cta):
    kw = dict(DSRELU_CASES[case])
    counts = kw.pop("counts", (256, 0, 512))
    spec = synth.small_dglu_spec(case, L=len(counts), counts=counts, act="dsrelu", **kw)
    x = synth.make_dglu_inputs(spec)
    gpu = run_dsrelu_gpu(spec, x, dev, sched=sched, cta=cta)
    assert gpu["status"] == 0, api.last_error()
    ref = run_dsrelu_oracle(spec, x)
    rows = oracle.expert_ranges(x["padded_offsets"].numpy())
    check_close("d_row", to_np(gpu["d_row"]), ref["d_row"], TOL[spec.d_dtype], rows)
    check_close("dprob", to_np(gpu["dprob"]), ref["dprob"], TOL_DPROB, rows)
    assert torch.equal(gpu["d_col"], gpu["d_row"])
    amax = gpu["amax"].numpy().astype(np.float64)
    for g, (lo, hi) in enumerate(rows):
        if hi == lo:
            assert amax[g] == 0.0
        else:
            assert abs(amax[g] - ref["amax"][g]) <= 2e-3 * ref["amax"][g], (g, amax[g], ref["amax"][g])
    tm, tn = api.dglu_bwd_tile_shape()
    want = oracle.dgrad_tiles(np.cumsum(spec.counts), spec.N, tm, tn)
    np.testing.assert_array_equal(tiles_from_log(gpu["tile_log"]), want)


def test_dsrelu_accumulates_dprob_and_optional_outputs_off(dev):
    spec = synth.small_dglu_spec("acc", act="dsrelu")
    x = synth.make_dglu_inputs(spec)
    dprob0 = torch.randn(spec.M, generator=torch.Generator().manual_seed(3))
    gpu = run_dsrelu_gpu(spec, x, dev, with_extras=False, dprob0=dprob0)
    assert gpu["status"] == 0
    ref = run_dsrelu_oracle(spec, x, dprob0=dprob0)
    check_close("d_row", to_np(gpu["d_row"]), ref["d_row"], TOL["bf16"])
    check_close("dprob", to_np(gpu["dprob"]), ref["dprob"], TOL_DPROB)


@pytest.mark.parametrize("cta", ["single", "pair"])
def test_dsrelu_all_experts_empty(dev, cta):
    """M = 0 (every expert empty; the per-row tensors are empty, with NULL data pointers): the call
    succeeds and the per-expert amax, which the call overwrites, is zero."""
    L, K, N = 3, 128, 128
    empty = dict(a=torch.empty(0, K, dtype=torch.bfloat16, device=dev),
                 c=torch.empty(0, N, dtype=torch.bfloat16, device=dev),
                 prob=torch.empty(0, device=dev), dprob=torch.empty(0, device=dev),
                 d_row=torch.empty(0, N, dtype=torch.bfloat16, device=dev))
    amax = torch.full((L,), 3.0, device=dev)
    ws = api.dsrelu_bwd(b=torch.randn(L, N, K, device=dev).to(torch.bfloat16),
                        padded_offsets=torch.zeros(L, dtype=torch.int32, device=dev),
                        alpha=torch.ones(L, device=dev), amax=amax, cta=cta, **empty)
    assert api.read_device_status(ws) == 0
    assert (amax == 0).all()


def test_dsrelu_bad_offsets_report_and_leave_outputs(dev):
    spec = synth.small_dglu_spec("bad", act="dsrelu")
    x = synth.make_dglu_inputs(spec)
    x["padded_offsets"] = torch.tensor([256, 128, 768], dtype=torch.int32)
    gpu = run_dsrelu_gpu(spec, x, dev)
    assert gpu["status"] == 5
    assert torch.isnan(gpu["d_row"].float()).all() and (gpu["dprob"] == 0).all()
    assert (gpu["amax"] == -1.0).all()  # untouched


@pytest.mark.parametrize("cta", ["single", "pair"])
@pytest.mark.parametrize("case", [dict(act="dgeglu", c_std=4.0), dict(act="dswiglu", d_dtype="fp32"),
                                  dict(act="dswiglu", K=4160, N=64, counts=(256, 512)),
                                  dict(act="dswiglu", c_dtype="fp32")])
def test_dglu_amax_and_d_col(dev, case, cta):
    kw = dict(case)
    counts = kw.pop("counts", (256, 0, 512))
    spec = synth.small_dglu_spec("amax", L=len(counts), counts=counts, **kw)
    x = synth.make_dglu_inputs(spec)
    M, N, L = spec.M, spec.N, spec.L
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    dt = synth.torch_dtype(spec.d_dtype)
    d_row = torch.empty(M, 2 * N, dtype=dt, device=dev)
    d_col = torch.full((M, 2 * N), float("nan"), dtype=dt, device=dev)
    amax = torch.full((L, 2), -1.0, dtype=torch.float32, device=dev)
    dprob = torch.zeros(M, dtype=torch.float32, device=dev)
    ws = api.dglu_bwd(a=g["a"], b=g["b"], c=g["c"], padded_offsets=g["padded_offsets"], alpha=g["alpha"],
                      beta=g["beta"], prob=g["prob"], dprob=dprob, d_row=d_row, act=spec.act, d_col=d_col,
                      amax=amax, cta=cta)
    assert api.read_device_status(ws) == 0
    ref = oracle.dglu_bwd(to_np(x["a"]), dglu_b_getter(spec, x["b"]), to_np(x["c"]), x["padded_offsets"].numpy(),
                          x["alpha"].numpy(), x["beta"].numpy(), x["prob"].numpy(), act=spec.act)
    assert torch.equal(d_col.cpu(), d_row.cpu())
    check_close("d_row", to_np(d_row.cpu()), ref["d_row"], TOL[spec.d_dtype])
    got = amax.cpu().numpy().astype(np.float64)
    for e, (lo, hi) in enumerate(oracle.expert_ranges(x["padded_offsets"].numpy())):
        if hi == lo:
            assert (got[e] == 0).all()
        else:
            np.testing.assert_allclose(got[e], ref["amax"][e], rtol=2e-3)
