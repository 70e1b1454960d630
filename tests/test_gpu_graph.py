"""CUDA-graph replay of the ABI calls (dGLU dgrad, dsReLU dgrad, wgrad) with caller-owned workspaces.

The pages' wgrad API lets callers keep a descriptor workspace alive for CUDA Graph replay
("Block-scaled contract"), and the wgrad class API accepts later calls with a different
token distribution.  Here one step (dprob reset, dgrad + dGLU, wgrad) is captured once and
replayed after the inputs were overwritten in place, including new offsets with the same
total: the offsets, pointer arrays and all scalars are read on the device at every replay, and
the tensor maps (built by the prep kernel from the captured template) follow them.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_persistent_gb300 import api, synth
from moe_grouped_gemm_persistent_gb300.build import build

from gpu_helpers import TOL, TOL_DPROB, rel_fro, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    build()
    return torch.device("cuda", 0)


def _fill_inputs(spec_d, spec_w, bufs, seed):
    """New values (same shapes) written in place into the captured buffers."""
    spec_d = synth.DgluSpec(**{**spec_d.__dict__, "seed": seed})
    spec_w = synth.WgradSpec(**{**spec_w.__dict__, "seed": seed})
    x = synth.make_dglu_inputs(spec_d)
    y = synth.make_wgrad_inputs(spec_w)
    for k in ("a", "b", "c", "alpha", "beta", "prob", "padded_offsets"):
        bufs["d"][k].copy_(x[k])
    for k in ("a", "b", "offsets"):
        bufs["w"][k].copy_(y[k])
    return x, y


def _check(spec_d, spec_w, x, y, d_row, dprob, out):
    ref = oracle.dglu_bwd(to_np(x["a"]), lambda g: to_np(x["b"][g]), to_np(x["c"]),
                          x["padded_offsets"].numpy(), x["alpha"].numpy(), x["beta"].numpy(), x["prob"].numpy())
    assert rel_fro(to_np(d_row.cpu()), ref["d_row"]) <= TOL["bf16"]
    assert rel_fro(to_np(dprob.cpu()), ref["dprob"]) <= TOL_DPROB
    wref = oracle.wgrad(to_np(y["a"]), to_np(y["b"]), y["offsets"].numpy(), spec_w.hidden, spec_w.inter)
    for e in range(spec_w.L):
        assert rel_fro(to_np(out[e].cpu()), wref[e]) <= TOL["fp32"], e


def _check_srelu(x, c_s, d_s, dprob_s, amax_s):
    ref = oracle.dsrelu_bwd(to_np(x["a"]), lambda g: to_np(x["b"][g]), to_np(c_s.cpu()), x["padded_offsets"].numpy(),
                            x["alpha"].numpy(), x["prob"].numpy())
    assert rel_fro(to_np(d_s.cpu()), ref["d_row"]) <= TOL["bf16"]
    assert rel_fro(to_np(dprob_s.cpu()), ref["dprob"]) <= TOL_DPROB
    np.testing.assert_allclose(amax_s.cpu().numpy(), ref["amax"], rtol=2e-3, atol=0)


@pytest.mark.parametrize("sched,cta", [("static", "single"), ("dynamic", "single"), ("dynamic", "pair")])
def test_graph_replay_with_new_values_and_new_offsets(dev, sched, cta):
    counts = np.array([512, 0, 256, 768], dtype=np.int64)
    spec_d = synth.small_dglu_spec("g", L=4, counts=counts, K=192, N=96)
    spec_w = synth.small_wgrad_spec("g", L=4, counts=counts, hidden=256, inter=128)
    x0 = synth.make_dglu_inputs(spec_d)
    y0 = synth.make_wgrad_inputs(spec_w)
    bufs = {"d": {k: v.to(dev) for k, v in x0.items()}, "w": {k: v.to(dev) for k, v in y0.items() if v is not None}}
    M, N, L = spec_d.M, spec_d.N, spec_d.L
    d_row = torch.empty(M, 2 * N, dtype=torch.bfloat16, device=dev)
    dprob = torch.zeros(M, dtype=torch.float32, device=dev)
    out = torch.empty(L, spec_w.hidden, spec_w.inter, dtype=torch.float32, device=dev)
    ws_d = api.new_workspace(api.dglu_bwd_workspace_size(L, N), dev)
    ws_w = api.new_workspace(api.wgrad_workspace_size(L), dev)
    d, w = bufs["d"], bufs["w"]
    # a dsReLU call on the same rows (C (M, N) drawn once; its weights are the dGLU call's)
    c_s = torch.randn(M, N, generator=torch.Generator().manual_seed(17)).to(torch.bfloat16).to(dev)
    d_s = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    dprob_s = torch.zeros(M, dtype=torch.float32, device=dev)
    amax_s = torch.empty(L, dtype=torch.float32, device=dev)
    ws_s = api.new_workspace(api.dsrelu_bwd_workspace_size(L), dev)

    def step(stream):
        dprob_s.zero_()
        api.dsrelu_bwd(a=d["a"], b=d["b"], c=c_s, padded_offsets=d["padded_offsets"], alpha=d["alpha"],
                       prob=d["prob"], dprob=dprob_s, d_row=d_s, amax=amax_s, workspace=ws_s, sched=sched,
                       stream=stream, cta=cta)
        dprob.zero_()
        api.dglu_bwd(a=d["a"], b=d["b"], c=d["c"], padded_offsets=d["padded_offsets"], alpha=d["alpha"],
                     beta=d["beta"], prob=d["prob"], dprob=dprob, d_row=d_row, workspace=ws_d, sched=sched,
                     stream=stream, cta=cta)
        api.wgrad(a=w["a"], b=w["b"], offsets=w["offsets"], hidden=spec_w.hidden, inter=spec_w.inter, out=out,
                  workspace=ws_w, sched=sched, stream=stream, cta=cta)

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        step(s)  # eager warm-up on the capture stream
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)

    # replay 1: new values, same offsets
    x, y = _fill_inputs(spec_d, spec_w, bufs, seed=11)
    g.replay()
    torch.cuda.synchronize(dev)
    assert api.read_device_status(ws_d) == 0 and api.read_device_status(ws_w) == 0
    _check(spec_d, spec_w, x, y, d_row, dprob, out)
    _check_srelu(x, c_s, d_s, dprob_s, amax_s)

    # replay 2: another token distribution with the same totals (offsets are device data)
    counts2 = np.array([256, 768, 0, 512], dtype=np.int64)
    spec_d2 = synth.DgluSpec(**{**spec_d.__dict__, "counts": counts2})
    spec_w2 = synth.WgradSpec(**{**spec_w.__dict__, "counts": counts2})
    x, y = _fill_inputs(spec_d2, spec_w2, bufs, seed=12)
    g.replay()
    torch.cuda.synchronize(dev)
    assert api.read_device_status(ws_d) == 0 and api.read_device_status(ws_w) == 0
    assert api.read_device_status(ws_s) == 0
    _check(spec_d2, spec_w2, x, y, d_row, dprob, out)
    _check_srelu(x, c_s, d_s, dprob_s, amax_s)


@pytest.mark.parametrize("cta", ["single", "pair"])
def test_graph_replay_with_pointer_arrays_rewritten(dev, cta):
    """Discrete weights and per-expert outputs under replay: the per-expert tensor maps are rebuilt
    on the device from the pointer arrays at every replay, so rewriting the arrays in place (here:
    the experts' weight and output buffers exchanged) redirects the replayed calls.  The dgrad is
    the dGeGLU with N-major weights, fp32 D_row and dbias; the wgrad reads ragged K-major operands
    and writes one FP32 matrix per expert."""
    counts = np.array([256, 512, 0, 256], dtype=np.int64)
    spec_d = synth.small_dglu_spec("gp", L=4, counts=counts, K=128, N=64, act="dgeglu", c_std=4.0,
                                   b_mode="discrete", b_major="n", d_dtype="fp32", dbias=True)
    spec_w = synth.small_wgrad_spec("gp", L=4, counts=counts, hidden=256, inter=192, input_order="tensor_ragged",
                                    out_mode="discrete")
    x = synth.make_dglu_inputs(spec_d)
    y = synth.make_wgrad_inputs(spec_w)
    M, N, L = spec_d.M, spec_d.N, spec_d.L
    d = {k: v.to(dev) for k, v in x.items() if isinstance(v, torch.Tensor)}
    weights = [t.to(dev) for t in x["b"]]
    b_ptrs = api.pointer_array(weights, dev)
    d_row = torch.empty(M, 2 * N, dtype=torch.float32, device=dev)
    dprob = torch.zeros(M, dtype=torch.float32, device=dev)
    dbias = torch.zeros(L, 2 * N, dtype=torch.bfloat16, device=dev)
    wa, wb, woffs = y["a"].to(dev), y["b"].to(dev), y["offsets"].to(dev)
    outs = [torch.full((spec_w.hidden, spec_w.inter), float("nan"), device=dev) for _ in range(L)]
    out_ptrs = api.pointer_array(outs, dev)
    ws_d = api.new_workspace(api.dglu_bwd_workspace_size(L, N), dev)
    ws_w = api.new_workspace(api.wgrad_workspace_size(L), dev)

    def step(stream):
        dprob.zero_()
        dbias.zero_()
        api.dglu_bwd(a=d["a"], b_ptrs=b_ptrs, b_major="n", N=N, c=d["c"], padded_offsets=d["padded_offsets"],
                     alpha=d["alpha"], beta=d["beta"], prob=d["prob"], dprob=dprob, d_row=d_row, dbias=dbias,
                     act="dgeglu", workspace=ws_d, stream=stream, cta=cta)
        api.wgrad(a=wa, b=wb, offsets=woffs, hidden=spec_w.hidden, inter=spec_w.inter, out_ptrs=out_ptrs,
                  out_dtype="fp32", input_order="tensor_ragged", workspace=ws_w, stream=stream, cta=cta)

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)

    def check(perm_w, perm_o):
        # the experts' weights as the pointer array now lists them; outputs as it now places them
        ref = oracle.dglu_bwd(to_np(x["a"]), lambda gg: to_np(x["b"][perm_w[gg]]).T, to_np(x["c"]),
                              x["padded_offsets"].numpy(), x["alpha"].numpy(), x["beta"].numpy(),
                              x["prob"].numpy(), act="dgeglu")
        assert rel_fro(to_np(d_row.cpu()), ref["d_row"]) <= TOL["fp32"]
        assert rel_fro(to_np(dprob.cpu()), ref["dprob"]) <= TOL_DPROB
        assert rel_fro(to_np(dbias.cpu()), ref["dbias"]) <= TOL["bf16"]
        wref = oracle.wgrad(to_np(y["a"]), to_np(y["b"]), y["offsets"].numpy(), spec_w.hidden, spec_w.inter,
                            input_order="tensor_ragged")
        for e in range(L):
            assert rel_fro(to_np(outs[perm_o[e]].cpu()), wref[e]) <= TOL["fp32"], e

    g.replay()
    torch.cuda.synchronize(dev)
    assert api.read_device_status(ws_d) == 0 and api.read_device_status(ws_w) == 0
    check([0, 1, 2, 3], [0, 1, 2, 3])
    # rewrite both pointer arrays in place: expert g now reads weights[perm[g]] and writes outs[perm[g]]
    perm = [3, 0, 1, 2]
    b_ptrs.copy_(api.pointer_array([weights[p] for p in perm], dev))
    out_ptrs.copy_(api.pointer_array([outs[p] for p in perm], dev))
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize(dev)
    assert api.read_device_status(ws_d) == 0 and api.read_device_status(ws_w) == 0
    check(perm, perm)
