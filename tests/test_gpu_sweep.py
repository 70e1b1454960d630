"""GPU parity over seeded random combinations of the options and shapes of every entry point.

The fixed parity cases exercise each option on its own; here a seeded generator draws whole
argument sets at once (activation, C and D dtypes, weight storage and major, dbias, block order
and filter, sched, CTA mode, expert counts with empty experts, K, N, hidden and inter with ragged
tails; for the wgrad the operand majors, input order, output mode and dtype, overwrite or
accumulate), so that options meet in combinations no hand-written case lists.  Every case is
checked against the CPU oracle with the tolerances of the other parity tests (relative Frobenius
error 1e-2 for 16-bit outputs, 2e-3 for fp32 outputs and dprob) and its tile log against the
oracle's schedule exactly.  Shapes follow the host requirements of the ABI (M and token counts
multiples of 256, K a multiple of 8, N a multiple of 32, hidden and inter multiples of 8).
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_persistent_gb300 import api, synth
from moe_grouped_gemm_persistent_gb300.build import build

from gpu_helpers import (TOL, TOL_DPROB, check_close, run_dglu_gpu, run_dglu_oracle, run_wgrad_gpu,
                         run_wgrad_oracle, tiles_from_log, to_np)
from test_gpu_dsrelu import run_dsrelu_gpu, run_dsrelu_oracle

N_DGRAD = 96
N_WGRAD = 96


@pytest.fixture(scope="module")
def dev():
    build()
    return torch.device("cuda", 0)


def _counts(rng, choices, p):
    """1 to 7 experts, empty ones among them, at least one with work (the all-empty call has tests
    of its own)."""
    L = int(rng.integers(1, 8))
    while True:
        c = tuple(int(v) for v in rng.choice(choices, size=L, p=p))
        if sum(c):
            return c


def dgrad_cases(n=N_DGRAD, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        act = str(rng.choice(["dswiglu", "dgeglu", "dsituglu", "dsrelu"], p=[0.3, 0.3, 0.2, 0.2]))
        b_mode = str(rng.choice(["dense", "discrete"]))
        c_dtype = str(rng.choice(["bf16", "fp16"] if act == "dsrelu" else ["bf16", "fp16", "fp32"]))
        kw = dict(
            act=act, b_mode=b_mode, b_major=str(rng.choice(["k", "n"])) if b_mode == "discrete" else "k",
            c_dtype=c_dtype, d_dtype=str(rng.choice(["bf16", "fp16", "fp32"])),
            dbias=act != "dsrelu" and bool(rng.integers(2)),
            c_std=1.0 if act in ("dswiglu", "dsrelu") else float(rng.choice([2.0, 4.0, 8.0])),
            K=int(rng.integers(1, 129)) * 8, N=int(rng.integers(1, 21)) * 32,
            counts=_counts(rng, [0, 256, 512, 768, 1024], [0.25, 0.35, 0.2, 0.1, 0.1]),
        )
        run = dict(gate_first=bool(rng.integers(2)), geglu_filter=str(rng.choice(["value", "indicator"])),
                   sched=str(rng.choice(["static", "dynamic"])), cta=str(rng.choice(["single", "pair", "auto"])))
        out.append((f"d{i:02d}", kw, run))
    return out


def wgrad_cases(n=N_WGRAD, seed=20261204):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        cta = str(rng.choice(["single", "pair", "auto"]))
        hidden = int(rng.integers(1, 3)) * 256 if cta == "pair" else int(rng.integers(1, 81)) * 8
        kw = dict(
            a_major=str(rng.choice(["k", "m"])), b_major=str(rng.choice(["n", "k"])),
            input_order=str(rng.choice(["tensor2d", "tensor_ragged"])),
            out_mode=str(rng.choice(["dense", "discrete"])), out_dtype=str(rng.choice(["fp32", "bf16", "fp16"])),
            accumulate=bool(rng.integers(2)), hidden=hidden, inter=int(rng.integers(1, 97)) * 8,
            counts=_counts(rng, [0, 256, 512, 1024, 1536], [0.25, 0.35, 0.2, 0.1, 0.1]),
        )
        out.append((f"w{i:02d}", kw, dict(sched=str(rng.choice(["static", "dynamic"])), cta=cta)))
    return out


def _ids(cases):
    return [f"{name}-" + "-".join(f"{v}" for v in list(kw.values())[:-1] + list(run.values()))
            for name, kw, run in cases]


DGRAD = dgrad_cases()
WGRAD = wgrad_cases()


def test_sweep_generators_are_seeded_and_cover_the_options():
    """The drawn sets are reproducible and reach every value of every option."""
    assert _ids(dgrad_cases()) == _ids(DGRAD) and _ids(wgrad_cases()) == _ids(WGRAD)
    seen = {}
    for _, kw, run in DGRAD:
        for k, v in {**kw, **run}.items():
            if k not in ("K", "N", "counts", "c_std"):
                seen.setdefault(k, set()).add(v)
    assert seen["act"] == {"dswiglu", "dgeglu", "dsituglu", "dsrelu"}
    assert seen["c_dtype"] == {"bf16", "fp16", "fp32"} and seen["d_dtype"] == {"bf16", "fp16", "fp32"}
    assert seen["cta"] == {"single", "pair", "auto"} and seen["sched"] == {"static", "dynamic"}
    assert seen["b_major"] == {"k", "n"} and seen["dbias"] == {False, True}
    seen = {}
    for _, kw, run in WGRAD:
        for k, v in {**kw, **run}.items():
            if k not in ("hidden", "inter", "counts"):
                seen.setdefault(k, set()).add(v)
    assert all(len(v) >= 2 for v in seen.values()), seen
    assert seen["out_dtype"] == {"fp32", "bf16", "fp16"} and seen["cta"] == {"single", "pair", "auto"}
    # ragged tails and empty experts occur
    assert any(kw["K"] % 64 for _, kw, _ in DGRAD) and any(kw["N"] % 256 for _, kw, _ in DGRAD)
    assert any(0 in kw["counts"] for _, kw, _ in DGRAD) and any(0 in kw["counts"] for _, kw, _ in WGRAD)
    assert any(kw["inter"] % 256 and kw["inter"] % 256 <= 128 for _, kw, _ in WGRAD)  # narrow last tile


@pytest.mark.gpu
@pytest.mark.parametrize("name,kw,run", DGRAD, ids=_ids(DGRAD))
def test_dgrad_sweep(dev, name, kw, run):
    kw = dict(kw)
    counts = kw.pop("counts")
    spec = synth.small_dglu_spec(name, L=len(counts), counts=counts, **kw)
    x = synth.make_dglu_inputs(spec)
    rows = oracle.expert_ranges(np.cumsum(spec.counts))
    if spec.act == "dsrelu":
        gpu = run_dsrelu_gpu(spec, x, dev, sched=run["sched"], cta=run["cta"])
        assert gpu["status"] == 0, api.last_error()
        ref = run_dsrelu_oracle(spec, x)
        assert torch.equal(gpu["d_col"], gpu["d_row"])
    else:
        gpu = run_dglu_gpu(spec, x, dev, gate_first=run["gate_first"], geglu_filter=run["geglu_filter"],
                           tile_log=True, sched=run["sched"], cta=run["cta"])
        assert gpu["status"] == 0, api.last_error()
        ref = run_dglu_oracle(spec, x, gate_first=run["gate_first"], geglu_filter=run["geglu_filter"])
        if spec.dbias:
            check_close("dbias", to_np(gpu["dbias"]), ref["dbias"], TOL["bf16"])
            for g, (lo, hi) in enumerate(rows):
                if hi == lo:
                    assert (gpu["dbias"][g] == 0).all()
    check_close("d_row", to_np(gpu["d_row"]), ref["d_row"], TOL[spec.d_dtype], rows)
    check_close("dprob", to_np(gpu["dprob"]), ref["dprob"], TOL_DPROB, rows)
    tm, tn = api.dglu_bwd_tile_shape()
    np.testing.assert_array_equal(tiles_from_log(gpu["tile_log"]),
                                  oracle.dgrad_tiles(np.cumsum(spec.counts), spec.N, tm, tn))


@pytest.mark.gpu
@pytest.mark.parametrize("name,kw,run", WGRAD, ids=_ids(WGRAD))
def test_wgrad_sweep(dev, name, kw, run):
    kw = dict(kw)
    counts = kw.pop("counts")
    spec = synth.small_wgrad_spec(name, L=len(counts), counts=counts, **kw)
    x = synth.make_wgrad_inputs(spec)
    gpu = run_wgrad_gpu(spec, x, dev, tile_log=True, sched=run["sched"], cta=run["cta"])
    assert gpu["status"] == 0, api.last_error()
    ref = run_wgrad_oracle(spec, x)
    for e in range(spec.L):
        check_close(f"wgrad[{e}]", to_np(gpu["out"][e]), ref[e], TOL[spec.out_dtype])
        if spec.counts[e] == 0:
            if spec.accumulate:
                old = x["out_old"][e].to(synth.torch_dtype(spec.out_dtype))
                assert torch.equal(gpu["out"][e], old)
            else:
                assert (gpu["out"][e] == 0).all()
    tm, tn = api.wgrad_tile_shape(spec.inter)
    np.testing.assert_array_equal(tiles_from_log(gpu["tile_log"]),
                                  oracle.wgrad_tiles(np.cumsum(spec.counts), spec.hidden, spec.inter, tm, tn,
                                                     spec.accumulate))
