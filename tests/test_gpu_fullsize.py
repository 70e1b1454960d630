"""Full-size parity: the four large workloads, run through the same ABI calls bench.py times,
checked against the CPU oracle on sampled rows / elements (the oracle evaluates them one
expert at a time), plus properties that hold at any size:

* dgrad: sampled D_row rows and dprob entries vs the oracle (per sampled expert as well);
  the tile log equals the oracle's schedule exactly; dbias of three whole experts (the
  smallest, the largest and a random one) vs the oracle's per-expert column sums, and for every
  expert the column sums of the kernel's own D_row, with zero rows for empty experts.
* dsReLU: the per-expert amax of whole experts vs the oracle's.
* wgrad: sampled output elements of many experts and every element of a few experts vs the
  oracle; accumulate leaves empty experts bit-identical; the tile log equals the schedule.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_persistent_gb300 import api, synth
from moe_grouped_gemm_persistent_gb300.build import build

from gpu_helpers import TOL, TOL_DPROB, rel_fro, tiles_from_log

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def dev():
    build()
    return torch.device("cuda", 0)


def f32(t):
    return t.detach().float().cpu().numpy()


def oracle_whole_expert(spec, x, g, chunk=2048):
    """The oracle on every row of expert g, evaluated as local one-expert problems over row chunks
    (the rows partition the expert, so the column sums add up and the maxima combine): returns
    (dbias row of expert g, amax entry of expert g)."""
    lo, hi = oracle.expert_ranges(np.cumsum(spec.counts))[g]
    bm = x["b"][g]
    b_g = f32(bm) if (spec.b_mode == "dense" or spec.b_major == "k") else f32(bm).T
    cols = spec.N if spec.act == "dsrelu" else 2 * spec.N
    dbias = np.zeros(cols)
    amax = None
    for r0 in range(lo, hi, chunk):
        r1 = min(hi, r0 + chunk)
        offs_local = np.zeros(spec.L, dtype=np.int64)
        offs_local[g:] = r1 - r0
        a_rows, c_rows, p_rows = f32(x["a"][r0:r1]), f32(x["c"][r0:r1]), f32(x["prob"][r0:r1])
        if spec.act == "dsrelu":
            res = oracle.dsrelu_bwd(a_rows, lambda e: b_g, c_rows, offs_local, f32(x["alpha"]), p_rows)
        else:
            res = oracle.dglu_bwd(a_rows, lambda e: b_g, c_rows, offs_local, f32(x["alpha"]), f32(x["beta"]), p_rows,
                                  act=spec.act)
            dbias += res["dbias"][g]
        amax = res["amax"][g] if amax is None else np.maximum(amax, res["amax"][g])
    return dbias, amax


def sampled_experts(counts, rng, n):
    nz = [g for g in range(len(counts)) if counts[g] > 0]
    if len(nz) <= n:
        return nz
    big = int(np.argmax(counts))
    small = int(min(nz, key=lambda g: counts[g]))
    pick = set(rng.choice(nz, size=n - 2, replace=False).tolist()) | {big, small}
    return sorted(pick)


def sample_rows(counts, experts, rng, edge=4, n_random=48):
    offs = np.cumsum(counts)
    ranges = oracle.expert_ranges(offs)
    rows = []
    for g in experts:
        lo, hi = ranges[g]
        rows += list(range(lo, min(lo + edge, hi))) + list(range(max(hi - edge, lo), hi))
        rows += rng.integers(lo, hi, size=max(1, n_random // len(experts))).tolist()
    return np.array(sorted(set(rows)), dtype=np.int64)


def run_dglu_full(spec, dev):
    x = synth.make_dglu_inputs(spec, device=dev)
    M, N, L = spec.M, spec.N, spec.L
    d_row = torch.full((M, 2 * N), float("nan"), dtype=synth.torch_dtype(spec.d_dtype), device=dev)
    dprob = torch.zeros(M, dtype=torch.float32, device=dev)
    dbias = torch.zeros(L, 2 * N, dtype=torch.bfloat16, device=dev) if spec.dbias else None
    if spec.b_mode == "discrete":
        kw = dict(b_ptrs=api.pointer_array(x["b"], dev), b_major=spec.b_major, N=N)
    else:
        kw = dict(b=x["b"])
    log = torch.empty(4 * api.dglu_bwd_num_tiles(M, N), dtype=torch.int32, device=dev)
    ws = api.dglu_bwd(a=x["a"], c=x["c"], padded_offsets=x["padded_offsets"], alpha=x["alpha"], beta=x["beta"],
                      prob=x["prob"], dprob=dprob, d_row=d_row, dbias=dbias, act=spec.act, tile_log=log, **kw)
    assert api.read_device_status(ws) == 0, api.last_error()
    return x, d_row, dprob, dbias, log


def check_dglu_sampled(spec, x, d_row, dprob, rng, n_experts):
    experts = sampled_experts(spec.counts, rng, n_experts)
    rows = sample_rows(spec.counts, experts, rng)
    offs = np.cumsum(spec.counts)
    ranges = oracle.expert_ranges(offs)
    got_all, ref_all, dp_got, dp_ref = [], [], [], []
    for g in experts:
        lo, hi = ranges[g]
        sel = rows[(rows >= lo) & (rows < hi)]
        bm = x["b"][g]
        b_g = f32(bm) if (spec.b_mode == "dense" or spec.b_major == "k") else f32(bm).T
        idx = torch.as_tensor(sel, device=x["a"].device)
        a_rows = f32(x["a"][idx])
        c_rows = f32(x["c"][idx])
        # local problem: expert g owns rows [0, len(sel)) of the gathered rows
        offs_local = np.zeros(spec.L, dtype=np.int64)
        offs_local[g:] = len(sel)
        res = oracle.dglu_bwd(a_rows, lambda e: b_g, c_rows, offs_local, f32(x["alpha"]), f32(x["beta"]),
                              f32(x["prob"][idx]), act=spec.act)
        got = f32(d_row[idx])
        assert not np.isnan(got).any()
        err = rel_fro(got, res["d_row"])
        assert err <= TOL[spec.d_dtype], f"expert {g}: d_row relative error {err:.3e}"
        got_all.append(got)
        ref_all.append(res["d_row"])
        dp_got.append(f32(dprob[idx]))
        dp_ref.append(res["dprob"])
    assert rel_fro(np.concatenate(got_all), np.concatenate(ref_all)) <= TOL[spec.d_dtype]
    assert rel_fro(np.concatenate(dp_got), np.concatenate(dp_ref)) <= TOL_DPROB


@pytest.mark.parametrize("name", ["mixtral", "geglu", "deepseek", "mixtral_situ"])
def test_dgrad_full_size(dev, name):
    spec, _ = synth.workload_specs(name)
    rng = np.random.default_rng(7)
    x, d_row, dprob, dbias, log = run_dglu_full(spec, dev)
    tm, tn = api.dglu_bwd_tile_shape()
    np.testing.assert_array_equal(tiles_from_log(log.cpu()), oracle.dgrad_tiles(np.cumsum(spec.counts), spec.N, tm, tn))
    check_dglu_sampled(spec, x, d_row, dprob, rng, n_experts=8 if spec.L <= 16 else 12)
    if dbias is not None:
        # dbias of whole experts against the oracle: the smallest, the largest and a random one
        nz = [g for g in range(spec.L) if spec.counts[g] > 0]
        pick = {min(nz, key=lambda g: spec.counts[g]), int(np.argmax(spec.counts)), int(rng.choice(nz))}
        for g in sorted(pick):
            want, _ = oracle_whole_expert(spec, x, g)
            err = rel_fro(f32(dbias[g]), want)
            assert err <= TOL["bf16"], f"dbias of expert {g} ({spec.counts[g]} rows): relative error {err:.3e}"
        # property at any size: dbias = per-expert column sums of the kernel's own D_row
        offs = np.cumsum(spec.counts)
        sums = torch.zeros(spec.L, 2 * spec.N, dtype=torch.float64, device=dev)
        for g, (lo, hi) in enumerate(oracle.expert_ranges(offs)):
            if hi > lo:
                sums[g] = d_row[lo:hi].double().sum(0)
            else:
                assert (dbias[g] == 0).all()
        assert rel_fro(f32(dbias), sums.cpu().numpy()) <= TOL["bf16"]
    del x, d_row, dprob, dbias
    torch.cuda.empty_cache()


def test_dsrelu_full_size(dev):
    """The Mixtral-shaped dsReLU layer: sampled D_row rows and dprob vs the oracle, the tile log
    vs the schedule, D_col = D_row bit for bit, amax = the per-expert max |D_row|."""
    spec, _ = synth.workload_specs("dsrelu")
    rng = np.random.default_rng(11)
    x = synth.make_dglu_inputs(spec, device=dev)
    M, N, L = spec.M, spec.N, spec.L
    d_row = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    d_col = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    dprob = torch.zeros(M, dtype=torch.float32, device=dev)
    amax = torch.full((L,), -1.0, dtype=torch.float32, device=dev)
    log = torch.empty(4 * api.dglu_bwd_num_tiles(M, N), dtype=torch.int32, device=dev)
    ws = api.dsrelu_bwd(a=x["a"], b=x["b"], c=x["c"], padded_offsets=x["padded_offsets"], alpha=x["alpha"],
                        prob=x["prob"], dprob=dprob, d_row=d_row, d_col=d_col, amax=amax, tile_log=log)
    assert api.read_device_status(ws) == 0, api.last_error()
    tm, tn = api.dglu_bwd_tile_shape()
    offs = np.cumsum(spec.counts)
    np.testing.assert_array_equal(tiles_from_log(log.cpu()), oracle.dgrad_tiles(offs, N, tm, tn))
    assert torch.equal(d_row.view(torch.int16), d_col.view(torch.int16))
    ranges = oracle.expert_ranges(offs)
    experts = sampled_experts(spec.counts, rng, 6)
    rows = sample_rows(spec.counts, experts, rng)
    got_all, ref_all, dp_got, dp_ref = [], [], [], []
    for g in experts:
        lo, hi = ranges[g]
        sel = rows[(rows >= lo) & (rows < hi)]
        idx = torch.as_tensor(sel, device=dev)
        b_g = f32(x["b"][g])
        offs_local = np.zeros(L, dtype=np.int64)
        offs_local[g:] = len(sel)
        res = oracle.dsrelu_bwd(f32(x["a"][idx]), lambda e: b_g, f32(x["c"][idx]), offs_local, f32(x["alpha"]),
                                f32(x["prob"][idx]))
        got = f32(d_row[idx])
        assert not np.isnan(got).any()
        err = rel_fro(got, res["d_row"])
        assert err <= TOL["bf16"], f"expert {g}: d_row relative error {err:.3e}"
        got_all.append(got)
        ref_all.append(res["d_row"])
        dp_got.append(f32(dprob[idx]))
        dp_ref.append(res["dprob"])
    assert rel_fro(np.concatenate(got_all), np.concatenate(ref_all)) <= TOL["bf16"]
    assert rel_fro(np.concatenate(dp_got), np.concatenate(dp_ref)) <= TOL_DPROB
    # amax of whole experts against the oracle (the smallest and the largest expert)
    nz = [g for g in range(L) if spec.counts[g] > 0]
    for g in sorted({min(nz, key=lambda e: spec.counts[e]), int(np.argmax(spec.counts))}):
        _, want_g = oracle_whole_expert(spec, x, g)
        assert abs(float(amax[g]) - want_g) <= 2e-3 * want_g, (g, float(amax[g]), want_g)
    # amax is taken on the fp32 values before rounding; the bf16 D_row is within 2^-8 of them
    want = torch.stack([d_row[lo:hi].float().abs().max() if hi > lo else torch.zeros((), device=dev)
                        for lo, hi in ranges])
    np.testing.assert_allclose(f32(amax), f32(want), rtol=4e-3, atol=0)
    del x, d_row, d_col, dprob
    torch.cuda.empty_cache()


def test_wgrad_full_size_accumulate_wgrad64(dev):
    _, spec = synth.workload_specs("wgrad64")
    rng = np.random.default_rng(8)
    y = synth.make_wgrad_inputs(spec, device=dev)
    L, h, i = spec.L, spec.hidden, spec.inter
    out = y["out_old"].clone()
    log = torch.empty(4 * api.wgrad_num_tiles(L, h, i), dtype=torch.int32, device=dev)
    ws = api.wgrad(a=y["a"], b=y["b"], offsets=y["offsets"], hidden=h, inter=i, out=out, a_major=spec.a_major,
                   b_major=spec.b_major, accumulate=True, tile_log=log)
    assert api.read_device_status(ws) == 0, api.last_error()
    tm, tn = api.wgrad_tile_shape(i)
    np.testing.assert_array_equal(tiles_from_log(log.cpu()),
                                  oracle.wgrad_tiles(np.cumsum(spec.counts), h, i, tm, tn, True))
    ranges = oracle.expert_ranges(np.cumsum(spec.counts))
    A = y["a"].view(h, spec.T)
    B = y["b"].view(spec.T, i)
    full = sampled_experts(spec.counts, rng, 6)
    for e in range(L):
        lo, hi = ranges[e]
        if hi == lo:
            assert torch.equal(out[e], y["out_old"][e]), f"empty expert {e} was modified"
            continue
        a_blk = f32(A[:, lo:hi]).reshape(-1)
        b_blk = f32(B[lo:hi]).reshape(-1)
        old = f32(y["out_old"][e])
        if e in full:
            ref = oracle.wgrad(a_blk, b_blk, [hi - lo], h, i, accumulate=True, out_old=[old])[0]
            err = rel_fro(f32(out[e]), ref)
        else:
            hh = rng.integers(0, h, 256)
            ii = rng.integers(0, i, 256)
            ref = oracle.wgrad_elements(a_blk, b_blk, [hi - lo], h, i, 0, hh, ii, accumulate=True,
                                        old_values=old[hh, ii])
            err = rel_fro(f32(out[e])[hh, ii], ref)
        assert err <= TOL["fp32"], f"expert {e}: relative error {err:.3e}"
    del y, out
    torch.cuda.empty_cache()


def test_wgrad_full_size_ragged_discrete_deepseek(dev):
    _, spec = synth.workload_specs("deepseek")
    rng = np.random.default_rng(9)
    y = synth.make_wgrad_inputs(spec, device=dev)
    L, h, i = spec.L, spec.hidden, spec.inter
    big = torch.full((L, h, i), float("nan"), dtype=torch.float32, device=dev)
    ptrs = api.pointer_array([big[e] for e in range(L)], dev)
    log = torch.empty(4 * api.wgrad_num_tiles(L, h, i), dtype=torch.int32, device=dev)
    ws = api.wgrad(a=y["a"], b=y["b"], offsets=y["offsets"], hidden=h, inter=i, out_ptrs=ptrs, out_dtype="fp32",
                   a_major="k", b_major="n", input_order="tensor_ragged", tile_log=log)
    assert api.read_device_status(ws) == 0, api.last_error()
    tm, tn = api.wgrad_tile_shape(i)
    np.testing.assert_array_equal(tiles_from_log(log.cpu()),
                                  oracle.wgrad_tiles(np.cumsum(spec.counts), h, i, tm, tn, False))
    assert not torch.isnan(big).any()
    ranges = oracle.expert_ranges(np.cumsum(spec.counts))
    full = set(sampled_experts(spec.counts, rng, 3))
    for e in sampled_experts(spec.counts, rng, 32):
        lo, hi = ranges[e]
        a_blk = f32(y["a"][lo * h:hi * h])          # ragged K-major block (h, K_e)
        b_blk = f32(y["b"].view(spec.T, i)[lo:hi]).reshape(-1)
        if e in full:
            ref = oracle.wgrad(a_blk, b_blk, [hi - lo], h, i)[0]
            err = rel_fro(f32(big[e]), ref)
        else:
            hh = rng.integers(0, h, 256)
            ii = rng.integers(0, i, 256)
            ref = oracle.wgrad_elements(a_blk, b_blk, [hi - lo], h, i, 0, hh, ii)
            err = rel_fro(f32(big[e])[hh, ii], ref)
        assert err <= TOL["fp32"], f"expert {e}: relative error {err:.3e}"
    del y, big
    torch.cuda.empty_cache()
