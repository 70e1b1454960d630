"""Shared helpers of the GPU parity tests: run the CUDA path and the CPU oracle on the same
seeded inputs and compare with the tolerances of the task (Frobenius-norm relative error:
<= 1e-2 for bf16/fp16 outputs, <= 2e-3 for fp32 outputs and for dprob)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_grouped_gemm_persistent_gb300 import api, synth

TOL = {"bf16": 1e-2, "fp16": 1e-2, "fp32": 2e-3}
TOL_DPROB = 2e-3


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def rel_fro(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0:
        return float(num)
    return float(num / den)


def check_close(name, got, ref, tol, per_expert_rows=None):
    err = rel_fro(got, ref)
    assert err <= tol, f"{name}: relative Frobenius error {err:.3e} > {tol}"
    if per_expert_rows is not None:
        for g, (lo, hi) in enumerate(per_expert_rows):
            if hi > lo:
                e = rel_fro(got[lo:hi], ref[lo:hi])
                assert e <= tol, f"{name} expert {g}: relative error {e:.3e} > {tol}"
    return err


def dglu_b_getter(spec, b):
    """Oracle view of the weights: (N, K) values of B_g whatever the storage."""
    if spec.b_mode == "dense":
        return lambda g: to_np(b[g])
    if spec.b_major == "k":
        return lambda g: to_np(b[g])
    return lambda g: to_np(b[g]).T  # stored (K, N) row-major = n-major (N, K)


def run_dglu_gpu(spec, x, dev, gate_first=True, geglu_filter="value", dprob0=None, dbias0=None, tile_log=False,
                 dbias=None, sched="static", situ=(4.0, 25.0), cta="auto"):
    """Runs mgg_dglu_bwd on inputs x (CPU tensors from synth) and returns the outputs on CPU."""
    M, N, L = spec.M, spec.N, spec.L
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    if spec.b_mode == "dense":
        b_kw = dict(b=g["b"])
        keep = None
    else:
        keep = [t.to(dev) for t in x["b"]]
        b_kw = dict(b_ptrs=api.pointer_array(keep, dev), b_major=spec.b_major, N=N)
    d_row = torch.full((M, 2 * N), float("nan"), dtype=synth.torch_dtype(spec.d_dtype), device=dev)
    dprob = (dprob0.to(dev).clone() if dprob0 is not None else torch.zeros(M, dtype=torch.float32, device=dev))
    want_dbias = spec.dbias if dbias is None else dbias
    db = None
    if want_dbias:
        db = (dbias0.to(dev).clone() if dbias0 is not None else torch.zeros(L, 2 * N, dtype=torch.bfloat16, device=dev))
    log = None
    if tile_log:
        log = torch.empty(4 * api.dglu_bwd_num_tiles(M, N), dtype=torch.int32, device=dev)
    ws = api.dglu_bwd(a=g["a"], c=g["c"], padded_offsets=g["padded_offsets"], alpha=g["alpha"], beta=g["beta"],
                      prob=g["prob"], dprob=dprob, d_row=d_row, dbias=db, act=spec.act, geglu_filter=geglu_filter,
                      gate_first=gate_first, tile_log=log, sched=sched, situ_beta1=situ[0], situ_beta2=situ[1],
                      cta=cta, **b_kw)
    status = api.read_device_status(ws)
    torch.cuda.synchronize()
    out = dict(status=status, d_row=d_row.cpu(), dprob=dprob.cpu(), dbias=None if db is None else db.cpu(),
               tile_log=None if log is None else log.cpu())
    del keep
    return out


def run_dglu_oracle(spec, x, gate_first=True, geglu_filter="value", dprob0=None, dbias0=None, rows=None,
                    situ=(4.0, 25.0)):
    b_get = dglu_b_getter(spec, x["b"])
    offs = x["padded_offsets"].numpy().astype(np.int64)
    c = to_np(x["c"]) if rows is None else to_np(x["c"][torch.as_tensor(rows)])
    return oracle.dglu_bwd(to_np(x["a"]), b_get, c, offs, x["alpha"].numpy(), x["beta"].numpy(), x["prob"].numpy(),
                           act=spec.act, gate_first=gate_first, geglu_filter=geglu_filter, rows=rows,
                           dprob_in=None if dprob0 is None else to_np(dprob0),
                           dbias_in=None if dbias0 is None else to_np(dbias0), situ_beta1=situ[0],
                           situ_beta2=situ[1])


def wgrad_pack(spec, x):
    """Device tensors of the flat storages, as the binding expects them."""
    return x["a"], x["b"]


def run_wgrad_gpu(spec, x, dev, tile_log=False, sched="static", cta="auto"):
    L, h, i = spec.L, spec.hidden, spec.inter
    a = x["a"].to(dev)
    b = x["b"].to(dev)
    offs = x["offsets"].to(dev)
    odt = synth.torch_dtype(spec.out_dtype)
    if spec.accumulate:
        init = x["out_old"].to(dev).to(odt)
    else:
        init = torch.full((L, h, i), float("nan"), dtype=odt, device=dev)
    if spec.out_mode == "dense":
        out = init.clone()
        kw = dict(out=out)
        outs = None
    else:
        outs = [init[e].clone() for e in range(L)]
        kw = dict(out_ptrs=api.pointer_array(outs, dev), out_dtype=spec.out_dtype)
    log = None
    if tile_log:
        log = torch.empty(4 * api.wgrad_num_tiles(L, h, i), dtype=torch.int32, device=dev)
    ws = api.wgrad(a=a, b=b, offsets=offs, hidden=h, inter=i, a_major=spec.a_major, b_major=spec.b_major,
                   input_order=spec.input_order, accumulate=spec.accumulate, tile_log=log, sched=sched, cta=cta,
                   **kw)
    status = api.read_device_status(ws)
    torch.cuda.synchronize()
    res = out.cpu() if outs is None else torch.stack([o.cpu() for o in outs])
    return dict(status=status, out=res, tile_log=None if log is None else log.cpu())


def run_wgrad_oracle(spec, x, experts=None):
    offs = x["offsets"].numpy().astype(np.int64)
    old = None if not spec.accumulate else to_np(x["out_old"].to(synth.torch_dtype(spec.out_dtype)))
    return oracle.wgrad(to_np(x["a"]), to_np(x["b"]), offs, spec.hidden, spec.inter, a_major=spec.a_major,
                        b_major=spec.b_major, input_order=spec.input_order, accumulate=spec.accumulate, out_old=old,
                        experts=experts)


def tiles_from_log(log: torch.Tensor) -> np.ndarray:
    arr = log.numpy().reshape(-1, 4)
    arr = arr[arr[:, 0] >= 0]
    return np.array(sorted(map(tuple, arr[:, :3].tolist())), dtype=np.int64).reshape(-1, 3)
