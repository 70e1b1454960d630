"""Torch-facing binding of the C ABI: argument marshalling only.

Every computation runs in libmgg's CUDA kernels; these functions only turn torch
tensors into device pointers, pick the current stream and raise on a bad status.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import (ACTS, CTA_MODES, DTYPES, FILTERS, MAJORS, ORDERS, SCHEDS, DgluBwdArgs, DsreluBwdArgs, WgradArgs,
                   check, load)

_TORCH_TO_DT = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    return t.data_ptr()


# The current stream's raw handle without building a torch Stream object (the public route
# costs a few microseconds per call, which small calls notice); the public route where torch
# lacks the raw query.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def dglu_bwd_workspace_size(L: int, N: int) -> int:
    return int(load().mgg_dglu_bwd_workspace_size(L, N))


def wgrad_workspace_size(L: int) -> int:
    return int(load().mgg_wgrad_workspace_size(L))


def dglu_bwd_num_tiles(M: int, N: int) -> int:
    return int(load().mgg_dglu_bwd_num_tiles(M, N))


def wgrad_num_tiles(L: int, hidden: int, inter: int) -> int:
    return int(load().mgg_wgrad_num_tiles(L, hidden, inter))


def dglu_bwd_tile_shape():
    import ctypes
    m, n = ctypes.c_int32(), ctypes.c_int32()
    load().mgg_dglu_bwd_tile_shape(ctypes.byref(m), ctypes.byref(n))
    return m.value, n.value


def wgrad_tile_shape(inter: int):
    import ctypes
    m, n = ctypes.c_int32(), ctypes.c_int32()
    load().mgg_wgrad_tile_shape(inter, ctypes.byref(m), ctypes.byref(n))
    return m.value, n.value


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A 256-byte aligned device scratch buffer of at least nbytes."""
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def make_dglu_args(*, a, c, padded_offsets, alpha, beta, prob, dprob, d_row, b=None, b_ptrs=None, N=None,
                   dbias=None, act="dswiglu", geglu_filter="value", gate_first=True, b_major="k",
                   sched="static", workspace=None, tile_log=None, situ_beta1=4.0, situ_beta2=25.0,
                   cta="auto", d_col=None, amax=None) -> DgluBwdArgs:
    M, K = a.shape
    L = padded_offsets.numel()
    if N is None:
        N = c.shape[1] // 2
    args = DgluBwdArgs()
    args.M, args.K, args.N, args.L = M, K, N, L
    args.a = _ptr(a)
    args.b = _ptr(b)
    args.b_ptrs = _ptr(b_ptrs)
    args.c = _ptr(c)
    args.padded_offsets = _ptr(padded_offsets)
    args.alpha, args.beta, args.prob = _ptr(alpha), _ptr(beta), _ptr(prob)
    args.dprob, args.d_row, args.dbias = _ptr(dprob), _ptr(d_row), _ptr(dbias)
    args.d_col, args.amax = _ptr(d_col), _ptr(amax)
    args.workspace = _ptr(workspace)
    args.workspace_bytes = workspace.numel() if workspace is not None else 0
    args.tile_log = _ptr(tile_log)
    args.tile_log_capacity = tile_log.numel() // 4 if tile_log is not None else 0
    args.b_major = MAJORS[b_major]
    args.c_dtype = DTYPES[_TORCH_TO_DT[c.dtype]]
    args.d_dtype = DTYPES[_TORCH_TO_DT[d_row.dtype]]
    args.act = ACTS[act]
    args.geglu_filter = FILTERS[geglu_filter]
    args.gate_first = 1 if gate_first else 0
    args.sched = SCHEDS[sched]
    args.cta_mode = CTA_MODES[cta]
    args.situ_beta1 = situ_beta1
    args.situ_beta2 = situ_beta2
    return args


def dglu_bwd(*, a: torch.Tensor, c: torch.Tensor, padded_offsets: torch.Tensor, alpha: torch.Tensor,
             beta: torch.Tensor, prob: torch.Tensor, dprob: torch.Tensor, d_row: torch.Tensor,
             b: Optional[torch.Tensor] = None, b_ptrs: Optional[torch.Tensor] = None, N: Optional[int] = None,
             dbias: Optional[torch.Tensor] = None, act: str = "dswiglu", geglu_filter: str = "value",
             gate_first: bool = True, b_major: str = "k", sched: str = "dynamic",
             workspace: Optional[torch.Tensor] = None, tile_log: Optional[torch.Tensor] = None, stream=None,
             situ_beta1: float = 4.0, situ_beta2: float = 25.0, cta: str = "auto",
             d_col: Optional[torch.Tensor] = None, amax: Optional[torch.Tensor] = None):
    """Grouped GEMM + dGLU backward (see include/mgg.h, mgg_dglu_bwd).

    ``cta`` is "auto", "single" (128-row tiles per CTA) or "pair" (256-row tiles per CTA pair).
    ``d_col`` (a second D_row) and ``amax`` (fp32 (L, 2), per expert max |dgate|, |dinput|) are
    optional outputs.

    d_row is written; dprob and dbias (when given) are accumulated into.  Returns the
    workspace used (allocated here when not given).
    """
    L = padded_offsets.numel()
    n = N if N is not None else c.shape[1] // 2
    if workspace is None:
        workspace = new_workspace(dglu_bwd_workspace_size(L, n), a.device)
    args = make_dglu_args(a=a, c=c, padded_offsets=padded_offsets, alpha=alpha, beta=beta, prob=prob, dprob=dprob,
                          d_row=d_row, b=b, b_ptrs=b_ptrs, N=n, dbias=dbias, act=act, geglu_filter=geglu_filter,
                          gate_first=gate_first, b_major=b_major, sched=sched, workspace=workspace,
                          tile_log=tile_log, situ_beta1=situ_beta1, situ_beta2=situ_beta2, cta=cta, d_col=d_col,
                          amax=amax)
    check(load().mgg_dglu_bwd(args, _stream(stream)))
    return workspace


def dsrelu_bwd_workspace_size(L: int) -> int:
    return int(load().mgg_dsrelu_bwd_workspace_size(L))


def make_dsrelu_args(*, a, c, padded_offsets, alpha, prob, dprob, d_row, b=None, b_ptrs=None, N=None, b_major="k",
                     d_col=None, amax=None, sched="static", workspace=None, tile_log=None, cta="auto") -> DsreluBwdArgs:
    M, K = a.shape
    args = DsreluBwdArgs()
    args.M, args.K, args.N, args.L = M, K, (N if N is not None else c.shape[1]), padded_offsets.numel()
    args.a, args.b, args.b_ptrs, args.c = _ptr(a), _ptr(b), _ptr(b_ptrs), _ptr(c)
    args.padded_offsets, args.alpha, args.prob = _ptr(padded_offsets), _ptr(alpha), _ptr(prob)
    args.dprob, args.d_row, args.d_col, args.amax = _ptr(dprob), _ptr(d_row), _ptr(d_col), _ptr(amax)
    args.workspace = _ptr(workspace)
    args.workspace_bytes = workspace.numel() if workspace is not None else 0
    args.tile_log = _ptr(tile_log)
    args.tile_log_capacity = tile_log.numel() // 4 if tile_log is not None else 0
    args.b_major = MAJORS[b_major]
    args.c_dtype = DTYPES[_TORCH_TO_DT[c.dtype]]
    args.d_dtype = DTYPES[_TORCH_TO_DT[d_row.dtype]]
    args.sched = SCHEDS[sched]
    args.cta_mode = CTA_MODES[cta]
    args.reserved = 0
    return args


def dsrelu_bwd(*, a: torch.Tensor, c: torch.Tensor, padded_offsets: torch.Tensor, alpha: torch.Tensor,
               prob: torch.Tensor, dprob: torch.Tensor, d_row: torch.Tensor, b: Optional[torch.Tensor] = None,
               b_ptrs: Optional[torch.Tensor] = None, N: Optional[int] = None, b_major: str = "k",
               d_col: Optional[torch.Tensor] = None, amax: Optional[torch.Tensor] = None, sched: str = "dynamic",
               workspace: Optional[torch.Tensor] = None, tile_log: Optional[torch.Tensor] = None, stream=None,
               cta: str = "auto"):
    """Grouped GEMM + dsReLU backward (see include/mgg.h, mgg_dsrelu_bwd): D_row = prob*2*C*relu(G),
    dprob += sum C*relu(G)^2 with G = alpha_g A_g B_g^T; optional D_col copy and per-expert amax (L,).
    Returns the workspace used."""
    L = padded_offsets.numel()
    if workspace is None:
        workspace = new_workspace(dsrelu_bwd_workspace_size(L), a.device)
    args = make_dsrelu_args(a=a, c=c, padded_offsets=padded_offsets, alpha=alpha, prob=prob, dprob=dprob,
                            d_row=d_row, b=b, b_ptrs=b_ptrs, N=N, b_major=b_major, d_col=d_col, amax=amax,
                            sched=sched, workspace=workspace, tile_log=tile_log, cta=cta)
    check(load().mgg_dsrelu_bwd(args, _stream(stream)))
    return workspace


def make_wgrad_args(*, a, b, offsets, hidden, inter, out=None, out_ptrs=None, out_dtype=None, a_major="k",
                    b_major="n", input_order="tensor2d", accumulate=False, sched="static", workspace=None,
                    tile_log=None, tokens_sum=None, cta="auto") -> WgradArgs:
    L = offsets.numel()
    args = WgradArgs()
    args.hidden, args.inter, args.L = hidden, inter, L
    args.tokens_sum = tokens_sum if tokens_sum is not None else a.numel() // hidden
    args.a, args.b, args.offsets = _ptr(a), _ptr(b), _ptr(offsets)
    args.out, args.out_ptrs = _ptr(out), _ptr(out_ptrs)
    args.workspace = _ptr(workspace)
    args.workspace_bytes = workspace.numel() if workspace is not None else 0
    args.tile_log = _ptr(tile_log)
    args.tile_log_capacity = tile_log.numel() // 4 if tile_log is not None else 0
    args.a_major = MAJORS[a_major]
    args.b_major = MAJORS[b_major]
    args.input_order = ORDERS[input_order]
    if out_dtype is None:
        out_dtype = _TORCH_TO_DT[out.dtype]
    args.out_dtype = DTYPES[out_dtype]
    args.accumulate = 1 if accumulate else 0
    args.sched = SCHEDS[sched]
    args.cta_mode = CTA_MODES[cta]
    args.reserved1 = 0
    return args


def wgrad(*, a: torch.Tensor, b: torch.Tensor, offsets: torch.Tensor, hidden: int, inter: int,
          out: Optional[torch.Tensor] = None, out_ptrs: Optional[torch.Tensor] = None,
          out_dtype: Optional[str] = None, a_major: str = "k", b_major: str = "n", input_order: str = "tensor2d",
          accumulate: bool = False, sched: str = "dynamic", workspace: Optional[torch.Tensor] = None,
          tile_log: Optional[torch.Tensor] = None, stream=None, cta: str = "auto"):
    """Grouped wgrad (see include/mgg.h, mgg_wgrad).  ``a``/``b`` are the flat bf16 storage
    of A (hidden, T) and B (T, inter) in the declared majors / input order; ``cta`` as in
    dglu_bwd ("pair" needs hidden % 256 == 0)."""
    L = offsets.numel()
    if workspace is None:
        workspace = new_workspace(wgrad_workspace_size(L), a.device)
    args = make_wgrad_args(a=a, b=b, offsets=offsets, hidden=hidden, inter=inter, out=out, out_ptrs=out_ptrs,
                           out_dtype=out_dtype, a_major=a_major, b_major=b_major, input_order=input_order,
                           accumulate=accumulate, sched=sched, workspace=workspace, tile_log=tile_log, cta=cta)
    check(load().mgg_wgrad(args, _stream(stream)))
    return workspace


def wgrad_noalloc(*, a: torch.Tensor, b: torch.Tensor, offsets: torch.Tensor, hidden: int, inter: int,
                  out: Optional[torch.Tensor] = None, out_ptrs: Optional[torch.Tensor] = None,
                  out_dtype: Optional[str] = None, a_major: str = "k", b_major: str = "n",
                  input_order: str = "tensor2d", accumulate: bool = False, sched: str = "dynamic",
                  tile_log: Optional[torch.Tensor] = None, stream=None, cta: str = "auto") -> None:
    """Grouped wgrad that allocates nothing (include/mgg.h, mgg_wgrad_noalloc): for callers that
    cannot allocate device memory; its scratch is a fixed array inside the library (<= 1024
    experts).  Calls share that array, so calls that may overlap on the GPU must be ordered.
    Its device-side checks are not reported: check offsets and output pointers on the host."""
    args = make_wgrad_args(a=a, b=b, offsets=offsets, hidden=hidden, inter=inter, out=out, out_ptrs=out_ptrs,
                           out_dtype=out_dtype, a_major=a_major, b_major=b_major, input_order=input_order,
                           accumulate=accumulate, sched=sched, workspace=None, tile_log=tile_log, cta=cta)
    check(load().mgg_wgrad_noalloc(args, _stream(stream)))


def read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises `stream` and returns the device-side status word of the workspace's last call."""
    return int(load().mgg_read_device_status(_ptr(workspace), _stream(stream)))


def last_error() -> str:
    return load().mgg_last_error().decode()


def pointer_array(tensors: Sequence[torch.Tensor], device) -> torch.Tensor:
    """Device int64 array of the tensors' addresses (discrete weights / outputs)."""
    return torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=device)
