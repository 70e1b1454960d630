"""Seeded synthetic inputs for the MoE grouped GEMM backward workloads.

This module draws random numbers and builds expert token counts; it holds
none of the operation's arithmetic.  Both the CUDA path (tests, bench) and
the CPU oracle's tests take their inputs from here, so that the two sides see
the same data.

Recipe (stated once, used everywhere):

* Expert counts come first, from ``numpy.random.default_rng(seed)``.
  - uniform router: ``rng.multinomial(M, [1/L]*L)``;
  - Zipf(s) router: weights ``r**-s`` for ranks r = 1..L, assigned to experts
    through ``rng.permutation(L)``; the last ``n_empty`` experts of that
    permutation get weight 0; weights are renormalised;
  - dgrad row counts: each multinomial count rounded up to a multiple of 256
    (the 256-row group alignment of the grouped dGLU page, "Shapes and
    Divisibility");
  - wgrad token counts: ``256 * rng.multinomial(T/256, p)`` so the sum is
    exactly T and every count is a multiple of 256 (grouped wgrad page, "BF16
    contract": every expert token count must be a multiple of 256).
* Tensors follow, from a ``torch.Generator`` seeded with the same seed on the
  device the tensors live on.  "N(mu, s)" means standard deviation s.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

ALIGN = 256


def ceil_to(x, m=ALIGN):
    return ((np.asarray(x, dtype=np.int64) + m - 1) // m) * m


def router_probs(rng: np.random.Generator, L: int, zipf_s: Optional[float], n_empty: int = 0) -> np.ndarray:
    """Expert selection probabilities: uniform when ``zipf_s`` is None, else Zipf(zipf_s)."""
    if zipf_s is None:
        p = np.full(L, 1.0 / L)
        return p
    ranks = np.arange(1, L + 1, dtype=np.float64)
    w = ranks ** (-float(zipf_s))
    perm = rng.permutation(L)
    p = np.empty(L, dtype=np.float64)
    p[perm] = w
    if n_empty:
        p[perm[L - n_empty:]] = 0.0
    return p / p.sum()


def dgrad_counts(seed: int, L: int, tokens: int, zipf_s: Optional[float], n_empty: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    p = router_probs(rng, L, zipf_s, n_empty)
    return ceil_to(rng.multinomial(tokens, p)).astype(np.int64)


def wgrad_counts(seed: int, L: int, tokens: int, zipf_s: Optional[float], n_empty: int = 0) -> np.ndarray:
    assert tokens % ALIGN == 0
    rng = np.random.default_rng(seed)
    p = router_probs(rng, L, zipf_s, n_empty)
    return (ALIGN * rng.multinomial(tokens // ALIGN, p)).astype(np.int64)


def offsets_from_counts(counts) -> np.ndarray:
    """Cumulative group ends (int32), the layout of ``padded_offsets`` / ``offsets_tensor``."""
    return np.cumsum(np.asarray(counts, dtype=np.int64)).astype(np.int32)


# --------------------------------------------------------------------------------------
# Workload descriptions
# --------------------------------------------------------------------------------------

@dataclasses.dataclass
class DgluSpec:
    name: str
    L: int
    K: int
    N: int
    counts: np.ndarray          # per-expert rows (multiples of 256)
    act: str = "dswiglu"        # "dswiglu" | "dgeglu" | "dsituglu" | "dsrelu" (C, D_row (M, N))
    b_mode: str = "dense"       # "dense" | "discrete"
    b_major: str = "k"          # "k" | "n" (discrete only)
    c_dtype: str = "bf16"
    d_dtype: str = "bf16"
    dbias: bool = False
    a_std: float = 1.0
    b_std: float = 1.0
    c_std: float = 1.0
    seed: int = 0

    @property
    def M(self) -> int:
        return int(np.sum(self.counts))

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


@dataclasses.dataclass
class WgradSpec:
    name: str
    L: int
    hidden: int
    inter: int
    counts: np.ndarray          # per-expert tokens (multiples of 256)
    a_major: str = "k"          # "k": (hidden, T) stride (T, 1); "m": stride (1, hidden)
    b_major: str = "n"          # "n": (T, inter) stride (inter, 1); "k": stride (1, T)
    input_order: str = "tensor2d"   # "tensor2d" | "tensor_ragged"
    out_mode: str = "dense"     # "dense" | "discrete"
    out_dtype: str = "fp32"
    accumulate: bool = False
    seed: int = 0

    @property
    def T(self) -> int:
        return int(np.sum(self.counts))

    @property
    def flops(self) -> float:
        return 2.0 * self.hidden * self.T * self.inter


def workload_specs(name: str):
    """Return (dglu_spec or None, wgrad_spec or None) for a named workload.

    tiny       : L=4, counts [256,0,512,256], K=hidden=256, N=128; dSwiGLU + wgrad (FP32 out)
    mixtral    : L=8, K=4096, N=14336, 32768 tokens uniform router; dSwiGLU, dense B
    geglu      : L=16, K=2048, N=5632, 49152 tokens Zipf(1.1), 2 empty; dGeGLU, discrete
                 n-major B, C ~ N(0,4), FP32 D_row, dbias
    wgrad64    : L=64, hidden=2048, inter=1408, T=65536 Zipf(1.2), 4 forced empty; FP32
                 dense accumulate
    deepseek   : L=256, K=hidden=7168, N=2048, 131072 tokens Zipf(1.0); dSwiGLU dense B,
                 then wgrad on the same ranges (A' ragged K-major), discrete FP32 outputs
    """
    if name == "tiny":
        counts = np.array([256, 0, 512, 256], dtype=np.int64)
        d = DgluSpec("tiny", L=4, K=256, N=128, counts=counts)
        w = WgradSpec("tiny", L=4, hidden=256, inter=128, counts=counts.copy())
        return d, w
    if name == "mixtral":
        counts = dgrad_counts(0, 8, 32768, None)
        return DgluSpec("mixtral", L=8, K=4096, N=14336, counts=counts, b_std=0.02), None
    if name == "geglu":
        counts = dgrad_counts(0, 16, 49152, 1.1, n_empty=2)
        return DgluSpec("geglu", L=16, K=2048, N=5632, counts=counts, act="dgeglu",
                        b_mode="discrete", b_major="n", c_std=4.0, d_dtype="fp32", dbias=True), None
    if name == "wgrad64":
        counts = wgrad_counts(0, 64, 65536, 1.2, n_empty=4)
        return None, WgradSpec("wgrad64", L=64, hidden=2048, inter=1408, counts=counts,
                               a_major="k", b_major="n", accumulate=True)
    if name == "deepseek":
        counts = dgrad_counts(0, 256, 131072, 1.0)
        d = DgluSpec("deepseek", L=256, K=7168, N=2048, counts=counts)
        w = WgradSpec("deepseek", L=256, hidden=7168, inter=2048, counts=counts.copy(),
                      a_major="k", b_major="n", input_order="tensor_ragged", out_mode="discrete")
        return d, w
    # the Mixtral-like layer with the dSiTU-GLU backward (beta1 = 4, beta2 = 25)
    if name == "mixtral_situ":
        counts = dgrad_counts(0, 8, 32768, None)
        return DgluSpec("mixtral_situ", L=8, K=4096, N=14336, counts=counts, b_std=0.02, act="dsituglu",
                        c_std=4.0), None
    # the Mixtral-like layer with the dsReLU backward (squared-ReLU experts: C, D_row (M, N))
    if name == "dsrelu":
        counts = dgrad_counts(0, 8, 32768, None)
        return DgluSpec("dsrelu", L=8, K=4096, N=14336, counts=counts, b_std=0.02, act="dsrelu"), None
    # reduced copies of the layers above, sized for profiler captures (a few GB on the device)
    if name == "mixtral_s":
        counts = dgrad_counts(0, 2, 8192, None)
        return DgluSpec("mixtral_s", L=2, K=4096, N=14336, counts=counts, b_std=0.02), None
    if name == "geglu_s":
        counts = dgrad_counts(0, 16, 12288, 1.1, n_empty=2)
        return DgluSpec("geglu_s", L=16, K=2048, N=5632, counts=counts, act="dgeglu", b_mode="discrete",
                        b_major="n", c_std=4.0, d_dtype="fp32", dbias=True), None
    if name == "dsrelu_s":
        counts = dgrad_counts(0, 2, 8192, None)
        return DgluSpec("dsrelu_s", L=2, K=4096, N=14336, counts=counts, b_std=0.02, act="dsrelu"), None
    if name == "deepseek_s":
        counts = dgrad_counts(0, 32, 16384, 1.0)
        d = DgluSpec("deepseek_s", L=32, K=7168, N=2048, counts=counts)
        w = WgradSpec("deepseek_s", L=32, hidden=7168, inter=2048, counts=counts.copy(),
                      a_major="k", b_major="n", input_order="tensor_ragged", out_mode="discrete")
        return d, w
    raise KeyError(name)


WORKLOADS = ("tiny", "mixtral", "geglu", "wgrad64", "deepseek")
PROFILE_WORKLOADS = ("mixtral_s", "geglu_s", "deepseek_s", "dsrelu_s")


# --------------------------------------------------------------------------------------
# Tensor generation (torch)
# --------------------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def torch_dtype(name: str):
    torch = _torch()
    return {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[name]


def _normal(gen, shape, std, dtype, device):
    torch = _torch()
    t = torch.empty(shape, dtype=dtype, device=device)
    t.normal_(0.0, std, generator=gen)
    return t


def _uniform(gen, shape, lo, hi, device):
    torch = _torch()
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.uniform_(lo, hi, generator=gen)
    return t


def make_dglu_inputs(spec: DgluSpec, device="cpu"):
    """Tensors for one dgrad + dGLU call.

    Returns a dict: a (M,K) bf16; b (L,N,K) bf16 dense or list of L per-expert matrices
    (each (N,K) K-major, or an (K,N) row-major tensor whose transpose view is the
    n-major (N,K) matrix); c (M,2N), or (M,N) for "dsrelu"; alpha, beta (L,) fp32 ~U(0.5,1.5);
    prob (M,) fp32 ~U(0,1); padded_offsets (L,) int32.
    """
    torch = _torch()
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    M, K, N, L = spec.M, spec.K, spec.N, spec.L
    bf16 = torch.bfloat16
    a = _normal(gen, (M, K), spec.a_std, bf16, device)
    if spec.b_mode == "dense":
        b = _normal(gen, (L, N, K), spec.b_std, bf16, device)
    else:
        b = []
        for _ in range(L):
            if spec.b_major == "k":
                b.append(_normal(gen, (N, K), spec.b_std, bf16, device))
            else:
                # n-major (N,K): element (n,k) at k*N + n -> a row-major (K,N) buffer
                b.append(_normal(gen, (K, N), spec.b_std, bf16, device))
    c = _normal(gen, (M, N if spec.act == "dsrelu" else 2 * N), spec.c_std, torch_dtype(spec.c_dtype), device)
    alpha = _uniform(gen, (L,), 0.5, 1.5, device)
    beta = _uniform(gen, (L,), 0.5, 1.5, device)
    prob = _uniform(gen, (M,), 0.0, 1.0, device)
    offs = torch.from_numpy(offsets_from_counts(spec.counts)).to(device)
    return dict(a=a, b=b, c=c, alpha=alpha, beta=beta, prob=prob, padded_offsets=offs)


def make_wgrad_inputs(spec: WgradSpec, device="cpu", old_std: float = 1.0):
    """Tensors for one grouped wgrad call.

    a: flat bf16 storage of A (hidden, T); b: flat bf16 storage of B (T, inter). Their
    element placement follows (a_major, b_major, input_order); ``a_view``/``b_view``
    helpers in the binding interpret them.  out_old: (L, hidden, inter) initial output
    contents (~N(0, old_std)) in the output dtype, used by accumulate mode.
    """
    torch = _torch()
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed + 1)
    h, i, T, L = spec.hidden, spec.inter, spec.T, spec.L
    bf16 = torch.bfloat16
    a = _normal(gen, (h * T,), 1.0, bf16, device)
    b = _normal(gen, (T * i,), 1.0, bf16, device)
    offs = torch.from_numpy(offsets_from_counts(spec.counts)).to(device)
    out_old = None
    if spec.accumulate:
        out_old = _normal(gen, (L, h, i), old_std, torch_dtype(spec.out_dtype), device)
    return dict(a=a, b=b, offsets=offs, out_old=out_old)


def small_dglu_spec(name="small", L=3, counts=(256, 0, 512), K=320, N=160, **kw) -> DgluSpec:
    """A parity-size dgrad case: a few tiles, an empty expert, ragged N and K tails."""
    return DgluSpec(name, L=L, K=K, N=N, counts=np.asarray(counts, dtype=np.int64), **kw)


def small_wgrad_spec(name="small", L=4, counts=(512, 0, 256, 768), hidden=192, inter=160, **kw) -> WgradSpec:
    return WgradSpec(name, L=L, hidden=hidden, inter=inter, counts=np.asarray(counts, dtype=np.int64), **kw)
