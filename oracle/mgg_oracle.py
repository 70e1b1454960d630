"""Plain float64 CPU oracle for the grouped dGLU and dsReLU dgrad and the grouped wgrad.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): only tests, the smoke
check and the benchmark's CPU-baseline leg may call this module.

Conventions.  Inputs are numpy arrays holding the exact values of the stored
BF16/FP16/FP32 numbers (the caller decodes storage); results are float64 before
any output rounding.  Matrix products use numpy's float64 matmul as a library
step; nothing is blocked, fused or reordered beyond the definitions.

Readings of the pages that the oracle fixes, where they are silent or ambiguous:

* gate/input block order: gate first by default (dGLU page, BF16 contract:
  "alternating 32-wide gate/input blocks"); ``gate_first=False`` gives the
  input-first order printed for the block-scaled step 2.
* X_g = beta_g * C_g is formed as one float32 product, as the kernel does, so the
  dGeGLU filter decisions (comparisons with +-7) are taken in the same precision
  on both sides; everything after that is float64.
* dGeGLU filters are "value-bearing" as printed (filter = raw value inside the
  range, 0 outside); ``geglu_filter="indicator"`` gives 1 inside the range, which
  is the analytic derivative of the clamped GeGLU.
* dprob is the row sum of R times the unscaled activation (no prob factor),
  added to the caller's dprob; dbias is the per-expert column sum of the
  pre-rounding D_row values, added to the caller's dbias.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

# Grouped GEMM + dGLU (SM100), BF16 contract: source GeGLU constants and the
# default linear offset of the dGeGLU equation.
GEGLU_ALPHA = 1.702
GLU_CLAMP_MAX = 7.0
GLU_CLAMP_MIN = -7.0
LINEAR_OFFSET = 1.0
# Grouped GEMM + dGLU (SM100), "Common Parameters": situ_beta1 / situ_beta2 defaults of dSiTU-GLU.
SITU_BETA1 = 4.0
SITU_BETA2 = 25.0
# Grouped GEMM + dGLU: X splits into alternating 32-wide gate/input blocks.
GLU_BLOCK = 32
# Grouped GEMM + dGLU, "Shapes and Divisibility": m_aligned = 256, at most 1024 experts.
M_ALIGNED = 256
MAX_EXPERTS = 1024


# --------------------------------------------------------------------------------------
# Group ranges
# --------------------------------------------------------------------------------------

def expert_ranges(offsets: Sequence[int]) -> List[Tuple[int, int]]:
    """Row (dgrad) or token (wgrad) range of each expert.

    Grouped GEMM + WGrad, "Operation": begin = 0 for the first expert and
    offsets[e-1] otherwise, end = offsets[e].  The dGLU page uses the same
    cumulative-end convention for padded_offsets ("rows m in
    [padded_offsets[g-1], padded_offsets[g])").
    """
    out = []
    for e, end in enumerate(offsets):
        begin = 0 if e == 0 else int(offsets[e - 1])
        out.append((begin, int(end)))
    return out


# --------------------------------------------------------------------------------------
# dGLU epilogue math (elementwise)
# --------------------------------------------------------------------------------------

def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def glu_columns(n: int, gate_first: bool = True) -> Tuple[np.ndarray, np.ndarray]:
    """Columns of X (width 2N) holding the gate and the input of compact column j < N.

    Grouped GEMM + dGLU: X is split into alternating 32-wide blocks; compact block
    b = j // 32 owns X columns [64b, 64b + 64): the first 32 belong to the gate
    (gate first) and the next 32 to the input.
    """
    j = np.arange(n)
    blk = j // GLU_BLOCK
    w = j % GLU_BLOCK
    first = 2 * GLU_BLOCK * blk + w
    second = first + GLU_BLOCK
    return (first, second) if gate_first else (second, first)


def dswiglu(R, prob, gate, inp):
    """dSwiGLU backward (dGLU page, BF16 contract; block-scaled step 2 for dprob).

    s = sigmoid(gate); dinput = R prob gate s; dgate = R prob input s (1 + gate (1 - s));
    the unscaled activation used by dprob is swish(gate) * input = gate s input.
    Returns (dgate, dinput, act).
    """
    R = np.asarray(R, np.float64)
    prob = np.asarray(prob, np.float64)
    gate = np.asarray(gate, np.float64)
    inp = np.asarray(inp, np.float64)
    s = sigmoid(gate)
    dinput = R * prob * (gate * s)
    dgate = R * prob * inp * s * (1.0 + gate * (1.0 - s))
    act = gate * s * inp
    return dgate, dinput, act


def dgeglu(R, prob, gate, inp, geglu_filter: str = "value"):
    """dGeGLU backward with clamp and filters (dGLU page, BF16 contract).

    clamped_gate = min(raw_gate, 7); clamped_input = clamp(raw_input, -7, 7);
    gate_filter = raw_gate if raw_gate <= 7 else 0;
    input_filter = raw_input if -7 <= raw_input <= 7 else 0;
    s = sigmoid(1.702 clamped_gate);
    dgate = R prob (clamped_input + 1) s (1 + 1.702 clamped_gate (1 - s)) gate_filter;
    dinput = R prob clamped_gate s input_filter.
    ``geglu_filter="indicator"`` replaces the raw value inside the range by 1.
    The unscaled activation for dprob is (clamped_input + 1) clamped_gate s.
    Returns (dgate, dinput, act).
    """
    R = np.asarray(R, np.float64)
    prob = np.asarray(prob, np.float64)
    raw_gate = np.asarray(gate, np.float64)
    raw_input = np.asarray(inp, np.float64)
    clamped_gate = np.minimum(raw_gate, GLU_CLAMP_MAX)
    clamped_input = np.clip(raw_input, GLU_CLAMP_MIN, GLU_CLAMP_MAX)
    gate_in = raw_gate <= GLU_CLAMP_MAX
    input_in = (raw_input >= GLU_CLAMP_MIN) & (raw_input <= GLU_CLAMP_MAX)
    if geglu_filter == "value":
        gate_filter = np.where(gate_in, raw_gate, 0.0)
        input_filter = np.where(input_in, raw_input, 0.0)
    elif geglu_filter == "indicator":
        gate_filter = np.where(gate_in, 1.0, 0.0)
        input_filter = np.where(input_in, 1.0, 0.0)
    else:
        raise ValueError(geglu_filter)
    s = sigmoid(GEGLU_ALPHA * clamped_gate)
    dgate = (R * prob * (clamped_input + LINEAR_OFFSET) * s
             * (1.0 + GEGLU_ALPHA * clamped_gate * (1.0 - s)) * gate_filter)
    dinput = R * prob * clamped_gate * s * input_filter
    act = (clamped_input + LINEAR_OFFSET) * clamped_gate * s
    return dgate, dinput, act


def dsituglu(R, prob, gate, inp, beta1: float = SITU_BETA1, beta2: float = SITU_BETA2):
    """dSiTU-GLU backward (dGLU page, block-scaled contract, "Equations").

    T_g = beta1 tanh(G / beta1) sigmoid(G);  T_u = beta2 tanh(U / beta2);
    dT_g/dG = (1 - tanh^2(G / beta1)) sigmoid(G) + beta1 tanh(G / beta1) sigmoid(G) (1 - sigmoid(G));
    dT_u/dU = 1 - tanh^2(U / beta2);
    dgate = R prob T_u dT_g/dG, dinput = R prob T_g dT_u/dU; the dprob activation is T_g T_u.
    G is the gate and U the input block of X.  Returns (dgate, dinput, act).
    """
    R = np.asarray(R, np.float64)
    prob = np.asarray(prob, np.float64)
    G = np.asarray(gate, np.float64)
    U = np.asarray(inp, np.float64)
    tg = np.tanh(G / beta1)
    sg = sigmoid(G)
    tu = np.tanh(U / beta2)
    T_g = beta1 * tg * sg
    T_u = beta2 * tu
    dT_g = (1.0 - tg * tg) * sg + beta1 * tg * sg * (1.0 - sg)
    dT_u = 1.0 - tu * tu
    return R * prob * T_u * dT_g, R * prob * T_g * dT_u, T_g * T_u


def scale_x(beta_g, c_values) -> np.ndarray:
    """X = beta_g * C as one float32 product per element (then widened to float64)."""
    x32 = np.float32(beta_g) * np.asarray(c_values, dtype=np.float32)
    return x32.astype(np.float64)


# --------------------------------------------------------------------------------------
# Grouped GEMM + dGLU
# --------------------------------------------------------------------------------------

def dglu_bwd(a: np.ndarray,
             get_b: Callable[[int], np.ndarray],
             c: np.ndarray,
             offsets: Sequence[int],
             alpha: Sequence[float],
             beta: Sequence[float],
             prob: Sequence[float],
             act: str = "dswiglu",
             gate_first: bool = True,
             geglu_filter: str = "value",
             rows: Optional[np.ndarray] = None,
             dprob_in: Optional[np.ndarray] = None,
             dbias_in: Optional[np.ndarray] = None,
             situ_beta1: float = SITU_BETA1,
             situ_beta2: float = SITU_BETA2) -> Dict[str, np.ndarray]:
    """Grouped GEMM + dGLU backward (dGLU page, BF16 contract).

    a: (M, K) values of A; get_b(g) -> (N, K) values of B_g (dense (N,K,L) slice or
    the discrete matrix, whatever its storage major); c: (M, 2N) values of C, or,
    when ``rows`` is given, the rows ``rows`` of C in that order (shape (len(rows), 2N));
    offsets: padded_offsets (cumulative ends); alpha, beta: (L,); prob: (M,).

    For each expert g and row m in its range:
      R[m, :] = alpha_g^2 * (A[m, :] @ B_g^T)
      X[m, :] = beta_g * C[m, :]
      (dgate, dinput) from the activation on the gate/input blocks, written back
      into the interleaved positions of D_row;
      dprob[m] = dprob_in[m] + sum_j R[m, j] * act[m, j];
      dbias[g, col] = dbias_in[g, col] + sum over the expert's rows of D_row[m, col].

    amax[g, 0] / amax[g, 1] = the largest |dgate| / |dinput| over the expert's rows (the
    per-group amax of shape (L, 2, 1) that the dGLU page lists among the outputs for 16-bit
    D_row; its two entries read as the gate and the input block), 0 for an empty expert.

    ``rows`` restricts the evaluation to those rows (dbias and amax are then not returned).
    Returns dict(d_row (R, 2N), dprob (R,), rows, [dbias (L, 2N), amax (L, 2)]), float64.
    """
    a = np.asarray(a)
    M = a.shape[0]
    L = len(offsets)
    ranges = expert_ranges(offsets)
    all_rows = rows is None
    if all_rows:
        rows = np.arange(M)
    rows = np.asarray(rows, dtype=np.int64)
    c = np.asarray(c)
    two_n = c.shape[1]
    n = two_n // 2
    gcol, icol = glu_columns(n, gate_first)
    d_row = np.zeros((len(rows), two_n), dtype=np.float64)
    dprob = np.zeros(len(rows), dtype=np.float64)
    if dprob_in is not None:
        dprob += np.asarray(dprob_in, np.float64)[rows]
    dbias = np.zeros((L, two_n), dtype=np.float64) if all_rows else None
    if all_rows and dbias_in is not None:
        dbias += np.asarray(dbias_in, np.float64)
    amax = np.zeros((L, 2), dtype=np.float64) if all_rows else None
    prob = np.asarray(prob, np.float64)
    for g, (lo, hi) in enumerate(ranges):
        sel = np.nonzero((rows >= lo) & (rows < hi))[0]
        if sel.size == 0:
            continue
        b_g = np.asarray(get_b(g), dtype=np.float64)
        a_rows = np.asarray(a[rows[sel]], dtype=np.float64)
        alpha_g = float(alpha[g])
        R = (alpha_g * alpha_g) * (a_rows @ b_g.T)
        c_rows = c[sel] if not all_rows else c[rows[sel]]
        X = scale_x(beta[g], c_rows)
        gate = X[:, gcol]
        inp = X[:, icol]
        p = prob[rows[sel]][:, None]
        if act == "dswiglu":
            dgate, dinput, a_unscaled = dswiglu(R, p, gate, inp)
        elif act == "dgeglu":
            dgate, dinput, a_unscaled = dgeglu(R, p, gate, inp, geglu_filter)
        elif act == "dsituglu":
            dgate, dinput, a_unscaled = dsituglu(R, p, gate, inp, situ_beta1, situ_beta2)
        else:
            raise ValueError(act)
        out = np.zeros((sel.size, two_n), dtype=np.float64)
        out[:, gcol] = dgate
        out[:, icol] = dinput
        d_row[sel] = out
        dprob[sel] += np.sum(R * a_unscaled, axis=1)
        if dbias is not None:
            dbias[g] += out.sum(axis=0)
        if amax is not None:
            amax[g, 0] = np.max(np.abs(dgate))
            amax[g, 1] = np.max(np.abs(dinput))
    res = dict(d_row=d_row, dprob=dprob, rows=rows)
    if dbias is not None:
        res["dbias"] = dbias
    if amax is not None:
        res["amax"] = amax
    return res


# --------------------------------------------------------------------------------------
# Grouped dgrad + dsReLU
# --------------------------------------------------------------------------------------

def dsrelu(G, prob, c):
    """dsReLU backward on one block (dsReLU page, "Equations").

    With relu(G) = max(G, 0): D_row = prob * 2 * C * relu(G) and the row terms of dprob are
    C * relu(G)^2.  G is the alpha-scaled GEMM result, C the forward tensor, prob the row's
    gating probability.  Returns (d_row, dprob_terms).
    """
    G = np.asarray(G, np.float64)
    c = np.asarray(c, np.float64)
    r = np.maximum(G, 0.0)
    return np.asarray(prob, np.float64) * 2.0 * c * r, c * r * r


def dsrelu_bwd(a: np.ndarray,
               get_b: Callable[[int], np.ndarray],
               c: np.ndarray,
               offsets: Sequence[int],
               alpha: Sequence[float],
               prob: Sequence[float],
               rows: Optional[np.ndarray] = None,
               dprob_in: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Grouped GEMM + dsReLU backward (dsReLU page, "Equations"), on BF16 operands.

    a: (M, K) values of A; get_b(g) -> (N, K) values of B_g; c: (M, N) values of C (rows
    ``rows`` of C when given); offsets: padded_offsets; alpha: (L,); prob: (M,).

    For each expert g and row m in its range:
      G[m, :] = alpha_g * (A[m, :] @ B_g^T)          (alpha, not alpha^2, as printed)
      D_row[m, n] = prob[m] * 2 * C[m, n] * relu(G[m, n])
      dprob[m] = dprob_in[m] + sum_n C[m, n] * relu(G[m, n])^2
      amax[g] = the largest |D_row| over the expert's rows (the (L, 1) Amax of 16-bit D_row).
    C and D_row are plain (M, N): no gate/input blocks, no beta.
    Returns dict(d_row (R, N), dprob (R,), rows, [amax (L,)]), float64.
    """
    a = np.asarray(a)
    M = a.shape[0]
    L = len(offsets)
    all_rows = rows is None
    if all_rows:
        rows = np.arange(M)
    rows = np.asarray(rows, dtype=np.int64)
    c = np.asarray(c)
    n = c.shape[1]
    d_row = np.zeros((len(rows), n), dtype=np.float64)
    dprob = np.zeros(len(rows), dtype=np.float64)
    if dprob_in is not None:
        dprob += np.asarray(dprob_in, np.float64)[rows]
    amax = np.zeros(L, dtype=np.float64) if all_rows else None
    prob = np.asarray(prob, np.float64)
    for g, (lo, hi) in enumerate(expert_ranges(offsets)):
        sel = np.nonzero((rows >= lo) & (rows < hi))[0]
        if sel.size == 0:
            continue
        b_g = np.asarray(get_b(g), dtype=np.float64)
        G = float(alpha[g]) * (np.asarray(a[rows[sel]], dtype=np.float64) @ b_g.T)
        c_rows = c[sel] if not all_rows else c[rows[sel]]
        d, terms = dsrelu(G, prob[rows[sel]][:, None], c_rows)
        d_row[sel] = d
        dprob[sel] += terms.sum(axis=1)
        if amax is not None:
            amax[g] = np.max(np.abs(d))
    res = dict(d_row=d_row, dprob=dprob, rows=rows)
    if amax is not None:
        res["amax"] = amax
    return res


# --------------------------------------------------------------------------------------
# Grouped wgrad
# --------------------------------------------------------------------------------------

def wgrad_a_block(a_flat: np.ndarray, hidden: int, T: int, begin: int, end: int,
                  a_major: str = "k", input_order: str = "tensor2d") -> np.ndarray:
    """A[:, begin:end] (hidden x K_e) from the flat storage of A (hidden, T).

    Grouped GEMM + WGrad, "BF16 contract": A is K-major (strides (T, 1)) or M-major
    (strides (1, hidden)).  With input_order "tensor_ragged" the token axis is stored as
    per-expert K-contiguous blocks concatenated in memory; only the unit-stride axis
    counts.  For K-major A the expert block is (hidden, K_e) with row length K_e,
    starting at element begin * hidden.  For M-major A the unit stride is along hidden,
    so the expert's rows are already one contiguous (K_e, hidden) block.
    """
    ke = end - begin
    if a_major == "k":
        if input_order == "tensor_ragged":
            return a_flat[begin * hidden:end * hidden].reshape(hidden, ke)
        return a_flat.reshape(hidden, T)[:, begin:end]
    if a_major == "m":
        return a_flat.reshape(T, hidden)[begin:end, :].T
    raise ValueError(a_major)


def wgrad_b_block(b_flat: np.ndarray, T: int, inter: int, begin: int, end: int,
                  b_major: str = "n", input_order: str = "tensor2d") -> np.ndarray:
    """B[begin:end, :] (K_e x inter) from the flat storage of B (T, inter).

    B is N-major (strides (inter, 1)) or K-major (strides (1, T)).  tensor_ragged: a
    K-major B stores each expert as an (inter, K_e) K-contiguous block at element
    begin * inter; an N-major B is already one contiguous (K_e, inter) block per expert.
    """
    ke = end - begin
    if b_major == "n":
        return b_flat.reshape(T, inter)[begin:end, :]
    if b_major == "k":
        if input_order == "tensor_ragged":
            return b_flat[begin * inter:end * inter].reshape(inter, ke).T
        return b_flat.reshape(inter, T)[:, begin:end].T
    raise ValueError(b_major)


def wgrad(a_flat: np.ndarray, b_flat: np.ndarray, offsets: Sequence[int], hidden: int, inter: int,
          a_major: str = "k", b_major: str = "n", input_order: str = "tensor2d",
          accumulate: bool = False, out_old: Optional[np.ndarray] = None,
          experts: Optional[Sequence[int]] = None) -> Dict[int, np.ndarray]:
    """Grouped wgrad (Grouped GEMM + WGrad, "Operation").

    Wgrad[e] = A[:, begin:end] @ B[begin:end, :]; with accumulate_on_output the result is
    added to the existing output (out_old[e]), otherwise it overwrites it and an empty
    expert produces zero.  Returns {e: (hidden, inter) float64} for ``experts`` (all by
    default).
    """
    T = int(offsets[-1]) if len(offsets) else 0
    ranges = expert_ranges(offsets)
    if experts is None:
        experts = range(len(offsets))
    out = {}
    for e in experts:
        begin, end = ranges[e]
        if end > begin:
            A_e = np.asarray(wgrad_a_block(a_flat, hidden, T, begin, end, a_major, input_order), np.float64)
            B_e = np.asarray(wgrad_b_block(b_flat, T, inter, begin, end, b_major, input_order), np.float64)
            w = A_e @ B_e
        else:
            w = np.zeros((hidden, inter), dtype=np.float64)
        if accumulate:
            w = np.asarray(out_old[e], np.float64) + w
        out[e] = w
    return out


def wgrad_elements(a_flat, b_flat, offsets, hidden, inter, e, hh, ii,
                   a_major="k", b_major="n", input_order="tensor2d",
                   accumulate=False, old_values=None) -> np.ndarray:
    """Selected elements Wgrad[e][hh[t], ii[t]] (same definition as ``wgrad``)."""
    T = int(offsets[-1])
    begin, end = expert_ranges(offsets)[e]
    hh = np.asarray(hh)
    ii = np.asarray(ii)
    if end > begin:
        A_e = np.asarray(wgrad_a_block(a_flat, hidden, T, begin, end, a_major, input_order), np.float64)
        B_e = np.asarray(wgrad_b_block(b_flat, T, inter, begin, end, b_major, input_order), np.float64)
        vals = np.einsum("tk,kt->t", A_e[hh, :], B_e[:, ii])
    else:
        vals = np.zeros(hh.shape, dtype=np.float64)
    if accumulate:
        vals = vals + np.asarray(old_values, np.float64)
    return vals


# --------------------------------------------------------------------------------------
# Tile schedules
# --------------------------------------------------------------------------------------

def dgrad_tiles(offsets: Sequence[int], N: int, tile_m: int, tile_n: int) -> np.ndarray:
    """Canonical output tiles (expert, m0, n0) of the grouped dgrad.

    Groups are contiguous row ranges (dGLU page, Overview); each expert owns the
    tile_m-row blocks inside its range (tile_m divides the 256-row alignment), empty
    experts own none; every block is split into ceil(N / tile_n) column tiles.
    Sorted by (expert, m0, n0).
    """
    tiles = []
    for g, (lo, hi) in enumerate(expert_ranges(offsets)):
        for m0 in range(lo, hi, tile_m):
            for n0 in range(0, N, tile_n):
                tiles.append((g, m0, n0))
    return np.asarray(tiles, dtype=np.int64).reshape(-1, 3)


def wgrad_tiles(offsets: Sequence[int], hidden: int, inter: int, tile_m: int, tile_n: int,
                accumulate: bool) -> np.ndarray:
    """Canonical output tiles (expert, h0, i0) of the grouped wgrad.

    Every non-empty expert contributes all tiles of its (hidden, inter) output.  An
    empty expert contributes its tiles only in overwrite mode (it must be written as
    zeros); under accumulate_on_output it is left untouched.  Sorted by (e, h0, i0).
    """
    tiles = []
    for e, (begin, end) in enumerate(expert_ranges(offsets)):
        if end == begin and accumulate:
            continue
        for h0 in range(0, hidden, tile_m):
            for i0 in range(0, inter, tile_n):
                tiles.append((e, h0, i0))
    return np.asarray(tiles, dtype=np.int64).reshape(-1, 3)


# --------------------------------------------------------------------------------------
# Validation rules the boundary enforces (pages' constraints), as plain predicates
# --------------------------------------------------------------------------------------

def offsets_valid(offsets: Sequence[int], total: int, align: int = M_ALIGNED) -> bool:
    """Non-decreasing cumulative ends, each count a multiple of ``align``, last == total.

    Grouped GEMM + WGrad, "BF16 contract"; grouped dGLU, "Shapes and Divisibility".
    """
    prev = 0
    for v in offsets:
        v = int(v)
        if v < prev or (v - prev) % align != 0:
            return False
        prev = v
    return prev == total


__all__ = [
    "GEGLU_ALPHA", "GLU_CLAMP_MAX", "GLU_CLAMP_MIN", "LINEAR_OFFSET", "GLU_BLOCK", "M_ALIGNED", "MAX_EXPERTS",
    "SITU_BETA1", "SITU_BETA2",
    "expert_ranges", "sigmoid", "glu_columns", "dswiglu", "dgeglu", "dsituglu", "scale_x", "dglu_bwd",
    "dsrelu", "dsrelu_bwd",
    "wgrad_a_block", "wgrad_b_block", "wgrad", "wgrad_elements", "dgrad_tiles", "wgrad_tiles",
    "offsets_valid",
]
