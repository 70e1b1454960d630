"""Pins of the CPU oracle against things other than itself.

Each test ties one oracle function to what the pages and the mathematics fix:
brute-force loops on tiny inputs, central finite differences of the forward
activations, closed forms, invariants and special cases.  A plausible mistake
(a dropped alpha square, swapped gate/input blocks, a wrong filter, a shifted
expert range, a transposed operand) fails at least one of them; the last tests
plant such mistakes in the oracle and check that they are caught.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import mgg_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------------------
# helpers (independent re-statements used only by the pins)
# --------------------------------------------------------------------------------------

def _sig(x):
    return 1.0 / (1.0 + math.exp(-x))


def fwd_swiglu(gate, inp):
    """Forward SwiGLU unit: input * gate * sigmoid(gate)."""
    return inp * gate * _sig(gate)


def fwd_geglu_clamped(gate, inp):
    """Forward clamped GeGLU unit with linear offset 1: (clip(in)+1) * g * sigmoid(1.702 g), g = min(gate, 7)."""
    g = min(gate, 7.0)
    x = min(max(inp, -7.0), 7.0)
    return (x + 1.0) * g * _sig(1.702 * g)


def fwd_situglu(gate, inp, b1=4.0, b2=25.0):
    """Forward SiTU-GLU unit: (b1 tanh(g/b1) sigmoid(g)) * (b2 tanh(u/b2))."""
    return (b1 * math.tanh(gate / b1) * _sig(gate)) * (b2 * math.tanh(inp / b2))


def fd(f, x, h=1e-6):
    return (f(x + h) - f(x - h)) / (2.0 * h)


def brute_dglu(a, bs, c, offsets, alpha, beta, prob, act, gate_first, filt):
    """Pure-python reference: explicit loops, expert found by scanning the ends, D by FD."""
    M, K = a.shape
    two_n = c.shape[1]
    N = two_n // 2
    L = len(offsets)
    D = np.zeros((M, two_n))
    dprob = np.zeros(M)
    dbias = np.zeros((L, two_n))
    fwd = {"dswiglu": fwd_swiglu, "dgeglu": fwd_geglu_clamped, "dsituglu": fwd_situglu}[act]
    for m in range(M):
        g = next(e for e in range(L) if m < offsets[e])
        for j in range(N):
            acc = 0.0
            for k in range(K):
                acc += float(a[m, k]) * float(bs[g][j, k])
            R = alpha[g] ** 2 * acc
            blk, w = divmod(j, 32)
            col_first, col_second = 64 * blk + w, 64 * blk + 32 + w
            cg, ci = (col_first, col_second) if gate_first else (col_second, col_first)
            gate = float(np.float32(beta[g]) * np.float32(c[m, cg]))
            inp = float(np.float32(beta[g]) * np.float32(c[m, ci]))
            dg = fd(lambda x: fwd(x, inp), gate)
            di = fd(lambda x: fwd(gate, x), inp)
            if act == "dgeglu" and filt == "value":
                dg *= gate   # value-bearing filters: the raw value replaces the 0/1 indicator
                di *= inp
            D[m, cg] = R * prob[m] * dg
            D[m, ci] = R * prob[m] * di
            dprob[m] += R * fwd(gate, inp)
        dbias[g] += D[m]
    return D, dprob, dbias


def tiny_case(seed, M_counts, K, N, c_std=1.0, avoid_kinks=False):
    rng = np.random.default_rng(seed)
    offsets = np.cumsum(M_counts).astype(np.int64)
    M = int(offsets[-1])
    L = len(M_counts)
    # bf16-representable values (8 significant bits) keep the float32 X products exact-ish
    q = lambda x: np.round(x * 64) / 64
    a = q(rng.normal(size=(M, K)))
    bs = [q(rng.normal(size=(N, K))) for _ in range(L)]
    c = q(rng.normal(scale=c_std, size=(M, 2 * N)))
    if avoid_kinks:  # keep FD away from the +-7 corners of the clamp
        bad = np.abs(np.abs(c) - 7.0 / 1.0) < 0.05
        c[bad] += 0.25
    alpha = rng.uniform(0.5, 1.5, L)
    beta = np.ones(L) if avoid_kinks else rng.uniform(0.5, 1.5, L)
    prob = rng.uniform(0, 1, M)
    return a, bs, c, offsets, alpha, beta, prob


# --------------------------------------------------------------------------------------
# constants and ranges
# --------------------------------------------------------------------------------------

def test_constants_match_pages_fixture():
    vals = {}
    with open(os.path.join(GOLDEN, "dglu_contract_constants.txt")) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            name, v = line.split()
            vals[name] = float(v)
    assert O.GEGLU_ALPHA == vals["geglu_alpha"]
    assert O.GLU_CLAMP_MAX == vals["glu_clamp_max"]
    assert O.GLU_CLAMP_MIN == vals["glu_clamp_min"]
    assert O.LINEAR_OFFSET == vals["linear_offset"]
    assert O.GLU_BLOCK == vals["glu_block"]
    assert O.M_ALIGNED == vals["m_aligned"] == vals["token_multiple"]
    assert O.MAX_EXPERTS == vals["max_experts"]
    assert O.SITU_BETA1 == vals["situ_beta1"] and O.SITU_BETA2 == vals["situ_beta2"]


def test_expert_ranges_cumulative_ends():
    # begin = 0 for the first expert, offsets[e-1] otherwise; end = offsets[e]
    assert O.expert_ranges([256, 256, 768, 1024]) == [(0, 256), (256, 256), (256, 768), (768, 1024)]
    assert O.expert_ranges([0, 0, 512]) == [(0, 0), (0, 0), (0, 512)]
    # ranges tile [0, last) without overlap
    offs = [256, 512, 512, 2048]
    covered = np.zeros(2048, int)
    for lo, hi in O.expert_ranges(offs):
        covered[lo:hi] += 1
    assert (covered == 1).all()


def test_offsets_valid_rules():
    assert O.offsets_valid([256, 256, 768, 1024], 1024)
    assert not O.offsets_valid([256, 128, 768, 1024], 1024)       # decreasing
    assert not O.offsets_valid([256, 300, 768, 1024], 1024)       # count not a multiple of 256
    assert not O.offsets_valid([256, 512], 1024)                  # last != total
    assert O.offsets_valid([0, 0, 0], 0)


def test_glu_columns_hand_values():
    g, i = O.glu_columns(96, gate_first=True)
    assert (g[0], i[0]) == (0, 32)
    assert (g[31], i[31]) == (31, 63)
    assert (g[32], i[32]) == (64, 96)
    assert (g[95], i[95]) == (159, 191)
    g2, i2 = O.glu_columns(96, gate_first=False)
    assert (g2 == i).all() and (i2 == g).all()
    # every X column is used exactly once
    assert sorted(np.concatenate([g, i]).tolist()) == list(range(192))


# --------------------------------------------------------------------------------------
# activation derivatives: finite differences and closed forms
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("gate,inp", [(0.3, -1.2), (-2.5, 0.7), (4.0, 3.0), (-9.0, 2.0), (1e-3, 5.0)])
def test_dswiglu_matches_fd(gate, inp):
    R, p = 1.7, 0.35
    dg, di, act = O.dswiglu(R, p, gate, inp)
    assert dg == pytest.approx(R * p * fd(lambda x: fwd_swiglu(x, inp), gate), rel=1e-7, abs=1e-12)
    assert di == pytest.approx(R * p * fd(lambda x: fwd_swiglu(gate, x), inp), rel=1e-7, abs=1e-12)
    assert act == pytest.approx(fwd_swiglu(gate, inp), rel=1e-12)


@pytest.mark.parametrize("gate,inp", [(0.3, -1.2), (-2.5, 0.7), (6.5, 6.9), (8.0, 2.0), (3.0, -8.5),
                                      (9.0, 9.0), (-12.0, -3.0), (2.0, 7.5)])
def test_dgeglu_indicator_matches_fd(gate, inp):
    R, p = -0.8, 0.6
    dg, di, act = O.dgeglu(R, p, gate, inp, "indicator")
    assert dg == pytest.approx(R * p * fd(lambda x: fwd_geglu_clamped(x, inp), gate), rel=1e-7, abs=1e-12)
    assert di == pytest.approx(R * p * fd(lambda x: fwd_geglu_clamped(gate, x), inp), rel=1e-7, abs=1e-12)
    assert act == pytest.approx(fwd_geglu_clamped(gate, inp), rel=1e-12)


@pytest.mark.parametrize("gate,inp", [(0.3, -1.2), (-2.5, 0.7), (6.0, 30.0), (-15.0, -40.0), (12.0, 3.0)])
@pytest.mark.parametrize("b1,b2", [(4.0, 25.0), (2.0, 5.0)])
def test_dsituglu_matches_fd(gate, inp, b1, b2):
    R, p = 1.1, 0.45
    dg, di, act = O.dsituglu(R, p, gate, inp, b1, b2)
    # central differences of an O(10) forward carry ~1e-9 absolute rounding noise
    assert dg == pytest.approx(R * p * fd(lambda x: fwd_situglu(x, inp, b1, b2), gate), rel=1e-7, abs=1e-8)
    assert di == pytest.approx(R * p * fd(lambda x: fwd_situglu(gate, x, b1, b2), inp), rel=1e-7, abs=1e-8)
    assert act == pytest.approx(fwd_situglu(gate, inp, b1, b2), rel=1e-12)


def test_dsituglu_closed_forms():
    # G = 0: tanh(0) = 0 and sigmoid(0) = 1/2, so T_g = 0 and dT_g/dG = 1/2
    dg, di, act = O.dsituglu(2.0, 0.5, 0.0, 10.0)
    assert di == 0.0 and act == 0.0
    assert dg == pytest.approx(2.0 * 0.5 * 25.0 * math.tanh(10.0 / 25.0) * 0.5)
    # U = 0: T_u = 0 and dT_u/dU = 1
    dg, di, act = O.dsituglu(2.0, 0.5, 1.5, 0.0)
    assert dg == 0.0 and act == 0.0
    assert di == pytest.approx(2.0 * 0.5 * 4.0 * math.tanh(1.5 / 4.0) / (1 + math.exp(-1.5)))
    # saturation: |U| >> beta2 gives dT_u/dU -> 0, T_u -> +-beta2
    dg, di, act = O.dsituglu(1.0, 1.0, 1.0, 1e4)
    assert abs(di) < 1e-12 and dg == pytest.approx(25.0 * ((1 - math.tanh(0.25) ** 2) / (1 + math.exp(-1.0))
                                                           + 4 * math.tanh(0.25) * _sig(1.0) * (1 - _sig(1.0))))


@pytest.mark.parametrize("gate,inp", [(0.3, -1.2), (6.5, 6.9), (8.0, 2.0), (3.0, -8.5), (7.0, -7.0)])
def test_dgeglu_value_filter_is_indicator_times_raw(gate, inp):
    R, p = 1.3, 0.9
    dgv, div, actv = O.dgeglu(R, p, gate, inp, "value")
    dgi, dii, acti = O.dgeglu(R, p, gate, inp, "indicator")
    assert dgv == pytest.approx(dgi * gate, rel=1e-14, abs=0)
    assert div == pytest.approx(dii * inp, rel=1e-14, abs=0)
    assert actv == acti


def test_closed_forms():
    R, p, x = 2.0, 0.5, 3.0
    # SwiGLU at gate = 0: s = 1/2 -> dinput = 0, dgate = R p x / 2, act = 0
    dg, di, act = O.dswiglu(R, p, 0.0, x)
    assert di == 0.0 and act == 0.0 and dg == pytest.approx(R * p * x / 2)
    # SwiGLU at gate = ln 3: s = 3/4
    g = math.log(3.0)
    dg, di, act = O.dswiglu(R, p, g, x)
    assert di == pytest.approx(R * p * g * 0.75)
    assert dg == pytest.approx(R * p * x * 0.75 * (1 + g / 4))
    # GeGLU at 1.702 g = ln 3 (s = 3/4), input inside the range
    g = math.log(3.0) / 1.702
    dg, di, act = O.dgeglu(R, p, g, x, "indicator")
    assert dg == pytest.approx(R * p * (x + 1) * 0.75 * (1 + math.log(3.0) / 4))
    assert di == pytest.approx(R * p * g * 0.75)
    assert act == pytest.approx((x + 1) * g * 0.75)
    # GeGLU: gate above the clamp -> dgate = 0; input below -7 -> dinput = 0, act uses -7 + 1
    dg, di, act = O.dgeglu(R, p, 8.0, -9.0, "value")
    assert dg == 0.0 and di == 0.0
    assert act == pytest.approx(-6.0 * 7.0 / (1 + math.exp(-1.702 * 7.0)))
    # Value filter at gate = 0 makes dgate vanish although the indicator form does not
    assert O.dgeglu(R, p, 0.0, x, "value")[0] == 0.0
    assert O.dgeglu(R, p, 0.0, x, "indicator")[0] == pytest.approx(R * p * (x + 1) * 0.5)
    # boundary ties: gate == 7 and input == +-7 pass the filters
    assert O.dgeglu(1.0, 1.0, 7.0, 1.0, "indicator")[0] != 0.0
    assert O.dgeglu(1.0, 1.0, 1.0, 7.0, "indicator")[1] != 0.0
    assert O.dgeglu(1.0, 1.0, 1.0, -7.0, "indicator")[1] != 0.0


def test_scale_x_is_single_float32_product():
    beta = 1.1
    c = np.array([3.3, -7.0, 6.37], dtype=np.float32)
    x = O.scale_x(beta, c)
    assert x.dtype == np.float64
    expect = [float(np.float32(np.float32(beta) * ci)) for ci in c]
    assert x.tolist() == expect


# --------------------------------------------------------------------------------------
# the full dgrad + dGLU against brute force
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("act,filt,gate_first", [
    ("dswiglu", "value", True), ("dswiglu", "value", False), ("dsituglu", "value", True), ("dsituglu", "value", False),
    ("dgeglu", "indicator", True), ("dgeglu", "value", True), ("dgeglu", "value", False)])
def test_dglu_bwd_bruteforce(act, filt, gate_first):
    a, bs, c, offsets, alpha, beta, prob = tiny_case(
        1, [3, 0, 2, 3], K=5, N=64, c_std=(4.0 if act == "dgeglu" else 1.0), avoid_kinks=(act == "dgeglu"))
    res = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, prob, act=act,
                     gate_first=gate_first, geglu_filter=filt)
    D, dprob, dbias = brute_dglu(a, bs, c, offsets, alpha, beta, prob, act, gate_first, filt)
    np.testing.assert_allclose(res["d_row"], D, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(res["dprob"], dprob, rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(res["dbias"], dbias, rtol=1e-6, atol=1e-7)
    if act == "dgeglu":  # the case must actually exercise both sides of the clamp
        X = c * 1.0
        assert (X > 7).any() and (X < -7).any() and (np.abs(X) <= 7).any()


def test_dglu_bwd_row_subset_equals_full():
    a, bs, c, offsets, alpha, beta, prob = tiny_case(2, [4, 4, 0, 4], K=7, N=32)
    full = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, prob)
    rows = np.array([11, 0, 5, 7])
    part = O.dglu_bwd(a, lambda g: bs[g], c[rows], offsets, alpha, beta, prob, rows=rows)
    np.testing.assert_array_equal(part["d_row"], full["d_row"][rows])
    np.testing.assert_array_equal(part["dprob"], full["dprob"][rows])


def test_dglu_single_expert_is_plain_matmul_times_alpha_squared():
    a, bs, c, offsets, alpha, beta, prob = tiny_case(3, [6], K=9, N=32)
    # with prob = 1, beta chosen so gate = 0: dgate = R * input / 2 exactly gives R back
    beta = np.ones(1)
    c = c.copy()
    gcol, icol = O.glu_columns(32)
    c[:, gcol] = 0.0
    c[:, icol] = 2.0
    res = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, np.ones(6))
    R_ref = alpha[0] ** 2 * np.einsum("mk,nk->mn", a, bs[0])
    np.testing.assert_allclose(res["d_row"][:, gcol], R_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(res["d_row"][:, icol], 0.0)


def test_dglu_special_cases_prob_zero_and_alpha_zero():
    a, bs, c, offsets, alpha, beta, prob = tiny_case(4, [2, 3], K=4, N=32)
    dprob_in = np.arange(5, dtype=np.float64)
    res = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, np.zeros(5), dprob_in=dprob_in)
    assert (res["d_row"] == 0).all()
    assert not np.allclose(res["dprob"], dprob_in)  # dprob has no prob factor
    res = O.dglu_bwd(a, lambda g: bs[g], c, offsets, np.zeros(2), beta, prob, dprob_in=dprob_in)
    assert (res["d_row"] == 0).all()
    np.testing.assert_array_equal(res["dprob"], dprob_in)


def test_dglu_linear_in_R_and_accumulates_inputs():
    a, bs, c, offsets, alpha, beta, prob = tiny_case(5, [3, 2], K=6, N=32)
    r1 = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, prob, act="dgeglu")
    r2 = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha * math.sqrt(2.0), beta, prob, act="dgeglu")
    np.testing.assert_allclose(r2["d_row"], 2 * r1["d_row"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r2["dprob"], 2 * r1["dprob"], rtol=1e-12, atol=1e-14)
    dprob_in = np.linspace(-1, 1, 5)
    dbias_in = np.linspace(0, 3, 2 * 64).reshape(2, 64)
    r3 = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, prob, act="dgeglu",
                    dprob_in=dprob_in, dbias_in=dbias_in)
    np.testing.assert_allclose(r3["dprob"], r1["dprob"] + dprob_in, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(r3["dbias"], r1["dbias"] + dbias_in, rtol=1e-14, atol=1e-14)


def test_dprob_is_derivative_in_prob():
    a, bs, c, offsets, alpha, beta, prob = tiny_case(6, [2, 2], K=3, N=32)

    def loss(p):
        # total forward contribution sum_{m,j} R * prob * act, via the brute-force forward
        _, dp, _ = brute_dglu(a, bs, c, offsets, alpha, beta, np.ones(4), "dswiglu", True, "value")
        return float(np.dot(p, dp))

    res = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, prob)
    for m in range(4):
        e = np.zeros(4)
        e[m] = 1.0
        g = (loss(prob + 1e-4 * e) - loss(prob - 1e-4 * e)) / 2e-4
        assert res["dprob"][m] == pytest.approx(g, rel=1e-8, abs=1e-10)


def test_dbias_is_per_expert_column_sum():
    a, bs, c, offsets, alpha, beta, prob = tiny_case(7, [3, 0, 4], K=4, N=64)
    res = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, prob)
    D = res["d_row"]
    np.testing.assert_allclose(res["dbias"][0], D[0:3].sum(0), rtol=1e-13)
    np.testing.assert_array_equal(res["dbias"][1], 0.0)   # empty expert
    np.testing.assert_allclose(res["dbias"][2], D[3:7].sum(0), rtol=1e-13)


# --------------------------------------------------------------------------------------
# grouped wgrad
# --------------------------------------------------------------------------------------

def brute_wgrad(A, B, offsets):
    """Loops over experts, rows, columns and the expert's tokens (A (h,T), B (T,i) dense)."""
    h, T = A.shape
    i = B.shape[1]
    out = []
    for e in range(len(offsets)):
        begin = 0 if e == 0 else offsets[e - 1]
        end = offsets[e]
        W = np.zeros((h, i))
        for r in range(h):
            for col in range(i):
                s = 0.0
                for t in range(begin, end):
                    s += A[r, t] * B[t, col]
                W[r, col] = s
        out.append(W)
    return out


def _wgrad_case(seed, counts, h, i):
    rng = np.random.default_rng(seed)
    offsets = np.cumsum(counts).astype(np.int64)
    T = int(offsets[-1])
    A = rng.normal(size=(h, T))
    B = rng.normal(size=(T, i))
    return A, B, offsets, T


def _store(A, B, offsets, a_major, b_major, order):
    """Flat storage of A (h,T) and B (T,i) in the requested majors / order (test-side packing)."""
    h, T = A.shape
    i = B.shape[1]
    ranges = O.expert_ranges(offsets)
    if a_major == "k":
        if order == "tensor_ragged":
            a_flat = np.concatenate([A[:, lo:hi].reshape(-1) for lo, hi in ranges])
        else:
            a_flat = A.reshape(-1)
    else:
        a_flat = A.T.copy().reshape(-1)
    if b_major == "n":
        b_flat = B.reshape(-1)
    else:
        if order == "tensor_ragged":
            b_flat = np.concatenate([B[lo:hi, :].T.reshape(-1) for lo, hi in ranges])
        else:
            b_flat = B.T.copy().reshape(-1)
    return a_flat, b_flat


def test_wgrad_bruteforce_tiny():
    A, B, offsets, T = _wgrad_case(10, [3, 0, 2, 4], 3, 4)
    ref = brute_wgrad(A, B, offsets)
    out = O.wgrad(A.reshape(-1), B.reshape(-1), offsets, 3, 4)
    for e in range(4):
        np.testing.assert_allclose(out[e], ref[e], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(out[1], 0.0)


@pytest.mark.parametrize("a_major", ["k", "m"])
@pytest.mark.parametrize("b_major", ["n", "k"])
@pytest.mark.parametrize("order", ["tensor2d", "tensor_ragged"])
def test_wgrad_layouts_and_orders_agree(a_major, b_major, order):
    A, B, offsets, T = _wgrad_case(11, [4, 2, 0, 3], 5, 6)
    ref = brute_wgrad(A, B, offsets)
    a_flat, b_flat = _store(A, B, offsets, a_major, b_major, order)
    out = O.wgrad(a_flat, b_flat, offsets, 5, 6, a_major=a_major, b_major=b_major, input_order=order)
    for e in range(4):
        np.testing.assert_allclose(out[e], ref[e], rtol=1e-12, atol=1e-12)


def test_wgrad_sum_over_experts_is_full_matmul():
    A, B, offsets, T = _wgrad_case(12, [5, 3, 7, 1], 6, 4)
    out = O.wgrad(A.reshape(-1), B.reshape(-1), offsets, 6, 4)
    total = sum(out[e] for e in range(4))
    np.testing.assert_allclose(total, np.einsum("ht,ti->hi", A, B), rtol=1e-12, atol=1e-12)


def test_wgrad_accumulate_is_old_plus_new_and_empty_untouched():
    A, B, offsets, T = _wgrad_case(13, [2, 0, 3], 3, 5)
    old = np.random.default_rng(0).normal(size=(3, 3, 5))
    new = O.wgrad(A.reshape(-1), B.reshape(-1), offsets, 3, 5)
    acc = O.wgrad(A.reshape(-1), B.reshape(-1), offsets, 3, 5, accumulate=True, out_old=old)
    for e in range(3):
        np.testing.assert_array_equal(acc[e], old[e] + new[e])
    np.testing.assert_array_equal(acc[1], old[1])
    np.testing.assert_array_equal(new[1], 0.0)


def test_wgrad_elements_match_full():
    A, B, offsets, T = _wgrad_case(14, [4, 0, 6], 7, 9)
    a_flat, b_flat = _store(A, B, offsets, "k", "n", "tensor_ragged")
    full = O.wgrad(a_flat, b_flat, offsets, 7, 9, input_order="tensor_ragged")
    hh = np.array([0, 6, 3])
    ii = np.array([8, 0, 4])
    for e in range(3):
        v = O.wgrad_elements(a_flat, b_flat, offsets, 7, 9, e, hh, ii, input_order="tensor_ragged")
        np.testing.assert_allclose(v, full[e][hh, ii], rtol=1e-13, atol=1e-13)
    old = np.ones(3)
    v = O.wgrad_elements(a_flat, b_flat, offsets, 7, 9, 1, hh, ii, input_order="tensor_ragged",
                         accumulate=True, old_values=old)
    np.testing.assert_array_equal(v, old)


# --------------------------------------------------------------------------------------
# schedules
# --------------------------------------------------------------------------------------

def test_dgrad_tiles_bruteforce():
    offsets = [256, 256, 1024, 1280]
    N, TM, TN = 300, 128, 128
    tiles = O.dgrad_tiles(offsets, N, TM, TN)
    brute = []
    for mb in range(1280 // TM):
        r = mb * TM
        g = next(e for e in range(len(offsets)) if r < offsets[e])
        # the whole block lies in that expert
        assert r + TM <= offsets[g]
        for nb in range(-(-N // TN)):
            brute.append((g, r, nb * TN))
    assert sorted(map(tuple, tiles.tolist())) == sorted(brute)
    assert len(tiles) == (1280 // TM) * 3
    assert 1 not in tiles[:, 0]


def _tiles_by_element_cover(offsets, hidden, inter, tm, tn, accumulate):
    """Tile origins derived from the output elements instead of from a tile loop: every element
    (e, h, i) an expert must write (all of them in overwrite mode, only non-empty experts under
    accumulate_on_output) belongs to the tile whose origin is (floor(h / tm) tm, floor(i / tn) tn)."""
    origins = set()
    prev = 0
    for e, end in enumerate(offsets):
        empty = int(end) == prev
        prev = int(end)
        if empty and accumulate:
            continue
        for h in range(hidden):
            for i in range(inter):
                origins.add((e, (h // tm) * tm, (i // tn) * tn))
    return sorted(origins)


@pytest.mark.parametrize("hidden,inter,tm,tn,accumulate", [
    (300, 200, 128, 128, False),   # tm == tn: a swapped (h0, i0) or i0 stepped by tm would pass a count check
    (200, 300, 128, 128, True),
    (384, 520, 128, 256, False),   # ragged inter tail
    (512, 136, 256, 128, True),    # pair-sized hidden tiles, inter just past one tile
    (130, 260, 128, 256, False),
])
def test_wgrad_tiles_bruteforce(hidden, inter, tm, tn, accumulate):
    offsets = [256, 256, 768, 768, 1024]  # experts 1 and 3 empty
    tiles = O.wgrad_tiles(offsets, hidden, inter, tm, tn, accumulate)
    assert sorted(map(tuple, tiles.tolist())) == _tiles_by_element_cover(offsets, hidden, inter, tm, tn, accumulate)
    # the tiles partition each written expert's output: every element lies in exactly one tile
    for e in sorted(set(tiles[:, 0].tolist())):
        cover = np.zeros((hidden, inter), dtype=np.int64)
        for _, h0, i0 in tiles[tiles[:, 0] == e]:
            cover[h0:h0 + tm, i0:i0 + tn] += 1
        assert (cover == 1).all()


def test_wgrad_tiles_overwrite_includes_empty_accumulate_skips():
    offsets = [512, 512, 768]
    t_ow = O.wgrad_tiles(offsets, 256, 384, 128, 256, accumulate=False)
    t_acc = O.wgrad_tiles(offsets, 256, 384, 128, 256, accumulate=True)
    per = 2 * 2
    assert len(t_ow) == 3 * per
    assert len(t_acc) == 2 * per
    assert 1 in t_ow[:, 0] and 1 not in t_acc[:, 0]


# --------------------------------------------------------------------------------------
# planted mistakes must be caught by the pins above
# --------------------------------------------------------------------------------------

def test_planted_mistakes_are_caught(monkeypatch):
    a, bs, c, offsets, alpha, beta, prob = tiny_case(1, [3, 0, 2, 3], K=5, N=64)
    D, dprob, _ = brute_dglu(a, bs, c, offsets, alpha, beta, prob, "dswiglu", True, "value")

    def run():
        return O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, prob)

    res = run()
    assert np.allclose(res["d_row"], D, rtol=1e-6, atol=1e-8)
    real_gc = O.glu_columns
    with monkeypatch.context() as mp:   # gate/input blocks swapped
        mp.setattr(O, "glu_columns", lambda n, gate_first=True: real_gc(n, not gate_first))
        r = run()
        assert not np.allclose(r["d_row"], D, rtol=1e-6, atol=1e-8)
    with monkeypatch.context() as mp:   # expert ranges shifted by one row
        mp.setattr(O, "expert_ranges", lambda offs: [(0, 2), (2, 2), (2, 5), (5, 8)])
        r = run()
        assert not np.allclose(r["d_row"], D, rtol=1e-6, atol=1e-8)
    with monkeypatch.context() as mp:
        real_sw = O.dswiglu
        mp.setattr(O, "dswiglu", lambda R, p, g, i: real_sw(R, p, i, g))  # gate/input roles swapped
        r = run()
        assert not np.allclose(r["d_row"], D, rtol=1e-6, atol=1e-8)
    with monkeypatch.context() as mp:
        mp.setattr(O, "sigmoid", lambda x: 1.0 / (1.0 + np.exp(x)))       # sign error
        r = run()
        assert not np.allclose(r["d_row"], D, rtol=1e-6, atol=1e-8)
    # alpha instead of alpha^2: rescale alpha so alpha^2 -> alpha
    r = O.dglu_bwd(a, lambda g: bs[g], c, offsets, np.sqrt(alpha), beta, prob)
    assert not np.allclose(r["d_row"], D, rtol=1e-6, atol=1e-8)
    # a transposed wgrad operand is caught by the brute force
    A, B, offs, T = _wgrad_case(10, [3, 0, 2, 4], 3, 4)
    ref = brute_wgrad(A, B, offs)
    bad = O.wgrad(A.reshape(-1), B.reshape(-1), offs, 3, 4, b_major="k")
    assert not all(np.allclose(bad[e], ref[e]) for e in (0, 2, 3))


def test_planted_tile_schedule_mistakes_are_caught():
    """Wrong wgrad schedules that a tile count (or expert membership) alone would accept."""
    offsets, hidden, inter, tm, tn = [256, 256, 768], 300, 200, 128, 128
    want = _tiles_by_element_cover(offsets, hidden, inter, tm, tn, False)
    good = sorted(map(tuple, O.wgrad_tiles(offsets, hidden, inter, tm, tn, False).tolist()))
    assert good == want
    swapped = sorted((e, i0, h0) for e, h0, i0 in good)                        # (h0, i0) swapped
    extents = sorted((e, h0, i0) for e in range(3) for h0 in range(0, inter, tm)  # hidden and inter swapped
                     for i0 in range(0, hidden, tn))
    assert len(swapped) == len(good) and swapped != want
    assert len(extents) == len(good) and extents != want


# --------------------------------------------------------------------------------------
# dsReLU (dsReLU page, "Equations") and the per-expert amax
# --------------------------------------------------------------------------------------

def fwd_srelu_unit(g, c):
    """Forward term whose derivatives the dsReLU backward gives: c * relu(g)^2."""
    return c * max(g, 0.0) ** 2


def brute_dsrelu(a, bs, c, offsets, alpha, prob):
    """Pure-python loops: expert found by scanning the ends, D by a central difference in G of
    prob * c * relu(G)^2, dprob as the forward term summed over the row, amax by a running max."""
    M, K = a.shape
    N = c.shape[1]
    L = len(offsets)
    D = np.zeros((M, N))
    dprob = np.zeros(M)
    amax = np.zeros(L)
    for m in range(M):
        g = next(e for e in range(L) if m < offsets[e])
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += float(a[m, k]) * float(bs[g][n, k])
            G = alpha[g] * acc
            D[m, n] = prob[m] * fd(lambda x: fwd_srelu_unit(x, c[m, n]), G, h=1e-7)
            dprob[m] += fwd_srelu_unit(G, c[m, n])
            amax[g] = max(amax[g], abs(D[m, n]))
    return D, dprob, amax


def srelu_case(seed, counts, K, N):
    rng = np.random.default_rng(seed)
    offsets = np.cumsum(counts).astype(np.int64)
    M = int(offsets[-1])
    q = lambda x: np.round(x * 64) / 64
    a = q(rng.normal(size=(M, K)))
    bs = [q(rng.normal(size=(N, K))) for _ in counts]
    c = q(rng.normal(size=(M, N)))
    alpha = rng.uniform(0.5, 1.5, len(counts))
    prob = rng.uniform(0, 1, M)
    return a, bs, c, offsets, alpha, prob


def test_dsrelu_bwd_bruteforce():
    a, bs, c, offsets, alpha, prob = srelu_case(21, [3, 0, 2, 3], K=5, N=40)
    res = O.dsrelu_bwd(a, lambda g: bs[g], c, offsets, alpha, prob)
    D, dprob, amax = brute_dsrelu(a, bs, c, offsets, alpha, prob)
    G_all = np.concatenate([alpha[g] * a[lo:hi] @ bs[g].T for g, (lo, hi) in enumerate(O.expert_ranges(offsets))])
    assert (G_all > 0).any() and (G_all < 0).any()  # both sides of the relu are exercised
    np.testing.assert_allclose(res["d_row"], D, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(res["dprob"], dprob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["amax"], amax, rtol=1e-6)
    assert res["amax"][1] == 0.0  # empty expert


def test_dsrelu_closed_forms_and_special_cases():
    a, bs, c, offsets, alpha, prob = srelu_case(22, [4, 4], K=6, N=32)
    G = np.concatenate([alpha[g] * a[lo:hi] @ bs[g].T for g, (lo, hi) in enumerate(O.expert_ranges(offsets))])
    # C = 1, prob = 1: D_row = 2 relu(G) and dprob = sum relu(G)^2 exactly
    res = O.dsrelu_bwd(a, lambda g: bs[g], np.ones_like(c), offsets, alpha, np.ones(8))
    np.testing.assert_allclose(res["d_row"], 2 * np.maximum(G, 0), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(res["dprob"], (np.maximum(G, 0) ** 2).sum(1), rtol=1e-13)
    # alpha (not alpha^2): doubling alpha doubles D_row and quadruples dprob
    r1 = O.dsrelu_bwd(a, lambda g: bs[g], c, offsets, alpha, prob)
    r2 = O.dsrelu_bwd(a, lambda g: bs[g], c, offsets, 2 * alpha, prob)
    np.testing.assert_allclose(r2["d_row"], 2 * r1["d_row"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(r2["dprob"], 4 * r1["dprob"], rtol=1e-13, atol=1e-13)
    # prob = 0 zeroes D_row but not dprob (no prob factor); negative G contributes nothing
    r0 = O.dsrelu_bwd(a, lambda g: bs[g], c, offsets, alpha, np.zeros(8), dprob_in=np.arange(8.0))
    assert (r0["d_row"] == 0).all()
    np.testing.assert_allclose(r0["dprob"], r1["dprob"] + np.arange(8.0), rtol=1e-13)
    neg = O.dsrelu_bwd(a, lambda g: -bs[g], c, offsets, alpha, prob)
    np.testing.assert_array_equal(neg["d_row"][G > 0], 0.0)
    # dprob is the derivative in prob of sum prob * C * relu(G)^2
    fwd = (c * np.maximum(G, 0) ** 2).sum(1)
    np.testing.assert_allclose(r1["dprob"], fwd, rtol=1e-13)
    rows = np.array([7, 1, 4])
    part = O.dsrelu_bwd(a, lambda g: bs[g], c[rows], offsets, alpha, prob, rows=rows)
    np.testing.assert_array_equal(part["d_row"], r1["d_row"][rows])


def test_dglu_amax_is_per_expert_block_max():
    a, bs, c, offsets, alpha, beta, prob = tiny_case(23, [3, 0, 4], K=4, N=64)
    res = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, prob, act="dgeglu")
    D = res["d_row"]
    gcol, icol = O.glu_columns(64)
    for g, (lo, hi) in enumerate(O.expert_ranges(offsets)):
        if hi == lo:
            assert (res["amax"][g] == 0).all()
            continue
        blk = D[lo:hi]
        assert res["amax"][g, 0] == np.abs(blk[:, gcol]).max()
        assert res["amax"][g, 1] == np.abs(blk[:, icol]).max()
    # gate/input roles: with the blocks swapped in the layout the two entries follow their block
    res2 = O.dglu_bwd(a, lambda g: bs[g], c, offsets, alpha, beta, prob, act="dgeglu", gate_first=False)
    g2, i2 = O.glu_columns(64, gate_first=False)
    assert res2["amax"][0, 0] == np.abs(res2["d_row"][0:3][:, g2]).max()


def test_dsrelu_planted_mistakes_are_caught(monkeypatch):
    a, bs, c, offsets, alpha, prob = srelu_case(24, [3, 0, 2, 3], K=5, N=40)
    D, dprob, amax = brute_dsrelu(a, bs, c, offsets, alpha, prob)

    def ok(r):
        return (np.allclose(r["d_row"], D, rtol=1e-6, atol=1e-8) and np.allclose(r["dprob"], dprob, rtol=1e-9)
                and np.allclose(r["amax"], amax, rtol=1e-6))

    assert ok(O.dsrelu_bwd(a, lambda g: bs[g], c, offsets, alpha, prob))
    assert not ok(O.dsrelu_bwd(a, lambda g: bs[g], c, offsets, alpha ** 2, prob))   # alpha^2 instead of alpha
    assert not ok(O.dsrelu_bwd(a, lambda g: bs[g][::-1], c, offsets, alpha, prob))    # permuted weight rows
    with monkeypatch.context() as mp:
        mp.setattr(O, "dsrelu", lambda G, p, cc: (p * 2.0 * np.asarray(cc) * np.abs(G),
                                                  np.asarray(cc) * np.asarray(G) ** 2))  # |G| instead of relu
        assert not ok(O.dsrelu_bwd(a, lambda g: bs[g], c, offsets, alpha, prob))
    with monkeypatch.context() as mp:
        mp.setattr(O, "expert_ranges", lambda offs: [(0, 2), (2, 2), (2, 5), (5, 8)])     # shifted ranges
        assert not ok(O.dsrelu_bwd(a, lambda g: bs[g], c, offsets, alpha, prob))
