"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by element,
on seeded inputs that span several tiles and ragged tails, in every supported mode."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_persistent_gb300 import api, synth
from moe_grouped_gemm_persistent_gb300.build import build

from gpu_helpers import (TOL, TOL_DPROB, check_close, rel_fro, run_dglu_gpu, run_dglu_oracle, run_wgrad_gpu,
                         run_wgrad_oracle, tiles_from_log, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    build()
    return torch.device("cuda", 0)


def _ranges(spec):
    return oracle.expert_ranges(np.cumsum(spec.counts))


def test_binding_queues_on_the_current_stream(dev):
    """The binding's default stream is torch's current stream of the current device, inside and
    outside a stream context."""
    assert api._stream(None) == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        assert api._stream(None) == s.cuda_stream == torch.cuda.current_stream().cuda_stream
    assert api._stream(s) == s.cuda_stream and api._stream(s.cuda_stream) == s.cuda_stream


# ------------------------------------------------------------------------------ tensor maps
def test_tensormap_replace_matches_host_encoding(dev):
    """Device-side rewriting of a descriptor equals the driver's encoding of the target (bytes)."""
    from moe_grouped_gemm_persistent_gb300 import _lib
    lib = _lib.load()
    buf = torch.empty(1 << 22, dtype=torch.bfloat16, device=dev)
    base = buf.data_ptr()
    import ctypes
    host = (ctypes.c_uint8 * 256)()
    off = (-ctypes.addressof(host)) % 64
    tmpl = ctypes.addressof(host) + off
    exp_host = (ctypes.c_uint8 * 256)()
    off2 = (-ctypes.addressof(exp_host)) % 64
    exp = ctypes.addressof(exp_host) + off2
    # template: dims {4096, 128}, stride 8192 B at base; target: dims {1536, 128}, stride 3072 B at base + 1 MiB
    _lib.check(lib.mgg_test_encode_tmap_2d(tmpl, base, 4096, 128, 8192, 64, 128))
    tgt = base + (1 << 20)
    _lib.check(lib.mgg_test_encode_tmap_2d(exp, tgt, 1536, 128, 3072, 64, 128))
    out = torch.zeros(256, dtype=torch.uint8, device=dev)
    optr = out.data_ptr() + ((-out.data_ptr()) % 128)
    _lib.check(lib.mgg_test_tmap_replace(tmpl, optr, tgt, 1536, 3072, 7, None))
    torch.cuda.synchronize()
    got = out.cpu().numpy()[(optr - out.data_ptr()):(optr - out.data_ptr()) + 128]
    want = np.frombuffer(bytes(exp_host)[off2:off2 + 128], dtype=np.uint8)
    assert got.tobytes() == want.tobytes()
    # address only
    _lib.check(lib.mgg_test_encode_tmap_2d(exp, tgt, 4096, 128, 8192, 64, 128))
    _lib.check(lib.mgg_test_tmap_replace(tmpl, optr, tgt, 0, 0, 1, None))
    torch.cuda.synchronize()
    got = out.cpu().numpy()[(optr - out.data_ptr()):(optr - out.data_ptr()) + 128]
    want = np.frombuffer(bytes(exp_host)[off2:off2 + 128], dtype=np.uint8)
    assert got.tobytes() == want.tobytes()


# ------------------------------------------------------------------------------ dgrad + dGLU
DGLU_CASES = {
    "swiglu_dense": dict(),
    "swiglu_ktail_ntail": dict(K=328, N=160),
    "geglu_value_fp32d_dbias": dict(act="dgeglu", c_std=4.0, d_dtype="fp32", dbias=True),
    "swiglu_fp16": dict(c_dtype="fp16", d_dtype="fp16"),
    "swiglu_fp32c": dict(c_dtype="fp32"),
    "discrete_k": dict(b_mode="discrete", b_major="k"),
    "discrete_n_geglu": dict(b_mode="discrete", b_major="n", act="dgeglu", c_std=4.0, dbias=True),
    # N % 64 == 0: N-major weights through one 3-D box of 64-column blocks per ring slot
    "discrete_n_blocked_fp32d": dict(b_mode="discrete", b_major="n", N=192, K=256, act="dgeglu", c_std=4.0,
                                     d_dtype="fp32", dbias=True),
    "wide_n": dict(N=544, K=192, counts=(512, 256)),
    # K >= 4096 selects the register path for 16-bit C
    "regpath_swiglu": dict(K=4096, N=96, counts=(256, 0, 256)),
    "regpath_geglu_fp32d_dbias": dict(K=4160, N=64, counts=(256, 512), act="dgeglu", c_std=4.0, d_dtype="fp32",
                                      dbias=True),
    "situglu": dict(act="dsituglu", c_std=4.0),
    "situglu_fp32d_dbias": dict(act="dsituglu", c_std=8.0, d_dtype="fp32", dbias=True),
    "regpath_situglu": dict(K=4096, N=64, counts=(256, 0, 256), act="dsituglu", c_std=4.0),
}


DGLU_SCHED = [(c, "static") for c in DGLU_CASES] + [("swiglu_dense", "dynamic"), ("discrete_n_geglu", "dynamic"),
                                                      ("many_experts", "dynamic")]
DGLU_CASES["many_experts"] = dict(K=128, N=64, counts=(256, 0, 0, 512, 256, 0, 768, 256, 256, 0, 512))
# one expert (L = 1): the grouped call is a plain alpha^2 A B^T with the dGLU epilogue
DGLU_CASES["single_expert"] = dict(K=192, N=96, counts=(768,))
DGLU_SCHED += [("single_expert", "static"), ("single_expert", "dynamic")]
# the operation's maximum of 1024 experts, most of them empty: 1024 per-expert weight maps built on
# the device, the expert search over 1024 offsets, dbias partial sums for every expert (zero rows
# for the empty ones) and the dGeGLU filters, through discrete N-major weights
_MAX_COUNTS = [0] * 1024
for _g in (0, 1, 300, 511, 512, 777, 1022, 1023):
    _MAX_COUNTS[_g] = 256
_MAX_COUNTS[300] = 512
DGLU_CASES["max_experts_discrete"] = dict(K=128, N=64, counts=tuple(_MAX_COUNTS), b_mode="discrete", b_major="n",
                                          act="dgeglu", c_std=4.0, dbias=True)
DGLU_SCHED += [("max_experts_discrete", "static"), ("max_experts_discrete", "dynamic")]


# "single": 128-row tiles, one CTA per SM; "pair": 256-row tiles on CTA pairs (cta_group::2).
CTAS = ["single", "pair"]


@pytest.mark.parametrize("cta", CTAS)
@pytest.mark.parametrize("case,sched", DGLU_SCHED)
def test_dglu_bwd_parity(dev, case, sched, cta):
    kw = dict(DGLU_CASES[case])
    counts = kw.pop("counts", (256, 0, 512))
    spec = synth.small_dglu_spec(case, L=len(counts), counts=counts, **kw)
    x = synth.make_dglu_inputs(spec)
    gpu = run_dglu_gpu(spec, x, dev, tile_log=True, sched=sched, cta=cta)
    assert gpu["status"] == 0
    ref = run_dglu_oracle(spec, x)
    rows = [(lo, hi) for lo, hi in _ranges(spec)]
    check_close("d_row", to_np(gpu["d_row"]), ref["d_row"], TOL[spec.d_dtype], rows)
    check_close("dprob", to_np(gpu["dprob"]), ref["dprob"], TOL_DPROB, rows)
    if spec.dbias:
        check_close("dbias", to_np(gpu["dbias"]), ref["dbias"], TOL["bf16"])
        for g, (lo, hi) in enumerate(rows):
            if hi == lo:
                assert (gpu["dbias"][g] == 0).all()
    tm, tn = api.dglu_bwd_tile_shape()
    want = oracle.dgrad_tiles(np.cumsum(spec.counts), spec.N, tm, tn)
    np.testing.assert_array_equal(tiles_from_log(gpu["tile_log"]), want)


@pytest.mark.parametrize("gate_first,filt,d_dtype", [(False, "value", "bf16"), (True, "indicator", "bf16"),
                                                     (False, "indicator", "bf16"), (False, "value", "fp32")])
def test_dglu_block_order_and_filter_modes(dev, gate_first, filt, d_dtype):
    # the fp32 case also sums dbias from the staged fp32 boxes with the input block first
    spec = synth.small_dglu_spec("modes", act="dgeglu", c_std=4.0, d_dtype=d_dtype, dbias=d_dtype == "fp32")
    x = synth.make_dglu_inputs(spec)
    gpu = run_dglu_gpu(spec, x, dev, gate_first=gate_first, geglu_filter=filt)
    ref = run_dglu_oracle(spec, x, gate_first=gate_first, geglu_filter=filt)
    check_close("d_row", to_np(gpu["d_row"]), ref["d_row"], TOL[d_dtype])
    check_close("dprob", to_np(gpu["dprob"]), ref["dprob"], TOL_DPROB)
    if spec.dbias:
        check_close("dbias", to_np(gpu["dbias"]), ref["dbias"], TOL["bf16"])


@pytest.mark.parametrize("betas", [(2.0, 5.0), (0.5, 40.0)])
def test_dsituglu_custom_betas(dev, betas):
    spec = synth.small_dglu_spec("situ_b", act="dsituglu", c_std=6.0)
    x = synth.make_dglu_inputs(spec)
    gpu = run_dglu_gpu(spec, x, dev, situ=betas)
    ref = run_dglu_oracle(spec, x, situ=betas)
    check_close("d_row", to_np(gpu["d_row"]), ref["d_row"], TOL["bf16"])
    check_close("dprob", to_np(gpu["dprob"]), ref["dprob"], TOL_DPROB)


# bf16-exact values on and just past the dGeGLU clamp / filter boundaries (one bf16 ulp at 7 is
# 2^-5), plus 0 (a value-bearing filter of 0) and -1 (clamped_input + 1 = 0)
TIE_VALUES = (7.0, -7.0, 7.0 + 2 ** -5, -7.0 - 2 ** -5, 0.0, -1.0)


def _plant_ties(spec, x, zero_prob_rows, zero_alpha_expert):
    """beta = 1 (X = C exactly), tie values planted over C, some prob rows 0, one expert's alpha 0."""
    c = x["c"].float()
    M, two_n = c.shape
    r = torch.arange(M)[:, None]
    col = torch.arange(two_n)[None, :]
    sel = ((r * 7 + col * 3) % 5) == 0
    vals = torch.tensor(TIE_VALUES)[((r + col) % len(TIE_VALUES)).expand(M, two_n)]
    c = torch.where(sel, vals, c)
    x["c"] = c.to(x["c"].dtype)
    assert torch.equal(x["c"].float()[sel], vals[sel])  # every planted value is exact in the C dtype
    x["beta"] = torch.ones_like(x["beta"])
    x["prob"][torch.as_tensor(zero_prob_rows)] = 0.0
    x["alpha"][zero_alpha_expert] = 0.0
    return x


@pytest.mark.parametrize("cta", CTAS)
@pytest.mark.parametrize("act,filt,d_dtype,K,N,counts", [
    ("dgeglu", "value", "bf16", 320, 160, (256, 0, 512, 256)),
    ("dgeglu", "indicator", "bf16", 320, 160, (256, 0, 512, 256)),
    ("dgeglu", "value", "fp32", 320, 160, (256, 0, 512, 256)),
    ("dgeglu", "indicator", "fp32", 192, 96, (512, 256)),
    ("dgeglu", "value", "bf16", 4096, 64, (256, 512)),        # register C path (single CTAs)
    ("dswiglu", "value", "bf16", 320, 160, (256, 0, 512, 256)),
    ("dsituglu", "value", "bf16", 320, 160, (256, 0, 512, 256)),
])
def test_dglu_exact_ties_zero_prob_rows_zero_alpha(dev, cta, act, filt, d_dtype, K, N, counts):
    """The clamp and filter decisions at X = +-7 and one ulp past them must be the oracle's, element
    by element (zero vs non-zero, bit-exact); prob = 0 rows give D = 0 but still add to dprob; an
    expert with alpha = 0 gives D = 0 and adds exactly nothing to dprob."""
    # C ~ N(0, 4) makes the dGeGLU clamps fire; the tanh-based sigmoid of dSwiGLU / dSiTU-GLU rounds to
    # exactly 0 or 1 in fp32 past |x| ~ 17, where float64 does not, so those keep |X| small
    spec = synth.small_dglu_spec("ties", L=len(counts), counts=counts, K=K, N=N, act=act,
                                 c_std=4.0 if act == "dgeglu" else 2.0, d_dtype=d_dtype, dbias=d_dtype == "fp32")
    x = synth.make_dglu_inputs(spec)
    ranges = _ranges(spec)
    zero_alpha = len(counts) - 1
    lo_first = ranges[0][0]
    zero_rows = [lo_first + 3, lo_first + 100, ranges[-2][1] - 1]
    x = _plant_ties(spec, x, zero_rows, zero_alpha)
    gpu = run_dglu_gpu(spec, x, dev, geglu_filter=filt, cta=cta)
    assert gpu["status"] == 0
    ref = run_dglu_oracle(spec, x, geglu_filter=filt)
    got = to_np(gpu["d_row"])
    check_close("d_row", got, ref["d_row"], TOL[d_dtype], [rg for rg in ranges if rg[1] > rg[0]][:-1])
    nz_dprob = [rg for g, rg in enumerate(ranges) if g != zero_alpha]
    check_close("dprob", to_np(gpu["dprob"])[:ranges[zero_alpha][0]], ref["dprob"][:ranges[zero_alpha][0]],
                TOL_DPROB, nz_dprob)
    np.testing.assert_array_equal(got == 0, ref["d_row"] == 0)  # every zero / non-zero decision
    lo, hi = ranges[zero_alpha]
    assert (gpu["d_row"][lo:hi] == 0).all() and (gpu["dprob"][lo:hi] == 0).all()
    for m in zero_rows:
        assert (gpu["d_row"][m] == 0).all() and gpu["dprob"][m] != 0
    if act == "dgeglu":  # the oracle itself took the tie decisions as the page prints them
        gcol, icol = oracle.glu_columns(N)
        c = x["c"].float().numpy()
        live = np.ones(spec.M, bool)
        live[zero_rows] = False
        live[lo:hi] = False
        gate_past = (c[:, gcol] == 7.0 + 2 ** -5) & live[:, None]
        inp_past = (np.abs(c[:, icol]) == 7.0 + 2 ** -5) & live[:, None]
        gate_on = (c[:, gcol] == 7.0) & live[:, None]
        inp_on = (np.abs(c[:, icol]) == 7.0) & live[:, None] & (c[:, gcol] != 0)  # gate 0 zeroes dinput
        assert gate_past.any() and inp_past.any() and gate_on.any() and inp_on.any()
        assert (ref["d_row"][:, gcol][gate_past] == 0).all() and (ref["d_row"][:, icol][inp_past] == 0).all()
        assert (ref["d_row"][:, icol][inp_on] != 0).all()
    if spec.dbias:
        check_close("dbias", to_np(gpu["dbias"]), ref["dbias"], TOL["bf16"])


def test_dglu_accumulates_into_dprob_and_dbias(dev):
    spec = synth.small_dglu_spec("acc", dbias=True)
    x = synth.make_dglu_inputs(spec)
    gen = torch.Generator().manual_seed(5)
    dprob0 = torch.randn(spec.M, generator=gen)
    dbias0 = torch.randn(spec.L, 2 * spec.N, generator=gen).to(torch.bfloat16)
    gpu = run_dglu_gpu(spec, x, dev, dprob0=dprob0, dbias0=dbias0)
    ref = run_dglu_oracle(spec, x, dprob0=dprob0, dbias0=dbias0)
    check_close("dprob", to_np(gpu["dprob"]), ref["dprob"], TOL_DPROB)
    check_close("dbias", to_np(gpu["dbias"]), ref["dbias"], TOL["bf16"])


def test_dglu_tiny_workload(dev):
    spec, _ = synth.workload_specs("tiny")
    x = synth.make_dglu_inputs(spec)
    gpu = run_dglu_gpu(spec, x, dev)
    ref = run_dglu_oracle(spec, x)
    check_close("d_row", to_np(gpu["d_row"]), ref["d_row"], TOL["bf16"], _ranges(spec))
    check_close("dprob", to_np(gpu["dprob"]), ref["dprob"], TOL_DPROB)


@pytest.mark.parametrize("cta", CTAS)
def test_dglu_all_experts_empty(dev, cta):
    """M = 0 (every expert empty; torch gives the empty per-row tensors NULL data pointers): the
    call succeeds, launches no GEMM tiles, and dbias (accumulated into) keeps its values."""
    L, K, N = 4, 128, 64
    a = torch.empty(0, K, dtype=torch.bfloat16, device=dev)
    c = torch.empty(0, 2 * N, dtype=torch.bfloat16, device=dev)
    prob, dprob = torch.empty(0, device=dev), torch.empty(0, device=dev)
    d_row = torch.empty(0, 2 * N, dtype=torch.bfloat16, device=dev)
    b = torch.randn(L, N, K, device=dev).to(torch.bfloat16)
    alpha = torch.ones(L, device=dev)
    beta = torch.ones(L, device=dev)
    offs = torch.zeros(L, dtype=torch.int32, device=dev)
    dbias = torch.full((L, 2 * N), 1.5, dtype=torch.bfloat16, device=dev)
    ws = api.dglu_bwd(a=a, c=c, padded_offsets=offs, alpha=alpha, beta=beta, prob=prob, dprob=dprob, d_row=d_row,
                      b=b, dbias=dbias, act="dgeglu", cta=cta)
    assert api.read_device_status(ws) == 0
    assert (dbias == 1.5).all()


@pytest.mark.parametrize("cta", CTAS)
@pytest.mark.parametrize("accumulate", [False, True])
def test_wgrad_all_experts_empty(dev, cta, accumulate):
    """T = 0 (every expert empty; the empty operands have NULL data pointers): overwrite writes zeros
    into every output, accumulate leaves every output as it was."""
    L, h, i = 3, 256, 128
    a = torch.empty(0, h, dtype=torch.bfloat16, device=dev)
    b = torch.empty(0, i, dtype=torch.bfloat16, device=dev)
    offs = torch.zeros(L, dtype=torch.int32, device=dev)
    out = torch.full((L, h, i), 2.5, dtype=torch.float32, device=dev)
    ws = api.wgrad(a=a, b=b, offsets=offs, hidden=h, inter=i, out=out, accumulate=accumulate, cta=cta,
                   input_order="tensor_ragged")
    assert api.read_device_status(ws) == 0
    if accumulate:
        assert (out == 2.5).all()
    else:
        assert (out == 0).all()


@pytest.mark.parametrize("cta", CTAS)
def test_dglu_bad_offsets_report_and_leave_outputs(dev, cta):
    spec = synth.small_dglu_spec("bad")
    x = synth.make_dglu_inputs(spec)
    x["padded_offsets"] = torch.tensor([256, 128, 768], dtype=torch.int32)  # decreasing
    gpu = run_dglu_gpu(spec, x, dev, cta=cta)
    assert gpu["status"] == 5
    assert torch.isnan(gpu["d_row"].float()).all()
    assert (gpu["dprob"] == 0).all()


# ------------------------------------------------------------------------------ wgrad
WGRAD_CASES = {
    "k_n_fp32": dict(),
    "k_n_fp32_acc": dict(accumulate=True),
    "k_n_bf16": dict(out_dtype="bf16"),
    "k_n_fp16_acc": dict(out_dtype="fp16", accumulate=True),
    "m_n": dict(a_major="m"),
    "k_k": dict(b_major="k"),
    "m_k": dict(a_major="m", b_major="k"),
    "ragged_k_n_discrete": dict(input_order="tensor_ragged", out_mode="discrete"),
    "ragged_k_k": dict(input_order="tensor_ragged", b_major="k"),
    "bn256": dict(inter=512, hidden=128, counts=(256, 768, 0)),
    # MN extents that are multiples of 64: MN-major operands through blocked 3-D maps
    "m_n_blocked": dict(a_major="m", hidden=256, inter=192),
    "m_n_blocked_acc_bf16": dict(a_major="m", hidden=320, inter=448, accumulate=True, out_dtype="bf16"),
    # FP32 outputs with inter % 64 == 0: one TMA copy stores two 32-column chunks (blocked output map),
    # for dense and per-expert outputs, overwrite and accumulate; hidden = 192 leaves warps with no rows
    "out_blocked_ragged_discrete": dict(input_order="tensor_ragged", out_mode="discrete", inter=320),
    "out_blocked_acc": dict(accumulate=True, inter=384),
    "out_blocked_discrete_acc": dict(out_mode="discrete", accumulate=True, inter=256),
    # inter % 256 in (0, 128]: the last column tile runs N = 128 MMAs (in a pair each CTA supplies
    # 64 of its columns), through every B path: K-major, ragged K-major, N-major in 64-column
    # boxes and N-major blocked; with 16-bit and FP32 outputs
    "narrow_k_k": dict(b_major="k", inter=384),
    "narrow_ragged_k_k_bf16": dict(input_order="tensor_ragged", b_major="k", inter=640, out_dtype="bf16"),
    "narrow_k_n_352": dict(inter=352),
    "narrow_m_n_blocked_acc": dict(a_major="m", hidden=256, inter=320, accumulate=True),
}


WGRAD_SCHED = [(c, "static") for c in WGRAD_CASES] + [("k_n_fp32", "dynamic"), ("k_n_fp32_acc", "dynamic"),
                                                        ("ragged_k_n_discrete", "dynamic"), ("many_experts", "dynamic"),
                                                        ("out_blocked_ragged_discrete", "dynamic"),
                                                        ("out_blocked_discrete_acc", "dynamic")]
WGRAD_CASES["many_experts"] = dict(hidden=256, inter=128, counts=(256, 0, 2048, 0, 512, 256, 0, 768, 256, 1024))
# 1024 experts (the maximum), most of them empty: the expert order over 1024 counts, 1024 ragged
# per-expert maps, zero outputs for the empty experts, and the long/short alternation of the
# dynamic schedule over a very uneven order
_WMAX = [0] * 1024
for _e, _c in ((0, 256), (5, 1024), (400, 256), (511, 512), (512, 256), (900, 768), (1023, 256)):
    _WMAX[_e] = _c
WGRAD_CASES["max_experts_ragged"] = dict(hidden=256, inter=128, counts=tuple(_WMAX), input_order="tensor_ragged")
# one expert (L = 1): A @ B over all tokens
WGRAD_CASES["single_expert"] = dict(hidden=256, inter=192, counts=(1280,))
WGRAD_SCHED += [("single_expert", "static"), ("single_expert", "dynamic")]
WGRAD_SCHED += [("max_experts_ragged", "static"), ("max_experts_ragged", "dynamic")]


@pytest.mark.parametrize("cta", CTAS)
@pytest.mark.parametrize("case,sched", WGRAD_SCHED)
def test_wgrad_parity(dev, case, sched, cta):
    kw = dict(WGRAD_CASES[case])
    counts = kw.pop("counts", (512, 0, 256, 768))
    if cta == "pair" and kw.get("hidden", 192) % 256 != 0:
        kw["hidden"] = 512  # CTA pairs tile hidden in 256-row blocks
    spec = synth.small_wgrad_spec(case, L=len(counts), counts=counts, **kw)
    x = synth.make_wgrad_inputs(spec)
    gpu = run_wgrad_gpu(spec, x, dev, tile_log=True, sched=sched, cta=cta)
    assert gpu["status"] == 0
    ref = run_wgrad_oracle(spec, x)
    tol = TOL[spec.out_dtype]
    for e in range(spec.L):
        got = to_np(gpu["out"][e])
        check_close(f"wgrad[{e}]", got, ref[e], tol)
        if spec.counts[e] == 0 and not spec.accumulate:
            assert (gpu["out"][e] == 0).all()
    tm, tn = api.wgrad_tile_shape(spec.inter)
    want = oracle.wgrad_tiles(np.cumsum(spec.counts), spec.hidden, spec.inter, tm, tn, spec.accumulate)
    np.testing.assert_array_equal(tiles_from_log(gpu["tile_log"]), want)


def test_wgrad_tiny_workload(dev):
    _, spec = synth.workload_specs("tiny")
    x = synth.make_wgrad_inputs(spec)
    gpu = run_wgrad_gpu(spec, x, dev)
    ref = run_wgrad_oracle(spec, x)
    for e in range(spec.L):
        check_close(f"wgrad[{e}]", to_np(gpu["out"][e]), ref[e], TOL["fp32"])


def test_wgrad_sum_over_experts_equals_full_matmul(dev):
    spec = synth.small_wgrad_spec("sum", counts=(256, 512, 256), L=3)
    x = synth.make_wgrad_inputs(spec)
    gpu = run_wgrad_gpu(spec, x, dev)
    A = to_np(x["a"]).reshape(spec.hidden, spec.T)
    B = to_np(x["b"]).reshape(spec.T, spec.inter)
    total = to_np(gpu["out"]).sum(0)
    assert rel_fro(total, A @ B) < TOL["fp32"]


@pytest.mark.parametrize("cta", CTAS)
def test_wgrad_bad_pointer_reports(dev, cta):
    spec = synth.small_wgrad_spec("badptr", out_mode="discrete", hidden=256)
    x = synth.make_wgrad_inputs(spec)
    L, h, i = spec.L, spec.hidden, spec.inter
    outs = [torch.zeros(h, i, device=dev) for _ in range(L)]
    ptrs = api.pointer_array(outs, dev)
    ptrs[1] += 4  # misaligned entry
    ws = api.wgrad(a=x["a"].to(dev), b=x["b"].to(dev), offsets=x["offsets"].to(dev), hidden=h, inter=i,
                   out_ptrs=ptrs, out_dtype="fp32", cta=cta)
    assert api.read_device_status(ws) == 6
    assert all((o == 0).all() for o in outs)


# ------------------------------------------------------------------------------ concurrency
def test_calls_on_two_streams_at_once(dev):
    """The ABI keeps no state between calls: dgrad and wgrad calls queued on two streams at once,
    each with its own workspace, give the oracle's results (three rounds, nothing synchronised
    between the calls of a round)."""
    d1 = synth.small_dglu_spec("conc_d1", L=3, counts=(512, 256, 768), K=256, N=320)
    d2 = synth.small_dglu_spec("conc_d2", L=4, counts=(256, 0, 512, 256), K=192, N=160, act="dgeglu", c_std=4.0,
                               b_mode="discrete", b_major="n", d_dtype="fp32", dbias=True, seed=1)
    w1 = synth.small_wgrad_spec("conc_w1", counts=(512, 0, 1024, 256), hidden=512, inter=384,
                                input_order="tensor_ragged", out_mode="discrete")
    xd1, xd2, xw1 = synth.make_dglu_inputs(d1), synth.make_dglu_inputs(d2), synth.make_wgrad_inputs(w1)
    ref_d1, ref_d2, ref_w1 = run_dglu_oracle(d1, xd1), run_dglu_oracle(d2, xd2), run_wgrad_oracle(w1, xw1)

    def dglu_call(spec, x):
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        keep = None
        if spec.b_mode == "dense":
            b_kw = dict(b=g["b"])
        else:
            keep = [t.to(dev) for t in x["b"]]
            b_kw = dict(b_ptrs=api.pointer_array(keep, dev), b_major=spec.b_major, N=spec.N)
        out = dict(d_row=torch.full((spec.M, 2 * spec.N), float("nan"), dtype=synth.torch_dtype(spec.d_dtype),
                                    device=dev),
                   dprob=torch.zeros(spec.M, device=dev),
                   dbias=torch.zeros(spec.L, 2 * spec.N, dtype=torch.bfloat16, device=dev) if spec.dbias else None,
                   ws=api.new_workspace(api.dglu_bwd_workspace_size(spec.L, spec.N), dev))

        def run():
            out["dprob"].zero_()
            if out["dbias"] is not None:
                out["dbias"].zero_()
            api.dglu_bwd(a=g["a"], c=g["c"], padded_offsets=g["padded_offsets"], alpha=g["alpha"], beta=g["beta"],
                         prob=g["prob"], dprob=out["dprob"], d_row=out["d_row"], dbias=out["dbias"], act=spec.act,
                         workspace=out["ws"], **b_kw)
        return run, out, keep

    def wgrad_call(spec, x):
        a, b, offs = x["a"].to(dev), x["b"].to(dev), x["offsets"].to(dev)
        outs = [torch.full((spec.hidden, spec.inter), float("nan"), device=dev) for _ in range(spec.L)]
        ptrs = api.pointer_array(outs, dev)
        out = dict(outs=outs, ws=api.new_workspace(api.wgrad_workspace_size(spec.L), dev))

        def run():
            api.wgrad(a=a, b=b, offsets=offs, hidden=spec.hidden, inter=spec.inter, out_ptrs=ptrs, out_dtype="fp32",
                      input_order=spec.input_order, workspace=out["ws"])
        return run, out, (a, b, offs, ptrs)

    r_d1, o_d1, k1 = dglu_call(d1, xd1)
    r_d2, o_d2, k2 = dglu_call(d2, xd2)
    r_w1, o_w1, k3 = wgrad_call(w1, xw1)
    r_w2, o_w2, k4 = wgrad_call(w1, xw1)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for _ in range(3):
        s1.wait_stream(torch.cuda.current_stream(dev))
        s2.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s1):
            r_d1()
            r_w1()
        with torch.cuda.stream(s2):
            r_w2()
            r_d2()
        torch.cuda.current_stream(dev).wait_stream(s1)
        torch.cuda.current_stream(dev).wait_stream(s2)
        torch.cuda.synchronize(dev)
        for o in (o_d1, o_d2, o_w1, o_w2):
            assert api.read_device_status(o["ws"]) == 0
        for spec, o, ref in ((d1, o_d1, ref_d1), (d2, o_d2, ref_d2)):
            rows = _ranges(spec)
            check_close("d_row", to_np(o["d_row"]), ref["d_row"], TOL[spec.d_dtype], rows)
            check_close("dprob", to_np(o["dprob"]), ref["dprob"], TOL_DPROB, rows)
            if spec.dbias:
                check_close("dbias", to_np(o["dbias"]), ref["dbias"], TOL["bf16"])
        for o in (o_w1, o_w2):
            for e in range(w1.L):
                check_close(f"wgrad[{e}]", to_np(o["outs"][e]), ref_w1[e], TOL["fp32"])
    del k1, k2, k3, k4
