"""The C-ABI library: it loads, exports what include/*.h declares, and its host-side
validation rejects malformed arguments before anything is queued (no GPU needed)."""
import ctypes
import glob
import os
import re

import pytest

from moe_grouped_gemm_persistent_gb300 import _lib
from moe_grouped_gemm_persistent_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(mgg_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "mgg_dglu_bwd" in names and "mgg_wgrad" in names and len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    bound = {s[0] for s in _lib.SIGNATURES}
    assert names <= bound, names - bound


def test_struct_layouts_match_library(lib):
    assert lib.mgg_abi_version() == 5
    assert lib.mgg_sizeof_dglu_bwd_args() == ctypes.sizeof(_lib.DgluBwdArgs)
    assert lib.mgg_sizeof_dsrelu_bwd_args() == ctypes.sizeof(_lib.DsreluBwdArgs)
    assert lib.mgg_sizeof_wgrad_args() == ctypes.sizeof(_lib.WgradArgs)


@pytest.mark.parametrize("which,struct", [(0, _lib.DgluBwdArgs), (1, _lib.DsreluBwdArgs), (2, _lib.WgradArgs)])
def test_struct_field_offsets_match_library(lib, which, struct):
    """Field by field: two swapped fields of equal size would pass a sizeof check."""
    n = lib.mgg_args_field_offsets(which, None, 0)
    assert n == len(struct._fields_)
    buf = (ctypes.c_size_t * n)()
    assert lib.mgg_args_field_offsets(which, buf, n) == n
    want = [getattr(struct, name).offset for name, _ in struct._fields_]
    assert list(buf) == want
    assert lib.mgg_args_field_offsets(3, None, 0) == -1


def test_struct_fields_follow_the_header_order():
    """The ctypes mirror lists the fields of include/mgg.h's structs in the header's order."""
    text = open(os.path.join(ROOT, "include", "mgg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    for cname, struct in (("mgg_dglu_bwd_args", _lib.DgluBwdArgs), ("mgg_dsrelu_bwd_args", _lib.DsreluBwdArgs),
                          ("mgg_wgrad_args", _lib.WgradArgs)):
        body = re.search(r"typedef struct %s \{(.*?)\} %s;" % (cname, cname), text, flags=re.S).group(1)
        names = []
        for decl in filter(None, (d.strip() for d in body.split(";"))):
            # "type a, b, c": the first declarator follows the type, the others follow commas
            parts = decl.split(",")
            names.append(re.split(r"[\s\*]+", parts[0].strip())[-1])
            names += [p.strip().lstrip("*") for p in parts[1:]]
        assert names == [f for f, _ in struct._fields_], cname


def test_sizes_and_tile_counts(lib):
    assert lib.mgg_dglu_bwd_workspace_size(4, 128) == 256 + 4 * 128 + 4 * 256 * 4
    assert lib.mgg_dsrelu_bwd_workspace_size(4) == 768  # 256-byte header + 4 tensor maps of 128 B
    assert lib.mgg_wgrad_workspace_size(64) % 256 == 0
    assert lib.mgg_wgrad_workspace_size(64) >= 256 + 3 * 64 * 128 + 64 * 4
    assert lib.mgg_dglu_bwd_num_tiles(1024, 128) == 8
    assert lib.mgg_dglu_bwd_num_tiles(33536, 14336) == 262 * 56
    assert lib.mgg_wgrad_num_tiles(64, 2048, 1408) == 64 * 16 * 6
    assert lib.mgg_wgrad_num_tiles(4, 256, 128) == 4 * 2 * 1
    assert lib.mgg_wgrad_num_tiles(256, 7168, 2048) == 256 * 56 * 8
    for s in range(9):
        assert lib.mgg_status_string(s).decode().startswith("MGG_")
    assert lib.mgg_status_string(8).decode() == "MGG_ERR_DEVICE_BOUNDS"


FAKE = 1 << 20  # an aligned address; validation never dereferences pointers


def dglu_args(**over):
    a = _lib.DgluBwdArgs()
    a.M, a.K, a.N, a.L = 1024, 256, 128, 4
    for f in ("a", "b", "c", "padded_offsets", "alpha", "beta", "prob", "dprob", "d_row", "workspace"):
        setattr(a, f, FAKE)
    a.workspace_bytes = 1 << 20
    a.gate_first = 1
    for k, v in over.items():
        setattr(a, k, v)
    return a


def dsrelu_args(**over):
    a = _lib.DsreluBwdArgs()
    a.M, a.K, a.N, a.L = 1024, 256, 128, 4
    for f in ("a", "b", "c", "padded_offsets", "alpha", "prob", "dprob", "d_row", "workspace"):
        setattr(a, f, FAKE)
    a.workspace_bytes = 1 << 20
    for k, v in over.items():
        setattr(a, k, v)
    return a


def wgrad_args(**over):
    a = _lib.WgradArgs()
    a.hidden, a.inter, a.L, a.tokens_sum = 256, 128, 4, 1024
    for f in ("a", "b", "offsets", "out", "workspace"):
        setattr(a, f, FAKE)
    a.workspace_bytes = 1 << 20
    a.out_dtype = 2
    a.b_major = 1
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,expect", [
    (dict(L=0), 1), (dict(L=1025), 1), (dict(M=1000), 1), (dict(K=100), 1), (dict(N=48), 1),
    (dict(b_ptrs=FAKE), 1), (dict(b=None), 1), (dict(b_major=1), 1), (dict(c_dtype=3), 1),
    (dict(d_dtype=-1), 1), (dict(act=3), 1), (dict(act=2, situ_beta1=-1.0), 1), (dict(act=2, situ_beta2=float("inf")), 1), (dict(geglu_filter=5), 1), (dict(gate_first=2), 1),
    (dict(a=FAKE + 8), 1), (dict(c=None), 1), (dict(dprob=FAKE + 4), 1), (dict(workspace=FAKE + 16), 1),
    (dict(workspace_bytes=100), 1), (dict(cta_mode=3), 1), (dict(cta_mode=-1), 1), (dict(dbias=FAKE + 2), 1),
    (dict(sched=7), 1), (dict(sched=-1), 1),
])
def test_dglu_validation_rejects_before_launch(lib, over, expect):
    st = lib.mgg_dglu_bwd(dglu_args(**over), None)
    assert st == expect, lib.mgg_last_error()
    assert lib.mgg_last_error()


@pytest.mark.parametrize("over,expect", [
    (dict(L=0), 1), (dict(hidden=100), 1), (dict(inter=4), 1), (dict(tokens_sum=1000), 1),
    (dict(out_ptrs=FAKE), 1), (dict(out=None), 1), (dict(a_major=3), 1), (dict(input_order=2), 1),
    (dict(out_dtype=9), 1), (dict(accumulate=2), 1), (dict(b=FAKE + 8), 1), (dict(offsets=None), 1),
    (dict(workspace_bytes=8), 1), (dict(reserved1=1), 1), (dict(sched=2), 1), (dict(cta_mode=3), 1),
    (dict(cta_mode=2, hidden=128), 1),
])
def test_wgrad_validation_rejects_before_launch(lib, over, expect):
    st = lib.mgg_wgrad(wgrad_args(**over), None)
    assert st == expect, lib.mgg_last_error()


def test_null_args(lib):
    assert lib.mgg_dglu_bwd(None, None) == 1
    assert lib.mgg_wgrad(None, None) == 1


def test_valid_args_without_device_report_arch(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.mgg_dglu_bwd(dglu_args(), None) == _lib.MGG_ERR_ARCH
    assert lib.mgg_wgrad(wgrad_args(), None) == _lib.MGG_ERR_ARCH


def test_empty_calls_accept_null_per_row_tensors(lib):
    """Without rows (M == 0) or tokens (tokens_sum == 0) the per-row tensors may be NULL: the host
    check passes them (no device here: the call then reports MGG_ERR_ARCH); with rows they may not."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rows = dict(a=None, c=None, prob=None, dprob=None, d_row=None)
    assert lib.mgg_dglu_bwd(dglu_args(M=0, **rows), None) == _lib.MGG_ERR_ARCH
    assert lib.mgg_dsrelu_bwd(dsrelu_args(M=0, **rows), None) == _lib.MGG_ERR_ARCH
    assert lib.mgg_wgrad(wgrad_args(tokens_sum=0, a=None, b=None), None) == _lib.MGG_ERR_ARCH
    for f in rows:
        assert lib.mgg_dglu_bwd(dglu_args(**{f: None}), None) == _lib.MGG_ERR_VALUE, f
    assert lib.mgg_wgrad(wgrad_args(a=None), None) == _lib.MGG_ERR_VALUE
    assert lib.mgg_wgrad(wgrad_args(b=None), None) == _lib.MGG_ERR_VALUE
    # the rest stays required without rows
    assert lib.mgg_dglu_bwd(dglu_args(M=0, padded_offsets=None), None) == _lib.MGG_ERR_VALUE
    assert lib.mgg_wgrad(wgrad_args(tokens_sum=0, offsets=None), None) == _lib.MGG_ERR_VALUE


@pytest.mark.parametrize("over,expect", [
    (dict(L=0), 1), (dict(M=1000), 1), (dict(K=100), 1), (dict(N=48), 1), (dict(b_ptrs=FAKE), 1), (dict(b=None), 1),
    (dict(b_major=1), 1), (dict(c_dtype=2), 2), (dict(c_dtype=7), 1), (dict(d_dtype=-1), 1), (dict(a=FAKE + 8), 1),
    (dict(c=None), 1), (dict(d_col=FAKE + 4), 1), (dict(amax=FAKE + 4), 1), (dict(workspace_bytes=512), 1),
    (dict(workspace=FAKE + 16), 1), (dict(sched=3), 1), (dict(cta_mode=5), 1), (dict(reserved=1), 1),
])
def test_dsrelu_validation_rejects_before_launch(lib, over, expect):
    st = lib.mgg_dsrelu_bwd(dsrelu_args(**over), None)
    assert st == expect, lib.mgg_last_error()
    assert lib.mgg_last_error()


def test_dglu_validation_of_new_outputs(lib):
    assert lib.mgg_dglu_bwd(dglu_args(d_col=FAKE + 8), None) == 1
    assert lib.mgg_dglu_bwd(dglu_args(amax=FAKE + 4), None) == 1
