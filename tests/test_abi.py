"""CPU tests of the C ABI: the library builds, loads, exports every symbol that
include/fa.h declares, and rejects bad arguments with the documented codes
before touching the GPU (all calls below fail validation, so no device is needed)."""
import os
import re

import pytest

from attn_bwd_gb300 import _lib
from attn_bwd_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
A = 0x100000       # a fake, 16-byte-aligned "device pointer": never dereferenced
W = 0x200000       # a fake, 256-byte-aligned workspace


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_strerror", "fa_last_device_error",
              "fa_bwd_preprocess", "fa_bwd_main", "fa_bwd_dq", "fa_selftest_wait_timeout"):
        assert s in syms, s


def test_library_exports_every_declared_symbol(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), f"{s} declared in include/fa.h but not exported"
        assert s in _lib._SIGNATURES, f"{s} has no binding"


def test_strerror_covers_all_codes(lib):
    for code in range(0, 12):
        assert _lib.fa_strerror(code) != "unknown fa_status"
    assert _lib.fa_strerror(1234) == "unknown fa_status"


def test_workspace_size_formula(lib):
    # 256 bytes for the call's abort word, then rows padded to 128: L*log2e and D (fp32 each),
    # plus the fp32 dQ accumulator in atomic mode
    rows = 2 * 4 * 128
    hdr = 256
    assert _lib.fa_bwd_workspace_size(2, 4, 4, 100, 100, 64, 1) == hdr + 2 * rows * 4
    assert _lib.fa_bwd_workspace_size(2, 4, 4, 100, 100, 64, 0) == hdr + 2 * rows * 4 + rows * 64 * 4
    assert _lib.fa_bwd_workspace_size(2, 4, 3, 100, 100, 64, 0) == 0     # GQA mismatch
    assert _lib.fa_bwd_workspace_size(2, 4, 4, 0, 100, 64, 0) == 0       # empty sequence
    assert _lib.fa_bwd_workspace_size(2, 4, 4, 100, 100, 100, 0) == 0    # head dim
    # other head dims use the accumulator width of the kernel that serves them (64 or 128)
    assert _lib.fa_bwd_workspace_size(2, 4, 4, 100, 100, 96, 0) == hdr + 2 * rows * 4 + rows * 128 * 4
    assert _lib.fa_bwd_workspace_size(2, 4, 4, 100, 100, 40, 0) == hdr + 2 * rows * 4 + rows * 64 * 4


def _bwd(**kw):
    args = dict(q=A, k=A, v=A, o=A, dO=A, lse=A, dq=A, dk=A, dv=A, B=1, Hq=2, Hkv=1, Nq=64, Nkv=64, d=64,
                scale=0.125, causal=0, dtype=_lib.FA_F16, deterministic=0, workspace=W, workspace_bytes=0)
    args.update(kw)
    return _lib.fa_bwd(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), _lib.FA_ERR_NULL),
    (dict(lse=None), _lib.FA_ERR_NULL),
    (dict(dv=None), _lib.FA_ERR_NULL),
    (dict(Nq=0), _lib.FA_ERR_SHAPE),
    (dict(Nkv=-3), _lib.FA_ERR_SHAPE),
    (dict(B=0), _lib.FA_ERR_SHAPE),
    (dict(Nq=(1 << 24) + 1), _lib.FA_ERR_SHAPE),
    (dict(d=100), _lib.FA_ERR_HEADDIM),
    (dict(d=4), _lib.FA_ERR_HEADDIM),
    (dict(d=136), _lib.FA_ERR_HEADDIM),
    (dict(d=256), _lib.FA_ERR_HEADDIM),
    (dict(Hq=3, Hkv=2), _lib.FA_ERR_GQA),
    (dict(dtype=7), _lib.FA_ERR_DTYPE),
    (dict(q=A + 8), _lib.FA_ERR_ALIGN),
    (dict(dk=A + 2), _lib.FA_ERR_ALIGN),
    (dict(workspace=None), _lib.FA_ERR_WORKSPACE),
    (dict(workspace=W + 16, workspace_bytes=1 << 30), _lib.FA_ERR_ALIGN),
    (dict(workspace_bytes=100), _lib.FA_ERR_WORKSPACE),
    (dict(scale=float("nan"), workspace_bytes=1 << 30), _lib.FA_ERR_ARG),
    (dict(scale=float("inf"), workspace_bytes=1 << 30), _lib.FA_ERR_ARG),
    (dict(causal=3, workspace_bytes=1 << 30), _lib.FA_ERR_ARG),
    (dict(causal=-1, workspace_bytes=1 << 30), _lib.FA_ERR_ARG),
])
def test_bwd_rejects_bad_arguments(lib, kw, code):
    assert _bwd(**kw) == code


def test_deterministic_workspace_is_smaller(lib):
    need_det = _lib.fa_bwd_workspace_size(1, 2, 1, 64, 64, 64, 1)
    need_atomic = _lib.fa_bwd_workspace_size(1, 2, 1, 64, 64, 64, 0)
    assert need_det < need_atomic
    # a deterministic-size workspace is too small for atomic mode
    assert _bwd(deterministic=0, workspace_bytes=need_det) == _lib.FA_ERR_WORKSPACE


def test_fwd_rejects_bad_arguments(lib):
    f = _lib.fa_fwd
    assert f(None, A, A, A, A, 1, 2, 1, 8, 8, 64, 0.1, 0, 0) == _lib.FA_ERR_NULL
    assert f(A, A, A, A, A, 1, 2, 1, 8, 8, 33, 0.1, 0, 0) == _lib.FA_ERR_HEADDIM
    assert f(A, A, A, A, A, 1, 3, 2, 8, 8, 64, 0.1, 0, 0) == _lib.FA_ERR_GQA
    assert f(A, A, A, A, A + 4, 1, 2, 1, 8, 8, 64, 0.1, 0, 0) == _lib.FA_ERR_ALIGN
    assert f(A, A, A, A, A, 1, 2, 1, 8, 8, 64, 0.1, 0, 2) == _lib.FA_ERR_DTYPE


def test_stage_entry_points_validate(lib):
    assert _lib.fa_bwd_preprocess(None, A, A, 1, 2, 1, 8, 8, 64, 0, 0, W, 1 << 30) == _lib.FA_ERR_NULL
    assert _lib.fa_bwd_main(A, A, A, A, A, A, 1, 2, 1, 8, 8, 64, 0.1, 0, 0, 0, W, 16) == _lib.FA_ERR_WORKSPACE
    assert _lib.fa_bwd_dq(A, A, A, A, None, 1, 2, 1, 8, 8, 64, 0.1, 0, 0, 1, W, 1 << 30) == _lib.FA_ERR_NULL
    assert _lib.fa_selftest_wait_timeout(0) == _lib.FA_ERR_ARG
    assert _lib.fa_selftest_wait_timeout(10_000_000) == _lib.FA_ERR_ARG


C = 0x300000       # fake, 4-byte-aligned device offset arrays


def _bwd_varlen(**kw):
    args = dict(q=A, k=A, v=A, o=A, dO=A, lse=A, dq=A, dk=A, dv=A, cu_q=C, cu_k=C + 64, B=2, Hq=2, Hkv=1,
                total_q=100, total_k=80, max_q=60, max_k=50, d=64, scale=0.125, causal=0, dtype=_lib.FA_BF16,
                deterministic=0, workspace=W, workspace_bytes=0)
    args.update(kw)
    return _lib.fa_bwd_varlen(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(cu_q=None), _lib.FA_ERR_NULL),
    (dict(cu_k=None), _lib.FA_ERR_NULL),
    (dict(dq=None), _lib.FA_ERR_NULL),
    (dict(cu_q=C + 2), _lib.FA_ERR_ALIGN),
    (dict(cu_k=C + 1), _lib.FA_ERR_ALIGN),
    (dict(q=A + 8), _lib.FA_ERR_ALIGN),
    (dict(total_q=0), _lib.FA_ERR_SHAPE),
    (dict(total_k=(1 << 30) + 1), _lib.FA_ERR_SHAPE),
    (dict(max_q=0), _lib.FA_ERR_SHAPE),
    (dict(max_k=(1 << 24) + 1), _lib.FA_ERR_SHAPE),
    (dict(B=0), _lib.FA_ERR_SHAPE),
    (dict(d=84), _lib.FA_ERR_HEADDIM),
    (dict(Hq=3, Hkv=2), _lib.FA_ERR_GQA),
    (dict(causal=5), _lib.FA_ERR_ARG),
    (dict(workspace_bytes=100), _lib.FA_ERR_WORKSPACE),
])
def test_bwd_varlen_rejects_bad_arguments(lib, kw, code):
    assert _bwd_varlen(**kw) == code


def test_fwd_varlen_rejects_bad_arguments(lib):
    f = _lib.fa_fwd_varlen
    ok = dict(q=A, k=A, v=A, o=A, lse=A, cu_q=C, cu_k=C, B=1, Hq=2, Hkv=1, total_q=10, total_k=10, max_q=10,
              max_k=10, d=64, scale=0.1, causal=1, dtype=0)
    assert f(**{**ok, "cu_k": None}) == _lib.FA_ERR_NULL
    assert f(**{**ok, "lse": A + 4}) == _lib.FA_ERR_ALIGN
    assert f(**{**ok, "total_q": -1}) == _lib.FA_ERR_SHAPE
    assert f(**{**ok, "scale": float("nan")}) == _lib.FA_ERR_ARG


def test_varlen_workspace_matches_dense_at_the_longest_length(lib):
    for det in (0, 1):
        assert (_lib.fa_bwd_varlen_workspace_size(3, 4, 2, 300, 200, 128, det)
                == _lib.fa_bwd_workspace_size(3, 4, 2, 300, 200, 128, det))


def _st(**over):
    base = dict(q=(4096, 1024, 64), k=(2048, 1024, 64), v=(2048, 1024, 64), o=(4096, 1024, 64),
                dO=(4096, 1024, 64), dq=(4096, 1024, 64), dk=(2048, 1024, 64), dv=(2048, 1024, 64),
                lse=(64, 16, 1))
    base.update(over)
    return _lib.make_strides(**base)


@pytest.mark.parametrize("over,code", [
    (dict(), None),
    (dict(q=(4096, 1024, 60)), _lib.FA_ERR_ARG),          # row stride not a multiple of 8 elements
    (dict(dk=(2048, 0, 64)), _lib.FA_ERR_ARG),            # zero head stride
    (dict(o=(-4096, 1024, 64)), _lib.FA_ERR_ARG),         # negative batch stride
    (dict(lse=(64, 16, 0)), _lib.FA_ERR_ARG),             # zero row stride of L
])
def test_bwd_strided_validates_strides(lib, over, code):
    st = _st(**over)
    # a workspace that is too small makes the valid layout stop at the workspace check instead
    r = _lib.fa_bwd_strided(A, A, A, A, A, A, A, A, A, st, None, None, 1, 2, 1, 16, 16, 0, 0, 64, 0.1, 0,
                            _lib.FA_BF16, 0, W, 16)
    assert r == (code if code is not None else _lib.FA_ERR_WORKSPACE)


def test_strided_offsets_must_come_in_pairs(lib):
    r = _lib.fa_fwd_strided(A, A, A, A, A, None, None, C, 1, 2, 1, 16, 16, 16, 16, 64, 0.1, 0, _lib.FA_BF16)
    assert r == _lib.FA_ERR_NULL


@pytest.mark.parametrize("kw,code", [
    (dict(bias=None, bs=(0, 0, 64)), _lib.FA_ERR_NULL),               # description without a bias
    (dict(bias=A + 8), _lib.FA_ERR_ALIGN),
    (dict(bs=(0, 0, 60)), _lib.FA_ERR_ARG),                          # query stride not a multiple of 8
    (dict(bs=(-8, 0, 64)), _lib.FA_ERR_ARG),
    (dict(dbias=A, dbs=(0, 4096, 64)), _lib.FA_ERR_ARG),             # dBias rows must not broadcast
    (dict(dbias=A + 4, dbs=(8192, 4096, 64)), _lib.FA_ERR_ALIGN),
])
def test_bwd_bias_validates(lib, kw, code):
    args = dict(bias=A, bs=(0, 0, 64), dbias=None, dbs=(0, 0, 0))
    args.update(kw)
    fb = _lib.make_bias(args["bias"], args["bs"], args["dbias"], args["dbs"])
    r = _lib.fa_bwd_bias(A, A, A, A, A, A, A, A, A, fb, None, None, None, 1, 2, 1, 64, 64, 0, 0, 64, 0.1, 1,
                         _lib.FA_BF16, 0, W, 1 << 30)
    assert r == code


def test_fwd_bias_takes_no_dbias(lib):
    fb = _lib.make_bias(A, (0, 0, 64), A, (8192, 4096, 64))
    assert _lib.fa_fwd_bias(A, A, A, A, A, fb, None, None, None, 1, 2, 1, 64, 64, 0, 0, 64, 0.1, 0,
                            _lib.FA_BF16) == _lib.FA_ERR_ARG


def test_host_pipeline_validation_and_staging_size(lib):
    # 5 sequences x 2 kv heads = 10 (batch, kv-head) groups of 2 query heads each
    one = _lib.fa_bwd_workspace_size(1, 2 * 3, 3, 100, 100, 64, 0)
    assert one > 0
    slot = _lib.fa_bwd_host_staging_size(5, 4, 2, 100, 100, 64, 0, 3, 1)
    assert slot > one
    assert _lib.fa_bwd_host_staging_size(5, 4, 2, 100, 100, 64, 0, 3, 2) == 2 * slot
    # never more slots than chunks: 10 groups in chunks of 3 -> 4 chunks
    assert _lib.fa_bwd_host_staging_size(5, 4, 2, 100, 100, 64, 0, 3, 8) == 4 * slot
    assert _lib.fa_bwd_host_staging_size(5, 4, 2, 100, 100, 64, 0, 10, 8) == \
        _lib.fa_bwd_host_staging_size(5, 4, 2, 100, 100, 64, 0, 10, 1)
    for cg, sl in ((0, 2), (11, 2), (3, 0), (3, _lib.FA_HOST_MAX_SLOTS + 1)):
        assert _lib.fa_bwd_host_staging_size(5, 4, 2, 100, 100, 64, 0, cg, sl) == 0
    assert _lib.fa_bwd_host_staging_size(5, 4, 3, 100, 100, 64, 0, 1, 2) == 0    # Hq % Hkv != 0
    args = [A] * 9 + [5, 4, 2, 100, 100, 64, 0.1, 1, _lib.FA_BF16, 0]
    assert _lib.fa_bwd_host(*args, 0, 2, W, 1 << 30) == _lib.FA_ERR_SHAPE
    assert _lib.fa_bwd_host(*args, 2, 0, W, 1 << 30) == _lib.FA_ERR_SHAPE
    assert _lib.fa_bwd_host(*args, 2, 2, None, 1 << 30) == _lib.FA_ERR_WORKSPACE
    assert _lib.fa_bwd_host(*args, 2, 2, W, 100) == _lib.FA_ERR_WORKSPACE
    assert _lib.fa_bwd_host(*args, 2, 2, W + 16, 1 << 30) == _lib.FA_ERR_ALIGN
    bad = [A] * 9 + [5, 4, 3, 100, 100, 64, 0.1, 1, _lib.FA_BF16, 0]
    assert _lib.fa_bwd_host(*bad, 1, 2, W, 1 << 30) == _lib.FA_ERR_GQA
    # dtype, scale and causal are rejected before any copy is queued (no CUDA call is made)
    base = [A] * 9 + [5, 4, 2, 100, 100, 64]
    assert _lib.fa_bwd_host(*base, 0.1, 1, 7, 0, 2, 2, W, 1 << 30) == _lib.FA_ERR_DTYPE
    assert _lib.fa_bwd_host(*base, float("nan"), 1, _lib.FA_BF16, 0, 2, 2, W, 1 << 30) == _lib.FA_ERR_ARG
    assert _lib.fa_bwd_host(*base, 0.1, 3, _lib.FA_BF16, 0, 2, 2, W, 1 << 30) == _lib.FA_ERR_ARG


def test_noalloc_checks_dtype_and_arguments_before_its_size_limit(lib):
    # the headline problem in atomic mode does not fit the static scratch ...
    assert _lib.fa_bwd_workspace_size(4, 32, 8, 8192, 8192, 128, 0) > _lib.FA_STATIC_SCRATCH_BYTES
    args = [A] * 9 + [4, 32, 8, 8192, 8192, 128]
    assert _lib.fa_bwd_noalloc(*args, 0.088, 1, _lib.FA_BF16, 0, None) == _lib.FA_ERR_WORKSPACE
    # ... but an unknown dtype, a scale that is not finite or an unknown causal mode is named first
    assert _lib.fa_bwd_noalloc(*args, 0.088, 1, 7, 0, None) == _lib.FA_ERR_DTYPE
    assert _lib.fa_bwd_noalloc(*args, float("nan"), 1, _lib.FA_BF16, 0, None) == _lib.FA_ERR_ARG
    assert _lib.fa_bwd_noalloc(*args, 0.088, 3, _lib.FA_BF16, 0, None) == _lib.FA_ERR_ARG
