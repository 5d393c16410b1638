"""The C ABI without a GPU: the library builds and loads, exports every entry
point its header declares, and rejects bad arguments on the host before
touching CUDA.

Every call below is built to fail validation, so no pointer it passes is ever
dereferenced and nothing reaches the GPU even when one is present.
"""

import ctypes
import os
import re

import pytest

import normalization_fwd_gb300 as nf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("normfuse.h", "normfuse_testing.h")]

OK, NULL, ALIGN, SHAPE, UNSUPPORTED, CUDA, WORKSPACE, INVALID, SCRATCH_LIMIT = range(9)


@pytest.fixture(scope="module")
def lib():
    nf.build_library()
    return nf.load_library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:ln_status|const char\*|int|size_t)\s+(ln_\w+)\s*\(",
                                text, flags=re.M))
    return sorted(names)


def test_every_header_is_checked():
    on_disk = sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))
    assert on_disk == sorted(os.path.basename(h) for h in HEADERS)


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(
        ["ln_fwd", "ln_fwd_ex", "ln_bwd", "ln_bwd_ex", "ln_bwd_workspace_bytes",
         "ln_status_string", "ln_last_cuda_error", "ln_device_error", "ln_bwd_noalloc",
         "ln_softmax_fwd", "ln_testing_select_kernels", "ln_fwd_from_partials",
         "ln_testing_plan"])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(nf.exported_symbols()) == declared_functions()


def test_binding_constants_match_the_header():
    text = re.sub(r"/\*.*?\*/", "", open(HEADERS[0]).read(), flags=re.S)
    enum = re.search(r"typedef enum \{([^{}]*)\} ln_status;", text, flags=re.S).group(1)
    codes = dict((k, int(v)) for k, v in re.findall(r"(LN_\w+)\s*=\s*(\d+)", enum))
    assert codes == {k: getattr(nf, k) for k in codes}
    assert len(codes) == 9
    m = re.search(r"#define LN_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert int(m.group(1)) << int(m.group(2)) == nf.LN_NOALLOC_SCRATCH_BYTES
    for k in ("LN_F32", "LN_BF16", "LN_F16"):
        assert re.search(rf"{k} = {getattr(nf, k)}\b", text), k


def test_status_strings(lib):
    for code in range(9):
        s = nf.ln_status_string(code)
        assert s.startswith("LN_"), s
    assert "unknown" in nf.ln_status_string(99)


# Fake, never-dereferenced device addresses (256-byte aligned like cudaMalloc).
X, RES, G, B, BIAS, S, Y, M, R, A = (0x7f0000000000 + i * 0x10000000 for i in range(10))


def fwd(lib, x=X, bias=BIAS, residual=RES, gamma=G, beta=B, eps=1e-5, mode=0, zc=0,
        out_sum=S, y=Y, mean=M, rstd=R, amax=A, rows=4, hidden=384, dtype=1):
    return lib.ln_fwd(x, bias, residual, gamma, beta, eps, mode, zc, out_sum, y, mean, rstd,
                      amax, None, rows, hidden, dtype)


@pytest.mark.parametrize("kw,want", [
    (dict(x=None), NULL),
    (dict(y=None), NULL),
    (dict(gamma=None), NULL),
    (dict(dtype=3), UNSUPPORTED),
    (dict(mode=2), UNSUPPORTED),
    (dict(rows=-1), SHAPE),
    (dict(hidden=0), SHAPE),
    (dict(hidden=16385), SHAPE),
    (dict(hidden=8200, dtype=0), SHAPE),           # fp32: 8192 max
    (dict(x=X + 1), ALIGN),                        # bf16 needs 2-byte alignment
    (dict(dtype=0, y=Y + 2), ALIGN),               # fp32 needs 4-byte alignment
    (dict(mean=M + 2), ALIGN),
    (dict(amax=A + 1), ALIGN),
    (dict(eps=float("nan")), INVALID),
    (dict(eps=-1.0), INVALID),
    (dict(eps=float("inf")), INVALID),
    (dict(y=X), INVALID),                          # output aliases input
    (dict(out_sum=Y + 64), INVALID),               # outputs overlap each other
    (dict(rstd=M + 8), INVALID),
    (dict(amax=G + 16), INVALID),
])
def test_fwd_rejects_on_host(lib, kw, want):
    assert fwd(lib, **kw) == want


def test_fwd_unaligned_hidden_beyond_scalar_limit_is_rejected(lib):
    # 16-byte misaligned rows fall to the scalar kernel, which stops at 8192.
    assert fwd(lib, x=X + 2, hidden=9000) == SHAPE
    assert fwd(lib, hidden=8194) == SHAPE          # 8194 * 2 bytes is not a multiple of 16


def bwd(lib, dy=X, xs=RES, gamma=G, mean=M, rstd=R, dx=Y, dg=S, db=B, rows=4, hidden=384,
        dtype=1, mode=0, zc=0, ws=A, ws_bytes=1 << 20):
    return lib.ln_bwd(dy, xs, gamma, mean, rstd, dx, dg, db, None, rows, hidden, dtype, mode,
                      zc, ws, ws_bytes)


@pytest.mark.parametrize("kw,want", [
    (dict(dy=None), NULL),
    (dict(xs=None), NULL),
    (dict(rstd=None), NULL),
    (dict(dx=None), NULL),
    (dict(dg=None), NULL),
    (dict(mean=None), NULL),                       # LayerNorm needs the mean
    (dict(dtype=-1), UNSUPPORTED),
    (dict(mode=5), UNSUPPORTED),
    (dict(rows=-3), SHAPE),
    (dict(hidden=0), SHAPE),
    (dict(dx=Y + 1), ALIGN),
    (dict(dg=S + 2), ALIGN),
    (dict(dx=X), INVALID),
    (dict(dg=M), INVALID),
    (dict(ws=R + 4), INVALID),
])
def test_bwd_rejects_on_host(lib, kw, want):
    assert bwd(lib, **kw) == want


def test_fwd_ex_validates_fp8_on_host(lib):
    F8, SC = 0x7f0000000000 + 12 * 0x10000000, 0x7f0000000000 + 13 * 0x10000000

    def call(y_fp8=F8, scale=SC, **kw):
        a = dict(x=X, bias=BIAS, residual=RES, gamma=G, beta=B, out_sum=S, y=Y, mean=M, rstd=R,
                 amax=A, rows=4, hidden=384, dtype=1)
        a.update(kw)
        return lib.ln_fwd_ex(a["x"], a["bias"], a["residual"], a["gamma"], a["beta"], 1e-5, 0, 0,
                             a["out_sum"], a["y"], a["mean"], a["rstd"], a["amax"], y_fp8, scale,
                             None, a["rows"], a["hidden"], a["dtype"])
    assert call(scale=None) == NULL            # a scale is required with y_fp8
    assert call(y_fp8=None, y=None) == NULL    # some output is required
    assert call(scale=SC + 2) == ALIGN
    assert call(y_fp8=X + 16) == INVALID       # overlaps x
    assert call(y_fp8=Y + 128) == INVALID      # overlaps y
    assert call(y_fp8=M) == INVALID            # overlaps mean


def test_bwd_ex_validates_dbias_on_host(lib):
    def call(dbias, **kw):
        a = dict(dy=X, xs=RES, gamma=G, mean=M, rstd=R, dx=Y, dg=S, db=B, rows=4, hidden=384,
                 dtype=1, mode=0, zc=0, ws=A, ws_bytes=1 << 20)
        a.update(kw)
        return lib.ln_bwd_ex(a["dy"], a["xs"], a["gamma"], a["mean"], a["rstd"], a["dx"], a["dg"],
                             a["db"], dbias, None, a["rows"], a["hidden"], a["dtype"], a["mode"],
                             a["zc"], a["ws"], a["ws_bytes"], a.get("gdt", 0))
    DBIAS = 0x7f0000000000 + 11 * 0x10000000
    assert call(DBIAS + 2) == ALIGN
    assert call(S + 16) == INVALID          # overlaps dgamma
    assert call(X + 64) == INVALID          # overlaps dy
    assert call(DBIAS, dy=None) == NULL
    assert call(DBIAS, gdt=3) == UNSUPPORTED       # grad_dtype must be f32, bf16 or f16
    assert call(DBIAS, gdt=1, dg=S + 1) == ALIGN    # bf16 grads need 2-byte alignment
    assert call(DBIAS, gdt=0, dg=S + 2) == ALIGN
    assert call(DBIAS, gdt=1, db=S + 512) == INVALID   # bf16 dgamma [384] is 768 bytes


@pytest.mark.parametrize("kw,want", [
    (dict(x=None), NULL),
    (dict(y=None), NULL),
    (dict(dtype=5), UNSUPPORTED),
    (dict(rows=-1), SHAPE),
    (dict(hidden=0), SHAPE),
    (dict(hidden=16385), SHAPE),
    (dict(hidden=8200, dtype=0), SHAPE),           # fp32: 8192 max
    (dict(x=X + 2, hidden=9000), SHAPE),           # unaligned rows: scalar path, 8192 max
    (dict(x=X + 1), ALIGN),
    (dict(y=Y + 2, dtype=0), ALIGN),
    (dict(y=X + 128), INVALID),                    # partial overlap (in place is y == x)
    (dict(x=Y + 768), INVALID),
])
def test_softmax_rejects_on_host(lib, kw, want):
    a = dict(x=X, y=Y, rows=4, hidden=384, dtype=1)
    a.update(kw)
    assert lib.ln_softmax_fwd(a["x"], a["y"], None, a["rows"], a["hidden"], a["dtype"]) == want


def test_rmsnorm_ignores_mean_and_dbeta(lib):
    # With mode = RMSNorm a NULL mean is fine; the call then fails on
    # something else (here a NULL dx), proving the mean was not required.
    assert bwd(lib, mode=1, mean=None, db=None, dx=None) == NULL
    assert bwd(lib, mode=1, mean=None, dx=Y + 1) == ALIGN


def test_workspace_query_on_host(lib):
    out = ctypes.c_size_t(123)
    assert lib.ln_bwd_workspace_bytes(0, 384, 1, 0, ctypes.byref(out)) == OK
    assert out.value == 0
    assert lib.ln_bwd_workspace_bytes(10, 384, 1, 0, None) == NULL
    assert lib.ln_bwd_workspace_bytes(-1, 384, 1, 0, ctypes.byref(out)) == SHAPE
    assert lib.ln_bwd_workspace_bytes(10, 0, 1, 0, ctypes.byref(out)) == SHAPE
    assert lib.ln_bwd_workspace_bytes(10, 384, 7, 0, ctypes.byref(out)) == UNSUPPORTED
    assert lib.ln_bwd_workspace_bytes(10, 20000, 1, 0, ctypes.byref(out)) == SHAPE


PS, PQ = 0x7f0100000000, 0x7f0110000000


def fwdp(lib, x=X, psum=PS, psq=PQ, n_tiles=3, tile_cols=128, kind=0, gamma=G, beta=B,
         eps=1e-5, mode=0, zc=0, y=Y, mean=M, rstd=R, amax=None, rows=8, hidden=384, dtype=1):
    return lib.ln_fwd_from_partials(x, psum, psq, n_tiles, tile_cols, kind, gamma, beta, eps,
                                    mode, zc, y, mean, rstd, amax, None, rows, hidden, dtype)


@pytest.mark.parametrize("kw,want", [
    ({"dtype": 7}, UNSUPPORTED),
    ({"mode": 3}, UNSUPPORTED),
    ({"kind": 2}, UNSUPPORTED),
    ({"rows": -1}, SHAPE),
    ({"hidden": 0}, SHAPE),
    ({"tile_cols": 0}, SHAPE),
    ({"n_tiles": 4}, SHAPE),                 # ceil(384 / 128) = 3
    ({"n_tiles": 2, "tile_cols": 100}, SHAPE),  # ceil(384 / 100) = 4
    ({"eps": -1.0}, INVALID),
    ({"eps": float("inf")}, INVALID),
    ({"gamma": None}, NULL),
    ({"x": None}, NULL),
    ({"psum": None}, NULL),
    ({"psq": None}, NULL),
    ({"y": None}, NULL),
    ({"psum": PS + 2}, ALIGN),
    ({"x": X + 1}, ALIGN),
    ({"y": X}, INVALID),                      # output overlaps an input
    ({"mean": PS}, INVALID),
])
def test_fwd_from_partials_rejects_on_host(lib, kw, want):
    assert fwdp(lib, **kw) == want


def test_kernel_family_hook_validates_on_host(lib):
    assert lib.ln_testing_select_kernels(2, 0, 0) == INVALID
    assert lib.ln_testing_select_kernels(0, -1, 0) == INVALID
    assert lib.ln_testing_select_kernels(0, 0, 0) == OK
    with pytest.raises(ValueError):
        nf.ln_testing_select_kernels(forward="registers")


def test_plan_hook_validates_on_host(lib):
    out = (ctypes.c_int * 6)()
    assert lib.ln_testing_plan(0, 16, 384, 1, 0, 1, None) == NULL
    assert lib.ln_testing_plan(4, 16, 384, 1, 0, 1, out) == UNSUPPORTED
    assert lib.ln_testing_plan(0, 16, 384, 7, 0, 1, out) == UNSUPPORTED
    assert lib.ln_testing_plan(1, 16, 384, 1, 5, 0, out) == UNSUPPORTED
    assert lib.ln_testing_plan(0, 0, 384, 1, 0, 1, out) == SHAPE
    assert lib.ln_testing_plan(0, 16, 0, 1, 0, 1, out) == SHAPE
    with pytest.raises(ValueError):
        nf.ln_testing_plan("sideways", 16, 384, 1)


def test_library_reads_no_environment():
    """Kernel choice depends on the arguments and the device only: no source
    of the library reads an environment variable."""
    csrc = os.path.join(ROOT, "normalization_fwd_gb300", "csrc")
    for name in os.listdir(csrc):
        if name.endswith((".cu", ".cuh", ".h")):
            assert "getenv" not in open(os.path.join(csrc, name)).read(), name


def test_device_error_query_rejects_null(lib):
    assert lib.ln_device_error(None, None) == NULL


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    mod = importlib.import_module("normalization_fwd_gb300")
    missing = str(tmp_path / "nope.so")
    saved = mod._lib
    mod._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            mod.load_library(missing)
    finally:
        mod._lib = saved


def test_cuda_errors_propagate_as_status_without_a_device(lib):
    # Where no CUDA device is usable, the calls that only query the device
    # (no launch, no pointer dereference) must return LN_ERR_CUDA and leave
    # the CUDA error code readable, never abort.
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible: covered by the GPU tests")
    out = ctypes.c_size_t(0)
    assert lib.ln_bwd_workspace_bytes(1024, 384, 1, 0, ctypes.byref(out)) == CUDA
    assert lib.ln_last_cuda_error() != 0
    flags = ctypes.c_uint(7)
    assert lib.ln_device_error(None, ctypes.byref(flags)) == CUDA
    out = (ctypes.c_int * 6)()
    assert lib.ln_testing_plan(0, 16, 384, 1, 0, 1, out) == CUDA
    assert nf.ln_status_string(CUDA).startswith("LN_ERR_CUDA")
