"""C-ABI boundary tests that need no GPU.

The library must load, export every function include/attn.h declares, and
reject bad arguments with the documented status code before any CUDA call.

The argument-validation cases hand the entry points made-up addresses that
are never dereferenced because validation rejects the call first. They run
only where no GPU is visible: on a machine with a GPU a regression in the
order of validation and launch could otherwise start a kernel on addresses
nobody owns. (The GPU tier checks the same rejections with real buffers.)
"""
import ctypes
import math
import os
import re

import pytest

from exact_scaled_dot_flash_gb300 import attn as A

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

codes = {}
for m in re.finditer(r"(ATTN_(?:OK|ERR_[A-Z_]+))\s*=\s*(-?\d+)", open(HEADER).read()):
    codes[m.group(1)] = int(m.group(2))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(A.library_path()):
        from exact_scaled_dot_flash_gb300 import build
        build.build()
    return A.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert {"attn_fwd", "attn_strerror", "attn_last_cuda_error", "attn_device_status",
            "attn_version"} <= set(declared_functions())


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libattn.so does not export {name}"


def test_strerror_and_version(lib):
    for name, code in codes.items():
        s = A.strerror(code)
        assert isinstance(s, str) and s and s != "unknown status code", name
    assert A.strerror(12345) == "unknown status code"
    assert lib.attn_version() >= 10000


def _shape(B=1, Hq=2, Hkv=2, Sq=8, Sk=8, D=64, bb=1, bh=1):
    return A.Shape(B, Hq, Hkv, Sq, Sk, D, bb, bh)


FAKE = 1 << 16  # 16-byte aligned, never dereferenced: validation fails first


def _gpu_visible():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


# made-up addresses only where no kernel can be launched on them
no_gpu_only = pytest.mark.skipif(_gpu_visible(), reason="made-up device addresses are passed only "
                                                       "where no GPU is visible")


def call(shape, q=FAKE, k=FAKE * 2, v=FAKE * 3, mask=0, lens=0, bias=0, scale=0.125, dtype=A.ATTN_BF16,
         out=FAKE * 64):
    lib = A.load_library()
    sp = ctypes.byref(shape) if shape is not None else None
    return lib.attn_fwd(sp, q or None, k or None, v or None, mask, lens or None, bias or None,
                        ctypes.c_float(scale), dtype, out or None, None)


@no_gpu_only
def test_null_shape(lib):
    assert call(None) == codes["ATTN_ERR_NULL"]


@no_gpu_only
@pytest.mark.parametrize("kw", [dict(B=-1), dict(Hq=0), dict(Hkv=0), dict(D=0), dict(Sq=-2), dict(Sk=-1),
                                dict(Hq=6, Hkv=4)])
def test_bad_shapes(lib, kw):
    assert call(_shape(**kw)) == codes["ATTN_ERR_SHAPE"]


@no_gpu_only
def test_bad_dtype(lib):
    assert call(_shape(), dtype=7) == codes["ATTN_ERR_DTYPE"]


@no_gpu_only
@pytest.mark.parametrize("dtype,D", [(A.ATTN_BF16, 16), (A.ATTN_F16, 96), (A.ATTN_BF16, 256),
                                     (A.ATTN_F32, 8), (A.ATTN_F32, 48)])
def test_unsupported_head_dim(lib, dtype, D):
    assert call(_shape(D=D), dtype=dtype) == codes["ATTN_ERR_HEAD_DIM"]


@no_gpu_only
@pytest.mark.parametrize("scale", [0.0, -0.5, math.inf, math.nan])
def test_bad_scale(lib, scale):
    assert call(_shape(), scale=scale) == codes["ATTN_ERR_SCALE"]


@no_gpu_only
def test_bad_mask(lib):
    assert call(_shape(), mask=4) == codes["ATTN_ERR_MASK"]
    assert call(_shape(), mask=A.MASK_KEY_PADDING) == codes["ATTN_ERR_MASK"]
    assert call(_shape(), mask=A.MASK_CAUSAL | A.MASK_KEY_PADDING) == codes["ATTN_ERR_MASK"]


@no_gpu_only
def test_bad_bias_dims(lib):
    assert call(_shape(B=2, bb=3), bias=FAKE * 200) == codes["ATTN_ERR_SHAPE"]
    assert call(_shape(Hq=4, Hkv=2, bh=2), bias=FAKE * 200) == codes["ATTN_ERR_SHAPE"]


@no_gpu_only
def test_null_tensors(lib):
    assert call(_shape(), q=0) == codes["ATTN_ERR_NULL"]
    assert call(_shape(), out=0) == codes["ATTN_ERR_NULL"]
    assert call(_shape(), k=0) == codes["ATTN_ERR_NULL"]


@no_gpu_only
def test_misaligned(lib):
    assert call(_shape(), q=FAKE + 8) == codes["ATTN_ERR_ALIGN"]
    assert call(_shape(), out=FAKE * 64 + 2) == codes["ATTN_ERR_ALIGN"]
    assert call(_shape(), bias=FAKE * 200 + 2) == codes["ATTN_ERR_ALIGN"]


@no_gpu_only
def test_overlap(lib):
    # out == q, and out overlapping the tail of v
    assert call(_shape(), out=FAKE) == codes["ATTN_ERR_OVERLAP"]
    assert call(_shape(), v=FAKE * 64 - 16) == codes["ATTN_ERR_OVERLAP"]


@no_gpu_only
def test_empty_problems_are_noops(lib):
    # B == 0 or Sq == 0: nothing to compute, nothing launched, success
    assert call(_shape(B=0)) == codes["ATTN_OK"]
    assert call(_shape(Sq=0)) == codes["ATTN_OK"]


def test_python_binding_missing_library_is_an_error(tmp_path, monkeypatch):
    monkeypatch.setattr(A, "_lib", None)
    monkeypatch.setattr(A, "_HERE", str(tmp_path))
    with pytest.raises(A.AttnError):
        A.load_library()


def call_split(shape, ns=2, ws=FAKE * 512, ws_bytes=1 << 30, lse=0, **kw):
    """attn_fwd_split with fake, never-dereferenced pointers (validation only)."""
    lib = A.load_library()
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, mask=0, lens=0, bias=0, scale=0.125, dtype=A.ATTN_BF16,
             out=FAKE * 64)
    a.update(kw)
    return lib.attn_fwd_split(ctypes.byref(shape), a["q"] or None, a["k"] or None, a["v"] or None, a["mask"],
                              a["lens"] or None, a["bias"] or None, ctypes.c_float(a["scale"]), a["dtype"],
                              ns, ws or None, ws_bytes, a["out"] or None, lse or None, None)


def ws_bytes(shape, ns):
    n = ctypes.c_size_t(0)
    rc = A.load_library().attn_split_workspace_bytes(ctypes.byref(shape), ns, ctypes.byref(n))
    return rc, n.value


def test_split_workspace_size(lib):
    s = _shape(B=2, Hq=3, Hkv=1, Sq=5, Sk=100, D=32)
    assert ws_bytes(s, 1) == (0, 0)
    rc, n = ws_bytes(s, 3)
    rows = 3 * 2 * 3 * 5
    o_bytes = rows * 32 * 4
    assert rc == 0 and n == (o_bytes + 255) // 256 * 256 + rows * 8
    assert ws_bytes(s, 0)[0] == codes["ATTN_ERR_SPLITS"]
    assert ws_bytes(s, 33)[0] == codes["ATTN_ERR_SPLITS"]
    assert ws_bytes(_shape(D=0), 2)[0] == codes["ATTN_ERR_SHAPE"]
    assert lib.attn_split_workspace_bytes(ctypes.byref(s), 2, None) == codes["ATTN_ERR_NULL"]


@no_gpu_only
@pytest.mark.parametrize("ns", [0, -1, 33, 1000])
def test_split_count_out_of_range(lib, ns):
    assert call_split(_shape(), ns=ns) == codes["ATTN_ERR_SPLITS"]


@no_gpu_only
def test_split_workspace_errors(lib):
    s = _shape()
    need = ws_bytes(s, 4)[1]
    assert call_split(s, ns=4, ws=0) == codes["ATTN_ERR_WORKSPACE"]
    assert call_split(s, ns=4, ws_bytes=need - 1) == codes["ATTN_ERR_WORKSPACE"]
    assert call_split(s, ns=4, ws=FAKE * 512 + 8, ws_bytes=need) == codes["ATTN_ERR_ALIGN"]
    # the workspace overlapping q, or the output
    assert call_split(s, ns=4, ws=FAKE, ws_bytes=need) == codes["ATTN_ERR_OVERLAP"]
    assert call_split(s, ns=4, ws=FAKE * 64, ws_bytes=need) == codes["ATTN_ERR_OVERLAP"]


@no_gpu_only
def test_split_lse_errors(lib):
    s = _shape()
    assert call_split(s, ns=1, ws=0, lse=FAKE * 300 + 2) == codes["ATTN_ERR_ALIGN"]
    assert call_split(s, ns=1, ws=0, lse=FAKE * 64) == codes["ATTN_ERR_OVERLAP"]  # lse inside out
    assert call_split(s, ns=2, ws=FAKE * 300, ws_bytes=1 << 20, lse=FAKE * 300 + 64) == \
        codes["ATTN_ERR_OVERLAP"]  # lse inside the workspace


@no_gpu_only
def test_split_empty_problem_is_noop(lib):
    assert call_split(_shape(B=0), ns=8, ws=0) == codes["ATTN_OK"]
    assert call_split(_shape(Sq=0), ns=8, ws=0) == codes["ATTN_OK"]


def test_library_exports_only_the_c_abi(lib):
    # hidden visibility: kernels and helpers stay internal, so two builds of
    # the library loaded in one process never bind to each other's kernels
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", A.library_path()], capture_output=True, text=True,
                         check=True).stdout
    names = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    names = {n for n in names if not n.startswith("_")}  # linker-provided markers
    assert names == set(declared_functions())


def _host_ws(lib, shape, dtype=A.ATTN_BF16, bias=False):
    n = ctypes.c_size_t(0)
    rc = lib.attn_fwd_host_workspace_bytes(ctypes.byref(shape), dtype, int(bias), ctypes.byref(n))
    return rc, n.value


def test_host_workspace_holds_two_chunk_slots(lib):
    # headline-sized problem: 4 batches x 32 kv heads in 8 chunks of 16 heads
    rc, n = _host_ws(lib, _shape(B=4, Hq=32, Hkv=32, Sq=4096, Sk=4096, D=128))
    assert rc == 0
    chunk = 16 * 4096 * 128 * 2                       # Q, K, V or O of one chunk
    assert 2 * 4 * chunk <= n <= 2 * 4 * chunk + 4096   # two slots of Q, K, V, O (+ padding)
    # a per-head bias adds one bias slice per slot; a broadcast bias one row block
    rc, nb = _host_ws(lib, _shape(B=4, Hq=32, Hkv=32, Sq=512, Sk=512, D=64, bb=1, bh=32), bias=True)
    rc0, n0 = _host_ws(lib, _shape(B=4, Hq=32, Hkv=32, Sq=512, Sk=512, D=64))
    assert rc == rc0 == 0 and nb - n0 >= 2 * 16 * 512 * 512 * 4
    rc, n1 = _host_ws(lib, _shape(B=4, Hq=32, Hkv=32, Sq=512, Sk=512, D=64, bb=4, bh=1), bias=True)
    assert rc == 0 and 2 * 512 * 512 * 4 <= n1 - n0 < 2 * 16 * 512 * 512 * 4
    # GQA: a chunk carries whole groups of query heads
    rc, ng = _host_ws(lib, _shape(B=1, Hq=32, Hkv=8, Sq=256, Sk=1024, D=128))
    assert rc == 0 and ng >= 2 * (2 * 4 * 256 * 128 * 2 + 2 * 1024 * 128 * 2)
    # F32 doubles the element size
    rc, nf = _host_ws(lib, _shape(B=2, Hq=4, Hkv=4, Sq=64, Sk=64, D=64), dtype=A.ATTN_F32)
    rc2, nh = _host_ws(lib, _shape(B=2, Hq=4, Hkv=4, Sq=64, Sk=64, D=64), dtype=A.ATTN_F16)
    assert rc == rc2 == 0 and nf > nh


def test_host_workspace_errors_and_empty(lib):
    assert _host_ws(lib, _shape(B=0))[1] == 0 and _host_ws(lib, _shape(B=0))[0] == 0
    assert _host_ws(lib, _shape(Sq=0)) == (0, 0)
    assert _host_ws(lib, _shape(Hq=3, Hkv=2))[0] == codes["ATTN_ERR_SHAPE"]
    assert _host_ws(lib, _shape(B=2, bb=3), bias=True)[0] == codes["ATTN_ERR_SHAPE"]
    assert _host_ws(lib, _shape(), dtype=7)[0] == codes["ATTN_ERR_DTYPE"]
    n = ctypes.c_size_t(0)
    assert lib.attn_fwd_host_workspace_bytes(None, 0, 0, ctypes.byref(n)) == codes["ATTN_ERR_NULL"]


@no_gpu_only
def test_host_call_argument_errors(lib):
    # rejected before any CUDA call (host pointers never dereferenced)
    s = _shape(B=2, Hq=2, Hkv=2, Sq=8, Sk=8, D=64)
    rc, need = _host_ws(lib, s)

    def call(shape=s, ws=FAKE, nbytes=need, out=FAKE * 8, scale=0.125, dtype=A.ATTN_BF16, mask=0):
        return lib.attn_fwd_host(ctypes.byref(shape), FAKE, FAKE * 2, FAKE * 3, mask, None, None,
                                 ctypes.c_float(scale), dtype, ws, nbytes, out, None)
    assert call(ws=None) == codes["ATTN_ERR_WORKSPACE"]
    assert call(nbytes=need - 1) == codes["ATTN_ERR_WORKSPACE"]
    assert call(ws=FAKE + 4) == codes["ATTN_ERR_ALIGN"]
    assert call(out=FAKE) == codes["ATTN_ERR_OVERLAP"]
    assert call(scale=-1.0) == codes["ATTN_ERR_SCALE"]
    assert call(mask=A.MASK_KEY_PADDING) == codes["ATTN_ERR_MASK"]
    assert call(shape=_shape(B=2, D=48)) == codes["ATTN_ERR_HEAD_DIM"]
    assert call(out=None) == codes["ATTN_ERR_NULL"]
    assert call(shape=_shape(B=0)) == 0


def _r256(x):
    return (x + 255) // 256 * 256


def test_paged_bwd_workspace_layout(lib):
    # row statistics (2 x rows floats), page counts, page offsets, the index,
    # the list of pages without exactly one reader
    s = A.PagedShape(3, 10, 4, 2, 64, 16, 7, 5, 4)
    n = ctypes.c_size_t(0)
    assert lib.attn_paged_bwd_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == 0
    assert n.value == 2 * _r256(40 * 4) + _r256(7 * 4) + _r256(8 * 4) + _r256(15 * 4) + _r256(8 * 4)
    m = A.MlaShape(3, 10, 16, 512, 64, 64, 700, 50, 4)
    assert lib.attn_paged_mla_bwd_workspace_bytes(ctypes.byref(m), ctypes.byref(n)) == 0
    assert n.value == 2 * _r256(160 * 4) + _r256(700 * 4) + _r256(701 * 4) + _r256(150 * 4) + _r256(701 * 4)
    assert lib.attn_paged_bwd_workspace_bytes(None, ctypes.byref(n)) == codes["ATTN_ERR_NULL"]
    bad = A.PagedShape(3, -1, 4, 2, 64, 16, 7, 5, 4)
    assert lib.attn_paged_bwd_workspace_bytes(ctypes.byref(bad), ctypes.byref(n)) == codes["ATTN_ERR_SHAPE"]


def _paged_bwd_call(lib, shape, ws=FAKE * 40, nbytes=1 << 20, dq=FAKE * 30, dk=FAKE * 31, dv=FAKE * 32,
                    dtype=A.ATTN_BF16, causal=1, scale=0.125, lse=FAKE * 12, table=FAKE * 20):
    # q, k, v, out, dout at FAKE x 1..5; metadata at FAKE x 20..23 (never dereferenced)
    return lib.attn_paged_bwd(ctypes.byref(shape), FAKE, FAKE * 2, FAKE * 3, table or None, FAKE * 21, FAKE * 22,
                              None, causal, ctypes.c_float(scale), dtype, FAKE * 4, FAKE * 5, lse or None,
                              ws or None, nbytes, dq or None, dk or None, dv or None, None)


@no_gpu_only
def test_paged_bwd_argument_errors(lib):
    s = A.PagedShape(2, 4, 2, 2, 64, 16, 3, 2, 2)
    n = ctypes.c_size_t(0)
    lib.attn_paged_bwd_workspace_bytes(ctypes.byref(s), ctypes.byref(n))
    need = n.value
    assert _paged_bwd_call(lib, s, ws=0) == codes["ATTN_ERR_WORKSPACE"]
    assert _paged_bwd_call(lib, s, nbytes=need - 1) == codes["ATTN_ERR_WORKSPACE"]
    assert _paged_bwd_call(lib, s, ws=FAKE * 40 + 4) == codes["ATTN_ERR_ALIGN"]
    assert _paged_bwd_call(lib, s, dq=FAKE * 4) == codes["ATTN_ERR_OVERLAP"]        # dq on out
    assert _paged_bwd_call(lib, s, dk=FAKE * 30) == codes["ATTN_ERR_OVERLAP"]       # dk on dq
    assert _paged_bwd_call(lib, s, ws=FAKE * 32) == codes["ATTN_ERR_OVERLAP"]       # workspace on dv
    assert _paged_bwd_call(lib, s, lse=0) == codes["ATTN_ERR_NULL"]
    assert _paged_bwd_call(lib, s, table=0) == codes["ATTN_ERR_NULL"]
    assert _paged_bwd_call(lib, s, dtype=9) == codes["ATTN_ERR_DTYPE"]
    assert _paged_bwd_call(lib, s, causal=2) == codes["ATTN_ERR_MASK"]
    assert _paged_bwd_call(lib, s, scale=float("inf")) == codes["ATTN_ERR_SCALE"]
    assert _paged_bwd_call(lib, A.PagedShape(2, 4, 2, 2, 96, 16, 3, 2, 2)) == codes["ATTN_ERR_HEAD_DIM"]
    assert _paged_bwd_call(lib, A.PagedShape(2, 4, 3, 2, 64, 16, 3, 2, 2)) == codes["ATTN_ERR_SHAPE"]
    # nothing asked for: validated, then a no-op (no workspace needed)
    assert _paged_bwd_call(lib, s, ws=0, dq=0, dk=0, dv=0) == codes["ATTN_OK"]


@no_gpu_only
def test_paged_mla_bwd_argument_errors(lib):
    m = A.MlaShape(2, 4, 8, 256, 64, 16, 3, 2, 2)

    def call(shape=m, ws=FAKE * 40, nbytes=1 << 20, dqp=FAKE * 33, qp=FAKE * 6, dtype=A.ATTN_BF16):
        return lib.attn_paged_mla_bwd(ctypes.byref(shape), FAKE, qp or None, FAKE * 2, FAKE * 3, FAKE * 20,
                                      FAKE * 21, FAKE * 22, None, 1, ctypes.c_float(0.1), dtype, FAKE * 4, FAKE * 5,
                                      FAKE * 12, ws or None, nbytes, FAKE * 30, dqp or None, FAKE * 31, FAKE * 32,
                                      None)
    assert call(ws=0) == codes["ATTN_ERR_WORKSPACE"]
    assert call(qp=0) == codes["ATTN_ERR_NULL"]
    assert call(dqp=FAKE * 6) == codes["ATTN_ERR_OVERLAP"]
    assert call(shape=A.MlaShape(2, 4, 8, 192, 64, 16, 3, 2, 2)) == codes["ATTN_ERR_HEAD_DIM"]
    assert call(shape=A.MlaShape(2, 4, 8, 256, 48, 16, 3, 2, 2)) == codes["ATTN_ERR_HEAD_DIM"]
    assert call(dtype=5) == codes["ATTN_ERR_DTYPE"]
