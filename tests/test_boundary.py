"""C-ABI boundary tests that need no GPU.

The library must load, export every function include/attn.h declares, and
reject bad arguments with the documented status code before any CUDA call.
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


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def call(shape, q=FAKE, k=FAKE * 2, v=FAKE * 3, mask=0, lens=0, bias=0, scale=0.125, dtype=A.ATTN_BF16,
         out=FAKE * 64):
    lib = A.load_library()
    sp = ctypes.byref(shape) if shape is not None else None
    return lib.attn_fwd(sp, q or None, k or None, v or None, mask, lens or None, bias or None,
                        ctypes.c_float(scale), dtype, out or None, None)


def test_null_shape(lib):
    assert call(None) == codes["ATTN_ERR_NULL"]


@pytest.mark.parametrize("kw", [dict(B=-1), dict(Hq=0), dict(Hkv=0), dict(D=0), dict(Sq=-2), dict(Sk=-1),
                                dict(Hq=6, Hkv=4)])
def test_bad_shapes(lib, kw):
    assert call(_shape(**kw)) == codes["ATTN_ERR_SHAPE"]


def test_bad_dtype(lib):
    assert call(_shape(), dtype=7) == codes["ATTN_ERR_DTYPE"]


@pytest.mark.parametrize("dtype,D", [(A.ATTN_BF16, 16), (A.ATTN_F16, 96), (A.ATTN_BF16, 256),
                                     (A.ATTN_F32, 8), (A.ATTN_F32, 48)])
def test_unsupported_head_dim(lib, dtype, D):
    assert call(_shape(D=D), dtype=dtype) == codes["ATTN_ERR_HEAD_DIM"]


@pytest.mark.parametrize("scale", [0.0, -0.5, math.inf, math.nan])
def test_bad_scale(lib, scale):
    assert call(_shape(), scale=scale) == codes["ATTN_ERR_SCALE"]


def test_bad_mask(lib):
    assert call(_shape(), mask=4) == codes["ATTN_ERR_MASK"]
    assert call(_shape(), mask=A.MASK_KEY_PADDING) == codes["ATTN_ERR_MASK"]
    assert call(_shape(), mask=A.MASK_CAUSAL | A.MASK_KEY_PADDING) == codes["ATTN_ERR_MASK"]


def test_bad_bias_dims(lib):
    assert call(_shape(B=2, bb=3), bias=FAKE * 200) == codes["ATTN_ERR_SHAPE"]
    assert call(_shape(Hq=4, Hkv=2, bh=2), bias=FAKE * 200) == codes["ATTN_ERR_SHAPE"]


def test_null_tensors(lib):
    assert call(_shape(), q=0) == codes["ATTN_ERR_NULL"]
    assert call(_shape(), out=0) == codes["ATTN_ERR_NULL"]
    assert call(_shape(), k=0) == codes["ATTN_ERR_NULL"]


def test_misaligned(lib):
    assert call(_shape(), q=FAKE + 8) == codes["ATTN_ERR_ALIGN"]
    assert call(_shape(), out=FAKE * 64 + 2) == codes["ATTN_ERR_ALIGN"]
    assert call(_shape(), bias=FAKE * 200 + 2) == codes["ATTN_ERR_ALIGN"]


def test_overlap(lib):
    # out == q, and out overlapping the tail of v
    assert call(_shape(), out=FAKE) == codes["ATTN_ERR_OVERLAP"]
    assert call(_shape(), v=FAKE * 64 - 16) == codes["ATTN_ERR_OVERLAP"]


def test_empty_problems_are_noops(lib):
    # B == 0 or Sq == 0: nothing to compute, nothing launched, success
    assert call(_shape(B=0)) == codes["ATTN_OK"]
    assert call(_shape(Sq=0)) == codes["ATTN_OK"]


def test_python_binding_missing_library_is_an_error(tmp_path, monkeypatch):
    monkeypatch.setattr(A, "_lib", None)
    monkeypatch.setattr(A, "_HERE", str(tmp_path))
    with pytest.raises(A.AttnError):
        A.load_library()
