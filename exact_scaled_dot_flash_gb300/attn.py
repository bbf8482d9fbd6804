"""ctypes binding of libattn.so (``include/attn.h``): argument marshalling only.

Every arithmetic step runs in the CUDA kernels behind ``attn_fwd``; this
module checks tensor devices, dtypes and contiguity, allocates the output with
PyTorch (PyTorch is used for device memory and streams only) and passes raw
pointers plus the current CUDA stream. When the library is missing the call
raises; there is no CPU fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBNAME = "libattn.so"
_lock = threading.Lock()
_lib = None

ATTN_F32, ATTN_F16, ATTN_BF16 = 0, 1, 2
MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING = 0, 1, 2


class AttnError(RuntimeError):
    """Raised when attn_fwd returns an error code or the library is missing."""

    def __init__(self, msg, code=None):
        super().__init__(msg)
        self.code = code


class Shape(ctypes.Structure):
    """attn_shape_t."""
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "Hq", "Hkv", "Sq", "Sk", "D", "bias_b", "bias_h")]


class PagedShape(ctypes.Structure):
    """attn_paged_shape_t."""
    _fields_ = [(n, ctypes.c_int32) for n in ("num_seqs", "num_queries", "Hq", "Hkv", "D", "page_size",
                                               "num_pages", "max_pages", "max_queries")]


class MlaShape(ctypes.Structure):
    """attn_mla_shape_t."""
    _fields_ = [(n, ctypes.c_int32) for n in ("num_seqs", "num_queries", "H", "R", "Pd", "page_size",
                                               "num_pages", "max_pages", "max_queries")]


def library_path() -> str:
    return os.path.join(_HERE, _LIBNAME)


def checked_library_path() -> str:
    """Path of the bounds-checked build (``build.build(checked=True)``)."""
    return os.path.join(_HERE, "libattn_checked.so")


def load_library():
    """Open libattn.so once; raise AttnError if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(library_path())
        return _lib


@contextlib.contextmanager
def use_library(path):
    """Route every call of this module through the library build at ``path``
    (for example the bounds-checked libattn_checked.so) while the block runs;
    its device status word is then the one :func:`device_status` reads."""
    global _lib
    lib = _open(path)
    with _lock:
        prev, _lib = _lib, lib
    try:
        yield lib
    finally:
        with _lock:
            _lib = prev


def _open(path):
    """Open a build of the library and declare its C signatures."""
    if not os.path.exists(path):
        raise AttnError(f"{path} is missing: build the CUDA library first "
                        "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    lib.attn_fwd.argtypes = [ctypes.POINTER(Shape), vp, vp, vp, ctypes.c_int, vp, vp,
                             ctypes.c_float, ctypes.c_int, vp, vp]
    lib.attn_fwd.restype = ctypes.c_int
    lib.attn_fwd_split.argtypes = [ctypes.POINTER(Shape), vp, vp, vp, ctypes.c_int, vp, vp,
                                   ctypes.c_float, ctypes.c_int, ctypes.c_int, vp, ctypes.c_size_t,
                                   vp, vp, vp]
    lib.attn_fwd_split.restype = ctypes.c_int
    lib.attn_split_workspace_bytes.argtypes = [ctypes.POINTER(Shape), ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_size_t)]
    lib.attn_split_workspace_bytes.restype = ctypes.c_int
    lib.attn_bwd.argtypes = [ctypes.POINTER(Shape), vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp,
                             ctypes.c_float, ctypes.c_int, vp, ctypes.c_size_t, vp, vp, vp, vp]
    lib.attn_bwd.restype = ctypes.c_int
    lib.attn_bwd_workspace_bytes.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(ctypes.c_size_t)]
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_int
    lib.attn_paged_fwd.argtypes = [ctypes.POINTER(PagedShape), vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                   ctypes.c_float, ctypes.c_int, ctypes.c_int, vp, ctypes.c_size_t, vp, vp, vp]
    lib.attn_paged_workspace_bytes.argtypes = [ctypes.POINTER(PagedShape), ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_size_t)]
    lib.attn_paged_workspace_bytes.restype = ctypes.c_int
    lib.attn_paged_fwd.restype = ctypes.c_int
    lib.attn_paged_mla.argtypes = [ctypes.POINTER(MlaShape), vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                   ctypes.c_float, ctypes.c_int, ctypes.c_int, vp, ctypes.c_size_t, vp, vp, vp]
    lib.attn_paged_mla.restype = ctypes.c_int
    lib.attn_paged_mla_workspace_bytes.argtypes = [ctypes.POINTER(MlaShape), ctypes.c_int,
                                                   ctypes.POINTER(ctypes.c_size_t)]
    lib.attn_paged_mla_workspace_bytes.restype = ctypes.c_int
    lib.attn_paged_bwd.argtypes = [ctypes.POINTER(PagedShape), vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                   ctypes.c_float, ctypes.c_int, vp, vp, vp, vp, ctypes.c_size_t, vp, vp, vp, vp]
    lib.attn_paged_bwd.restype = ctypes.c_int
    lib.attn_paged_bwd_workspace_bytes.argtypes = [ctypes.POINTER(PagedShape), ctypes.POINTER(ctypes.c_size_t)]
    lib.attn_paged_bwd_workspace_bytes.restype = ctypes.c_int
    lib.attn_paged_mla_bwd.argtypes = [ctypes.POINTER(MlaShape), vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                       ctypes.c_float, ctypes.c_int, vp, vp, vp, vp, ctypes.c_size_t, vp, vp,
                                       vp, vp, vp]
    lib.attn_paged_mla_bwd.restype = ctypes.c_int
    lib.attn_paged_mla_bwd_workspace_bytes.argtypes = [ctypes.POINTER(MlaShape),
                                                       ctypes.POINTER(ctypes.c_size_t)]
    lib.attn_paged_mla_bwd_workspace_bytes.restype = ctypes.c_int
    lib.attn_fwd_host.argtypes = [ctypes.POINTER(Shape), vp, vp, vp, ctypes.c_int, vp, vp, ctypes.c_float,
                                  ctypes.c_int, vp, ctypes.c_size_t, vp, vp]
    lib.attn_fwd_host.restype = ctypes.c_int
    lib.attn_fwd_host_workspace_bytes.argtypes = [ctypes.POINTER(Shape), ctypes.c_int, ctypes.c_int,
                                                  ctypes.POINTER(ctypes.c_size_t)]
    lib.attn_fwd_host_workspace_bytes.restype = ctypes.c_int
    lib.attn_strerror.argtypes = [ctypes.c_int]
    lib.attn_strerror.restype = ctypes.c_char_p
    lib.attn_last_cuda_error.argtypes = []
    lib.attn_last_cuda_error.restype = ctypes.c_int
    lib.attn_device_status.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.c_int]
    lib.attn_device_status.restype = ctypes.c_int
    lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint, ctypes.c_void_p]
    lib.attn_selftest_wait_timeout.restype = ctypes.c_int
    lib.attn_version.argtypes = []
    lib.attn_version.restype = ctypes.c_int
    return lib


def strerror(code: int) -> str:
    return load_library().attn_strerror(int(code)).decode()


def check(code: int):
    if code != 0:
        lib = load_library()
        extra = ""
        if code == -9:
            extra = f" (cudaError {lib.attn_last_cuda_error()})"
        raise AttnError(f"attn_fwd failed: {strerror(code)}{extra}", code)


def device_status(device: int = 0, clear: bool = False) -> int:
    """Sticky kernel error flags of ``device`` (0 = no bounded wait expired)."""
    flags = ctypes.c_int(0)
    check(load_library().attn_device_status(int(device), ctypes.byref(flags), int(bool(clear))))
    return flags.value


def _dtype_code(t):
    import torch
    codes = {torch.float32: ATTN_F32, torch.float16: ATTN_F16, torch.bfloat16: ATTN_BF16}
    if t.dtype not in codes:
        raise AttnError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def call(shape: Shape, q_ptr, k_ptr, v_ptr, mask: int, kv_lens_ptr, bias_ptr, scale: float,
         dtype: int, out_ptr, stream_handle) -> None:
    """Raw attn_fwd call with integer pointers (0 for NULL); raises on error."""
    lib = load_library()
    check(lib.attn_fwd(ctypes.byref(shape), q_ptr or None, k_ptr or None, v_ptr or None, int(mask),
                       kv_lens_ptr or None, bias_ptr or None, float(scale), int(dtype),
                       out_ptr or None, stream_handle or None))


def call_split(shape: Shape, q_ptr, k_ptr, v_ptr, mask: int, kv_lens_ptr, bias_ptr, scale: float,
               dtype: int, num_splits: int, ws_ptr, ws_bytes: int, out_ptr, lse_ptr,
               stream_handle) -> None:
    """Raw attn_fwd_split call with integer pointers (0 for NULL); raises on error."""
    lib = load_library()
    check(lib.attn_fwd_split(ctypes.byref(shape), q_ptr or None, k_ptr or None, v_ptr or None,
                             int(mask), kv_lens_ptr or None, bias_ptr or None, float(scale), int(dtype),
                             int(num_splits), ws_ptr or None, int(ws_bytes), out_ptr or None,
                             lse_ptr or None, stream_handle or None))


def split_workspace_bytes(shape: Shape, num_splits: int) -> int:
    """Workspace bytes attn_fwd_split needs for ``shape`` and ``num_splits``."""
    n = ctypes.c_size_t(0)
    check(load_library().attn_split_workspace_bytes(ctypes.byref(shape), int(num_splits),
                                                    ctypes.byref(n)))
    return n.value


def fwd(q, k, v, *, causal: bool = False, kv_lens=None, bias=None, scale: float | None = None,
        out=None, stream=None, num_splits: int = 1, return_lse: bool = False, workspace=None, lse_out=None):
    """O = softmax(Q K^T * scale + mask + bias) V on the GPU.

    q: [B,Hq,Sq,D]; k, v: [B,Hkv,Sk,D]; float32, float16 or bfloat16, contiguous.
    kv_lens: int32 [B] valid key counts (enables the key-padding mask).
    bias: float32 [bias_b, bias_h, Sq, Sk], bias_b in {1,B}, bias_h in {1,Hq}.
    scale: defaults to 1/sqrt(D).
    num_splits: 1..32 key-range splits (attn_fwd_split); the fp32 workspace is
    taken from ``workspace`` (a CUDA uint8 tensor) or allocated here.
    return_lse: also return the float32 [B,Hq,Sq] row log-sum-exp (written
    into ``lse_out`` when given).
    Tensors on a CUDA device run on ``stream`` (default: the current stream)
    and the result is returned without synchronising. Host tensors run through
    attn_fwd_host on the current CUDA device (chunked uploads, kernels and
    downloads overlapped; synchronising); pinned host memory makes the copies
    asynchronous DMA.
    """
    import torch

    if q.device.type == "cpu":
        if num_splits != 1 or return_lse:
            raise AttnError("host tensors support num_splits=1 without lse only")
        return _fwd_host(q, k, v, causal=causal, kv_lens=kv_lens, bias=bias, scale=scale, out=out)
    dev = q.device
    for name, t in (("k", k), ("v", v)):
        if t.device != dev:
            raise AttnError(f"{name} is on {t.device}, q on {dev}")
        if t.dtype != q.dtype:
            raise AttnError(f"{name} dtype {t.dtype} differs from q dtype {q.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dim() != 4:
            raise AttnError(f"{name} must be 4-D [B, H, S, D]")
        if not t.is_contiguous():
            raise AttnError(f"{name} must be contiguous")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if tuple(k.shape) != (B, Hkv, Sk, D) or tuple(v.shape) != tuple(k.shape):
        raise AttnError("k and v must be [B, Hkv, Sk, D] matching q")
    mask = MASK_CAUSAL if causal else MASK_NONE
    kv_ptr = 0
    if kv_lens is not None:
        if kv_lens.device != dev or kv_lens.dtype != torch.int32 or tuple(kv_lens.shape) != (B,):
            raise AttnError("kv_lens must be int32 [B] on q's device")
        kv_lens = kv_lens.contiguous()
        mask |= MASK_KEY_PADDING
        kv_ptr = kv_lens.data_ptr()
    bb = bh = 1
    b_ptr = 0
    if bias is not None:
        if bias.device != dev or bias.dtype != torch.float32 or bias.dim() != 4 or not bias.is_contiguous():
            raise AttnError("bias must be a contiguous float32 [bias_b, bias_h, Sq, Sk] tensor on q's device")
        bb, bh = int(bias.shape[0]), int(bias.shape[1])
        if tuple(bias.shape[2:]) != (Sq, Sk):
            raise AttnError("bias must be [bias_b, bias_h, Sq, Sk]")
        b_ptr = bias.data_ptr()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or out.device != dev or not out.is_contiguous():
        raise AttnError("out must be a contiguous tensor like q")
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    shape = Shape(B, Hq, Hkv, Sq, Sk, D, bb, bh)
    if num_splits == 1 and not return_lse:
        call(shape, q.data_ptr(), k.data_ptr(), v.data_ptr(), mask, kv_ptr, b_ptr, scale,
             _dtype_code(q), out.data_ptr(), stream.cuda_stream)
        return out
    lse = _lse_buffer(lse_out, (B, Hq, Sq), dev) if return_lse else None
    need = split_workspace_bytes(shape, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    elif workspace.device != dev or workspace.numel() * workspace.element_size() < need:
        raise AttnError(f"workspace must hold {need} bytes on q's device")
    call_split(shape, q.data_ptr(), k.data_ptr(), v.data_ptr(), mask, kv_ptr, b_ptr, scale,
               _dtype_code(q), num_splits, workspace.data_ptr() if need else 0, need,
               out.data_ptr(), lse.data_ptr() if lse is not None else 0, stream.cuda_stream)
    return (out, lse) if return_lse else out


def host_workspace_bytes(shape: Shape, dtype_code: int, with_bias: bool) -> int:
    """Device workspace attn_fwd_host needs for ``shape``."""
    n = ctypes.c_size_t(0)
    check(load_library().attn_fwd_host_workspace_bytes(ctypes.byref(shape), int(dtype_code), int(bool(with_bias)),
                                                      ctypes.byref(n)))
    return n.value


def _fwd_host(q, k, v, *, causal, kv_lens, bias, scale, out, workspace=None):
    """Host tensors in, host tensor out (attn_fwd_host): chunked uploads, the
    kernel per chunk and downloads overlapped on three streams; synchronises."""
    import torch

    for name, t in (("k", k), ("v", v), ("kv_lens", kv_lens), ("bias", bias), ("out", out)):
        if t is not None and t.device.type != "cpu":
            raise AttnError(f"{name} must be a host tensor like q")
    for name, t in (("k", k), ("v", v)):
        if t.dtype != q.dtype:
            raise AttnError(f"{name} dtype {t.dtype} differs from q dtype {q.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dim() != 4 or not t.is_contiguous():
            raise AttnError(f"{name} must be a contiguous 4-D [B, H, S, D] tensor")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if tuple(k.shape) != (B, Hkv, Sk, D) or tuple(v.shape) != tuple(k.shape):
        raise AttnError("k and v must be [B, Hkv, Sk, D] matching q")
    mask = MASK_CAUSAL if causal else MASK_NONE
    if kv_lens is not None:
        if kv_lens.dtype != torch.int32 or tuple(kv_lens.shape) != (B,) or not kv_lens.is_contiguous():
            raise AttnError("kv_lens must be a contiguous int32 [B] host tensor")
        mask |= MASK_KEY_PADDING
    bb = bh = 1
    if bias is not None:
        if bias.dtype != torch.float32 or bias.dim() != 4 or not bias.is_contiguous() or \
                tuple(bias.shape[2:]) != (Sq, Sk):
            raise AttnError("bias must be a contiguous float32 [bias_b, bias_h, Sq, Sk] host tensor")
        bb, bh = int(bias.shape[0]), int(bias.shape[1])
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise AttnError("out must be a contiguous host tensor like q")
    dev = torch.device("cuda", torch.cuda.current_device())
    shape = Shape(B, Hq, Hkv, Sq, Sk, D, bb, bh)
    need = host_workspace_bytes(shape, _dtype_code(q), bias is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    elif workspace.device != dev or workspace.numel() * workspace.element_size() < need:
        raise AttnError(f"workspace must hold {need} bytes on the current device")
    stream = torch.cuda.current_stream(dev)
    ptr = lambda t: (t.data_ptr() or None) if t is not None else None
    check(load_library().attn_fwd_host(ctypes.byref(shape), ptr(q), ptr(k), ptr(v), mask, ptr(kv_lens), ptr(bias),
                                       ctypes.c_float(scale), _dtype_code(q), ptr(workspace) if need else None, need,
                                       ptr(out), stream.cuda_stream or None))
    stream.synchronize()
    return out


def bwd_workspace_bytes(shape: Shape) -> int:
    """Workspace bytes attn_bwd needs for ``shape``."""
    n = ctypes.c_size_t(0)
    check(load_library().attn_bwd_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)))
    return n.value


def bwd(q, k, v, out, dout, lse, *, causal: bool = False, kv_lens=None, bias=None,
        scale: float | None = None, workspace=None, stream=None, dq=None, dk=None, dv=None):
    """Gradients (dq, dk, dv) of attention for dL/dO = ``dout`` (attn_bwd).

    q, k, v, kv_lens, bias, scale, causal: as given to the forward; ``out`` its
    output and ``lse`` its float32 [B,Hq,Sq] row log-sum-exp (``fwd(...,
    return_lse=True)``); ``dout`` like ``out``. All on one CUDA device,
    contiguous. Returns dq (like q), dk and dv (like k and v): the given
    ``dq``/``dk``/``dv`` tensors when passed, else new ones.
    """
    import torch

    dev = q.device
    for name, t in (("k", k), ("v", v), ("out", out), ("dout", dout)):
        if t.device != dev or t.dtype != q.dtype or not t.is_contiguous():
            raise AttnError(f"{name} must be a contiguous {q.dtype} tensor on {dev}")
    if not q.is_contiguous() or q.dim() != 4 or k.dim() != 4:
        raise AttnError("q, k, v must be contiguous 4-D tensors")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if tuple(out.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape) or tuple(v.shape) != tuple(k.shape):
        raise AttnError("out and dout must be like q, v like k")
    if lse.device != dev or lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Sq) or not lse.is_contiguous():
        raise AttnError("lse must be a contiguous float32 [B, Hq, Sq] tensor on q's device")
    mask = MASK_CAUSAL if causal else MASK_NONE
    kv_ptr = 0
    if kv_lens is not None:
        if kv_lens.device != dev or kv_lens.dtype != torch.int32 or tuple(kv_lens.shape) != (B,):
            raise AttnError("kv_lens must be int32 [B] on q's device")
        kv_lens = kv_lens.contiguous()
        mask |= MASK_KEY_PADDING
        kv_ptr = kv_lens.data_ptr()
    bb = bh = 1
    b_ptr = 0
    if bias is not None:
        if bias.device != dev or bias.dtype != torch.float32 or bias.dim() != 4 or not bias.is_contiguous():
            raise AttnError("bias must be a contiguous float32 [bias_b, bias_h, Sq, Sk] tensor on q's device")
        bb, bh = int(bias.shape[0]), int(bias.shape[1])
        b_ptr = bias.data_ptr()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    shape = Shape(B, Hq, Hkv, Sq, Sk, D, bb, bh)
    need = bwd_workspace_bytes(shape)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    elif workspace.device != dev or workspace.numel() * workspace.element_size() < need:
        raise AttnError(f"workspace must hold {need} bytes on q's device")
    for name, t, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t is not None and (t.shape != like.shape or t.dtype != like.dtype or t.device != dev
                              or not t.is_contiguous()):
            raise AttnError(f"{name} must be a contiguous tensor like {'q' if like is q else 'k'}")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    check(load_library().attn_bwd(ctypes.byref(shape), q.data_ptr() or None, k.data_ptr() or None,
                                  v.data_ptr() or None, out.data_ptr() or None, dout.data_ptr() or None,
                                  lse.data_ptr() or None, mask, kv_ptr or None, b_ptr or None, float(scale),
                                  _dtype_code(q), workspace.data_ptr() if need else None, need,
                                  dq.data_ptr() or None, dk.data_ptr() or None, dv.data_ptr() or None,
                                  stream.cuda_stream or None))
    return dq, dk, dv


def _lse_buffer(lse_out, shape, dev):
    import torch
    if lse_out is None:
        return torch.empty(shape, dtype=torch.float32, device=dev)
    if (tuple(lse_out.shape) != tuple(shape) or lse_out.dtype != torch.float32 or lse_out.device != dev
            or not lse_out.is_contiguous()):
        raise AttnError(f"lse_out must be a contiguous float32 {list(shape)} tensor on q's device")
    return lse_out


def _grad_buffer(name, given, like):
    import torch
    if given is None:
        return torch.empty_like(like)
    if (given.shape != like.shape or given.dtype != like.dtype or given.device != like.device
            or not given.is_contiguous()):
        raise AttnError(f"{name} must be a contiguous tensor shaped like its input")
    return given


def paged_workspace_bytes(shape: PagedShape, num_splits: int) -> int:
    """Workspace bytes attn_paged_fwd needs for ``shape`` and ``num_splits``."""
    n = ctypes.c_size_t(0)
    check(load_library().attn_paged_workspace_bytes(ctypes.byref(shape), int(num_splits), ctypes.byref(n)))
    return n.value


def paged_fwd(q, k_cache, v_cache, block_table, seq_lens, q_offsets, *, positions=None, causal: bool = True,
              scale: float | None = None, max_queries: int | None = None, return_lse: bool = False, out=None,
              stream=None, num_splits: int = 1, workspace=None, lse_out=None):
    """Attention of packed queries over a paged key/value cache (attn_paged_fwd).

    q [queries, Hq, D]; k_cache, v_cache [pages, page_size, Hkv, D] (same
    dtype, CUDA, contiguous); block_table int32 [num_seqs, max_pages];
    seq_lens int32 [num_seqs]; q_offsets int32 [num_seqs + 1]; positions
    int32 [queries] or None. ``max_queries`` bounds the queries of one
    sequence (computed from q_offsets, with a host sync, when None).
    ``num_splits`` splits the keys of decode-shaped calls (workspace taken
    from ``workspace``, a CUDA uint8 tensor, or allocated here).
    Returns out [queries, Hq, D] (and lse float32 [queries, Hq], written into
    ``lse_out`` when given).
    """
    import torch

    dev = q.device
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if t.device != dev or t.dtype != q.dtype or not t.is_contiguous() or t.dim() != 4:
            raise AttnError(f"{name} must be a contiguous 4-D {q.dtype} tensor on {dev}")
    if q.dim() != 3 or not q.is_contiguous():
        raise AttnError("q must be a contiguous [queries, Hq, D] tensor")
    nq, Hq, D = q.shape
    pages, P, Hkv, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape:
        raise AttnError("k_cache and v_cache must be [pages, page_size, Hkv, D] with q's D")
    ints = {}
    for name, t in (("block_table", block_table), ("seq_lens", seq_lens), ("q_offsets", q_offsets),
                    ("positions", positions)):
        if t is None:
            continue
        if t.device != dev or t.dtype != torch.int32 or not t.is_contiguous():
            raise AttnError(f"{name} must be a contiguous int32 tensor on q's device")
        ints[name] = t
    ns = int(seq_lens.shape[0])
    if block_table.dim() != 2 or block_table.shape[0] != ns or tuple(q_offsets.shape) != (ns + 1,):
        raise AttnError("block_table must be [num_seqs, max_pages] and q_offsets [num_seqs + 1]")
    if positions is not None and tuple(positions.shape) != (nq,):
        raise AttnError("positions must be int32 [queries]")
    if max_queries is None:
        max_queries = int((q_offsets[1:] - q_offsets[:-1]).max().item()) if ns else 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    lse = _lse_buffer(lse_out, (nq, Hq), dev) if return_lse else None
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    shape = PagedShape(ns, nq, Hq, Hkv, D, P, pages, int(block_table.shape[1]), int(max_queries))
    need = paged_workspace_bytes(shape, num_splits)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    elif need and (workspace.device != dev or workspace.numel() * workspace.element_size() < need):
        raise AttnError(f"workspace must hold {need} bytes on q's device")
    ptr = lambda t: (t.data_ptr() or None) if t is not None else None
    check(load_library().attn_paged_fwd(ctypes.byref(shape), ptr(q), ptr(k_cache), ptr(v_cache), ptr(block_table),
                                        ptr(seq_lens), ptr(q_offsets), ptr(positions), int(bool(causal)),
                                        float(scale), _dtype_code(q), int(num_splits),
                                        ptr(workspace) if need else None, need, ptr(out), ptr(lse),
                                        stream.cuda_stream or None))
    return (out, lse) if return_lse else out


def mla_workspace_bytes(shape: MlaShape, num_splits: int) -> int:
    """Workspace bytes attn_paged_mla needs for ``shape`` and ``num_splits``."""
    n = ctypes.c_size_t(0)
    check(load_library().attn_paged_mla_workspace_bytes(ctypes.byref(shape), int(num_splits), ctypes.byref(n)))
    return n.value


def paged_mla(q, qp, latent, kpos, block_table, seq_lens, q_offsets, *, positions=None, causal: bool = True,
              scale: float, max_queries: int | None = None, return_lse: bool = False, out=None, stream=None,
              num_splits: int = 1, workspace=None, lse_out=None):
    """MLA with absorbed projections over a paged latent cache (attn_paged_mla).

    q [queries, H, R]; qp [queries, H, Pd]; latent [pages, page_size, 1, R];
    kpos [pages, page_size, 1, Pd]; metadata as for :func:`paged_fwd`;
    ``scale`` is the original model's QK scale. ``num_splits`` splits the key
    range of every 128-row block (workspace taken from ``workspace``, a CUDA
    uint8 tensor, or allocated here). Returns out [queries, H, R] (and lse
    float32 [queries, H], written into ``lse_out`` when given).
    """
    import torch

    dev = q.device
    for name, t in (("qp", qp), ("latent", latent), ("kpos", kpos)):
        if t.device != dev or t.dtype != q.dtype or not t.is_contiguous():
            raise AttnError(f"{name} must be a contiguous {q.dtype} tensor on {dev}")
    if q.dim() != 3 or not q.is_contiguous() or latent.dim() != 4 or latent.shape[2] != 1:
        raise AttnError("q [queries, H, R] and latent [pages, page_size, 1, R]")
    nq, H, R = q.shape
    pages, P = int(latent.shape[0]), int(latent.shape[1])
    Pd = int(qp.shape[2])
    if tuple(latent.shape) != (pages, P, 1, R) or tuple(kpos.shape) != (pages, P, 1, Pd) or \
            tuple(qp.shape) != (nq, H, Pd):
        raise AttnError("qp [queries, H, Pd], kpos [pages, page_size, 1, Pd] must match q and latent")
    for name, t in (("block_table", block_table), ("seq_lens", seq_lens), ("q_offsets", q_offsets),
                    ("positions", positions)):
        if t is not None and (t.device != dev or t.dtype != torch.int32 or not t.is_contiguous()):
            raise AttnError(f"{name} must be a contiguous int32 tensor on q's device")
    ns = int(seq_lens.shape[0])
    if max_queries is None:
        max_queries = int((q_offsets[1:] - q_offsets[:-1]).max().item()) if ns else 0
    if out is None:
        out = torch.empty_like(q)
    lse = _lse_buffer(lse_out, (nq, H), dev) if return_lse else None
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    shape = MlaShape(ns, nq, H, R, Pd, P, pages, int(block_table.shape[1]), int(max_queries))
    need = mla_workspace_bytes(shape, num_splits)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    elif need and (workspace.device != dev or workspace.numel() * workspace.element_size() < need):
        raise AttnError(f"workspace must hold {need} bytes on q's device")
    ptr = lambda t: (t.data_ptr() or None) if t is not None else None
    check(load_library().attn_paged_mla(ctypes.byref(shape), ptr(q), ptr(qp), ptr(latent), ptr(kpos),
                                        ptr(block_table), ptr(seq_lens), ptr(q_offsets), ptr(positions),
                                        int(bool(causal)), float(scale), _dtype_code(q), int(num_splits),
                                        ptr(workspace) if need else None, need, ptr(out), ptr(lse),
                                        stream.cuda_stream or None))
    return (out, lse) if return_lse else out


def paged_bwd_workspace_bytes(shape: PagedShape) -> int:
    """Workspace bytes attn_paged_bwd needs for ``shape``."""
    n = ctypes.c_size_t(0)
    check(load_library().attn_paged_bwd_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)))
    return n.value


def _workspace(need, workspace, dev):
    import torch
    if workspace is None:
        return torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if workspace.device != dev or workspace.numel() * workspace.element_size() < need:
        raise AttnError(f"workspace must hold {need} bytes on q's device")
    return workspace


def paged_bwd(q, k_cache, v_cache, block_table, seq_lens, q_offsets, dout, *, out=None, lse=None, positions=None,
              causal: bool = True, scale: float | None = None, max_queries: int | None = None,
              grads=("dq", "dk", "dv"), workspace=None, stream=None, dq=None, dk=None, dv=None):
    """Gradients of :func:`paged_fwd` for dL/dO = ``dout`` (attn_paged_bwd, ordered).

    Arguments as for :func:`paged_fwd`; ``out`` and ``lse`` are the forward's
    output and float32 [queries, Hq] log-sum-exp (when either is None the
    forward runs here first to recompute them). ``grads`` names the gradients
    wanted; ``dq``/``dk``/``dv`` receive them when given. Returns (dq
    [queries, Hq, D], dk, dv [pages, page_size, Hkv, D]), None in place of a
    gradient not asked for.
    """
    import torch

    dev = q.device
    if dout.device != dev or dout.dtype != q.dtype or tuple(dout.shape) != tuple(q.shape) or not dout.is_contiguous():
        raise AttnError("dout must be a contiguous tensor like q")
    nq, Hq, D = q.shape
    pages, P, Hkv, _ = k_cache.shape
    ns = int(seq_lens.shape[0])
    if max_queries is None:
        max_queries = int((q_offsets[1:] - q_offsets[:-1]).max().item()) if ns else 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None or lse is None:
        out, lse = paged_fwd(q, k_cache, v_cache, block_table, seq_lens, q_offsets, positions=positions,
                             causal=causal, scale=scale, max_queries=max_queries, return_lse=True, stream=stream)
    if out.device != dev or out.dtype != q.dtype or tuple(out.shape) != tuple(q.shape) or not out.is_contiguous():
        raise AttnError("out must be a contiguous tensor like q")
    if lse.device != dev or lse.dtype != torch.float32 or tuple(lse.shape) != (nq, Hq) or not lse.is_contiguous():
        raise AttnError("lse must be a contiguous float32 [queries, Hq] tensor on q's device")
    shape = PagedShape(ns, nq, Hq, Hkv, D, P, pages, int(block_table.shape[1]), int(max_queries))
    need = paged_bwd_workspace_bytes(shape)
    workspace = _workspace(need, workspace, dev)
    dq = _grad_buffer("dq", dq, q) if "dq" in grads else None
    dk = _grad_buffer("dk", dk, k_cache) if "dk" in grads else None
    dv = _grad_buffer("dv", dv, v_cache) if "dv" in grads else None
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    ptr = lambda t: (t.data_ptr() or None) if t is not None else None
    check(load_library().attn_paged_bwd(ctypes.byref(shape), ptr(q), ptr(k_cache), ptr(v_cache), ptr(block_table),
                                        ptr(seq_lens), ptr(q_offsets), ptr(positions), int(bool(causal)),
                                        float(scale), _dtype_code(q), ptr(out), ptr(dout), ptr(lse),
                                        ptr(workspace), need, ptr(dq), ptr(dk), ptr(dv), stream.cuda_stream or None))
    return dq, dk, dv


def mla_bwd_workspace_bytes(shape: MlaShape) -> int:
    """Workspace bytes attn_paged_mla_bwd needs for ``shape``."""
    n = ctypes.c_size_t(0)
    check(load_library().attn_paged_mla_bwd_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)))
    return n.value


def paged_mla_bwd(q, qp, latent, kpos, block_table, seq_lens, q_offsets, dout, *, out=None, lse=None,
                  positions=None, causal: bool = True, scale: float, max_queries: int | None = None,
                  grads=("dq", "dqp", "dlatent", "dkpos"), workspace=None, stream=None, dq=None, dqp=None,
                  dlatent=None, dkpos=None):
    """Gradients of :func:`paged_mla` for dL/dO = ``dout`` (attn_paged_mla_bwd, ordered).

    Returns (dq [queries, H, R], dqp [queries, H, Pd], dlatent [pages,
    page_size, 1, R] with its key and value parts, dkpos [pages, page_size, 1,
    Pd]), None in place of a gradient not asked for (or of dqp, dkpos when
    Pd == 0); the given ``dq``/``dqp``/``dlatent``/``dkpos`` tensors receive
    them. ``out``/``lse`` as for :func:`paged_bwd`.
    """
    import torch

    dev = q.device
    if dout.device != dev or dout.dtype != q.dtype or tuple(dout.shape) != tuple(q.shape) or not dout.is_contiguous():
        raise AttnError("dout must be a contiguous tensor like q")
    nq, H, R = q.shape
    pages, P = int(latent.shape[0]), int(latent.shape[1])
    Pd = int(qp.shape[2])
    ns = int(seq_lens.shape[0])
    if max_queries is None:
        max_queries = int((q_offsets[1:] - q_offsets[:-1]).max().item()) if ns else 0
    if out is None or lse is None:
        out, lse = paged_mla(q, qp, latent, kpos, block_table, seq_lens, q_offsets, positions=positions,
                             causal=causal, scale=scale, max_queries=max_queries, return_lse=True, stream=stream)
    if out.device != dev or out.dtype != q.dtype or tuple(out.shape) != tuple(q.shape) or not out.is_contiguous():
        raise AttnError("out must be a contiguous tensor like q")
    if lse.device != dev or lse.dtype != torch.float32 or tuple(lse.shape) != (nq, H) or not lse.is_contiguous():
        raise AttnError("lse must be a contiguous float32 [queries, H] tensor on q's device")
    shape = MlaShape(ns, nq, H, R, Pd, P, pages, int(block_table.shape[1]), int(max_queries))
    need = mla_bwd_workspace_bytes(shape)
    workspace = _workspace(need, workspace, dev)
    dq = _grad_buffer("dq", dq, q) if "dq" in grads else None
    dqp = _grad_buffer("dqp", dqp, qp) if "dqp" in grads and Pd else None
    dlat = _grad_buffer("dlatent", dlatent, latent) if "dlatent" in grads else None
    dkp = _grad_buffer("dkpos", dkpos, kpos) if "dkpos" in grads and Pd else None
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    ptr = lambda t: (t.data_ptr() or None) if t is not None else None
    check(load_library().attn_paged_mla_bwd(ctypes.byref(shape), ptr(q), ptr(qp), ptr(latent), ptr(kpos),
                                            ptr(block_table), ptr(seq_lens), ptr(q_offsets), ptr(positions),
                                            int(bool(causal)), float(scale), _dtype_code(q), ptr(out), ptr(dout),
                                            ptr(lse), ptr(workspace), need, ptr(dq), ptr(dqp), ptr(dlat), ptr(dkp),
                                            stream.cuda_stream or None))
    return dq, dqp, dlat, dkp
