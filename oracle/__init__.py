"""Float64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY: the slow, plain definition the CUDA kernels are
checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import it. It shares no
code with the CUDA library and never consumes a value the CUDA path produced;
the one thing both sides share is the seeded input generator
(``exact_scaled_dot_flash_gb300.synth``), which holds no attention arithmetic.

The arithmetic lives in ``attn_ref.c`` (plain C, float64, threaded over
heads); this module widens the stored inputs exactly to float64, compiles the
C file on first use (gcc) and calls it through ctypes.

Every function is pinned by ``tests/test_oracle_pins.py`` (forward, LSE),
``tests/test_oracle_bwd_pins.py`` (backward), the paged and MLA pins and
``tests/test_oracle_paged_bwd_pins.py`` (paged and MLA backward) against closed forms, invariants,
a 50-digit brute force of the pages' raw-exp kernel, finite differences of the
forward, and textbook reductions; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MASK_CAUSAL, MASK_KEY_PADDING = 1, 2


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "Hq", "Hkv", "Sq", "Sk", "D", "bias_b", "bias_h")]


def build(force: bool = False) -> str:
    """Compile attn_ref.c into liboracle.so (skipped when up to date)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_attention.argtypes = [ctypes.POINTER(_Shape), dp, dp, dp, ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_int32), dp, ctypes.c_double,
                                             dp, dp, dp, ctypes.c_int]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention_rows.argtypes = [ctypes.POINTER(_Shape), dp, dp, dp, ctypes.c_int,
                                                  ctypes.POINTER(ctypes.c_int32), dp, ctypes.c_double,
                                                  ctypes.c_int64, ctypes.POINTER(ctypes.c_int64),
                                                  dp, dp, ctypes.c_int]
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_attention_bwd.argtypes = [ctypes.POINTER(_Shape), dp, dp, dp, ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_int32), dp, ctypes.c_double,
                                                 dp, dp, dp, dp, ctypes.c_int]
            lib.oracle_attention_bwd.restype = ctypes.c_int
            ip = ctypes.POINTER(ctypes.c_int32)
            i64 = ctypes.c_int64
            lib.oracle_paged_attention.argtypes = [i64, i64, i64, i64, i64, i64, dp, dp, dp, ip, ip, ip, ip,
                                                   ctypes.c_int, ctypes.c_double, dp, dp]
            lib.oracle_paged_attention.restype = ctypes.c_int
            lib.oracle_paged_mla.argtypes = [i64, i64, i64, i64, i64, i64, dp, dp, dp, dp, ip, ip, ip, ip,
                                             ctypes.c_int, ctypes.c_double, dp, dp]
            lib.oracle_paged_mla.restype = ctypes.c_int
            lib.oracle_paged_attention_bwd.argtypes = [i64] * 8 + [dp, dp, dp, ip, ip, ip, ip, ctypes.c_int,
                                                                   ctypes.c_double, dp, dp, dp, dp]
            lib.oracle_paged_attention_bwd.restype = ctypes.c_int
            lib.oracle_paged_mla_bwd.argtypes = [i64] * 8 + [dp, dp, dp, dp, ip, ip, ip, ip, ctypes.c_int,
                                                             ctypes.c_double, dp, dp, dp, dp, dp]
            lib.oracle_paged_mla_bwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exactly widen stored values to float64.

    ``dtype`` is "f32", "f16" or "bf16"; bf16 values arrive as uint16 bit
    patterns and become float32 by placing them in the high half of the word.
    """
    if dtype == "bf16":
        bits = np.ascontiguousarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype in ("f16", "f32", "f64"):
        return np.ascontiguousarray(x).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def _dptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) if a is not None else None


def _prepare(q, k, v, kv_lens, bias, dtype):
    q64 = widen(q, dtype) if dtype else np.ascontiguousarray(q, dtype=np.float64)
    k64 = widen(k, dtype) if dtype else np.ascontiguousarray(k, dtype=np.float64)
    v64 = widen(v, dtype) if dtype else np.ascontiguousarray(v, dtype=np.float64)
    B, Hq, Sq, D = q64.shape
    Bk, Hkv, Sk, Dk = k64.shape
    if (Bk, Dk) != (B, D) or v64.shape != k64.shape:
        raise ValueError("shape mismatch between q, k and v")
    shape = _Shape(B, Hq, Hkv, Sq, Sk, D, 1, 1)
    b64 = None
    if bias is not None:
        b64 = np.ascontiguousarray(bias, dtype=np.float64)
        if b64.ndim != 4 or b64.shape[2:] != (Sq, Sk):
            raise ValueError("bias must be [bias_b, bias_h, Sq, Sk]")
        shape.bias_b, shape.bias_h = b64.shape[0], b64.shape[1]
    lens = None
    if kv_lens is not None:
        lens = np.ascontiguousarray(kv_lens, dtype=np.int32)
    return q64, k64, v64, lens, b64, shape


def attention(q, k, v, *, mask: int = 0, kv_lens=None, bias=None, scale: float,
              dtype: str | None = None, weights: bool = False, lse: bool = False, threads: int = 0):
    """Float64 attention output for every row.

    q: [B,Hq,Sq,D], k/v: [B,Hkv,Sk,D] in storage format of ``dtype`` (or any
    float array when ``dtype`` is None); kv_lens: int32 [B] (key padding);
    bias: float [bias_b,bias_h,Sq,Sk]. Returns O [B,Hq,Sq,D] float64; with
    ``weights`` also the weights [B,Hq,Sq,Sk]; with ``lse`` also the row
    log-sum-exp [B,Hq,Sq] (natural log, -inf for a row with no visible key).
    """
    lib = _load()
    q64, k64, v64, lens, b64, shape = _prepare(q, k, v, kv_lens, bias, dtype)
    out = np.empty(q64.shape, dtype=np.float64)
    w = np.empty(q64.shape[:3] + (k64.shape[2],), dtype=np.float64) if weights else None
    ls = np.empty(q64.shape[:3], dtype=np.float64) if lse else None
    rc = lib.oracle_attention(ctypes.byref(shape), _dptr(q64), _dptr(k64), _dptr(v64), int(mask),
                              lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if lens is not None else None,
                              _dptr(b64), float(scale), _dptr(out), _dptr(w), _dptr(ls), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention rejected its arguments (rc={rc})")
    res = (out,) + ((w,) if weights else ()) + ((ls,) if lse else ())
    return res if len(res) > 1 else out


def attention_rows(q, k, v, rows, *, mask: int = 0, kv_lens=None, bias=None, scale: float,
                   dtype: str | None = None, threads: int = 0, widened=None, lse: bool = False):
    """Float64 output rows O[b,hq,i,:] for the (b, hq, i) triples in ``rows``.

    ``widened`` may carry a tuple from :func:`prepare` to avoid re-widening
    large inputs between calls. Returns [len(rows), D] float64.
    """
    lib = _load()
    if widened is None:
        widened = prepare(q, k, v, kv_lens=kv_lens, bias=bias, dtype=dtype)
    q64, k64, v64, lens, b64, shape = widened
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    out = np.empty((r.shape[0], q64.shape[3]), dtype=np.float64)
    ls = np.empty(r.shape[0], dtype=np.float64) if lse else None
    rc = lib.oracle_attention_rows(ctypes.byref(shape), _dptr(q64), _dptr(k64), _dptr(v64), int(mask),
                                   lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if lens is not None else None,
                                   _dptr(b64), float(scale), r.shape[0],
                                   r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _dptr(out), _dptr(ls),
                                   int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_rows rejected its arguments (rc={rc})")
    return (out, ls) if lse else out


def attention_bwd(q, k, v, dout, *, mask: int = 0, kv_lens=None, bias=None, scale: float,
                  dtype: str | None = None, threads: int = 0):
    """Float64 gradients (dq, dk, dv) of a loss whose gradient w.r.t. O is ``dout``.

    Inputs as for :func:`attention`; ``dout`` [B,Hq,Sq,D] in the same storage
    format (widened exactly). Returns dq [B,Hq,Sq,D] and dk, dv [B,Hkv,Sk,D]
    in float64; dk and dv sum over the query heads of a GQA group. The bias is
    a constant. A row with no visible key contributes nothing (its dq is 0).
    """
    lib = _load()
    q64, k64, v64, lens, b64, shape = _prepare(q, k, v, kv_lens, bias, dtype)
    g64 = widen(dout, dtype) if dtype else np.ascontiguousarray(dout, dtype=np.float64)
    if g64.shape != q64.shape:
        raise ValueError("dout must have the shape of q")
    dq = np.empty(q64.shape, dtype=np.float64)
    dk = np.empty(k64.shape, dtype=np.float64)
    dv = np.empty(v64.shape, dtype=np.float64)
    rc = lib.oracle_attention_bwd(ctypes.byref(shape), _dptr(q64), _dptr(k64), _dptr(v64), int(mask),
                                  lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if lens is not None else None,
                                  _dptr(b64), float(scale), _dptr(g64), _dptr(dq), _dptr(dk), _dptr(dv),
                                  int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd rejected its arguments (rc={rc})")
    return dq, dk, dv


def paged_attention(q, k_cache, v_cache, block_table, seq_lens, q_offsets, *, positions=None,
                    causal: bool = True, scale: float, dtype: str | None = None, lse: bool = False):
    """Float64 attention over a paged key/value cache with packed queries.

    q [queries, Hq, D]; k_cache, v_cache [pages, page_size, Hkv, D];
    block_table int32 [num_seqs, max_pages]; seq_lens int32 [num_seqs];
    q_offsets int32 [num_seqs + 1] (queries of sequence s are rows
    q_offsets[s]..q_offsets[s+1]-1); positions int32 [queries] or None (the
    newest tokens). Returns out [queries, Hq, D] (and lse [queries, Hq]).
    """
    lib = _load()
    q64 = widen(q, dtype) if dtype else np.ascontiguousarray(q, dtype=np.float64)
    k64 = widen(k_cache, dtype) if dtype else np.ascontiguousarray(k_cache, dtype=np.float64)
    v64 = widen(v_cache, dtype) if dtype else np.ascontiguousarray(v_cache, dtype=np.float64)
    nq, Hq, D = q64.shape
    pages, P, Hkv, Dk = k64.shape
    if Dk != D or v64.shape != k64.shape:
        raise ValueError("k_cache and v_cache must be [pages, page_size, Hkv, D]")
    tab = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    offs = np.ascontiguousarray(q_offsets, dtype=np.int32)
    ns = lens.shape[0]
    if tab.ndim != 2 or tab.shape[0] != ns or offs.shape != (ns + 1,) or offs[-1] != nq:
        raise ValueError("block_table [num_seqs, max_pages], q_offsets [num_seqs + 1] ending at queries")
    for s_ in range(ns):
        used = tab[s_, :(int(lens[s_]) + P - 1) // P]
        if lens[s_] > tab.shape[1] * P or ((used < 0) | (used >= pages)).any():
            raise ValueError("block_table does not cover the sequence inside the cache")
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int32)
    out = np.empty((nq, Hq, D), dtype=np.float64)
    ls = np.empty((nq, Hq), dtype=np.float64) if lse else None
    ip = ctypes.POINTER(ctypes.c_int32)
    rc = lib.oracle_paged_attention(ns, Hq, Hkv, D, P, tab.shape[1], _dptr(q64), _dptr(k64), _dptr(v64),
                                    tab.ctypes.data_as(ip), lens.ctypes.data_as(ip), offs.ctypes.data_as(ip),
                                    pos.ctypes.data_as(ip) if pos is not None else None, int(bool(causal)),
                                    float(scale), _dptr(out), _dptr(ls))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention rejected its arguments (rc={rc})")
    return (out, ls) if lse else out


def paged_mla(q, qp, latent, kpos, block_table, seq_lens, q_offsets, *, positions=None, causal: bool = True,
              scale: float, dtype: str | None = None, lse: bool = False):
    """Float64 MLA over a paged latent cache (absorbed projections).

    q [queries, H, R]; qp [queries, H, P]; latent [pages, page_size, 1, R];
    kpos [pages, page_size, 1, P]; paging, packing and positions as in
    :func:`paged_attention`. Returns out [queries, H, R] (and lse [queries, H]).
    """
    lib = _load()
    w = (lambda a: widen(a, dtype)) if dtype else (lambda a: np.ascontiguousarray(a, dtype=np.float64))
    q64, qp64, lat64, kp64 = w(q), w(qp), w(latent), w(kpos)
    nq, H, R = q64.shape
    pages, P, one, R2 = lat64.shape
    Pd = qp64.shape[2]
    if one != 1 or R2 != R or kp64.shape != (pages, P, 1, Pd) or qp64.shape[:2] != (nq, H):
        raise ValueError("latent [pages, page_size, 1, R], kpos [pages, page_size, 1, P], qp [queries, H, P]")
    tab = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    offs = np.ascontiguousarray(q_offsets, dtype=np.int32)
    ns = lens.shape[0]
    if tab.ndim != 2 or tab.shape[0] != ns or offs.shape != (ns + 1,) or offs[-1] != nq:
        raise ValueError("block_table [num_seqs, max_pages], q_offsets [num_seqs + 1] ending at queries")
    for s_ in range(ns):
        used = tab[s_, :(int(lens[s_]) + P - 1) // P]
        if lens[s_] > tab.shape[1] * P or ((used < 0) | (used >= pages)).any():
            raise ValueError("block_table does not cover the sequence inside the cache")
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int32)
    out = np.empty((nq, H, R), dtype=np.float64)
    ls = np.empty((nq, H), dtype=np.float64) if lse else None
    ip = ctypes.POINTER(ctypes.c_int32)
    rc = lib.oracle_paged_mla(ns, H, R, Pd, P, tab.shape[1], _dptr(q64), _dptr(qp64), _dptr(lat64), _dptr(kp64),
                              tab.ctypes.data_as(ip), lens.ctypes.data_as(ip), offs.ctypes.data_as(ip),
                              pos.ctypes.data_as(ip) if pos is not None else None, int(bool(causal)),
                              float(scale), _dptr(out), _dptr(ls))
    if rc != 0:
        raise ValueError(f"oracle_paged_mla rejected its arguments (rc={rc})")
    return (out, ls) if lse else out


def _paged_meta(block_table, seq_lens, q_offsets, positions, nq):
    tab = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    offs = np.ascontiguousarray(q_offsets, dtype=np.int32)
    ns = lens.shape[0]
    if tab.ndim != 2 or tab.shape[0] != ns or offs.shape != (ns + 1,) or offs[-1] != nq:
        raise ValueError("block_table [num_seqs, max_pages], q_offsets [num_seqs + 1] ending at queries")
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int32)
    return tab, lens, offs, pos


def paged_attention_bwd(q, k_cache, v_cache, dout, block_table, seq_lens, q_offsets, *, positions=None,
                        causal: bool = True, scale: float, dtype: str | None = None):
    """Float64 gradients of :func:`paged_attention` for dL/dO = ``dout``.

    Returns dq [queries, Hq, D] and dk, dv in the cache's shape [pages,
    page_size, Hkv, D]: a page read by several sequences (or blocks) gets the
    sum of every read's contribution, a page nobody reads gets zero.
    """
    lib = _load()
    w = (lambda a: widen(a, dtype)) if dtype else (lambda a: np.ascontiguousarray(a, dtype=np.float64))
    q64, k64, v64, g64 = w(q), w(k_cache), w(v_cache), w(dout)
    nq, Hq, D = q64.shape
    pages, P, Hkv, Dk = k64.shape
    if Dk != D or v64.shape != k64.shape or g64.shape != q64.shape:
        raise ValueError("k_cache, v_cache [pages, page_size, Hkv, D]; dout like q")
    tab, lens, offs, pos = _paged_meta(block_table, seq_lens, q_offsets, positions, nq)
    dq = np.empty_like(q64)
    dk = np.empty_like(k64)
    dv = np.empty_like(v64)
    ip = ctypes.POINTER(ctypes.c_int32)
    rc = lib.oracle_paged_attention_bwd(lens.shape[0], Hq, Hkv, D, P, tab.shape[1], pages, nq, _dptr(q64),
                                        _dptr(k64), _dptr(v64), tab.ctypes.data_as(ip), lens.ctypes.data_as(ip),
                                        offs.ctypes.data_as(ip), pos.ctypes.data_as(ip) if pos is not None else None,
                                        int(bool(causal)), float(scale), _dptr(g64), _dptr(dq), _dptr(dk), _dptr(dv))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention_bwd rejected its arguments (rc={rc})")
    return dq, dk, dv


def paged_mla_bwd(q, qp, latent, kpos, dout, block_table, seq_lens, q_offsets, *, positions=None,
                  causal: bool = True, scale: float, dtype: str | None = None):
    """Float64 gradients of :func:`paged_mla` for dL/dO = ``dout`` [queries, H, R].

    Returns dq [queries, H, R], dqp [queries, H, P], and the cache-shaped
    dlatent [pages, page_size, 1, R] (key and value contributions summed) and
    dkpos [pages, page_size, 1, P].
    """
    lib = _load()
    w = (lambda a: widen(a, dtype)) if dtype else (lambda a: np.ascontiguousarray(a, dtype=np.float64))
    q64, qp64, lat64, kp64, g64 = w(q), w(qp), w(latent), w(kpos), w(dout)
    nq, H, R = q64.shape
    pages, P, one, R2 = lat64.shape
    Pd = qp64.shape[2]
    if (one != 1 or R2 != R or kp64.shape != (pages, P, 1, Pd) or qp64.shape[:2] != (nq, H)
            or g64.shape != q64.shape):
        raise ValueError("latent [pages, page_size, 1, R], kpos [pages, page_size, 1, P], qp [queries, H, P]")
    tab, lens, offs, pos = _paged_meta(block_table, seq_lens, q_offsets, positions, nq)
    dq, dqp, dlat, dkp = (np.empty_like(a) for a in (q64, qp64, lat64, kp64))
    ip = ctypes.POINTER(ctypes.c_int32)
    rc = lib.oracle_paged_mla_bwd(lens.shape[0], H, R, Pd, P, tab.shape[1], pages, nq, _dptr(q64), _dptr(qp64),
                                  _dptr(lat64), _dptr(kp64), tab.ctypes.data_as(ip), lens.ctypes.data_as(ip),
                                  offs.ctypes.data_as(ip), pos.ctypes.data_as(ip) if pos is not None else None,
                                  int(bool(causal)), float(scale), _dptr(g64), _dptr(dq), _dptr(dqp), _dptr(dlat),
                                  _dptr(dkp))
    if rc != 0:
        raise ValueError(f"oracle_paged_mla_bwd rejected its arguments (rc={rc})")
    return dq, dqp, dlat, dkp


def prepare(q, k, v, *, kv_lens=None, bias=None, dtype: str | None = None):
    """Widen inputs once for repeated :func:`attention_rows` calls."""
    return _prepare(q, k, v, kv_lens, bias, dtype)
