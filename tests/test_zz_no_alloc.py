"""GPU test of attn_fwd_split_noalloc, the split-KV entry point that takes its
scratch from a static device array inside the library instead of a caller
workspace (for callers that may not call cudaMalloc: plugins given buffers
but no allocator, services with no device allocation after start-up).

The entry point is called through the C ABI and its output and row
log-sum-exp are compared with attn_fwd_split given an ordinary workspace, on
two calls in a row of different problems, so that the second call runs on
scratch the first one left behind. Tolerance: the same as every parity test
here (max|O - O_ref| / max|O_ref| <= 1.6e-2 BF16, 4e-3 F16; lse within
1e-4 * max(1, |lse|)). The file sorts last so that a stop at its first
failure has already run the other tests; it also passes alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest

from exact_scaled_dot_flash_gb300 import synth
from tests.gpu_util import TOL, rel_err, to_device, to_f64

pytestmark = pytest.mark.gpu
LSE_TOL = 1e-4
ATTN_ERR_SCRATCH = -13
SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module", autouse=True)
def _clean_status():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    torch.cuda.synchronize()
    attn.device_status(torch.cuda.current_device(), clear=True)
    yield
    torch.cuda.synchronize()
    assert attn.device_status(torch.cuda.current_device(), clear=True) == 0, "a kernel wait timed out"


def _lib():
    from exact_scaled_dot_flash_gb300 import attn
    lib = attn.load_library()
    vp = ctypes.c_void_p
    lib.attn_fwd_split_noalloc.argtypes = [ctypes.POINTER(attn.Shape), vp, vp, vp, ctypes.c_int, vp, vp,
                                           ctypes.c_float, ctypes.c_int, ctypes.c_int, vp, vp, vp]
    lib.attn_fwd_split_noalloc.restype = ctypes.c_int
    return lib


def _prepare(w):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    x = synth.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in ("q", "k", "v"))
    lens = to_device(x["kv_lens"], "i32") if x["kv_lens"] is not None else None
    shape = attn.Shape(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, 1, 1)
    mask = (synth.MASK_CAUSAL if w.causal else 0) | (synth.MASK_KEY_PADDING if lens is not None else 0)
    dtype = {"bf16": attn.ATTN_BF16, "f16": attn.ATTN_F16, "f32": attn.ATTN_F32}[w.dtype]
    out = torch.full_like(q, 777.0)
    lse = torch.full((w.B, w.Hq, w.Sq), 777.0, dtype=torch.float32, device=q.device)
    return x, q, k, v, lens, shape, mask, dtype, out, lse


def _noalloc(w, num_splits):
    import torch
    x, q, k, v, lens, shape, mask, dtype, out, lse = _prepare(w)
    rc = _lib().attn_fwd_split_noalloc(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(), mask,
                                       lens.data_ptr() if lens is not None else None, None,
                                       ctypes.c_float(x["scale"]), dtype, num_splits, out.data_ptr(),
                                       lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, f"attn_fwd_split_noalloc returned {rc}"
    torch.cuda.synchronize()
    return x, q, k, v, lens, to_f64(out), lse.cpu().numpy().astype(np.float64)


def _reference(w, x, q, k, v, lens, num_splits):
    from exact_scaled_dot_flash_gb300 import attn
    o, lse = attn.fwd(q, k, v, causal=w.causal, kv_lens=lens, scale=x["scale"], num_splits=num_splits,
                      return_lse=True)
    return to_f64(o), lse.cpu().numpy().astype(np.float64)


def _lse_err(got, ref):
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf)
    fin = ~ninf
    return float(np.max(np.abs(got[fin] - ref[fin]) / np.maximum(1.0, np.abs(ref[fin])))) if fin.any() else 0.0


CASES = [
    (synth.Workload("noalloc_gqa_causal", "bf16", 1, 8, 2, 256, 4096, 128, mask=synth.MASK_CAUSAL, seed=31), 4),
    (synth.Workload("noalloc_padding", "f16", 2, 4, 4, 100, 1500, 64, mask=synth.MASK_KEY_PADDING, seed=32,
                    kv_len_range=(1, 1500)), 7),
]


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import torch
    torch.cuda.synchronize()
    for w, ns in CASES:  # two calls in a row; the second reuses the first's scratch
        x, q, k, v, lens, got, got_lse = _noalloc(w, ns)
        ref, ref_lse = _reference(w, x, q, k, v, lens, ns)
        err = rel_err(got, ref)
        assert err <= TOL[w.dtype], f"{w.name}: O rel err {err:.3e}"
        assert _lse_err(got_lse, ref_lse) <= LSE_TOL, w.name


def test_noalloc_rejects_problems_beyond_the_scratch():
    from exact_scaled_dot_flash_gb300 import attn
    # 32 splits of 64 heads x 1024 rows x D=128 need about 1 GiB of partials
    shape = attn.Shape(1, 64, 64, 1024, 4096, 128, 1, 1)
    assert attn.split_workspace_bytes(shape, 32) > SCRATCH_BYTES
    rc = _lib().attn_fwd_split_noalloc(ctypes.byref(shape), 0x10000, 0x20000, 0x30000, 0, None, None,
                                       ctypes.c_float(0.1), attn.ATTN_BF16, 32, 0x40000, None, None)
    assert rc == ATTN_ERR_SCRATCH
