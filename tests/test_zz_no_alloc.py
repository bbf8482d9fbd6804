"""GPU test of attn_fwd_split_noalloc, the split-KV entry point that takes its
scratch from a static device array inside the library instead of a caller
workspace (for callers that may not call cudaMalloc: plugins given buffers
but no allocator, services with no device allocation after start-up).

The entry point is called through the C ABI on several problems in a row,
the first one the largest with the most splits, so that every later call runs
on scratch an earlier call filled with other partials. Each result must be
bit for bit the result of attn_fwd_split given a fresh workspace (the same
kernels on the same inputs; a stale partial that leaked would change bits),
and must match the float64 oracle within the tolerance of every parity test
here (max|O - O_ref| / max|O_ref| <= 1e-5 F32, 4e-3 F16, 1.6e-2 BF16; lse
within 1e-4 * max(1, |lse|)). The F32 case runs the fp32 FMA partial writer,
the others the tensor-core one. The file sorts last so that a stop at its
first failure has already run the other tests; it also passes alone in a
fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
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


def _dtype_code(dtype):
    from exact_scaled_dot_flash_gb300 import attn
    return {"bf16": attn.ATTN_BF16, "f16": attn.ATTN_F16, "f32": attn.ATTN_F32}[dtype]


def _noalloc(w, x, q, k, v, lens, num_splits):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    shape = attn.Shape(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, 1, 1)
    mask = (synth.MASK_CAUSAL if w.causal else 0) | (synth.MASK_KEY_PADDING if lens is not None else 0)
    out = torch.full_like(q, 777.0)
    lse = torch.full((w.B, w.Hq, w.Sq), 777.0, dtype=torch.float32, device=q.device)
    rc = _lib().attn_fwd_split_noalloc(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(), mask,
                                       lens.data_ptr() if lens is not None else None, None,
                                       ctypes.c_float(x["scale"]), _dtype_code(w.dtype), num_splits,
                                       out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, f"attn_fwd_split_noalloc returned {rc}"
    torch.cuda.synchronize()
    return out, lse


def _with_workspace(w, x, q, k, v, lens, num_splits):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    ws = torch.empty(attn.split_workspace_bytes(attn.Shape(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, 1, 1),
                                                num_splits), dtype=torch.uint8, device=q.device)
    o, lse = attn.fwd(q, k, v, causal=w.causal, kv_lens=lens, scale=x["scale"], num_splits=num_splits,
                      return_lse=True, workspace=ws)
    torch.cuda.synchronize()
    return o, lse


def _bits(t):
    import torch
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


def _lse_err(got, ref):
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf)
    assert not np.isnan(got).any()
    fin = ~ninf
    return float(np.max(np.abs(got[fin] - ref[fin]) / np.maximum(1.0, np.abs(ref[fin])))) if fin.any() else 0.0


# The first case fills most of the scratch (14 splits of 16 heads x 256 rows
# x D 128: 28.4 MiB of partials); the later ones are smaller and use other
# layouts (fewer splits, D 64, F32), so stale partials lie under them.
CASES = [
    (synth.Workload("noalloc_big", "bf16", 1, 16, 4, 256, 4096, 128, mask=synth.MASK_CAUSAL, seed=30), 14),
    (synth.Workload("noalloc_gqa_causal", "bf16", 1, 8, 2, 256, 4096, 128, mask=synth.MASK_CAUSAL, seed=31), 4),
    (synth.Workload("noalloc_padding", "f16", 2, 4, 4, 100, 1500, 64, mask=synth.MASK_KEY_PADDING, seed=32,
                    kv_len_range=(1, 1500)), 7),
    (synth.Workload("noalloc_f32", "f32", 1, 4, 2, 70, 600, 32, mask=synth.MASK_CAUSAL, seed=33), 5),
]


def test_noalloc_matches_workspace_entry_point_and_oracle():
    import torch
    torch.cuda.synchronize()
    for w, ns in CASES:  # calls in a row; each later one runs on the scratch the earlier ones left
        x = synth.make_inputs(w)
        q, k, v = (to_device(x[n], w.dtype) for n in ("q", "k", "v"))
        lens = to_device(x["kv_lens"], "i32") if x["kv_lens"] is not None else None
        out, lse = _noalloc(w, x, q, k, v, lens, ns)
        ref_o, ref_lse = _with_workspace(w, x, q, k, v, lens, ns)
        assert np.array_equal(_bits(out), _bits(ref_o)), f"{w.name}: O differs from attn_fwd_split"
        assert np.array_equal(_bits(lse), _bits(ref_lse)), f"{w.name}: lse differs from attn_fwd_split"
        o64, l64 = oracle.attention(x["q"], x["k"], x["v"], mask=w.mask, kv_lens=x["kv_lens"], scale=x["scale"],
                                    dtype=w.dtype, lse=True)
        err = rel_err(to_f64(out), o64)
        assert err <= TOL[w.dtype], f"{w.name}: O rel err {err:.3e} against the oracle"
        e2 = _lse_err(lse.cpu().numpy().astype(np.float64), l64)
        assert e2 <= LSE_TOL, f"{w.name}: lse err {e2:.3e} against the oracle"


def test_noalloc_rejects_problems_beyond_the_scratch():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    # 32 splits of 64 heads x 1024 rows x D=128 need about 1 GiB of partials;
    # the size check rejects the call before any buffer is touched, and the
    # buffers passed are small real device tensors all the same
    shape = attn.Shape(1, 64, 64, 1024, 4096, 128, 1, 1)
    assert attn.split_workspace_bytes(shape, 32) > SCRATCH_BYTES
    q, k, v, out = (torch.zeros(16, dtype=torch.bfloat16, device="cuda") for _ in range(4))
    rc = _lib().attn_fwd_split_noalloc(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(), 0, None,
                                       None, ctypes.c_float(0.1), attn.ATTN_BF16, 32, out.data_ptr(), None,
                                       torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == ATTN_ERR_SCRATCH
    assert not bool(out.any())
