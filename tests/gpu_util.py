"""Helpers shared by the GPU parity tests: moving seeded inputs to the device,
reading outputs back exactly, and the error metric with its tolerances."""
import numpy as np

# max|O_gpu - O_ref| / max|O_ref| bounds per input dtype
TOL = {"f32": 1e-5, "f16": 4e-3, "bf16": 1.6e-2}


def to_device(x, dtype, device="cuda"):
    import torch
    if x is None:
        return None
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(device)


def to_f64(t):
    """Exact widening of a float32/float16/bfloat16 tensor to a float64 array."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def rel_err(got, ref):
    """max|got - ref| / max|ref| over entries where ref is finite.

    Entries where ref is NaN (rows with no visible key) must be NaN in got.
    """
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref), "NaN pattern differs"
    fin = ~nan_ref
    if not fin.any():
        return 0.0
    denom = np.max(np.abs(ref[fin]))
    return float(np.max(np.abs(got[fin] - ref[fin])) / max(denom, 1e-300))


def run_gpu(x, dtype, causal=None, stream=None):
    """Run the library on the seeded inputs ``x`` (dict from synth.make_inputs)."""
    from exact_scaled_dot_flash_gb300 import attn
    q, k, v = (to_device(x[n], dtype) for n in ("q", "k", "v"))
    lens = to_device(x["kv_lens"], "i32") if x["kv_lens"] is not None else None
    bias = to_device(x["bias"], "f32") if x["bias"] is not None else None
    causal = bool(x["mask"] & 1) if causal is None else causal
    out = torch_full_like(q, 777.0)  # sentinel: a tile the kernel skips cannot pass as a result
    return attn.fwd(q, k, v, causal=causal, kv_lens=lens, bias=bias, scale=x["scale"], stream=stream,
                    out=out)


def torch_full_like(t, value):
    import torch
    return torch.full_like(t, value)
