"""GPU tests of attn_fwd_host (host tensors in and out, chunked uploads,
kernels and downloads overlapped on three streams).

Each chunk runs the same kernel on the same rows as one whole-problem attn_fwd
call, so the host path must return exactly (bit for bit) what attn_fwd returns
on device copies of the inputs; one case is also held to the float64 oracle
with the dense forward's tolerance.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_flash_gb300 import synth
from tests.gpu_util import TOL, rel_err, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _clean_status():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    torch.cuda.synchronize()
    attn.device_status(torch.cuda.current_device(), clear=True)
    yield
    torch.cuda.synchronize()
    assert attn.device_status(torch.cuda.current_device(), clear=True) == 0, "a kernel wait timed out"


def host(a, dtype, pin=True):
    import torch
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16) if dtype == "bf16" \
        else torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pin else t.clone()


def run_both(w, pin=True):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    x = synth.make_inputs(w)
    args = dict(causal=w.causal, scale=x["scale"])
    dev = attn.fwd(*(to_device(x[n], w.dtype) for n in ("q", "k", "v")),
                   kv_lens=to_device(x["kv_lens"], "i32") if x["kv_lens"] is not None else None,
                   bias=to_device(x["bias"], "f32") if x["bias"] is not None else None, **args)
    torch.cuda.synchronize()
    out = host(np.zeros_like(x["q"]), w.dtype, pin)
    got = attn.fwd(*(host(x[n], w.dtype, pin) for n in ("q", "k", "v")),
                   kv_lens=host(x["kv_lens"], "i32", pin), bias=host(x["bias"], "f32", pin), out=out, **args)
    assert got.data_ptr() == out.data_ptr() and got.device.type == "cpu"
    return x, got, dev.cpu()


def bits(t):
    import torch
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).numpy()


W = synth.Workload
CASES = [
    # B x Hkv units split into chunks within a batch index (2 per batch here)
    W("host_bf16_causal", "bf16", 4, 8, 8, 300, 300, 128, mask=synth.MASK_CAUSAL, seed=1),
    # GQA groups stay whole inside a chunk; one batch, eight chunks
    W("host_f16_gqa", "f16", 1, 32, 8, 200, 700, 64, seed=2),
    # padding (kv_lens slice per chunk) and a per-(batch, head) bias
    W("host_bf16_pad_bias_bh", "bf16", 3, 4, 2, 130, 260, 64, mask=synth.MASK_KEY_PADDING, bias=True,
      bias_b=3, bias_h=4, seed=3, kv_len_range=(0, 260)),
    # bias broadcast over batches and heads, and over heads only
    W("host_f16_bias_11", "f16", 2, 6, 3, 64, 96, 32, bias=True, bias_b=1, bias_h=1, seed=4),
    W("host_bf16_bias_b1", "bf16", 5, 2, 1, 90, 90, 64, mask=synth.MASK_CAUSAL, bias=True, bias_b=5, bias_h=1,
      seed=5),
    # F32 runs the fp32 kernel per chunk; more batches than target chunks
    W("host_f32_many_b", "f32", 11, 2, 2, 40, 70, 32, mask=synth.MASK_CAUSAL, seed=6),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_host_path_equals_device_path(w):
    x, got, dev = run_both(w)
    np.testing.assert_array_equal(bits(got), bits(dev))


def test_host_path_matches_oracle():
    w = CASES[2]
    x, got, _ = run_both(w)
    ref = oracle.attention(x["q"], x["k"], x["v"], mask=w.mask, kv_lens=x["kv_lens"], bias=x["bias"],
                           scale=x["scale"], dtype=w.dtype)
    assert rel_err(to_f64(got), ref) <= TOL[w.dtype]


def test_host_path_pageable_memory_and_empty_keys():
    # pageable (not pinned) host tensors: the copies block but the result is the same
    w = W("host_pageable", "bf16", 2, 4, 4, 128, 200, 64, mask=synth.MASK_CAUSAL, seed=7)
    x, got, dev = run_both(w, pin=False)
    np.testing.assert_array_equal(bits(got), bits(dev))
    # no keys at all: every row is NaN
    w0 = W("host_no_keys", "f16", 2, 2, 2, 16, 0, 64, seed=8)
    x0, got0, dev0 = run_both(w0)
    assert np.isnan(got0.float().numpy()).all() and np.isnan(dev0.float().numpy()).all()


def test_host_path_back_to_back_calls_share_nothing():
    # two calls in a row on one device: the library's copy streams are reused,
    # and each call's result is its own
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    wa = W("host_a", "bf16", 2, 4, 4, 256, 256, 128, seed=9)
    wb = W("host_b", "bf16", 2, 4, 4, 256, 256, 128, seed=10)
    xa, xb = synth.make_inputs(wa), synth.make_inputs(wb)
    oa = attn.fwd(*(host(xa[n], "bf16") for n in ("q", "k", "v")), scale=xa["scale"])
    ob = attn.fwd(*(host(xb[n], "bf16") for n in ("q", "k", "v")), scale=xb["scale"])
    da = attn.fwd(*(to_device(xa[n], "bf16") for n in ("q", "k", "v")), scale=xa["scale"]).cpu()
    db = attn.fwd(*(to_device(xb[n], "bf16") for n in ("q", "k", "v")), scale=xb["scale"]).cpu()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(oa), bits(da))
    np.testing.assert_array_equal(bits(ob), bits(db))
