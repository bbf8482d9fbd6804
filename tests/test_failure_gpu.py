"""Failure detection on the GPU without a GPU fault.

A kernel whose mbarrier wait can never complete must give up after its
bounded limit, report ATTN timeout through the device status word, and leave
the context usable for the next attention call.
"""
import ctypes
import time

import numpy as np
import pytest

import oracle
from exact_scaled_dot_flash_gb300 import attn, synth
from tests.gpu_util import TOL, rel_err, run_gpu, to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    dev = torch.cuda.current_device()
    torch.cuda.synchronize()
    attn.device_status(dev, clear=True)
    lib = attn.load_library()
    t0 = time.perf_counter()
    attn.check(lib.attn_selftest_wait_timeout(20000, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert attn.device_status(dev, clear=True) == 1, "the expired wait was not reported"
    assert 0.015 < elapsed < 5.0, f"the 20 ms limit took {elapsed:.3f} s"
    assert attn.device_status(dev) == 0
    # the context is healthy: a normal call still matches the oracle
    w = synth.Workload("after_timeout", "bf16", 1, 2, 2, 200, 200, 64, mask=synth.MASK_CAUSAL, seed=5)
    x = synth.make_inputs(w)
    out = run_gpu(x, w.dtype)
    ref = oracle.attention(x["q"], x["k"], x["v"], mask=w.mask, scale=x["scale"], dtype=w.dtype)
    assert rel_err(to_f64(out), ref) <= TOL[w.dtype]
    assert attn.device_status(dev) == 0


def test_selftest_rejects_bad_limits():
    lib = attn.load_library()
    assert lib.attn_selftest_wait_timeout(0, None) == -2
    assert lib.attn_selftest_wait_timeout(10_000_000, None) == -2
