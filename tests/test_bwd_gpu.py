"""GPU parity of the attention backward (attn_bwd) against the float64 oracle.

The pipeline is the user's: the CUDA forward with its row log-sum-exp, then
the CUDA backward on (q, k, v, out, dout, lse); the oracle computes dq, dk, dv
from (q, k, v, dout) alone. Tolerance per gradient tensor: max|g - g_ref| /
max|g_ref| <= 1e-5 (F32), 4e-3 (F16), 1.6e-2 (BF16), the forward's bounds:
the backward adds the rounding of the forward output (used for
D_i = dout_i . out_i) in the same dtype and fp32 arithmetic, so its error
scale is the same as the forward's.
"""
import math

import numpy as np
import pytest

import oracle
from exact_scaled_dot_flash_gb300 import synth
from tests.gpu_util import TOL, to_device, to_f64

pytestmark = pytest.mark.gpu
CAUSAL, PAD = synth.MASK_CAUSAL, synth.MASK_KEY_PADDING


@pytest.fixture(scope="module", autouse=True)
def _clean_status():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    torch.cuda.synchronize()
    attn.device_status(torch.cuda.current_device(), clear=True)
    yield
    torch.cuda.synchronize()
    assert attn.device_status(torch.cuda.current_device(), clear=True) == 0, "a kernel wait timed out"


def grad_err(got, ref):
    assert not np.isnan(got).any(), "gradient has NaN"
    denom = np.abs(ref).max()
    return float(np.abs(got - ref).max() / max(denom, 1e-300))


def run_bwd(w, x, dout_store):
    from exact_scaled_dot_flash_gb300 import attn
    q, k, v = (to_device(x[n], w.dtype) for n in ("q", "k", "v"))
    lens = to_device(x["kv_lens"], "i32") if x["kv_lens"] is not None else None
    bias = to_device(x["bias"], "f32") if x["bias"] is not None else None
    g = to_device(dout_store, w.dtype)
    causal = bool(w.mask & CAUSAL)
    out, lse = attn.fwd(q, k, v, causal=causal, kv_lens=lens, bias=bias, scale=x["scale"], return_lse=True)
    dq, dk, dv = attn.bwd(q, k, v, out, g, lse, causal=causal, kv_lens=lens, bias=bias, scale=x["scale"])
    return to_f64(dq), to_f64(dk), to_f64(dv)


def check(w, x=None, seed_g=None):
    x = x if x is not None else synth.make_inputs(w)
    g32 = synth.normal_f32(w.seed if seed_g is None else seed_g, 7, (w.B, w.Hq, w.Sq, w.D))
    g = synth.to_storage(g32, w.dtype)
    got = run_bwd(w, x, g)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], g, mask=w.mask, kv_lens=x["kv_lens"], bias=x["bias"],
                               scale=x["scale"], dtype=w.dtype)
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        err = grad_err(a, b)
        assert err <= TOL[w.dtype], f"{w.name} {name}: rel err {err:.3e} > {TOL[w.dtype]}"
    return x, g, got, ref


def W(name, dtype, B, Hq, Hkv, Sq, Sk, D, **kw):
    return synth.Workload(name, dtype, B, Hq, Hkv, Sq, Sk, D, **kw)


CASES = [
    W("bwd_f32_d16_causal", "f32", 2, 2, 2, 64, 64, 16, mask=CAUSAL, seed=0),
    W("bwd_f32_d64_gqa", "f32", 1, 4, 2, 100, 130, 64, mask=CAUSAL, seed=1),
    W("bwd_bf16_d128_causal", "bf16", 2, 4, 2, 200, 200, 128, mask=CAUSAL, seed=2),
    W("bwd_bf16_d64_full", "bf16", 1, 2, 2, 150, 333, 64, seed=3),
    W("bwd_f16_d32_causal_sq_gt_sk", "f16", 1, 2, 1, 160, 96, 32, mask=CAUSAL, seed=4),
    W("bwd_f16_d64_padding_bias", "f16", 3, 2, 2, 80, 190, 64, mask=PAD, bias=True, bias_b=1, bias_h=2,
      seed=5, kv_len_range=(1, 190)),
    W("bwd_bf16_d128_both_bias", "bf16", 2, 2, 1, 96, 96, 128, mask=CAUSAL | PAD, bias=True, bias_b=2,
      bias_h=1, seed=6, kv_len_range=(40, 96)),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_bwd_matches_oracle(w):
    check(w)


def test_bwd_rows_without_keys():
    # kv_len 0 for one batch: its rows have no visible key; dq = 0 there, and
    # the other batch is unaffected
    w = W("bwd_empty_rows", "bf16", 2, 2, 2, 70, 90, 64, mask=PAD, seed=8)
    x = synth.make_inputs(w)
    x["kv_lens"] = np.array([0, 57], dtype=np.int32)
    _, _, got, _ = check(w, x)
    assert (got[0][0] == 0).all() and (got[1][0] == 0).all() and (got[2][0] == 0).all()
    assert (got[1][1, :, 57:] == 0).all() and (got[2][1, :, 57:] == 0).all()


def test_bwd_is_deterministic():
    w = W("bwd_det", "bf16", 1, 4, 1, 300, 300, 128, mask=CAUSAL, seed=9)
    x = synth.make_inputs(w)
    g = synth.to_storage(synth.normal_f32(9, 7, (1, 4, 300, 128)), "bf16")
    a = run_bwd(w, x, g)
    b = run_bwd(w, x, g)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_bwd_empty_axes():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    dev = torch.device("cuda")
    # Sk = 0: dq = 0; Sq = 0: dk = dv = 0
    q = torch.randn(1, 2, 8, 64, device=dev, dtype=torch.bfloat16)
    k = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    out = torch.randn_like(q)
    lse = torch.full((1, 2, 8), float("-inf"), device=dev)
    dq, dk, dv = attn.bwd(q, k, k, out, out, lse)
    assert (dq == 0).all() and dk.numel() == 0
    q0 = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    k1 = torch.randn(1, 2, 5, 64, device=dev, dtype=torch.bfloat16)
    dq, dk, dv = attn.bwd(q0, k1, k1, q0, q0, torch.empty(1, 2, 0, device=dev))
    assert (dk == 0).all() and (dv == 0).all()


def test_bwd_argument_errors():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    dev = torch.device("cuda")
    q = torch.randn(1, 2, 8, 64, device=dev, dtype=torch.bfloat16)
    out = torch.randn_like(q)
    lse = torch.zeros(1, 2, 8, device=dev)
    shape = attn.Shape(1, 2, 2, 8, 8, 64, 1, 1)
    need = attn.bwd_workspace_bytes(shape)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    lib = attn.load_library()
    args = lambda **o: [o.get(n, d) for n, d in (
        ("q", q.data_ptr()), ("k", q.data_ptr()), ("v", q.data_ptr()), ("out", out.data_ptr()),
        ("dout", out.data_ptr()), ("lse", lse.data_ptr()), ("mask", 0), ("lens", None), ("bias", None),
        ("scale", 0.125), ("dtype", attn.ATTN_BF16), ("ws", ws.data_ptr()), ("wsb", need), ("dq", dq.data_ptr()),
        ("dk", dk.data_ptr()), ("dv", dv.data_ptr()), ("st", None))]
    import ctypes
    call = lambda **o: lib.attn_bwd(ctypes.byref(shape), *args(**o))
    assert call() == 0
    torch.cuda.synchronize()
    assert call(wsb=need - 1) == -12                    # workspace too small
    assert call(dq=q.data_ptr()) == -8                  # dq overlaps q
    assert call(dk=dq.data_ptr()) == -8                 # dk overlaps dq
    assert call(ws=dv.data_ptr()) == -8                 # workspace overlaps dv
    assert call(lse=None) == -1
    assert call(scale=math.nan) == -6


@pytest.mark.parametrize("D", [64, 128])
def test_bwd_zero_bias_equals_no_bias_bitwise(D):
    # the backward kernels with bias read it per element, which changes their
    # timing; adding a zero bias is exact, so on the same forward outputs the
    # gradients must be bit-identical to the bias-free call (the forward's own
    # bias and bias-free paths round differently, so it runs once)
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = W(f"bwd_zero_bias_d{D}", "bf16", 2, 2, 1, 256, 384, D, mask=CAUSAL, seed=12)
    x = synth.make_inputs(w)
    q, k, v = (to_device(x[n], "bf16") for n in ("q", "k", "v"))
    g = to_device(synth.to_storage(synth.normal_f32(12, 7, (2, 2, 256, D)), "bf16"), "bf16")
    zero = torch.zeros(1, 2, 256, 384, device=q.device)
    out, lse = attn.fwd(q, k, v, causal=True, scale=x["scale"], return_lse=True)
    res = [attn.bwd(q, k, v, out, g, lse, causal=True, bias=bias, scale=x["scale"]) for bias in (None, zero)]
    torch.cuda.synchronize()
    for a, b in zip(*res):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
