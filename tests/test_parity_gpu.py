"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle.

Every workload, including the long-context ones at full size in the launch
the benchmark times, is compared element by element over every output with
the oracle run on all host cores. Tolerance: max|O_gpu - O_ref| / max|O_ref| <= 1e-5 (F32), 4e-3 (F16),
1.6e-2 (BF16); rows with no visible key must be NaN on both sides; causal
row 0 must equal V[0] bit for bit.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_flash_gb300 import synth
from tests.gpu_util import TOL, rel_err, run_gpu, to_device, to_f64

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


def full_check(w, x=None):
    x = x if x is not None else synth.make_inputs(w)
    out = run_gpu(x, w.dtype)
    ref = oracle.attention(x["q"], x["k"], x["v"], mask=w.mask, kv_lens=x["kv_lens"], bias=x["bias"],
                           scale=x["scale"], dtype=w.dtype)
    got = to_f64(out)
    err = rel_err(got, ref)
    assert err <= TOL[w.dtype], f"{w.name}: rel err {err:.3e} > {TOL[w.dtype]}"
    return x, got, ref


def full_size_check(w, capsys):
    """The whole output of a full-size workload against the oracle, plus the
    size-independent invariant that causal row 0 equals V[0] bit for bit."""
    import torch
    x = synth.make_inputs(w)
    out = run_gpu(x, w.dtype)
    torch.cuda.synchronize()
    got = to_f64(out)
    ref = oracle.attention(x["q"], x["k"], x["v"], mask=w.mask, kv_lens=x["kv_lens"], bias=x["bias"],
                           scale=x["scale"], dtype=w.dtype)
    err = rel_err(got, ref)
    with capsys.disabled():
        print(f"\n{w.name}: max|O_gpu - O_ref| / max|O_ref| = {err:.3e} over {got.size} elements "
              f"(tol {TOL[w.dtype]:.1e})")
    assert err <= TOL[w.dtype], f"{w.name}: rel err {err:.3e} > {TOL[w.dtype]}"
    del ref
    if w.causal and w.Sq == w.Sk:
        v0 = to_f64(to_device(x["v"], w.dtype)[:, :, 0, :])
        g = w.Hq // w.Hkv
        np.testing.assert_array_equal(got[:, :, 0, :], np.repeat(v0, g, axis=1))
    return out


# ------------------------------------------------------------------ the workloads
@pytest.mark.parametrize("name", ["f32_causal_small", "bf16_block_d32", "bf16_block_d64"])
def test_workload_full(name):
    full_check(synth.WORKLOADS[name])


def test_padding_bias_workload_full():
    """F16 key padding + fp32 bias [1,16,1024,1024], every output element."""
    full_check(synth.WORKLOADS["f16_padding_bias"])


@pytest.mark.parametrize("name", ["bf16_causal_4k", "bf16_causal_4k_wide", "bf16_gqa_8k"])
def test_workload_full_size(name, capsys):
    """The headline workloads at full size, every output element."""
    full_size_check(synth.WORKLOADS[name], capsys)


# ------------------------------------------------------------------ coverage grid
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("mask", [0, CAUSAL, PAD, CAUSAL | PAD])
def test_tensor_core_grid(dtype, D, mask):
    """Several tiles in both directions, ragged tails, GQA group 2."""
    w = synth.Workload(f"grid_{dtype}_{D}_{mask}", dtype, 2, 4, 2, 300, 333, D, mask=mask,
                       seed=11 + D + mask, kv_len_range=(1, 333))
    full_check(w)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("bias_bh", [(1, 1), (2, 1), (1, 4), (2, 4)])
def test_bias_broadcasts(dtype, bias_bh):
    D = 64 if dtype != "f32" else 32
    w = synth.Workload("bias", dtype, 2, 4, 4, 200, 260, D, mask=CAUSAL | PAD, bias=True,
                       bias_b=bias_bh[0], bias_h=bias_bh[1], seed=21, kv_len_range=(100, 260))
    full_check(w)


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("mask", [0, CAUSAL, PAD, CAUSAL | PAD])
def test_f32_grid(D, mask):
    w = synth.Workload("f32grid", "f32", 2, 4, 2, 150, 170, D, mask=mask, seed=31 + D,
                       kv_len_range=(1, 170))
    full_check(w)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_gqa_groups(dtype, group):
    D = 128 if dtype == "bf16" else 64
    w = synth.Workload("gqa", dtype, 2, 8, 8 // group, 256, 256, D, mask=CAUSAL, seed=41 + group)
    full_check(w)


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("sq_sk", [(1, 1), (1, 300), (300, 1), (129, 127), (256, 256), (257, 513),
                                   (513, 200)])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_and_unequal_lengths(dtype, sq_sk, causal):
    """Bottom-right causal alignment; Sq > Sk leaves early rows with no key (NaN)."""
    Sq, Sk = sq_sk
    D = 64 if dtype != "f32" else 32
    w = synth.Workload("ragged", dtype, 1, 2, 1, Sq, Sk, D, mask=CAUSAL if causal else 0, seed=51)
    full_check(w)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_key_padding_extremes(dtype):
    """kv_len 0 (NaN rows), negative (clamped to 0), above Sk (clamped to Sk), 1, exact tile edges."""
    D = 128 if dtype == "bf16" else 32
    w = synth.Workload("pad", dtype, 7, 2, 2, 140, 384, D, mask=PAD, seed=61)
    x = synth.make_inputs(w.replace(kv_len_range=(0, 1)))
    x["kv_lens"] = np.array([0, -5, 1000, 1, 128, 256, 383], dtype=np.int32)
    full_check(w, x)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_no_keys_gives_nan(dtype):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    D = 64 if dtype != "f32" else 32
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]
    q = torch.randn(2, 2, 5, D, device="cuda").to(tdt)
    k = torch.empty(2, 2, 0, D, device="cuda", dtype=tdt)
    out = attn.fwd(q, k, k.clone())
    assert torch.isnan(out).all()


def test_empty_batch_is_noop():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    q = torch.empty(0, 2, 5, 64, device="cuda", dtype=torch.bfloat16)
    out = attn.fwd(q, q.clone(), q.clone())
    assert out.shape == q.shape


def test_minus_inf_bias_everywhere_gives_nan_rows():
    w = synth.Workload("ninf", "bf16", 1, 2, 2, 130, 140, 64, bias=True, bias_b=1, bias_h=2, seed=71)
    x = synth.make_inputs(w)
    x["bias"][:, :, 5, :] = -np.inf   # row 5: every key -inf
    x["bias"][:, :, 7, 3:] = -np.inf  # row 7: only keys 0..2 remain
    full_check(w, x)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_causal_row0_exact(dtype):
    D = 128 if dtype != "f32" else 64
    w = synth.Workload("row0", dtype, 2, 4, 4, 512, 512, D, mask=CAUSAL, seed=81, sigma_qk=3.0)
    x = synth.make_inputs(w)
    out = run_gpu(x, dtype)
    v = to_device(x["v"], dtype)
    assert torch_equal(out[:, :, 0, :], v[:, :, 0, :])


def torch_equal(a, b):
    import torch
    return bool(torch.equal(a, b))


def test_deterministic_and_guard_bands():
    """Two runs give identical bits; nothing outside `out` is written."""
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = synth.Workload("det", "bf16", 2, 4, 4, 384, 384, 128, mask=CAUSAL, seed=91)
    x = synth.make_inputs(w)
    q, k, v = (to_device(x[n], "bf16") for n in ("q", "k", "v"))
    n = q.numel()
    pad = 4096
    buf = torch.full((n + 2 * pad,), 1234.5, device="cuda", dtype=torch.bfloat16)
    out = buf[pad:pad + n].view(q.shape)
    attn.fwd(q, k, v, causal=True, scale=x["scale"], out=out)
    first = out.clone()
    attn.fwd(q, k, v, causal=True, scale=x["scale"], out=out)
    torch.cuda.synchronize()
    assert torch.equal(first, out)
    assert bool((buf[:pad] == 1234.5).all()) and bool((buf[pad + n:] == 1234.5).all())


def test_side_stream_and_host_buffers():
    """A non-default stream, and host tensors in/out (copies around the kernel)."""
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = synth.Workload("host", "f16", 2, 4, 2, 200, 300, 64, mask=CAUSAL, seed=101)
    x = synth.make_inputs(w)
    ref = oracle.attention(x["q"], x["k"], x["v"], mask=w.mask, scale=x["scale"], dtype="f16")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = run_gpu(x, "f16")
    s.synchronize()
    assert rel_err(to_f64(out), ref) <= TOL["f16"]
    qh, kh, vh = (to_device(x[n], "f16", "cpu").pin_memory() for n in ("q", "k", "v"))
    out_h = attn.fwd(qh, kh, vh, causal=True, scale=x["scale"])
    assert out_h.device.type == "cpu"
    assert rel_err(to_f64(out_h), ref) <= TOL["f16"]


def test_binding_rejects_bad_tensors():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    q = torch.randn(1, 2, 8, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(attn.AttnError):
        attn.fwd(q, q.half(), q)  # dtype mismatch
    with pytest.raises(attn.AttnError):
        attn.fwd(q.transpose(2, 3), q, q)  # not contiguous
    with pytest.raises(attn.AttnError):
        attn.fwd(q, q, q, scale=-1.0)  # C-ABI scale check
    with pytest.raises(attn.AttnError):
        attn.fwd(q[..., :48].contiguous(), q[..., :48].contiguous(), q[..., :48].contiguous())  # D=48


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D,Sk,path", [(32, 300, "staged"), (64, 516, "staged"), (64, 259, "direct"),
                                       (128, 260, "direct"), (128, 131, "direct")])
def test_bias_staged_and_direct_paths(dtype, D, Sk, path):
    """The bias goes through a TMA-staged shared-memory ring for D <= 64 with
    16-byte rows, and is read directly otherwise; both must match the oracle,
    with key padding, causal masking and per-head bias on several key tiles."""
    w = synth.Workload("biaspath", dtype, 2, 4, 2, 290, Sk, D, mask=CAUSAL | PAD, bias=True,
                       bias_b=2, bias_h=4, seed=111 + D + Sk, kv_len_range=(Sk // 3, Sk))
    full_check(w)
