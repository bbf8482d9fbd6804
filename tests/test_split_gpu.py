"""GPU parity of split-KV attention with the row log-sum-exp output
(attn_fwd_split) against the float64 oracle.

Split-KV (ruDNN user guide, section 9) cuts each row's keys into parts with
FP32 partial statistics and merges them; the merged output is the same
softmax as the unsplit one, so O is held to the same tolerance as attn_fwd
(max|O_gpu - O_ref| / max|O_ref| <= 1e-5 F32, 4e-3 F16, 1.6e-2 BF16).

LSE tolerance: the log-sum-exp is computed from fp32 scores, an fp32 running
max and an fp32 sum of exp2 terms (relative error of a few 2^-22 per term), so
its absolute error is a few 1e-6 times max(1, |lse|) plus the scores' own
rounding; the tests allow 1e-4 * max(1, |lse|), three orders of magnitude
below the effect of any plausible mistake (a missing ln 2 factor, a dropped
maximum, a lost part). Rows with no visible key must be NaN in O and -inf in
lse on both sides.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_flash_gb300 import synth
from tests.gpu_util import TOL, rel_err, to_device, to_f64

pytestmark = pytest.mark.gpu
CAUSAL, PAD = synth.MASK_CAUSAL, synth.MASK_KEY_PADDING
LSE_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _clean_status():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    torch.cuda.synchronize()
    attn.device_status(torch.cuda.current_device(), clear=True)
    yield
    torch.cuda.synchronize()
    assert attn.device_status(torch.cuda.current_device(), clear=True) == 0, "a kernel wait timed out"


def run_split(x, dtype, num_splits, workspace=None):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    q, k, v = (to_device(x[n], dtype) for n in ("q", "k", "v"))
    lens = to_device(x["kv_lens"], "i32") if x["kv_lens"] is not None else None
    bias = to_device(x["bias"], "f32") if x["bias"] is not None else None
    out = torch.full_like(q, 777.0)  # sentinel: a row the kernels skip cannot pass
    o, lse = attn.fwd(q, k, v, causal=bool(x["mask"] & CAUSAL), kv_lens=lens, bias=bias, scale=x["scale"],
                      out=out, num_splits=num_splits, return_lse=True, workspace=workspace)
    return to_f64(o), lse.cpu().numpy().astype(np.float64)


def lse_err(got, ref):
    """max |got - ref| / max(1, |ref|) over finite ref; -inf positions must agree."""
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf), "-inf pattern of lse differs"
    assert not np.isnan(got).any(), "lse has NaN"
    fin = ~ninf
    if not fin.any():
        return 0.0
    return float(np.max(np.abs(got[fin] - ref[fin]) / np.maximum(1.0, np.abs(ref[fin]))))


def check(w, splits, x=None):
    x = x if x is not None else synth.make_inputs(w)
    ref, ref_lse = oracle.attention(x["q"], x["k"], x["v"], mask=w.mask, kv_lens=x["kv_lens"], bias=x["bias"],
                                    scale=x["scale"], dtype=w.dtype, lse=True)
    for ns in splits:
        got, lse = run_split(x, w.dtype, ns)
        err = rel_err(got, ref)
        assert err <= TOL[w.dtype], f"{w.name} splits={ns}: O rel err {err:.3e}"
        e2 = lse_err(lse, ref_lse)
        assert e2 <= LSE_TOL, f"{w.name} splits={ns}: lse err {e2:.3e}"
    return x, ref, ref_lse


def W(name, dtype, B, Hq, Hkv, Sq, Sk, D, **kw):
    return synth.Workload(name, dtype, B, Hq, Hkv, Sq, Sk, D, **kw)


# Sq below one 256-row block and above it; Sk over several 128-key tiles with
# a ragged tail; splits from 1 to more than the number of tiles.
TC_CASES = [
    W("split_bf16_d128_causal", "bf16", 2, 4, 2, 100, 1000, 128, mask=CAUSAL, seed=11),
    W("split_bf16_d128_full", "bf16", 1, 4, 4, 300, 777, 128, seed=12),
    W("split_f16_d64_causal", "f16", 2, 2, 1, 333, 900, 64, mask=CAUSAL, seed=13),
    W("split_bf16_d32_full", "bf16", 1, 3, 3, 64, 1500, 32, seed=14),
]


@pytest.mark.parametrize("w", TC_CASES, ids=lambda w: w.name)
def test_split_tensor_core(w):
    check(w, (1, 2, 3, 7, 32))


@pytest.mark.parametrize("D", [16, 64, 128])
def test_split_f32(D):
    w = W(f"split_f32_d{D}", "f32", 2, 2, 1, 70, 500, D, mask=CAUSAL, seed=15)
    check(w, (1, 2, 5, 32))


@pytest.mark.parametrize("dtype,D", [("f16", 64), ("bf16", 128), ("f32", 32)])
def test_split_padding_bias(dtype, D):
    # key padding with every length case (0 keys, partial tile, full) and a
    # per-head bias; D=64 takes the TMA-staged bias ring, D=128 the direct read
    w = W(f"split_pad_bias_{dtype}", dtype, 4, 2, 2, 130, 600, D, mask=PAD, bias=True, bias_b=1, bias_h=2,
          seed=16, kv_len_range=(0, 600))
    x = synth.make_inputs(w)
    x["kv_lens"] = np.array([0, 1, 129, 600], dtype=np.int32)
    check(w, (1, 3, 8), x)


def test_split_causal_more_queries_than_keys():
    # bottom-right causal with Sq > Sk: the top Sq - Sk rows see no key
    w = W("split_causal_sq_gt_sk", "bf16", 1, 2, 2, 400, 300, 64, mask=CAUSAL, seed=17)
    x, ref, ref_lse = check(w, (1, 2, 4))
    assert np.isneginf(ref_lse[..., :100]).all() and np.isfinite(ref_lse[..., 100:]).all()


def test_split_no_keys():
    w = W("split_no_keys", "bf16", 1, 2, 2, 16, 0, 64, seed=18)
    x = synth.make_inputs(w)
    for ns in (1, 4):
        got, lse = run_split(x, "bf16", ns)
        assert np.isnan(got).all() and np.isneginf(lse).all()


def test_one_split_matches_attn_fwd_bitwise():
    # num_splits == 1 runs the attn_fwd kernel itself: O is bit-identical
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = W("split_one", "bf16", 2, 4, 2, 300, 700, 128, mask=CAUSAL, seed=19)
    x = synth.make_inputs(w)
    q, k, v = (to_device(x[n], "bf16") for n in ("q", "k", "v"))
    a = attn.fwd(q, k, v, causal=True, scale=x["scale"])
    b, lse = attn.fwd(q, k, v, causal=True, scale=x["scale"], num_splits=1, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_split_workspace_reuse_is_deterministic():
    # the same workspace, dirty from an earlier call of another shape, gives
    # bit-identical results on repeated calls
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = W("split_reuse", "bf16", 1, 8, 2, 200, 2000, 128, mask=CAUSAL, seed=20)
    x = synth.make_inputs(w)
    ws = torch.full((64 << 20,), 0xFF, dtype=torch.uint8, device="cuda")
    other = synth.make_inputs(W("split_other", "bf16", 2, 8, 8, 256, 512, 128, seed=21))
    run_split(other, "bf16", 6, workspace=ws)
    o1, l1 = run_split(x, "bf16", 5, workspace=ws)
    o2, l2 = run_split(x, "bf16", 5, workspace=ws)
    assert np.array_equal(o1, o2, equal_nan=True) and np.array_equal(l1, l2)
    ref = oracle.attention(x["q"], x["k"], x["v"], mask=w.mask, scale=x["scale"], dtype="bf16")
    assert rel_err(o1, ref) <= TOL["bf16"]


def test_split_workspace_too_small_is_an_error():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = W("split_small_ws", "bf16", 1, 2, 2, 64, 512, 64, seed=22)
    x = synth.make_inputs(w)
    q, k, v = (to_device(x[n], "bf16") for n in ("q", "k", "v"))
    shape = attn.Shape(1, 2, 2, 64, 512, 64, 1, 1)
    need = attn.split_workspace_bytes(shape, 4)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.call_split(shape, q.data_ptr(), k.data_ptr(), v.data_ptr(), 0, 0, 0, x["scale"], attn.ATTN_BF16,
                        4, ws.data_ptr(), need - 16, torch.empty_like(q).data_ptr(), 0,
                        torch.cuda.current_stream().cuda_stream)
    assert e.value.code == -12


def test_split_chunk_32k_sampled():
    # the benchmark's split-KV workload at full size, in the launch the
    # benchmark times, on sampled rows (newest and oldest rows of every head)
    import bench
    w = synth.WORKLOADS["bf16_gqa_chunk_32k"]
    x = synth.make_inputs(w)
    got, lse = run_split(x, w.dtype, bench.SPLITS[w.name])
    rng = np.random.default_rng(3)
    rows = [(0, h, i) for h in range(0, w.Hq, 5) for i in sorted({0, 1, 127, 128, 255} |
                                                                  set(int(r) for r in rng.integers(0, w.Sq, 4)))]
    ref, ref_lse = oracle.attention_rows(x["q"], x["k"], x["v"], rows, mask=w.mask, scale=x["scale"],
                                         dtype=w.dtype, lse=True)
    g = np.stack([got[b, h, i] for b, h, i in rows])
    gl = np.array([lse[b, h, i] for b, h, i in rows])
    assert rel_err(g, ref) <= TOL["bf16"]
    assert lse_err(gl, ref_lse) <= LSE_TOL
