"""GPU parity of attention over a paged key/value cache with packed queries
(attn_paged_fwd) against the float64 oracle (ruDNN user guide, section 9).

Tolerance: max|O_gpu - O_ref| / max|O_ref| as for the dense forward (1e-5
F32, 4e-3 F16, 1.6e-2 BF16); rows that see no key must be NaN on both sides;
lse within 1e-4 * max(1, |lse|), -inf where the oracle has -inf.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_flash_gb300 import synth
from tests.gpu_util import TOL, rel_err, to_device, to_f64

pytestmark = pytest.mark.gpu
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


def run_paged(w, x, num_splits=1):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    q, k, v = (to_device(x[n], w.dtype) for n in ("q", "k_cache", "v_cache"))
    ints = {n: to_device(x[n], "i32") for n in ("block_table", "seq_lens", "q_offsets")}
    pos = to_device(x["positions"], "i32") if x["positions"] is not None else None
    out = torch.full_like(q, 777.0)  # sentinel: a row the kernel skips cannot pass
    o, lse = attn.paged_fwd(q, k, v, ints["block_table"], ints["seq_lens"], ints["q_offsets"], positions=pos,
                            causal=w.causal, scale=x["scale"], return_lse=True, out=out, num_splits=num_splits)
    return to_f64(o), lse.cpu().numpy().astype(np.float64)


def check(w, x=None, num_splits=1):
    x = x if x is not None else synth.make_paged_inputs(w)
    got, lse = run_paged(w, x, num_splits)
    ref, ref_lse = oracle.paged_attention(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["seq_lens"],
                                          x["q_offsets"], positions=x["positions"], causal=w.causal,
                                          scale=x["scale"], dtype=w.dtype, lse=True)
    err = rel_err(got, ref)
    assert err <= TOL[w.dtype], f"{w.name}: rel err {err:.3e}"
    ninf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), ninf)
    fin = ~ninf
    if fin.any():
        e2 = np.max(np.abs(lse[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin])))
        assert e2 <= LSE_TOL, f"{w.name}: lse err {e2:.3e}"
    return x, got, ref


def PW(name, dtype, ns, Hq, Hkv, D, P, ctx, qr, **kw):
    return synth.PagedWorkload(name, dtype, ns, Hq, Hkv, D, P, ctx, qr, **kw)


CASES = [
    PW("paged_bf16_d128_p16_prefill", "bf16", 4, 8, 2, 128, 16, (100, 700), (50, 300), seed=1),
    PW("paged_bf16_d128_p128_decode", "bf16", 9, 8, 2, 128, 128, (1, 1500), (1, 1), seed=2),
    PW("paged_f16_d64_p64_mixed", "f16", 6, 4, 4, 64, 64, (1, 900), (1, 200), seed=3),
    PW("paged_f32_d32_p8_positions", "f32", 5, 4, 1, 32, 8, (5, 300), (1, 60), seed=4, explicit_positions=True),
    PW("paged_bf16_d64_p256_noncausal", "bf16", 3, 6, 2, 64, 256, (200, 800), (10, 100), seed=5, causal=False),
    PW("paged_f16_d16_p1", "f16", 3, 2, 2, 16, 1, (1, 40), (1, 20), seed=6),
    # tensor-core kernel, GQA heads packed into the rows: group 8 prefill with
    # positions, group 6 (does not divide 128: one head per CTA), MQA group 32
    PW("paged_bf16_d128_g8_positions", "bf16", 3, 32, 4, 128, 32, (60, 500), (20, 90), seed=9,
       explicit_positions=True),
    PW("paged_f16_d64_g6_prefill", "f16", 3, 12, 2, 64, 16, (40, 400), (5, 70), seed=10),
    PW("paged_bf16_d64_mqa_g32", "bf16", 4, 32, 1, 64, 64, (1, 600), (1, 6), seed=11),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_paged_matches_oracle(w):
    check(w)


def test_paged_empty_sequences_and_no_queries():
    # a sequence with no keys (its queries are NaN) and one with no queries
    w = PW("paged_edges", "bf16", 4, 4, 2, 64, 16, (0, 120), (0, 30), seed=7, explicit_positions=True)
    x = synth.make_paged_inputs(w)
    x["seq_lens"][1] = 0
    nq = np.diff(x["q_offsets"])
    x["block_table"][1, :] = -1
    check(w, x)
    assert (nq >= 0).all()


def test_paged_decode_equals_dense():
    # one query per sequence at its last position over the same keys as a dense call
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = PW("paged_vs_dense", "bf16", 3, 8, 2, 128, 32, (300, 300), (1, 1), seed=8)
    x = synth.make_paged_inputs(w)
    got, _ = run_paged(w, x)
    # rebuild the dense caches from the pages and run the dense forward
    P, L = 32, 300
    kd = np.stack([np.concatenate([x["k_cache"][x["block_table"][s, p]] for p in range((L + P - 1) // P)])[:L]
                   for s in range(3)]).transpose(0, 2, 1, 3)
    vd = np.stack([np.concatenate([x["v_cache"][x["block_table"][s, p]] for p in range((L + P - 1) // P)])[:L]
                   for s in range(3)]).transpose(0, 2, 1, 3)
    qd = x["q"].reshape(3, 1, 8, 128).transpose(0, 2, 1, 3)
    dense = attn.fwd(*(to_device(np.ascontiguousarray(a), "bf16") for a in (qd, kd, vd)), causal=True,
                     scale=x["scale"])
    torch.cuda.synchronize()
    ref = to_f64(dense).transpose(0, 2, 1, 3).reshape(3, 8, 128)
    assert rel_err(got, ref) <= TOL["bf16"]


def test_paged_argument_errors():
    import ctypes
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    lib = attn.load_library()
    dev = torch.device("cuda")
    q = torch.zeros(4, 2, 64, device=dev, dtype=torch.bfloat16)
    kc = torch.zeros(3, 16, 2, 64, device=dev, dtype=torch.bfloat16)
    tab = torch.zeros(1, 3, dtype=torch.int32, device=dev)
    lens = torch.tensor([40], dtype=torch.int32, device=dev)
    offs = torch.tensor([0, 4], dtype=torch.int32, device=dev)
    out = torch.empty_like(q)

    def call(shape=None, causal=1, scale=0.125, o=out):
        shape = shape or attn.PagedShape(1, 4, 2, 2, 64, 16, 3, 3, 4)
        return lib.attn_paged_fwd(ctypes.byref(shape), q.data_ptr(), kc.data_ptr(), kc.data_ptr(), tab.data_ptr(),
                                  lens.data_ptr(), offs.data_ptr(), None, causal, ctypes.c_float(scale),
                                  attn.ATTN_BF16, 1, None, 0, o.data_ptr(), None, None)
    assert call() == 0
    torch.cuda.synchronize()
    assert call(shape=attn.PagedShape(1, 4, 3, 2, 64, 16, 3, 3, 4)) == -2   # Hq % Hkv
    assert call(shape=attn.PagedShape(1, 4, 2, 2, 48, 16, 3, 3, 4)) == -4   # head dim
    assert call(causal=2) == -7
    assert call(scale=0.0) == -6
    assert call(o=q) == -8                                                  # out overlaps q


@pytest.mark.parametrize("splits", [2, 5, 32])
def test_paged_decode_splits(splits):
    # decode-shaped calls with the key range split and merged (every length
    # case: fewer chunks than splits, a sequence without keys, explicit positions)
    w = PW(f"paged_decode_split{splits}", "bf16", 7, 8, 2, 128, 32, (0, 2000), (1, 2), seed=30 + splits,
           explicit_positions=True)
    check(w, num_splits=splits)
    w2 = PW(f"paged_decode_split{splits}_f32", "f32", 5, 4, 4, 64, 16, (1, 700), (1, 1), seed=40 + splits)
    check(w2, num_splits=splits)
    # tensor-core decode: group 6 (one head per CTA) and group 8 with two queries
    w3 = PW(f"paged_decode_split{splits}_g6", "f16", 4, 12, 2, 64, 128, (1, 1200), (1, 1), seed=60 + splits)
    check(w3, num_splits=splits)
    w4 = PW(f"paged_decode_split{splits}_g4q2", "bf16", 5, 16, 4, 128, 64, (2, 2500), (2, 2), seed=70 + splits,
            causal=splits % 2 == 0)
    check(w4, num_splits=splits)


def test_paged_split_workspace_errors():
    from exact_scaled_dot_flash_gb300 import attn
    decode = attn.PagedShape(4, 4, 8, 2, 128, 16, 10, 5, 1)   # 1 query x group 4 <= 8 rows: decode kernel
    prefill = attn.PagedShape(4, 40, 8, 2, 128, 16, 10, 5, 10)
    assert attn.paged_workspace_bytes(decode, 1) == 0
    assert attn.paged_workspace_bytes(decode, 4) > 0
    assert attn.paged_workspace_bytes(prefill, 4) == 0       # the prefill kernel does not split
    with pytest.raises(attn.AttnError):
        attn.paged_workspace_bytes(decode, 33)
