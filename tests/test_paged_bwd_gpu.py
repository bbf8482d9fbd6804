"""GPU parity of the backward over a paged cache (attn_paged_bwd and
attn_paged_mla_bwd) against the float64 oracle. F16/BF16 cases with D in
{64, 128} (paged attention) or R in {256, 512} and Pd in {0, 64} (MLA) and
page sizes of 8..256 take the tensor-core kernels (with the fp32 FMA key-major
kernel for shared and unread pages); the others the fp32 FMA kernels
throughout.

The pipeline is the user's: the CUDA paged forward with its log-sum-exp, then
the CUDA backward on (inputs, out, dout, lse); the oracle computes every
gradient from the inputs and dout alone. Tolerance per gradient tensor:
max|g - g_ref| / max|g_ref| <= 1e-5 (F32), 4e-3 (F16), 1.6e-2 (BF16), the
bounds of the dense backward. The cache gradients cover every physical page
(pages nobody reads must come back zero), and shared-prefix cases give two
sequences the same physical pages, whose gradients then sum both readers.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_flash_gb300 import synth
from tests.gpu_util import TOL, to_device, to_f64

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


def grad_err(name, got, ref):
    assert not np.isnan(got).any(), f"{name} has NaN"
    denom = np.abs(ref).max()
    return float(np.abs(got - ref).max() / max(denom, 1e-300))


def share_prefix(x, P, blocks):
    """Sequence 1 reads sequence 0's first ``blocks`` physical pages in place
    of its own (a shared prefix); its old pages become nobody's."""
    lens, table = x["seq_lens"], x["block_table"].copy()
    blocks = min(blocks, int(lens[0]) // P, (int(lens[1]) + P - 1) // P)
    assert blocks > 0, "the first two sequences are too short to share a page"
    freed = table[1, :blocks].copy()
    table[1, :blocks] = table[0, :blocks]
    return {**x, "block_table": table}, freed


def dout_like(seed, q, dtype):
    return synth.to_storage(synth.normal_f32(seed, 9, q.shape), dtype)


def ints(x):
    d = {n: to_device(x[n], "i32") for n in ("block_table", "seq_lens", "q_offsets")}
    d["positions"] = to_device(x["positions"], "i32") if x["positions"] is not None else None
    return d


def max_q(x):
    return int(np.diff(x["q_offsets"]).max()) if len(x["seq_lens"]) else 0


def run_paged(w, x, g, grads=("dq", "dk", "dv")):
    from exact_scaled_dot_flash_gb300 import attn
    q, kc, vc = (to_device(x[n], w.dtype) for n in ("q", "k_cache", "v_cache"))
    m = ints(x)
    return attn.paged_bwd(q, kc, vc, m["block_table"], m["seq_lens"], m["q_offsets"], to_device(g, w.dtype),
                          positions=m["positions"], causal=w.causal, scale=x["scale"], max_queries=max_q(x),
                          grads=grads)


def check_paged(w, x=None):
    x = x if x is not None else synth.make_paged_inputs(w)
    g = dout_like(w.seed, x["q"], w.dtype)
    got = [to_f64(t) for t in run_paged(w, x, g)]
    ref = oracle.paged_attention_bwd(x["q"], x["k_cache"], x["v_cache"], g, x["block_table"], x["seq_lens"],
                                     x["q_offsets"], positions=x["positions"], causal=w.causal, scale=x["scale"],
                                     dtype=w.dtype)
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        err = grad_err(name, a, b)
        assert err <= TOL[w.dtype], f"{w.name} {name}: rel err {err:.3e} > {TOL[w.dtype]}"
    return x, got, ref


PW = synth.PagedWorkload
PAGED_CASES = [
    PW("pbwd_f32_d16_p1", "f32", 3, 2, 2, 16, 1, (5, 40), (1, 6), seed=1),
    PW("pbwd_f32_d64_gqa4_p16_pos", "f32", 4, 8, 2, 64, 16, (20, 200), (1, 40), seed=2, explicit_positions=True),
    PW("pbwd_bf16_d128_gqa4_p64", "bf16", 5, 8, 2, 128, 64, (64, 700), (1, 130), seed=3),
    PW("pbwd_f16_d32_p96_full", "f16", 4, 4, 4, 32, 96, (1, 400), (1, 20), seed=4, causal=False),
    PW("pbwd_bf16_d64_mqa_p256", "bf16", 3, 4, 1, 64, 256, (300, 900), (1, 70), seed=5),
    PW("pbwd_bf16_d128_decode_p16", "bf16", 8, 16, 4, 128, 16, (100, 1500), (1, 1), seed=6),
    PW("pbwd_f16_d128_prefill_p8_pos", "f16", 3, 4, 2, 128, 8, (100, 300), (50, 300), seed=7,
       explicit_positions=True),
    # a group of 6 (does not divide 128): one head per tile on the tensor cores
    PW("pbwd_bf16_d64_g6_p32", "bf16", 3, 12, 2, 64, 32, (100, 400), (1, 150), seed=8),
    PW("pbwd_f16_d64_p128_full", "f16", 3, 4, 2, 64, 128, (200, 700), (1, 200), seed=9, causal=False),
]


@pytest.mark.parametrize("w", PAGED_CASES, ids=lambda w: w.name)
def test_paged_bwd_matches_oracle(w):
    check_paged(w)


# The key-major kernel streams the key blocks of a (sequence, kv head) through
# one CTA per run of 8 blocks when the query side is a single tile (every head
# of the group in one block, at most 128 (query, head) pairs): decode steps and
# short chunks; with at most 32 pairs, on 32-pair tiles. Sequences of several
# runs, page sizes below and above a block, explicit positions and the
# non-causal form.
STREAM_CASES = [
    PW("pbwd_stream_bf16_d128_p8_long", "bf16", 4, 16, 4, 128, 8, (1500, 3100), (1, 1), seed=41),
    PW("pbwd_stream_f16_d64_p256_pos", "f16", 5, 8, 2, 64, 256, (200, 2600), (1, 12), seed=42,
       explicit_positions=True),
    PW("pbwd_stream_bf16_d128_p32_full", "bf16", 3, 8, 1, 128, 32, (900, 1400), (1, 16), seed=43, causal=False),
    # at most 32 pairs: the narrow variant (32-pair tiles)
    PW("pbwd_narrow_f16_d64_p64_pos", "f16", 4, 8, 2, 64, 64, (300, 2100), (1, 6), seed=44, explicit_positions=True),
    PW("pbwd_narrow_bf16_d128_p128_full", "bf16", 3, 16, 2, 128, 128, (500, 1500), (1, 4), seed=45, causal=False),
]


@pytest.mark.parametrize("w", STREAM_CASES, ids=lambda w: w.name)
def test_paged_bwd_streamed_key_blocks(w):
    check_paged(w)


@pytest.mark.parametrize("P", [16, 64, 256])
def test_paged_bwd_shared_prefix_pages_sum_both_readers(P):
    w = PW(f"pbwd_share_p{P}", "bf16", 4, 8, 2, 64, P, (2 * P + 5, 4 * P), (1, 9), seed=10 + P)
    x, freed = share_prefix(synth.make_paged_inputs(w), P, 2)
    _, got, ref = check_paged(w, x)
    # the pages sequence 1 no longer reads get nothing
    assert not got[1][freed].any() and not got[2][freed].any()


def test_paged_bwd_empty_sequences_rows_without_keys_and_spare_pages():
    # sequence 1 has queries but no keys (its rows see nothing: dq = 0);
    # sequence 2 has keys but no queries (its pages get zero gradients)
    w = PW("pbwd_edges", "f16", 4, 4, 2, 64, 16, (30, 90), (2, 5), seed=21, spare_pages=5)
    x = synth.make_paged_inputs(w)
    lens, offs = x["seq_lens"].copy(), x["q_offsets"].copy()
    lens[1] = 0
    n2 = offs[3] - offs[2]
    q = np.concatenate([x["q"][:offs[2]], x["q"][offs[3]:]])
    offs = np.concatenate([offs[:3], offs[3:] - n2]).astype(np.int32)
    x = {**x, "q": q, "seq_lens": lens, "q_offsets": offs}
    _, got, _ = check_paged(w, x)
    assert not got[0][offs[1]:offs[2]].any()
    used2 = x["block_table"][2, :(int(lens[2]) + 15) // 16]
    assert not got[1][used2].any() and not got[2][used2].any()


def test_paged_bwd_is_deterministic_and_skips_unwanted_gradients():
    import torch
    w = PAGED_CASES[2]
    x = synth.make_paged_inputs(w)
    g = dout_like(w.seed, x["q"], w.dtype)
    a = run_paged(w, x, g)
    b = run_paged(w, x, g)
    only_dk = run_paged(w, x, g, grads=("dk",))
    only_dq = run_paged(w, x, g, grads=("dq",))
    torch.cuda.synchronize()
    for t, u in zip(a, b):
        assert torch.equal(t.view(torch.int16), u.view(torch.int16))
    assert only_dk[0] is None and only_dk[2] is None and torch.equal(only_dk[1], a[1])
    assert only_dq[1] is None and only_dq[2] is None and torch.equal(only_dq[0], a[0])


def test_paged_bwd_without_queries_zeroes_the_cache_gradients():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    kc = torch.randn(5, 16, 2, 64, device="cuda", dtype=torch.float16)
    vc = torch.randn_like(kc)
    q = torch.empty(0, 4, 64, device="cuda", dtype=torch.float16)
    table = torch.zeros(2, 3, dtype=torch.int32, device="cuda")
    lens = torch.tensor([20, 30], dtype=torch.int32, device="cuda")
    offs = torch.zeros(3, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(0, 4, dtype=torch.float32, device="cuda")
    dq, dk, dv = attn.paged_bwd(q, kc, vc, table, lens, offs, torch.empty_like(q), out=out, lse=lse,
                                scale=0.125, max_queries=0)
    torch.cuda.synchronize()
    assert dq.numel() == 0 and not dk.any() and not dv.any()


# ------------------------------------------------------------------- MLA

def run_mla(w, x, g, grads=("dq", "dqp", "dlatent", "dkpos")):
    from exact_scaled_dot_flash_gb300 import attn
    q, qp, lat, kp = (to_device(x[n], w.dtype) for n in ("q", "qp", "latent", "kpos"))
    m = ints(x)
    return attn.paged_mla_bwd(q, qp, lat, kp, m["block_table"], m["seq_lens"], m["q_offsets"], to_device(g, w.dtype),
                              positions=m["positions"], causal=w.causal, scale=x["scale"], max_queries=max_q(x),
                              grads=grads)


def check_mla(w, x=None):
    x = x if x is not None else synth.make_mla_inputs(w)
    g = dout_like(w.seed, x["q"], w.dtype)
    got = run_mla(w, x, g)
    ref = oracle.paged_mla_bwd(x["q"], x["qp"], x["latent"], x["kpos"], g, x["block_table"], x["seq_lens"],
                               x["q_offsets"], positions=x["positions"], causal=w.causal, scale=x["scale"],
                               dtype=w.dtype)
    out = []
    for name, a, b in zip(("dq", "dqp", "dlatent", "dkpos"), got, ref):
        if w.Pd == 0 and name in ("dqp", "dkpos"):
            assert a is None
            out.append(None)
            continue
        a = to_f64(a)
        err = grad_err(name, a, b)
        assert err <= TOL[w.dtype], f"{w.name} {name}: rel err {err:.3e} > {TOL[w.dtype]}"
        out.append(a)
    return x, out, ref


MW = synth.MlaWorkload
MLA_CASES = [
    MW("mbwd_f32_r128_pd16_p16", "f32", 3, 4, 128, 16, 16, (10, 100), (1, 10), seed=41),
    MW("mbwd_bf16_r512_pd64_p64", "bf16", 4, 16, 512, 64, 64, (64, 400), (1, 3), seed=42),
    MW("mbwd_f16_r256_pd0_p32_pos", "f16", 3, 8, 256, 0, 32, (30, 300), (1, 20), seed=43, explicit_positions=True),
    MW("mbwd_bf16_r512_pd32_decode", "bf16", 4, 128, 512, 32, 64, (100, 600), (1, 1), seed=44),
    MW("mbwd_f16_r128_pd64_p8_full", "f16", 3, 8, 128, 64, 8, (20, 120), (1, 12), seed=45, causal=False),
    # tensor-core kernels: decode-shaped (one 128-row tile per sequence, the
    # query-major kernel longest sequence first), several row tiles per
    # sequence, page sizes 8 and 128..256, no causal mask, Pd 0 and 64
    MW("mbwd_bf16_r512_pd64_decode_h128", "bf16", 5, 128, 512, 64, 64, (100, 700), (1, 1), seed=47),
    MW("mbwd_f16_r512_pd64_p128_prefill", "f16", 3, 16, 512, 64, 128, (200, 700), (5, 30), seed=48),
    MW("mbwd_bf16_r256_pd64_p8_full", "bf16", 3, 8, 256, 64, 8, (20, 200), (1, 12), seed=49, causal=False),
    MW("mbwd_bf16_r512_pd0_p256", "bf16", 3, 32, 512, 0, 256, (100, 600), (1, 6), seed=50),
    MW("mbwd_f16_r512_pd64_p16_pos", "f16", 3, 16, 512, 64, 16, (40, 300), (2, 17), seed=51, explicit_positions=True),
]


@pytest.mark.parametrize("w", MLA_CASES, ids=lambda w: w.name)
def test_mla_bwd_matches_oracle(w):
    check_mla(w)


def test_mla_bwd_shared_prefix_and_determinism():
    import torch
    w = MW("mbwd_share", "bf16", 3, 16, 512, 64, 16, (40, 120), (1, 4), seed=46)
    x, freed = share_prefix(synth.make_mla_inputs(w), 16, 2)
    _, got, _ = check_mla(w, x)
    assert not got[2][freed].any() and not got[3][freed].any()
    g = dout_like(w.seed, x["q"], w.dtype)
    a, b = run_mla(w, x, g), run_mla(w, x, g)
    torch.cuda.synchronize()
    for t, u in zip(a, b):
        assert torch.equal(t.view(torch.int16), u.view(torch.int16))


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64)])
def test_paged_bwd_invalid_page_entry_reads_zeros(dtype, D):
    # a table entry outside the cache inside a sequence's range reads as zero
    # keys and values (as in the forward) and receives nothing: the same as a
    # valid page of zeros, whose own gradient is simply not kept
    import torch
    w = PW(f"pbwd_invalid_{dtype}", dtype, 3, 8, 2, D, 16, (40, 120), (2, 9), seed=31, spare_pages=2)
    x = synth.make_paged_inputs(w)
    pages = x["k_cache"].shape[0]
    zero = np.zeros_like(x["k_cache"][:1])
    x_zero = {**x, "k_cache": np.concatenate([x["k_cache"], zero]), "v_cache": np.concatenate([x["v_cache"], zero])}
    t_zero = x["block_table"].copy()
    t_bad = x["block_table"].copy()
    t_zero[0, 1] = pages       # the appended zero page
    t_bad[0, 1] = pages + 50   # outside the cache
    g = dout_like(w.seed, x["q"], w.dtype)
    a = run_paged(w, {**x_zero, "block_table": t_zero}, g)
    b = run_paged(w, {**x, "block_table": t_bad}, g)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_f64(b[0]), to_f64(a[0]))
    for i in (1, 2):
        np.testing.assert_array_equal(to_f64(b[i]), to_f64(a[i])[:pages])
