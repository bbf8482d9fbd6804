"""Pins for the float64 oracle: facts fixed by the pages and by mathematics.

None of these re-types the oracle's formula. Each checks the oracle against
something independent of it: the worked values the pages print, closed forms
(identical keys, a single key, a dominant score), invariants (row-stochastic
weights, shift and permutation invariance, the convex hull of V), a textbook
single-head routine, and a 50-digit brute force of the pages' raw-exp kernel
(no max subtraction) on tiny inputs. Together they catch a dropped term, a
wrong sign or index, a transposed operand, a wrong head mapping or mask edge.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from exact_scaled_dot_flash_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CAUSAL, PAD = oracle.MASK_CAUSAL, oracle.MASK_KEY_PADDING


def rnd(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def run(q, k, v, **kw):
    kw.setdefault("scale", 1.0 / math.sqrt(q.shape[-1]))
    return oracle.attention(q, k, v, **kw)


# --------------------------------------------------------------- pages' values
def test_golden_single_row_service_example():
    """HOF Flash Attention in Rust, sections 3-5: a 1 x d row has one key, so O = V."""
    g = json.load(open(os.path.join(GOLDEN, "p3_single_row.json")))
    q, k, v = (np.array(g[n], dtype=np.float64) for n in ("q", "k", "v"))
    out, w = oracle.attention(q, k, v, scale=g["scale"], weights=True)
    np.testing.assert_array_equal(out, np.array(g["expected_out"]))
    np.testing.assert_array_equal(w, np.array(g["expected_weights"]))


def test_golden_tensai_causal_mask_pattern():
    """tensai autograd guide, assembling attention: 0 on/below the diagonal, -inf above."""
    g = json.load(open(os.path.join(GOLDEN, "tensai_causal_mask_seq4.json")))
    S = g["seq"]
    masked = np.array([[e == "-inf" for e in row] for row in g["mask"]])
    q, k, v = rnd(1, 2, 3, S, 5), rnd(2, 2, 3, S, 5), rnd(3, 2, 3, S, 5)
    _, w = run(q, k, v, mask=CAUSAL, weights=True)
    for b in range(2):
        for h in range(3):
            assert np.all(w[b, h][masked] == 0.0)
            assert np.all(w[b, h][~masked] > 0.0)


# --------------------------------------------------------------- closed forms
@pytest.mark.parametrize("mask", [0, CAUSAL, PAD, CAUSAL | PAD])
def test_identical_keys_give_mean_of_visible_values(mask):
    """All keys equal: every visible weight is 1/n, so O is a mean of V rows."""
    B, H, S, D = 2, 3, 37, 8
    q = rnd(4, B, H, S, D)
    k = np.broadcast_to(rnd(5, 1, 1, 1, D), (B, H, S, D)).copy()
    v = rnd(6, B, H, S, D)
    lens = np.array([S, 11], dtype=np.int32)
    out = run(q, k, v, mask=mask, kv_lens=lens if mask & PAD else None)
    for b in range(B):
        L = int(lens[b]) if mask & PAD else S
        csum = np.cumsum(v[b], axis=1)  # prefix sums over keys, [H, S, D]
        for i in range(S):
            n = min(L, i + 1) if mask & CAUSAL else L
            expect = csum[:, n - 1, :] / n
            np.testing.assert_allclose(out[b, :, i, :], expect, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_causal_row0_is_v0_exactly(dtype):
    """Causal row 0 sees only key 0: weight 1, so O[0] == V[0] bit for bit."""
    w = synth.WORKLOADS["f32_causal_small"].replace(dtype=dtype, seed=7)
    x = synth.make_inputs(w)
    out = oracle.attention(x["q"], x["k"], x["v"], mask=CAUSAL, scale=x["scale"], dtype=dtype)
    np.testing.assert_array_equal(out[:, :, 0, :], oracle.widen(x["v"], dtype)[:, :, 0, :])


def test_single_key_returns_that_value_row():
    q, k, v = rnd(8, 1, 2, 5, 4), rnd(9, 1, 2, 1, 4), rnd(10, 1, 2, 1, 4)
    out = run(q, k, v)
    np.testing.assert_array_equal(out, np.broadcast_to(v, out.shape))


@pytest.mark.parametrize("how", ["bias", "key"])
def test_one_dominant_score_selects_its_value_row(how):
    """A score 1e4 above the rest gets weight 1 - O(e^-1e4): O[i] = V[j*]."""
    B, H, S, D = 1, 2, 9, 4
    q, k, v = rnd(11, B, H, S, D), rnd(12, B, H, S, D), rnd(13, B, H, S, D)
    jstar = [(3 * i + 2) % S for i in range(S)]
    if how == "bias":
        bias = np.zeros((1, 1, S, S))
        for i, j in enumerate(jstar):
            bias[0, 0, i, j] = 1e4
        out = run(q, k, v, bias=bias)
        for i, j in enumerate(jstar):
            np.testing.assert_allclose(out[0, :, i], v[0, :, j], rtol=0, atol=1e-12)
    else:
        # single query row per head; K[j*] = c * Q[i] dominates Q.K
        q1 = q[:, :, :1, :]
        k2 = k.copy() * 1e-3
        k2[:, :, 5, :] = q1[:, :, 0, :] * 1e4
        out = run(q1, k2, v, scale=1.0)
        np.testing.assert_allclose(out[:, :, 0, :], v[:, :, 5, :], rtol=0, atol=1e-12)


def test_hand_solved_two_by_two():
    """Q=[[1,0],[0,1]], K=[[1,0],[0,0]], V=[[1,2],[3,4]], scale 1, solved by hand."""
    q = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    k = np.array([[[[1.0, 0.0], [0.0, 0.0]]]])
    v = np.array([[[[1.0, 2.0], [3.0, 4.0]]]])
    e = math.e
    out = run(q, k, v, scale=1.0)
    # row 0: scores (1, 0) -> weights (e, 1)/(e + 1); row 1: scores (0, 0) -> (1/2, 1/2)
    np.testing.assert_allclose(out[0, 0, 0], [(e + 3) / (e + 1), (2 * e + 4) / (e + 1)], rtol=1e-15)
    np.testing.assert_allclose(out[0, 0, 1], [2.0, 3.0], rtol=1e-15)
    out_c = run(q, k, v, scale=1.0, mask=CAUSAL)
    np.testing.assert_array_equal(out_c[0, 0, 0], [1.0, 2.0])
    np.testing.assert_allclose(out_c[0, 0, 1], [2.0, 3.0], rtol=1e-15)


# --------------------------------------------------------------- invariants
@pytest.mark.parametrize("mask", [0, CAUSAL, PAD, CAUSAL | PAD])
def test_weights_are_row_stochastic_and_zero_where_masked(mask):
    """HOF Flash Attention in Rust, section 4: A is row-stochastic."""
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 19, 23, 8
    q, k, v = rnd(14, B, Hq, Sq, D, scale=2), rnd(15, B, Hkv, Sk, D, scale=2), rnd(16, B, Hkv, Sk, D)
    lens = np.array([23, 7], dtype=np.int32)
    bias = rnd(17, 1, Hq, Sq, Sk)
    _, w = run(q, k, v, mask=mask, kv_lens=lens if mask & PAD else None, bias=bias, weights=True)
    assert np.all(np.abs(w.sum(-1) - 1.0) <= 1e-12)
    assert np.all(w >= 0)
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    for b in range(B):
        masked = np.zeros((Sq, Sk), bool)
        if mask & CAUSAL:
            masked |= j > i + (Sk - Sq)
        if mask & PAD:
            masked |= j >= lens[b]
        assert np.all(w[b][:, masked] == 0.0)
        assert np.all(w[b][:, ~masked] > 0.0)


def test_output_in_convex_hull_of_visible_values():
    B, H, S, D = 2, 2, 31, 6
    q, k, v = rnd(18, B, H, S, D, scale=3), rnd(19, B, H, S, D, scale=3), rnd(20, B, H, S, D)
    out = run(q, k, v, mask=CAUSAL)
    for i in range(S):
        lo = v[:, :, : i + 1, :].min(axis=2)
        hi = v[:, :, : i + 1, :].max(axis=2)
        assert np.all(out[:, :, i, :] >= lo - 1e-12) and np.all(out[:, :, i, :] <= hi + 1e-12)


def test_per_row_constant_bias_leaves_output_unchanged():
    B, H, S, D = 1, 3, 17, 8
    q, k, v = rnd(21, B, H, S, D), rnd(22, B, H, S, D), rnd(23, B, H, S, D)
    c = rnd(24, 1, H, S, 1) * 50
    bias = np.broadcast_to(c, (1, H, S, S)).copy()
    np.testing.assert_allclose(run(q, k, v, bias=bias, mask=CAUSAL), run(q, k, v, mask=CAUSAL),
                               rtol=0, atol=1e-12)


def test_scaling_q_against_scale_leaves_output_unchanged():
    B, H, S, D = 1, 2, 13, 8
    q, k, v = rnd(25, B, H, S, D), rnd(26, B, H, S, D), rnd(27, B, H, S, D)
    a = 4.0  # a power of two keeps a*q exact
    np.testing.assert_allclose(run(q * a, k, v, scale=0.3 / a), run(q, k, v, scale=0.3),
                               rtol=0, atol=1e-13)


def test_joint_permutation_of_keys_and_values():
    B, H, S, D = 2, 2, 21, 8
    q, k, v = rnd(28, B, H, S, D), rnd(29, B, H, S, D), rnd(30, B, H, S, D)
    perm = np.random.default_rng(31).permutation(S)
    np.testing.assert_allclose(run(q, k[:, :, perm], v[:, :, perm]), run(q, k, v), rtol=0, atol=1e-13)


# --------------------------------------------------------------- equivalences
def test_gqa_equals_mha_with_repeated_kv_heads():
    """ruDNN guide, section 9: Hq a multiple of Hkv; query head hq reads kv head hq // g."""
    B, Hq, Hkv, S, D = 2, 8, 2, 16, 8
    q, k, v = rnd(32, B, Hq, S, D), rnd(33, B, Hkv, S, D), rnd(34, B, Hkv, S, D)
    g = Hq // Hkv
    ref = run(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), mask=CAUSAL)
    np.testing.assert_array_equal(run(q, k, v, mask=CAUSAL), ref)


def test_key_padding_equals_truncated_keys():
    B, H, S, D = 3, 2, 40, 8
    q, k, v = rnd(35, B, H, S, D), rnd(36, B, H, S, D), rnd(37, B, H, S, D)
    lens = np.array([40, 17, 1], dtype=np.int32)
    out = run(q, k, v, mask=PAD, kv_lens=lens)
    for b in range(B):
        L = int(lens[b])
        ref = run(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L])
        np.testing.assert_array_equal(out[b:b + 1], ref)


def test_causal_row_equals_unmasked_prefix():
    B, H, S, D = 1, 2, 12, 4
    q, k, v = rnd(38, B, H, S, D), rnd(39, B, H, S, D), rnd(40, B, H, S, D)
    out = run(q, k, v, mask=CAUSAL)
    for i in range(S):
        ref = run(q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1])
        np.testing.assert_array_equal(out[:, :, i:i + 1], ref)


def test_minus_inf_bias_equals_masking():
    B, H, S, D = 1, 2, 10, 4
    q, k, v = rnd(41, B, H, S, D), rnd(42, B, H, S, D), rnd(43, B, H, S, D)
    bias = np.where(np.arange(S)[None, :] > np.arange(S)[:, None], -np.inf, 0.0)[None, None]
    np.testing.assert_array_equal(run(q, k, v, bias=bias), run(q, k, v, mask=CAUSAL))


def test_bias_broadcast_axes():
    """A [1,1,Sq,Sk] bias equals the same bias repeated to [B,Hq,Sq,Sk]."""
    B, H, S, D = 2, 3, 9, 4
    q, k, v = rnd(44, B, H, S, D), rnd(45, B, H, S, D), rnd(46, B, H, S, D)
    b11 = rnd(47, 1, 1, S, S)
    ref = run(q, k, v, bias=np.broadcast_to(b11, (B, H, S, S)).copy())
    np.testing.assert_array_equal(run(q, k, v, bias=b11), ref)
    b1h = rnd(48, 1, H, S, S)
    np.testing.assert_array_equal(run(q, k, v, bias=b1h),
                                  run(q, k, v, bias=np.broadcast_to(b1h, (B, H, S, S)).copy()))


def test_fully_masked_rows_are_nan():
    """No visible key: the softmax is undefined; the oracle returns NaN rows."""
    B, H, Sq, Sk, D = 2, 1, 6, 4, 4
    q, k, v = rnd(49, B, H, Sq, D), rnd(50, B, H, Sk, D), rnd(51, B, H, Sk, D)
    out = run(q, k, v, mask=CAUSAL)  # bottom-right: rows i < Sq - Sk see no key
    assert np.all(np.isnan(out[:, :, : Sq - Sk]))
    assert np.all(np.isfinite(out[:, :, Sq - Sk:]))
    out = run(q, k, v, mask=PAD, kv_lens=np.array([0, 2], np.int32))
    assert np.all(np.isnan(out[0])) and np.all(np.isfinite(out[1]))


# --------------------------------------------------------------- textbook routine
def test_single_head_textbook_softmax():
    """tensai guide, recurrent networks: single-head softmax(Q K^T / sqrt(d)) V."""
    from scipy.special import softmax
    S, D = 33, 16
    q, k, v = rnd(52, S, D), rnd(53, S, D), rnd(54, S, D)
    ref = softmax(q @ k.T / math.sqrt(D), axis=-1) @ v
    out = run(q[None, None], k[None, None], v[None, None])[0, 0]
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)


# --------------------------------------------------------------- brute force
def _brute_force_raw_exp(q, k, v, mask, lens, bias, scale):
    """The pages' dense kernel in 50-digit arithmetic: raw exp, no max shift.

    HOF Flash Attention in Rust, section 4: scores = q.k^T scaled, exp, divide
    by the row sum, times V. Mask: tensai's -inf above the (bottom-right)
    diagonal; key padding drops keys >= kv_len; GQA via repeated kv heads.
    """
    import mpmath
    mpmath.mp.dps = 50
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    kk = np.repeat(k, Hq // Hkv, axis=1)
    vv = np.repeat(v, Hq // Hkv, axis=1)
    out = np.full(q.shape, np.nan)
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                terms = []
                for j in range(Sk):
                    if (mask & CAUSAL) and j - i > Sk - Sq:
                        continue
                    if (mask & PAD) and j >= lens[b]:
                        continue
                    dot = mpmath.fsum(mpmath.mpf(float(q[b, h, i, d])) * mpmath.mpf(float(kk[b, h, j, d]))
                                      for d in range(D))
                    sc = mpmath.mpf(float(scale)) * dot
                    if bias is not None:
                        sc += mpmath.mpf(float(bias[b % bias.shape[0], h % bias.shape[1], i, j]))
                    terms.append((mpmath.exp(sc), j))
                if not terms:
                    continue
                tot = mpmath.fsum(t for t, _ in terms)
                for d in range(D):
                    out[b, h, i, d] = float(mpmath.fsum(t * mpmath.mpf(float(vv[b, h, j, d]))
                                                        for t, j in terms) / tot)
    return out


@pytest.mark.parametrize("mask", [0, CAUSAL, PAD, CAUSAL | PAD])
@pytest.mark.parametrize("bias_shape", [None, (1, 1), (2, 1), (1, 4), (2, 4)])
@pytest.mark.parametrize("sq_sk", [(3, 3), (2, 5), (5, 3)])
def test_brute_force_tiny(mask, bias_shape, sq_sk):
    Sq, Sk = sq_sk
    B, Hq, Hkv, D = 2, 4, 2, 3
    seed = 100 + mask * 10 + (0 if bias_shape is None else sum(bias_shape)) + Sq * 3 + Sk
    q = rnd(seed, B, Hq, Sq, D, scale=0.7)
    k = rnd(seed + 1, B, Hkv, Sk, D, scale=0.7)
    v = rnd(seed + 2, B, Hkv, Sk, D)
    lens = np.array([Sk, max(1, Sk - 2)], dtype=np.int32)
    bias = None if bias_shape is None else rnd(seed + 3, *bias_shape, Sq, Sk, scale=0.5)
    scale = 0.61
    out = run(q, k, v, mask=mask, kv_lens=lens if mask & PAD else None, bias=bias, scale=scale)
    ref = _brute_force_raw_exp(q, k, v, mask, lens, bias, scale)
    np.testing.assert_array_equal(np.isnan(out), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_allclose(out[ok], ref[ok], rtol=0, atol=1e-14)


# --------------------------------------------------------------- sampled rows
def test_rows_entry_matches_full_entry():
    w = synth.WORKLOADS["f16_padding_bias"].replace(B=3, Hq=4, Hkv=4, Sq=70, Sk=90, bias_h=4,
                                                    kv_len_range=(20, 90))
    x = synth.make_inputs(w)
    full = oracle.attention(x["q"], x["k"], x["v"], mask=w.mask, kv_lens=x["kv_lens"], bias=x["bias"],
                            scale=x["scale"], dtype=w.dtype)
    rows = [(0, 0, 0), (2, 3, 69), (1, 2, 33), (2, 0, 5)]
    part = oracle.attention_rows(x["q"], x["k"], x["v"], rows, mask=w.mask, kv_lens=x["kv_lens"],
                                 bias=x["bias"], scale=x["scale"], dtype=w.dtype)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(part[n], full[b, h, i])


def test_widen_is_exact():
    x = np.array([1.0, -2.5, 3.140625, 65504.0, 2.0 ** -24], dtype=np.float32)
    np.testing.assert_array_equal(oracle.widen(synth.to_storage(x, "f16"), "f16"),
                                  x.astype(np.float16).astype(np.float64))
    bits = synth.to_storage(np.array([1.0, -2.5, 3.140625, 1.00390625, 1.01171875], np.float32), "bf16")
    # 1.00390625 = 1 + 2^-8 is a tie between bf16 neighbours 1 and 1 + 2^-7: even -> 1.0
    # 1.01171875 = 1 + 3*2^-8 ties between 1 + 2^-7 and 1 + 2^-6: even mantissa -> 1 + 2^-6
    np.testing.assert_array_equal(oracle.widen(bits, "bf16"), [1.0, -2.5, 3.140625, 1.0, 1.015625])


# --------------------------------------------------------------- log-sum-exp
def test_lse_hand_solved_and_single_key():
    """Row log-sum-exp: the 2x2 hand case gives log(e + 1) and log 2; one key gives its score."""
    q = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    k = np.array([[[[1.0, 0.0], [0.0, 0.0]]]])
    v = np.array([[[[1.0, 2.0], [3.0, 4.0]]]])
    _, lse = run(q, k, v, scale=1.0, lse=True)
    np.testing.assert_allclose(lse[0, 0], [math.log(math.e + 1.0), math.log(2.0)], rtol=0, atol=1e-15)
    _, lse_c = run(q, k, v, scale=1.0, mask=CAUSAL, lse=True)
    np.testing.assert_allclose(lse_c[0, 0], [1.0, math.log(2.0)], rtol=0, atol=1e-15)
    q1, k1, v1 = rnd(60, 1, 2, 3, 4), rnd(61, 1, 2, 1, 4), rnd(62, 1, 2, 1, 4)
    _, lse1 = run(q1, k1, v1, scale=0.7, lse=True)
    np.testing.assert_allclose(lse1, 0.7 * np.einsum("bhid,bhjd->bhi", q1, k1), rtol=0, atol=1e-14)


@pytest.mark.parametrize("mask", [0, CAUSAL, PAD])
def test_lse_identical_keys_is_score_plus_log_count(mask):
    B, H, S, D = 2, 2, 20, 8
    q = rnd(63, B, H, S, D)
    k = np.broadcast_to(rnd(64, 1, 1, 1, D), (B, H, S, D)).copy()
    v = rnd(65, B, H, S, D)
    lens = np.array([S, 7], dtype=np.int32)
    _, lse = run(q, k, v, mask=mask, kv_lens=lens if mask & PAD else None, scale=0.3, lse=True)
    s = 0.3 * np.einsum("bhid,d->bhi", q, k[0, 0, 0])
    for b in range(B):
        L = int(lens[b]) if mask & PAD else S
        n = np.array([min(L, i + 1) if mask & CAUSAL else L for i in range(S)])
        np.testing.assert_allclose(lse[b], s[b] + np.log(n)[None, :], rtol=0, atol=1e-13)


def test_lse_merges_two_key_halves():
    """Splitting the keys into two ranges and merging by log-sum-exp gives the whole row:
    lse = log(e^lseA + e^lseB), O = (e^lseA O_A + e^lseB O_B) / e^lse."""
    B, H, Sk, D = 2, 3, 50, 8
    q, k, v = rnd(66, B, H, 7, D, scale=2), rnd(67, B, H, Sk, D, scale=2), rnd(68, B, H, Sk, D)
    o, lse = run(q, k, v, lse=True)
    oa, la = run(q, k[:, :, :21], v[:, :, :21], lse=True)
    ob, lb = run(q, k[:, :, 21:], v[:, :, 21:], lse=True)
    m = np.maximum(la, lb)
    wa, wb = np.exp(la - m), np.exp(lb - m)
    np.testing.assert_allclose(lse, m + np.log(wa + wb), rtol=0, atol=1e-13)
    np.testing.assert_allclose(o, (wa[..., None] * oa + wb[..., None] * ob) / (wa + wb)[..., None],
                               rtol=0, atol=1e-13)


def test_lse_empty_row_is_minus_inf():
    q, k, v = rnd(69, 1, 1, 5, 4), rnd(70, 1, 1, 3, 4), rnd(71, 1, 1, 3, 4)
    _, lse = run(q, k, v, mask=CAUSAL, lse=True)  # rows 0, 1 see no key (bottom-right)
    assert np.all(lse[0, 0, :2] == -np.inf) and np.all(np.isfinite(lse[0, 0, 2:]))


def test_lse_brute_force_tiny():
    """50-digit log of the raw exp-sum, all masks and a per-head bias."""
    import mpmath
    mpmath.mp.dps = 50
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 4, 6, 3
    q, k = rnd(72, B, Hq, Sq, D, scale=0.8), rnd(73, B, Hkv, Sk, D, scale=0.8)
    v = rnd(74, B, Hkv, Sk, D)
    bias = rnd(75, 1, Hq, Sq, Sk, scale=0.5)
    lens = np.array([6, 3], dtype=np.int32)
    for mask in (0, CAUSAL, PAD, CAUSAL | PAD):
        _, lse = run(q, k, v, mask=mask, kv_lens=lens if mask & PAD else None, bias=bias, scale=0.45, lse=True)
        kk = np.repeat(k, Hq // Hkv, axis=1)
        for b in range(B):
            for h in range(Hq):
                for i in range(Sq):
                    terms = []
                    for j in range(Sk):
                        if (mask & CAUSAL) and j - i > Sk - Sq:
                            continue
                        if (mask & PAD) and j >= lens[b]:
                            continue
                        dot = mpmath.fsum(mpmath.mpf(float(q[b, h, i, d])) * mpmath.mpf(float(kk[b, h, j, d]))
                                          for d in range(D))
                        terms.append(mpmath.exp(mpmath.mpf(0.45) * dot + mpmath.mpf(float(bias[0, h, i, j]))))
                    ref = float(mpmath.log(mpmath.fsum(terms))) if terms else -math.inf
                    assert abs(lse[b, h, i] - ref) <= 1e-13 or lse[b, h, i] == ref
