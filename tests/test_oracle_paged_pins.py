"""Pins of the oracle's paged, packed-query attention (ruDNN user guide,
section 9) to the dense oracle, which test_oracle_pins ties to the pages'
kernel, closed forms and a 50-digit brute force.

- Equal-length sequences whose pages are laid out in order, with the default
  positions (the newest tokens), are dense attention with the bottom-right
  causal mask; variable lengths without the causal mask are dense attention
  with key padding.
- Renaming the physical pages (a permutation of the cache and the tables)
  changes nothing; explicit positions equal to the defaults change nothing;
  positions past the end of the keys turn the causal mask off; a decode step
  (one query at the last position) sees every key.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_flash_gb300 import synth
from tests.test_oracle_pins import CAUSAL, PAD, rnd


def dense_to_paged(k, v, page_size, rng=None):
    """[B, Hkv, S, D] caches -> ([pages, P, Hkv, D] x2, table [B, max_pages]), pages in
    order (or shuffled by ``rng``)."""
    B, Hkv, S, D = k.shape
    npg = (S + page_size - 1) // page_size
    pages = B * npg
    kc = np.zeros((pages, page_size, Hkv, D))
    vc = np.zeros((pages, page_size, Hkv, D))
    phys = np.arange(pages) if rng is None else rng.permutation(pages)
    table = np.zeros((B, npg), dtype=np.int32)
    for b in range(B):
        for p in range(npg):
            pg = phys[b * npg + p]
            table[b, p] = pg
            rows = slice(p * page_size, min(S, (p + 1) * page_size))
            n = rows.stop - rows.start
            kc[pg, :n] = k[b, :, rows].transpose(1, 0, 2)
            vc[pg, :n] = v[b, :, rows].transpose(1, 0, 2)
    return kc, vc, table


def packed_q(q):
    """[B, Hq, Sq, D] -> [B*Sq, Hq, D] packed by sequence."""
    B, Hq, Sq, D = q.shape
    return q.transpose(0, 2, 1, 3).reshape(B * Sq, Hq, D)


def unpack(o, B, Sq):
    return o.reshape(B, Sq, o.shape[1], o.shape[2]).transpose(0, 2, 1, 3)


@pytest.mark.parametrize("page_size", [1, 4, 16])
@pytest.mark.parametrize("sq_sk", [(5, 5), (3, 11), (1, 9)])
def test_equal_lengths_equal_dense_bottom_right_causal(page_size, sq_sk):
    Sq, Sk = sq_sk
    B, Hq, Hkv, D = 3, 4, 2, 5
    q, k, v = rnd(1, B, Hq, Sq, D), rnd(2, B, Hkv, Sk, D), rnd(3, B, Hkv, Sk, D)
    kc, vc, table = dense_to_paged(k, v, page_size)
    lens = np.full(B, Sk, dtype=np.int32)
    offs = np.arange(B + 1, dtype=np.int32) * Sq
    out, lse = oracle.paged_attention(packed_q(q), kc, vc, table, lens, offs, causal=True, scale=0.4, lse=True)
    ref, ref_lse = oracle.attention(q, k, v, mask=CAUSAL, scale=0.4, lse=True)
    np.testing.assert_allclose(unpack(out, B, Sq), ref, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse.reshape(B, Sq, Hq).transpose(0, 2, 1), ref_lse, rtol=0, atol=1e-14)


def test_variable_lengths_non_causal_equal_dense_key_padding():
    B, Hq, Hkv, Sq, Sk, D = 4, 2, 1, 3, 13, 4
    q, k, v = rnd(4, B, Hq, Sq, D), rnd(5, B, Hkv, Sk, D), rnd(6, B, Hkv, Sk, D)
    lens = np.array([13, 1, 7, 0], dtype=np.int32)
    kc, vc, table = dense_to_paged(k, v, 4)
    offs = np.arange(B + 1, dtype=np.int32) * Sq
    out = oracle.paged_attention(packed_q(q), kc, vc, table, lens, offs, causal=False, scale=0.7)
    ref = oracle.attention(q, k, v, mask=PAD, kv_lens=lens, scale=0.7)
    got = unpack(out, B, Sq)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))  # the length-0 sequence is NaN
    ok = ~np.isnan(ref)
    np.testing.assert_allclose(got[ok], ref[ok], rtol=0, atol=1e-14)


def test_renaming_physical_pages_changes_nothing():
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 4, 19, 3
    q, k, v = rnd(7, B, Hq, Sq, D), rnd(8, B, Hkv, Sk, D), rnd(9, B, Hkv, Sk, D)
    lens = np.array([19, 11], dtype=np.int32)
    offs = np.array([0, 4, 8], dtype=np.int32)
    a = oracle.paged_attention(packed_q(q), *dense_to_paged(k, v, 4), lens, offs, causal=True, scale=0.5)
    b = oracle.paged_attention(packed_q(q), *dense_to_paged(k, v, 4, np.random.default_rng(3)), lens, offs,
                               causal=True, scale=0.5)
    np.testing.assert_array_equal(a, b)


def test_positions():
    w = synth.PagedWorkload("pin", synth.F32, 5, 4, 2, 8, 8, (1, 40), (1, 12), seed=11)
    x = synth.make_paged_inputs(w)
    args = (x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["seq_lens"], x["q_offsets"])
    default = oracle.paged_attention(*args, causal=True, scale=0.3)
    lens, offs = x["seq_lens"], x["q_offsets"]
    pos = np.concatenate([np.arange(L - (offs[s + 1] - offs[s]), L) for s, L in enumerate(lens)]).astype(np.int32)
    np.testing.assert_array_equal(oracle.paged_attention(*args, positions=pos, causal=True, scale=0.3), default)
    far = np.full_like(pos, 10 ** 6)
    np.testing.assert_array_equal(oracle.paged_attention(*args, positions=far, causal=True, scale=0.3),
                                  oracle.paged_attention(*args, causal=False, scale=0.3))
    # position -1 sees no key at all: NaN rows, as in the dense definition
    none = np.full_like(pos, -1)
    assert np.isnan(oracle.paged_attention(*args, positions=none, causal=True, scale=0.3)).all()


def test_decode_step_sees_every_key():
    B, Hq, Hkv, Sk, D = 3, 4, 1, 17, 6
    q, k, v = rnd(12, B, Hq, 1, D), rnd(13, B, Hkv, Sk, D), rnd(14, B, Hkv, Sk, D)
    kc, vc, table = dense_to_paged(k, v, 8, np.random.default_rng(1))
    out = oracle.paged_attention(packed_q(q), kc, vc, table, np.full(B, Sk, dtype=np.int32),
                                 np.arange(B + 1, dtype=np.int32), causal=True, scale=0.45)
    ref = oracle.attention(q, k, v, scale=0.45)
    np.testing.assert_allclose(unpack(out, B, 1), ref, rtol=0, atol=1e-14)
