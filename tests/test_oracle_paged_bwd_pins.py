"""Pins of the oracle's paged-cache and MLA backward (ruDNN user guide,
section 11: dq and the cache-shaped history gradients dk, dv; for MLA dq, dqp,
dlatent with its key and value parts, dkp) to things other than itself.

- Finite differences of the paged forward oracle (itself pinned to the dense
  oracle): central differences of L = sum(O * dout) over every element of q
  and of both caches, with a physical page shared by two sequences, GQA, a
  page nobody reads, a sequence without queries and a query row that sees no
  key.
- The dense backward oracle (pinned by finite differences, a 50-digit
  brute force and PyTorch autograd): pages laid out in order with the default
  positions are dense attention with the bottom-right causal mask.
- Invariants: splitting a shared page into private copies and summing the
  copies' gradients gives the shared page's gradient; renaming physical pages
  permutes the gradients; pages that no query reads get zero.
- MLA reduces to paged attention with one key/value head: keys [c | kp], values
  [c | 0] and dout [g | 0] give dq = [dq | dqp], dlatent = dk[:R] + dv[:R] and
  dkp = dk[R:]; and MLA's own finite differences.
"""
import numpy as np
import pytest

import oracle
from tests.test_oracle_paged_pins import dense_to_paged, packed_q, unpack
from tests.test_oracle_pins import CAUSAL, rnd


def fd(loss, arrays, h=1e-5):
    """Central differences of loss(*arrays) for every element of every array."""
    out = []
    for x in arrays:
        gx = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            fp = loss(*arrays)
            x[idx] = old - h
            fm = loss(*arrays)
            x[idx] = old
            gx[idx] = (fp - fm) / (2 * h)
        out.append(gx)
    return out


def shared_case(seed=0, D=3, Hq=4, Hkv=2, P=2):
    """Three sequences over 6 pages: 0 and 1 share page 0 (a common prefix),
    sequence 2 (page 4) has no queries, page 5 belongs to nobody."""
    rng = np.random.default_rng(seed)
    pages = 6
    kc = rng.standard_normal((pages, P, Hkv, D)) * 0.8
    vc = rng.standard_normal((pages, P, Hkv, D))
    table = np.array([[0, 1, 2], [0, 3, -1], [4, -1, -1]], dtype=np.int32)
    lens = np.array([5, 3, 2], dtype=np.int32)
    offs = np.array([0, 3, 5, 5], dtype=np.int32)
    nq = 5
    q = rng.standard_normal((nq, Hq, D)) * 0.8
    g = rng.standard_normal((nq, Hq, D))
    return q, kc, vc, g, table, lens, offs


def paged_loss(table, lens, offs, g, positions, causal, scale):
    def L(q, kc, vc):
        o = oracle.paged_attention(q, kc, vc, table, lens, offs, positions=positions, causal=causal, scale=scale)
        return float(np.nansum(o * g))
    return L


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("positions", [None, [4, 1, 3, -1, 2]])
def test_paged_bwd_matches_finite_differences(causal, positions):
    # explicit positions: query 3 (sequence 1) at -1 sees no key under the causal mask
    q, kc, vc, g, table, lens, offs = shared_case(seed=3)
    pos = None if positions is None else np.array(positions, dtype=np.int32)
    dq, dk, dv = oracle.paged_attention_bwd(q, kc, vc, g, table, lens, offs, positions=pos, causal=causal,
                                            scale=0.61)
    fq, fk, fv = fd(paged_loss(table, lens, offs, g, pos, causal, 0.61), [q.copy(), kc.copy(), vc.copy()])
    for got, ref in ((dq, fq), (dk, fk), (dv, fv)):
        np.testing.assert_allclose(got, ref, rtol=0, atol=2e-8)
    # pages 4 (sequence without queries) and 5 (nobody's) get nothing
    assert not dk[4:].any() and not dv[4:].any()
    assert np.abs(dk[0]).max() > 0 and np.abs(dv[0]).max() > 0


@pytest.mark.parametrize("page_size", [1, 3, 4])
def test_in_order_pages_equal_dense_bottom_right_causal(page_size):
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 3, 7, 5
    q, k, v, g = rnd(11, B, Hq, Sq, D), rnd(12, B, Hkv, Sk, D), rnd(13, B, Hkv, Sk, D), rnd(14, B, Hq, Sq, D)
    kc, vc, table = dense_to_paged(k, v, page_size)
    lens = np.full(B, Sk, dtype=np.int32)
    offs = np.arange(B + 1, dtype=np.int32) * Sq
    dq, dk, dv = oracle.paged_attention_bwd(packed_q(q), kc, vc, packed_q(g), table, lens, offs, causal=True,
                                            scale=0.4)
    rq, rk, rv = oracle.attention_bwd(q, k, v, g, mask=CAUSAL, scale=0.4)
    np.testing.assert_allclose(unpack(dq, B, Sq), rq, rtol=0, atol=1e-13)
    dkd, dvd, _ = dense_to_paged(rk, rv, page_size)  # the dense key gradients laid out as pages
    np.testing.assert_allclose(dk, dkd, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dvd, rtol=0, atol=1e-13)


def test_shared_page_gradient_is_the_sum_over_private_copies():
    q, kc, vc, g, table, lens, offs = shared_case(seed=5)
    dq, dk, dv = oracle.paged_attention_bwd(q, kc, vc, g, table, lens, offs, causal=True, scale=0.5)
    # give sequence 1 a private copy of page 0 (as page 6)
    kc2, vc2 = np.concatenate([kc, kc[:1]]), np.concatenate([vc, vc[:1]])
    t2 = table.copy()
    t2[1, 0] = 6
    dq2, dk2, dv2 = oracle.paged_attention_bwd(q, kc2, vc2, g, t2, lens, offs, causal=True, scale=0.5)
    np.testing.assert_allclose(dq2, dq, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk2[0] + dk2[6], dk[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv2[0] + dv2[6], dv[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk2[1:6], dk[1:6], rtol=0, atol=1e-14)
    assert np.abs(dk2[6]).max() > 0 and np.abs(dk2[0] - dk[0]).max() > 1e-6


def test_renaming_pages_permutes_the_gradients():
    q, kc, vc, g, table, lens, offs = shared_case(seed=6)
    perm = np.random.default_rng(0).permutation(kc.shape[0])  # new page perm[i] holds old page i
    inv = np.argsort(perm)
    t2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1).astype(np.int32)
    dq, dk, dv = oracle.paged_attention_bwd(q, kc, vc, g, table, lens, offs, causal=True, scale=0.7)
    dq2, dk2, dv2 = oracle.paged_attention_bwd(q, kc[inv], vc[inv], g, t2, lens, offs, causal=True, scale=0.7)
    np.testing.assert_array_equal(dq2, dq)
    np.testing.assert_array_equal(dk2, dk[inv])
    np.testing.assert_array_equal(dv2, dv[inv])


def mla_case(seed, R=4, Pd=2, H=3, P=2):
    rng = np.random.default_rng(seed)
    pages = 5
    lat = rng.standard_normal((pages, P, 1, R)) * 0.7
    kp = rng.standard_normal((pages, P, 1, Pd)) * 0.7
    table = np.array([[0, 1, 2], [0, 3, -1]], dtype=np.int32)
    lens = np.array([6, 3], dtype=np.int32)
    offs = np.array([0, 2, 4], dtype=np.int32)
    q = rng.standard_normal((4, H, R)) * 0.7
    qp = rng.standard_normal((4, H, Pd)) * 0.7
    g = rng.standard_normal((4, H, R))
    return q, qp, lat, kp, g, table, lens, offs


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("pd", [0, 2])
def test_mla_bwd_is_paged_bwd_over_concatenated_keys(causal, pd):
    q, qp, lat, kp, g, table, lens, offs = mla_case(8 + pd, Pd=pd)
    R = q.shape[2]
    dq, dqp, dlat, dkp = oracle.paged_mla_bwd(q, qp, lat, kp, g, table, lens, offs, causal=causal, scale=0.45)
    kc = np.concatenate([lat, kp], axis=3)
    vc = np.concatenate([lat, np.zeros_like(kp)], axis=3)
    qq = np.concatenate([q, qp], axis=2)
    gg = np.concatenate([g, np.zeros_like(qp)], axis=2)
    rq, rk, rv = oracle.paged_attention_bwd(qq, kc, vc, gg, table, lens, offs, causal=causal, scale=0.45)
    np.testing.assert_allclose(dq, rq[..., :R], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dqp, rq[..., R:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dlat, rk[..., :R] + rv[..., :R], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dkp, rk[..., R:], rtol=0, atol=1e-13)
    assert not rv[..., R:].any()


def test_mla_bwd_matches_finite_differences():
    q, qp, lat, kp, g, table, lens, offs = mla_case(21)
    pos = np.array([5, 2, 0, 2], dtype=np.int32)

    def L(q_, qp_, lat_, kp_):
        o = oracle.paged_mla(q_, qp_, lat_, kp_, table, lens, offs, positions=pos, causal=True, scale=0.52)
        return float(np.nansum(o * g))
    got = oracle.paged_mla_bwd(q, qp, lat, kp, g, table, lens, offs, positions=pos, causal=True, scale=0.52)
    ref = fd(L, [q.copy(), qp.copy(), lat.copy(), kp.copy()])
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, b, rtol=0, atol=2e-8)
    assert not got[2][4].any() and not got[3][4].any()  # page 4: nobody's
