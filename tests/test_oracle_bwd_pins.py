"""Pins of the oracle's backward (dq, dk, dv) to things other than itself.

- Finite differences of the forward oracle (tensai autograd guide, section
  "演算" (operations): every op's gradient is checked against numerical
  differentiation): central differences of L = sum(O * dout) in float64.
- The pages' raw-exp dense kernel (HOF Flash Attention in Rust, section 4) in
  50-digit arithmetic, differentiated by central differences with a tiny
  step: a gradient of the plain definition with no float64 rounding at all.
- A library routine: PyTorch CPU autograd through softmax(QK^T*scale + bias)V
  in float64 for single heads.
- Closed forms and invariants: the key gradients of a (b, kv head) sum to
  zero (every softmax row's Jacobian annihilates constants); identical keys
  make the output independent of q (dq = 0); a single key gives dq = dk = 0
  and dv = the sum of dout over the rows that see it; masked keys and rows
  with no visible key receive and contribute nothing.
"""
import math

import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import CAUSAL, PAD, rnd


def loss_grad_fd(q, k, v, g, h=1e-5, **kw):
    """Central differences of L(q, k, v) = sum(attention(q, k, v) * g)."""
    def L(qq, kk, vv):
        o = oracle.attention(qq, kk, vv, **kw)
        return float(np.nansum(o * g))
    grads = []
    for which in range(3):
        base = [q.copy(), k.copy(), v.copy()]
        x = base[which]
        gx = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            fp = L(*base)
            x[idx] = old - h
            fm = L(*base)
            x[idx] = old
            gx[idx] = (fp - fm) / (2 * h)
        grads.append(gx)
    return grads


def case(seed, B=2, Hq=4, Hkv=2, Sq=4, Sk=5, D=3, mask=0, bias_shape=None):
    q = rnd(seed, B, Hq, Sq, D, scale=0.8)
    k = rnd(seed + 1, B, Hkv, Sk, D, scale=0.8)
    v = rnd(seed + 2, B, Hkv, Sk, D)
    g = rnd(seed + 3, B, Hq, Sq, D)
    lens = np.array([Sk, max(1, Sk - 2)][:B], dtype=np.int32)
    bias = None if bias_shape is None else rnd(seed + 4, *bias_shape, Sq, Sk, scale=0.5)
    kw = dict(mask=mask, kv_lens=lens if mask & PAD else None, bias=bias, scale=0.57)
    return q, k, v, g, kw


@pytest.mark.parametrize("mask", [0, CAUSAL, PAD, CAUSAL | PAD])
@pytest.mark.parametrize("bias_shape", [None, (1, 4), (2, 1)])
@pytest.mark.parametrize("sq_sk", [(4, 4), (3, 6), (6, 3)])
def test_matches_finite_differences_of_the_forward(mask, bias_shape, sq_sk):
    Sq, Sk = sq_sk
    q, k, v, g, kw = case(7 + mask + Sq * 5 + Sk, Sq=Sq, Sk=Sk, mask=mask, bias_shape=bias_shape)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, **kw)
    fq, fk, fv = loss_grad_fd(q, k, v, g, **kw)
    for got, ref in ((dq, fq), (dk, fk), (dv, fv)):
        np.testing.assert_allclose(got, ref, rtol=0, atol=2e-8)


def _raw_exp_loss(q, k, v, g, mask, lens, scale, mp):
    """sum(O * g) of the pages' raw-exp kernel in mpmath (q, k, v mp matrices)."""
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    total = mp.mpf(0)
    for b in range(B):
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            for i in range(Sq):
                terms = []
                for j in range(Sk):
                    if (mask & CAUSAL) and j - i > Sk - Sq:
                        continue
                    if (mask & PAD) and j >= lens[b]:
                        continue
                    dot = mp.fsum(q[b, h, i, d] * k[b, hk, j, d] for d in range(D))
                    terms.append((mp.exp(scale * dot), j))
                if not terms:
                    continue
                tot = mp.fsum(t for t, _ in terms)
                for d in range(D):
                    total += g[b, h, i, d] * mp.fsum(t * v[b, hk, j, d] for t, j in terms) / tot
    return total


@pytest.mark.parametrize("mask", [0, CAUSAL | PAD])
def test_matches_50_digit_raw_exp_gradient(mask):
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = 50
    q, k, v, g, kw = case(40 + mask, B=2, Hq=2, Hkv=1, Sq=3, Sk=4, D=2, mask=mask)
    lens = kw["kv_lens"] if kw["kv_lens"] is not None else np.array([4, 4], dtype=np.int32)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, **kw)
    conv = np.vectorize(lambda x: mp.mpf(float(x)), otypes=[object])
    Q, K, V, G = conv(q), conv(k), conv(v), conv(g)
    sc = mp.mpf(kw["scale"])
    h = mp.mpf("1e-20")
    for arr, got in ((Q, dq), (K, dk), (V, dv)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            fp = _raw_exp_loss(Q, K, V, G, mask, lens, sc, mp)
            arr[idx] = old - h
            fm = _raw_exp_loss(Q, K, V, G, mask, lens, sc, mp)
            arr[idx] = old
            ref = float((fp - fm) / (2 * h))
            assert abs(got[idx] - ref) <= 1e-13 * max(1.0, abs(ref)), (idx, got[idx], ref)


def test_matches_torch_autograd_single_heads():
    torch = pytest.importorskip("torch")
    q, k, v, g, kw = case(60, B=1, Hq=2, Hkv=2, Sq=7, Sk=9, D=5, mask=CAUSAL, bias_shape=(1, 2))
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, **kw)
    for h in range(2):
        qt = torch.tensor(q[0, h], dtype=torch.float64, requires_grad=True)
        kt = torch.tensor(k[0, h], dtype=torch.float64, requires_grad=True)
        vt = torch.tensor(v[0, h], dtype=torch.float64, requires_grad=True)
        Sq, Sk = 7, 9
        i = torch.arange(Sq)[:, None]
        j = torch.arange(Sk)[None, :]
        mask = torch.where(j <= i + (Sk - Sq), 0.0, float("-inf")).to(torch.float64)
        s = qt @ kt.T * kw["scale"] + torch.tensor(kw["bias"][0, h]) + mask
        o = torch.softmax(s, dim=-1) @ vt
        (o * torch.tensor(g[0, h])).sum().backward()
        np.testing.assert_allclose(dq[0, h], qt.grad.numpy(), rtol=0, atol=1e-13)
        np.testing.assert_allclose(dk[0, h], kt.grad.numpy(), rtol=0, atol=1e-13)
        np.testing.assert_allclose(dv[0, h], vt.grad.numpy(), rtol=0, atol=1e-13)


@pytest.mark.parametrize("mask", [0, CAUSAL, PAD, CAUSAL | PAD])
def test_key_gradients_sum_to_zero(mask):
    q, k, v, g, kw = case(80 + mask, Sq=6, Sk=7, D=4, mask=mask, bias_shape=(2, 4))
    _, dk, _ = oracle.attention_bwd(q, k, v, g, **kw)
    assert np.abs(dk.sum(axis=2)).max() < 1e-13
    assert np.abs(dk).max() > 1e-3  # and the gradients themselves are not trivially zero


def test_identical_keys_give_zero_query_gradient():
    q, k, v, g, kw = case(90, Sq=5, Sk=6, D=4, mask=CAUSAL)
    k[:] = k[:, :, :1, :]
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, **kw)
    assert np.abs(dq).max() < 1e-14
    assert np.abs(dv).max() > 1e-3


def test_single_key():
    q, k, v, g, kw = case(100, Sq=5, Sk=1, D=3)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, **kw)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    # dv of kv head hk = sum of dout over every row of its query heads (weight 1)
    group = q.shape[1] // k.shape[1]
    for b in range(q.shape[0]):
        for hk in range(k.shape[1]):
            ref = g[b, hk * group:(hk + 1) * group].sum(axis=(0, 1))
            np.testing.assert_allclose(dv[b, hk, 0], ref, rtol=0, atol=1e-13)


def test_masked_keys_and_empty_rows_get_and_give_nothing():
    q, k, v, g, kw = case(110, B=2, Sq=4, Sk=6, D=3, mask=PAD)
    kw["kv_lens"] = np.array([0, 3], dtype=np.int32)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, **kw)
    assert not np.isnan(dq).any() and not np.isnan(dk).any() and not np.isnan(dv).any()
    assert (dq[0] == 0).all() and (dk[0] == 0).all() and (dv[0] == 0).all()  # batch 0 sees no key
    assert (dk[1, :, 3:] == 0).all() and (dv[1, :, 3:] == 0).all()           # padded keys
    assert np.abs(dv[1, :, :3]).max() > 1e-3


def test_gqa_gradients_equal_mha_with_summed_heads():
    q, k, v, g, kw = case(120, B=1, Hq=4, Hkv=2, Sq=5, Sk=5, D=3, mask=CAUSAL)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, **kw)
    kr, vr = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    dq2, dk2, dv2 = oracle.attention_bwd(q, kr, vr, g, **kw)
    np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(dk, dk2.reshape(1, 2, 2, 5, 3).sum(axis=2), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, dv2.reshape(1, 2, 2, 5, 3).sum(axis=2), rtol=0, atol=1e-14)


def test_dtype_widening_matches_float_inputs():
    from exact_scaled_dot_flash_gb300 import synth
    x = synth.to_storage(rnd(130, 1, 2, 3, 8).astype(np.float32), "bf16")
    y = synth.to_storage(rnd(131, 1, 2, 4, 8).astype(np.float32), "bf16")
    z = synth.to_storage(rnd(132, 1, 2, 4, 8).astype(np.float32), "bf16")
    gg = synth.to_storage(rnd(133, 1, 2, 3, 8).astype(np.float32), "bf16")
    a = oracle.attention_bwd(x, y, z, gg, scale=1 / math.sqrt(8), dtype="bf16")
    b = oracle.attention_bwd(*(oracle.widen(t, "bf16") for t in (x, y, z, gg)), scale=1 / math.sqrt(8))
    for u, w in zip(a, b):
        np.testing.assert_array_equal(u, w)
