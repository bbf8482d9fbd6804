"""Pins of the oracle's MLA (ruDNN user guide, section 9: absorbed query,
positional query, shared latent and positional caches) to the paged
attention oracle, which test_oracle_paged_pins ties to the dense oracle.

MLA with latent rows c_j and positional rows kp_j is attention with one key
head whose keys are [c_j, kp_j], whose queries are [q, qp], and whose values
are c_j: the paged oracle with D = R + P, values [c_j, 0], gives the same
output in its first R columns and the same log-sum-exp.
"""
import numpy as np
import pytest

import oracle
from exact_scaled_dot_flash_gb300 import synth


def as_paged_attention(x):
    q = np.concatenate([oracle.widen(x["q"], "bf16"), oracle.widen(x["qp"], "bf16")], axis=2)
    lat, kp = oracle.widen(x["latent"], "bf16"), oracle.widen(x["kpos"], "bf16")
    k = np.concatenate([lat, kp], axis=3)
    v = np.concatenate([lat, np.zeros_like(kp)], axis=3)
    return q, k, v


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("positions", [False, True])
@pytest.mark.parametrize("pd", [16, 0])
def test_mla_is_single_head_attention_over_concatenated_keys(causal, positions, pd):
    w = synth.MlaWorkload("pin", synth.BF16, 4, 6, 32, pd, 8, (1, 70), (1, 12), seed=3 + pd,
                          causal=causal, explicit_positions=positions)
    x = synth.make_mla_inputs(w)
    meta = (x["block_table"], x["seq_lens"], x["q_offsets"])
    out, lse = oracle.paged_mla(x["q"], x["qp"], x["latent"], x["kpos"], *meta, positions=x["positions"],
                                causal=causal, scale=x["scale"], dtype="bf16", lse=True)
    q, k, v = as_paged_attention(x)
    ref, ref_lse = oracle.paged_attention(q, k, v, *meta, positions=x["positions"], causal=causal,
                                          scale=x["scale"], lse=True)
    R = w.R
    np.testing.assert_array_equal(np.isnan(out), np.isnan(ref[..., :R]))
    ok = ~np.isnan(out)
    np.testing.assert_allclose(out[ok], ref[..., :R][ok], rtol=0, atol=1e-13)
    assert np.abs(ref[..., R:][~np.isnan(ref[..., R:])]).max(initial=0.0) == 0.0
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-13)


def test_mla_single_key_returns_its_latent_row():
    w = synth.MlaWorkload("pin1", synth.BF16, 3, 4, 16, 8, 4, (1, 1), (1, 1), seed=9)
    x = synth.make_mla_inputs(w)
    out = oracle.paged_mla(x["q"], x["qp"], x["latent"], x["kpos"], x["block_table"], x["seq_lens"],
                           x["q_offsets"], scale=x["scale"], dtype="bf16")
    lat = oracle.widen(x["latent"], "bf16")
    for s in range(3):
        row = lat[x["block_table"][s, 0], 0, 0]
        np.testing.assert_array_equal(out[s], np.broadcast_to(row, out[s].shape))
