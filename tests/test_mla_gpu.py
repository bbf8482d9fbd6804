"""GPU parity of MLA over a paged latent cache (attn_paged_mla) against the
float64 oracle (ruDNN user guide, section 9). Tolerances as for the dense
forward (max|O - O_ref| / max|O_ref| <= 1e-5 F32, 4e-3 F16, 1.6e-2 BF16; NaN
rows must match) and lse within 1e-4 * max(1, |lse|).
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


def run_mla(w, x):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    q, qp, lat, kp = (to_device(x[n], w.dtype) for n in ("q", "qp", "latent", "kpos"))
    ints = {n: to_device(x[n], "i32") for n in ("block_table", "seq_lens", "q_offsets")}
    pos = to_device(x["positions"], "i32") if x["positions"] is not None else None
    out = torch.full_like(q, 777.0)
    o, lse = attn.paged_mla(q, qp, lat, kp, ints["block_table"], ints["seq_lens"], ints["q_offsets"],
                            positions=pos, causal=w.causal, scale=x["scale"], return_lse=True, out=out)
    return to_f64(o), lse.cpu().numpy().astype(np.float64)


def MW(name, dtype, ns, H, R, Pd, P, ctx, qr, **kw):
    return synth.MlaWorkload(name, dtype, ns, H, R, Pd, P, ctx, qr, **kw)


CASES = [
    MW("mla_bf16_r512_p64_decode", "bf16", 6, 16, 512, 64, 64, (1, 900), (1, 1), seed=1),
    MW("mla_bf16_r512_p64_prefill", "bf16", 3, 8, 512, 64, 16, (50, 400), (10, 60), seed=2),
    MW("mla_f16_r256_p32_positions", "f16", 4, 4, 256, 32, 32, (1, 300), (1, 40), seed=3,
       explicit_positions=True),
    MW("mla_f32_r128_p16", "f32", 3, 4, 128, 16, 8, (1, 120), (1, 20), seed=4),
    MW("mla_bf16_r128_p0_noncausal", "bf16", 3, 8, 128, 0, 64, (1, 500), (1, 30), seed=5, causal=False),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_mla_matches_oracle(w):
    x = synth.make_mla_inputs(w)
    got, lse = run_mla(w, x)
    ref, ref_lse = oracle.paged_mla(x["q"], x["qp"], x["latent"], x["kpos"], x["block_table"], x["seq_lens"],
                                    x["q_offsets"], positions=x["positions"], causal=w.causal, scale=x["scale"],
                                    dtype=w.dtype, lse=True)
    err = rel_err(got, ref)
    assert err <= TOL[w.dtype], f"{w.name}: rel err {err:.3e}"
    ninf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), ninf)
    fin = ~ninf
    if fin.any():
        assert np.max(np.abs(lse[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin]))) <= LSE_TOL


def test_mla_argument_errors():
    import ctypes
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    lib = attn.load_library()
    dev = torch.device("cuda")
    q = torch.zeros(2, 4, 512, device=dev, dtype=torch.bfloat16)
    qp = torch.zeros(2, 4, 64, device=dev, dtype=torch.bfloat16)
    lat = torch.zeros(2, 16, 1, 512, device=dev, dtype=torch.bfloat16)
    kp = torch.zeros(2, 16, 1, 64, device=dev, dtype=torch.bfloat16)
    tab = torch.zeros(1, 2, dtype=torch.int32, device=dev)
    lens = torch.tensor([20], dtype=torch.int32, device=dev)
    offs = torch.tensor([0, 2], dtype=torch.int32, device=dev)
    out = torch.empty_like(q)

    def call(R=512, Pd=64, o=out):
        shape = attn.MlaShape(1, 2, 4, R, Pd, 16, 2, 2, 2)
        return lib.attn_paged_mla(ctypes.byref(shape), q.data_ptr(), qp.data_ptr(), lat.data_ptr(), kp.data_ptr(),
                                  tab.data_ptr(), lens.data_ptr(), offs.data_ptr(), None, 1, ctypes.c_float(0.04),
                                  attn.ATTN_BF16, o.data_ptr(), None, None)
    assert call() == 0
    torch.cuda.synchronize()
    assert call(R=96) == -4
    assert call(Pd=48) == -4
    assert call(o=q) == -8
