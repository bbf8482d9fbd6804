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


def run_mla(w, x, num_splits=1):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    q, qp, lat, kp = (to_device(x[n], w.dtype) for n in ("q", "qp", "latent", "kpos"))
    ints = {n: to_device(x[n], "i32") for n in ("block_table", "seq_lens", "q_offsets")}
    pos = to_device(x["positions"], "i32") if x["positions"] is not None else None
    out = torch.full_like(q, 777.0)  # sentinel: a row the kernel skips cannot pass
    o, lse = attn.paged_mla(q, qp, lat, kp, ints["block_table"], ints["seq_lens"], ints["q_offsets"],
                            positions=pos, causal=w.causal, scale=x["scale"], return_lse=True, out=out,
                            num_splits=num_splits)
    return to_f64(o), lse.cpu().numpy().astype(np.float64)


def check(w, x=None, num_splits=1):
    x = x if x is not None else synth.make_mla_inputs(w)
    got, lse = run_mla(w, x, num_splits)
    ref, ref_lse = oracle.paged_mla(x["q"], x["qp"], x["latent"], x["kpos"], x["block_table"], x["seq_lens"],
                                    x["q_offsets"], positions=x["positions"], causal=w.causal, scale=x["scale"],
                                    dtype=w.dtype, lse=True)
    err = rel_err(got, ref)
    assert err <= TOL[w.dtype], f"{w.name}: rel err {err:.3e}"
    ninf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), ninf)
    fin = ~ninf
    if fin.any():
        e2 = np.max(np.abs(lse[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin])))
        assert e2 <= LSE_TOL, f"{w.name}: lse err {e2:.3e}"
    return x, got, ref


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
    check(w)


# Tensor-core kernel (F16/BF16, R in {256, 512}, Pd in {0, 64}, page sizes
# 8, 16, 32 or multiples of 64): 128-row blocks of (query, head) rows, a cluster
# of R/128 CTAs per block (one 128-column output slice each) that deal the
# 64-key tiles' scores round-robin and exchange the P tiles; several tiles and a
# ragged last tile.
TC_CASES = [
    MW("mla_tc_bf16_r512_p64_h128_decode", "bf16", 5, 128, 512, 64, 64, (1, 700), (1, 1), seed=11),
    MW("mla_tc_bf16_r512_p64_h16_p8", "bf16", 4, 16, 512, 64, 8, (30, 400), (1, 3), seed=12),
    MW("mla_tc_f16_r512_p0_h24_mtp", "f16", 3, 24, 512, 0, 32, (100, 500), (2, 11), seed=13),
    MW("mla_tc_bf16_r256_p64_p16_positions", "bf16", 4, 8, 256, 64, 16, (1, 300), (1, 40), seed=14,
       explicit_positions=True),
    MW("mla_tc_f16_r256_p0_p128_noncausal", "f16", 3, 32, 256, 0, 128, (40, 600), (1, 9), seed=15, causal=False),
    MW("mla_tc_bf16_r512_p64_prefill_p192", "bf16", 2, 8, 512, 64, 192, (150, 420), (40, 150), seed=16),
]


@pytest.mark.parametrize("w", TC_CASES, ids=lambda w: w.name)
def test_mla_tensor_core_matches_oracle(w):
    check(w)


@pytest.mark.parametrize("splits", [2, 7, 32])
def test_mla_tensor_core_splits(splits):
    # key runs per 128-row block merged from fp32 partials, including runs
    # with no tile (short sequences) and rows with no visible key
    w = MW(f"mla_tc_split{splits}", "bf16", 6, 64, 512, 64, 32, (0, 1500), (1, 2), seed=20 + splits,
           explicit_positions=True)
    check(w, num_splits=splits)
    w2 = MW(f"mla_tc_split{splits}_r256", "f16", 3, 16, 256, 0, 16, (1, 900), (1, 1), seed=50 + splits,
            causal=False)
    check(w2, num_splits=splits)


def _scale_key_rows(w, x, factor):
    """Multiply the latent and positional rows of every cached key by
    factor(position in its sequence, sequence length), rounded back to the
    storage dtype."""
    def widen(a):
        if w.dtype == "bf16":
            return (a.astype(np.uint32) << 16).view(np.float32)
        return a.astype(np.float32)
    lat, kp = widen(x["latent"]).copy(), widen(x["kpos"]).copy()
    P = w.page_size
    for s_ in range(len(x["seq_lens"])):
        L = int(x["seq_lens"][s_])
        for j in range(L):
            pg = x["block_table"][s_, j // P]
            lat[pg, j % P] *= factor(j, L)
            kp[pg, j % P] *= factor(j, L)
    x["latent"], x["kpos"] = synth.to_storage(lat, w.dtype), synth.to_storage(kp, w.dtype)
    return x


@pytest.mark.parametrize("dtype,R,Pd,kind", [("bf16", 512, 64, "grow"), ("f16", 256, 0, "grow"),
                                             ("bf16", 512, 64, "spike"), ("bf16", 512, 0, "shrink")])
def test_mla_tensor_core_reference_changes(dtype, R, Pd, kind):
    # The CTAs of a cluster compute the scores of alternate 64-key tiles, each
    # against a reference row maximum shared through the P tiles. Scores that
    # grow along the sequence (about 4 to 55 in log2 units per tile maximum)
    # make owners raise the reference mid-run: receivers rescale their output
    # rows, and tiles made against an older reference are scaled down (the
    # owner's own copy only after its peers have received it). A spike makes
    # one tile's maximum jump; shrinking scores keep the first tiles' maxima,
    # exchanged before the first P, as the reference.
    w = MW(f"mla_tc_ref_{kind}_{dtype}_r{R}", dtype, 4, 16, R, Pd, 64, (1500, 3200), (1, 1), seed=70 + R + Pd)
    x = synth.make_mla_inputs(w)
    if kind == "grow":
        f = lambda j, L: 1.0 + 15.0 * j / L
    elif kind == "shrink":
        f = lambda j, L: 16.0 - 15.0 * j / L
    else:
        f = lambda j, L: 40.0 if j == L // 2 else 1.0
    x = _scale_key_rows(w, x, f)
    check(w, x)
    if kind == "grow":
        check(w, x, num_splits=2)


def test_mla_tensor_core_edges():
    # a sequence without keys (NaN rows), sequences without queries, and
    # page-table entries past each sequence's pages that name no page of the
    # cache (a 32-key tile may reach into them; they must read as masked keys)
    w = MW("mla_tc_edges", "bf16", 5, 16, 512, 64, 16, (0, 200), (0, 3), seed=61, explicit_positions=True)
    x = synth.make_mla_inputs(w)
    x["seq_lens"][1] = 0
    pages = x["latent"].shape[0]
    for s_ in range(5):
        used = (int(x["seq_lens"][s_]) + 15) // 16
        x["block_table"][s_, used:] = pages + 5 if s_ % 2 else -7
    for ns in (1, 3):
        check(w, x, num_splits=ns)


def test_mla_splits_ignored_on_fma_path():
    # the fp32 FMA kernel (here F32, and a page size of 96) takes the workspace
    # but does not split
    w = MW("mla_f32_split", "f32", 3, 4, 128, 16, 8, (1, 120), (1, 4), seed=62)
    check(w, num_splits=4)
    w2 = MW("mla_bf16_p96_split", "bf16", 2, 8, 512, 64, 96, (150, 420), (1, 3), seed=63)
    check(w2, num_splits=3)


def test_mla_workspace_errors():
    import ctypes
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    lib = attn.load_library()
    dev = torch.device("cuda")
    shape = attn.MlaShape(1, 2, 4, 512, 64, 16, 2, 2, 2)
    need = attn.mla_workspace_bytes(shape, 3)
    assert need >= 3 * 2 * 4 * (4 * 512 + 8) and attn.mla_workspace_bytes(shape, 1) == 0
    q = torch.zeros(2, 4, 512, device=dev, dtype=torch.bfloat16)
    qp = torch.zeros(2, 4, 64, device=dev, dtype=torch.bfloat16)
    lat = torch.zeros(2, 16, 1, 512, device=dev, dtype=torch.bfloat16)
    kp = torch.zeros(2, 16, 1, 64, device=dev, dtype=torch.bfloat16)
    tab = torch.zeros(1, 2, dtype=torch.int32, device=dev)
    lens = torch.tensor([20], dtype=torch.int32, device=dev)
    offs = torch.tensor([0, 2], dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def call(ns, w, nbytes):
        return lib.attn_paged_mla(ctypes.byref(shape), q.data_ptr(), qp.data_ptr(), lat.data_ptr(), kp.data_ptr(),
                                  tab.data_ptr(), lens.data_ptr(), offs.data_ptr(), None, 1, ctypes.c_float(0.04),
                                  attn.ATTN_BF16, ns, w, nbytes, out.data_ptr(), None, None)
    assert call(3, ws.data_ptr(), need) == 0
    torch.cuda.synchronize()
    assert call(3, None, need) == -12
    assert call(3, ws.data_ptr(), need - 1) == -12
    assert call(0, None, 0) == -11
    assert call(33, ws.data_ptr(), need) == -11
    assert call(3, q.data_ptr(), need) == -8                                # workspace overlaps q


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
                                  attn.ATTN_BF16, 1, None, 0, o.data_ptr(), None, None)
    assert call() == 0
    torch.cuda.synchronize()
    assert call(R=96) == -4
    assert call(Pd=48) == -4
    assert call(o=q) == -8
