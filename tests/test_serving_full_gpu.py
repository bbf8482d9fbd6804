"""The serving workloads (paged decode, paged prefill, MLA decode) at full size,
launched exactly as bench.py times them (same shapes, same key splits), checked
against the float64 oracle on sampled query rows of sampled sequences.

The oracle cannot widen the whole cache (gigabytes in float64), so each check
builds a compact problem from the sampled rows only: their sequences' pages copied
into a small cache, their page-table rows remapped, their query rows repacked.
Rows of a sequence depend on nothing else, so the GPU's rows for those
sequences must match the oracle on the compact problem. Tolerances as for the
dense forward (bf16: max|O - O_ref| / max|O_ref| <= 1.6e-2; lse within 1e-4).
"""
import numpy as np
import pytest

import bench
import oracle
from exact_scaled_dot_flash_gb300 import synth
from tests.gpu_util import TOL, rel_err, to_device, to_f64

pytestmark = pytest.mark.gpu
LSE_TOL = 1e-4


def pick(x, n, seed):
    """Sampled sequences: the longest, the shortest and n-2 random others."""
    lens = x["seq_lens"]
    rest = np.random.default_rng(seed).permutation(len(lens))
    chosen = [int(np.argmax(lens)), int(np.argmin(lens))] + [int(s) for s in rest]
    out = []
    for s in chosen:
        if s not in out and np.diff(x["q_offsets"])[s] > 0:
            out.append(s)
        if len(out) == n:
            break
    return out


def compact(x, seqs, caches, P, per_seq=4, seed=0):
    """The sub-problem of sequences ``seqs``, each keeping at most ``per_seq``
    of its queries (its first, its last and random others) at their absolute
    positions: (dict of arrays, query rows of the full problem in the order of
    the sub-problem)."""
    table, lens, offs = x["block_table"], x["seq_lens"], x["q_offsets"]
    g = np.random.default_rng(seed)
    pages = []
    for s in seqs:
        pages += [int(p) for p in table[s, :(int(lens[s]) + P - 1) // P]]
    remap = {p: i for i, p in enumerate(pages)}
    sub = {c: np.ascontiguousarray(x[c][np.array(pages, dtype=np.int64)]) for c in caches}
    width = max(1, max((int(lens[s]) + P - 1) // P for s in seqs))
    sub["block_table"] = np.full((len(seqs), width), -1, dtype=np.int32)
    rows, pos = [], []
    sub_offs = [0]
    for i, s in enumerate(seqs):
        used = (int(lens[s]) + P - 1) // P
        sub["block_table"][i, :used] = [remap[int(p)] for p in table[s, :used]]
        lo, hi = int(offs[s]), int(offs[s + 1])
        keep = sorted({lo, hi - 1} | set(int(r) for r in g.integers(lo, hi, size=max(0, per_seq - 2))))
        rows += keep
        # absolute positions: explicit ones, else the newest-token default of the full problem
        pos += [int(x["positions"][r]) if x["positions"] is not None else int(lens[s]) - (hi - lo) + (r - lo)
                for r in keep]
        sub_offs.append(len(rows))
    sub["seq_lens"] = lens[np.array(seqs)].astype(np.int32)
    sub["q_offsets"] = np.array(sub_offs, dtype=np.int32)
    sub["positions"] = np.array(pos, dtype=np.int32)
    return sub, np.array(rows)


def check_rows(got, lse, ref, ref_lse, dtype, name):
    assert rel_err(got, ref) <= TOL[dtype], f"{name}: rel err {rel_err(got, ref):.3e}"
    ninf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), ninf)
    fin = ~ninf
    if fin.any():
        e2 = np.max(np.abs(lse[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin])))
        assert e2 <= LSE_TOL, f"{name}: lse err {e2:.3e}"


@pytest.mark.parametrize("name", sorted(synth.PAGED_WORKLOADS))
def test_paged_workload_full_size_sampled(name):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = synth.PAGED_WORKLOADS[name]
    x = synth.make_paged_inputs(w)
    q, kc, vc = (to_device(x[n], w.dtype) for n in ("q", "k_cache", "v_cache"))
    ints = {n: to_device(x[n], "i32") for n in ("block_table", "seq_lens", "q_offsets")}
    pos = to_device(x["positions"], "i32") if x["positions"] is not None else None
    max_q = int(np.diff(x["q_offsets"]).max())
    o, lse = attn.paged_fwd(q, kc, vc, ints["block_table"], ints["seq_lens"], ints["q_offsets"], positions=pos,
                            causal=w.causal, scale=x["scale"], max_queries=max_q, return_lse=True,
                            num_splits=bench.PAGED_SPLITS.get(name, 1))
    torch.cuda.synchronize()
    got, got_lse = to_f64(o), lse.cpu().numpy().astype(np.float64)
    seqs = pick(x, 4, seed=1)
    sub, rows = compact(x, seqs, ("k_cache", "v_cache"), w.page_size, seed=1)
    ref, ref_lse = oracle.paged_attention(x["q"][rows], sub["k_cache"], sub["v_cache"], sub["block_table"],
                                          sub["seq_lens"], sub["q_offsets"], positions=sub["positions"],
                                          causal=w.causal, scale=x["scale"], dtype=w.dtype, lse=True)
    check_rows(got[rows], got_lse[rows], ref, ref_lse, w.dtype, name)


@pytest.mark.parametrize("name", sorted(synth.MLA_WORKLOADS))
def test_mla_workload_full_size_sampled(name):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = synth.MLA_WORKLOADS[name]
    x = synth.make_mla_inputs(w)
    q, qp, lat, kp = (to_device(x[n], w.dtype) for n in ("q", "qp", "latent", "kpos"))
    ints = {n: to_device(x[n], "i32") for n in ("block_table", "seq_lens", "q_offsets")}
    pos = to_device(x["positions"], "i32") if x["positions"] is not None else None
    max_q = int(np.diff(x["q_offsets"]).max())
    o, lse = attn.paged_mla(q, qp, lat, kp, ints["block_table"], ints["seq_lens"], ints["q_offsets"],
                            positions=pos, causal=w.causal, scale=x["scale"], max_queries=max_q, return_lse=True,
                            num_splits=bench.PAGED_SPLITS.get(name, 1))
    torch.cuda.synchronize()
    got, got_lse = to_f64(o), lse.cpu().numpy().astype(np.float64)
    seqs = pick(x, 4, seed=2)
    sub, rows = compact(x, seqs, ("latent", "kpos"), w.page_size, seed=2)
    ref, ref_lse = oracle.paged_mla(x["q"][rows], x["qp"][rows], sub["latent"], sub["kpos"], sub["block_table"],
                                    sub["seq_lens"], sub["q_offsets"], positions=sub["positions"], causal=w.causal,
                                    scale=x["scale"], dtype=w.dtype, lse=True)
    check_rows(got[rows], got_lse[rows], ref, ref_lse, w.dtype, name)


def compact_all_rows(x, seqs, caches, P):
    """The sub-problem of sequences ``seqs`` with all their queries (so the
    default positions stay the same): (sub-problem, query rows of the full
    problem in order, physical pages of the full problem in the order of the
    sub-problem's cache)."""
    table, lens, offs = x["block_table"], x["seq_lens"], x["q_offsets"]
    pages = []
    for s in seqs:
        pages += [int(p) for p in table[s, :(int(lens[s]) + P - 1) // P]]
    remap = {p: i for i, p in enumerate(pages)}
    sub = {c: np.ascontiguousarray(x[c][np.array(pages, dtype=np.int64)]) for c in caches}
    width = max(1, max((int(lens[s]) + P - 1) // P for s in seqs))
    sub["block_table"] = np.full((len(seqs), width), -1, dtype=np.int32)
    rows, sub_offs = [], [0]
    for i, s in enumerate(seqs):
        used = (int(lens[s]) + P - 1) // P
        sub["block_table"][i, :used] = [remap[int(p)] for p in table[s, :used]]
        rows += list(range(int(offs[s]), int(offs[s + 1])))
        sub_offs.append(len(rows))
    sub["seq_lens"] = lens[np.array(seqs)].astype(np.int32)
    sub["q_offsets"] = np.array(sub_offs, dtype=np.int32)
    sub["positions"] = None if x["positions"] is None else x["positions"][np.array(rows)]
    return sub, np.array(rows), np.array(pages)


def cheapest(x, n):
    """The n sequences (with queries) of least oracle work (keys x queries)."""
    cost = x["seq_lens"].astype(np.int64) * np.diff(x["q_offsets"])
    order = [int(s) for s in np.argsort(cost, kind="stable") if np.diff(x["q_offsets"])[s] > 0]
    return order[:n]


def check_grads(got, ref, dtype, name):
    for gname, a, b in zip(name[1], got, ref):
        err = float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))
        assert err <= TOL[dtype], f"{name[0]} {gname}: rel err {err:.3e}"


def test_paged_prefill_backward_full_size_sampled():
    # the full-size call; no page is shared, so a page's gradients come from its
    # own sequence alone and the compact sub-problem reproduces them
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = synth.PAGED_WORKLOADS["bf16_paged_prefill"]
    x = synth.make_paged_inputs(w)
    q, kc, vc = (to_device(x[n], w.dtype) for n in ("q", "k_cache", "v_cache"))
    ints = {n: to_device(x[n], "i32") for n in ("block_table", "seq_lens", "q_offsets")}
    g = synth.to_storage(synth.normal_f32(w.seed, 9, x["q"].shape), w.dtype)
    dq, dk, dv = attn.paged_bwd(q, kc, vc, ints["block_table"], ints["seq_lens"], ints["q_offsets"],
                                to_device(g, w.dtype), causal=w.causal, scale=x["scale"])
    torch.cuda.synchronize()
    seqs = cheapest(x, 2)
    sub, rows, pages = compact_all_rows(x, seqs, ("k_cache", "v_cache"), w.page_size)
    ref = oracle.paged_attention_bwd(x["q"][rows], sub["k_cache"], sub["v_cache"], g[rows], sub["block_table"],
                                     sub["seq_lens"], sub["q_offsets"], positions=sub["positions"],
                                     causal=w.causal, scale=x["scale"], dtype=w.dtype)
    got = (to_f64(dq)[rows], to_f64(dk)[pages], to_f64(dv)[pages])
    check_grads(got, ref, w.dtype, (w.name, ("dq", "dk", "dv")))


def test_mla_decode_backward_full_size_sampled():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    w = synth.MLA_WORKLOADS["bf16_mla_decode"]
    x = synth.make_mla_inputs(w)
    q, qp, lat, kp = (to_device(x[n], w.dtype) for n in ("q", "qp", "latent", "kpos"))
    ints = {n: to_device(x[n], "i32") for n in ("block_table", "seq_lens", "q_offsets")}
    g = synth.to_storage(synth.normal_f32(w.seed, 9, x["q"].shape), w.dtype)
    grads = attn.paged_mla_bwd(q, qp, lat, kp, ints["block_table"], ints["seq_lens"], ints["q_offsets"],
                               to_device(g, w.dtype), causal=w.causal, scale=x["scale"])
    torch.cuda.synchronize()
    seqs = cheapest(x, 3)
    sub, rows, pages = compact_all_rows(x, seqs, ("latent", "kpos"), w.page_size)
    ref = oracle.paged_mla_bwd(x["q"][rows], x["qp"][rows], sub["latent"], sub["kpos"], g[rows],
                               sub["block_table"], sub["seq_lens"], sub["q_offsets"], positions=sub["positions"],
                               causal=w.causal, scale=x["scale"], dtype=w.dtype)
    dq, dqp, dlat, dkp = (to_f64(t) for t in grads)
    got = (dq[rows], dqp[rows], dlat[pages], dkp[pages])
    check_grads(got, ref, w.dtype, (w.name, ("dq", "dqp", "dlatent", "dkpos")))
