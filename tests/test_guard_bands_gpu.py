"""Guard bands around every output and workspace of the split, backward,
paged and MLA entry points, in the normal and in the bounds-checked build.

Each output (and workspace) is a view into the middle of a larger device
buffer whose bytes on both sides hold a sentinel pattern; after the call the
sentinel bytes must be untouched, so a write one element (or one row, one
page) past either end of any buffer is caught. The kernels index these
buffers through computed row, page and split offsets (the page tables of the
ruDNN user guide, section 9, in particular), where an off-by-one would land
in a neighbouring allocation. Every element of an output must also have been
written, and the device status word must stay clear. Shapes are small but span several tiles with
ragged tails; the tensor-core and the fp32 FMA kernels both run.

Every case runs twice: through libattn.so and through libattn_checked.so,
the same sources built with ATTN_CHECKED, whose kernels test every computed
global and shared-memory index and set ATTN_STATUS_BOUNDS in the status word
instead of making an out-of-range access. The checked run must leave that
word clear, and its outputs must be bit for bit those of the normal build
(the checks change no arithmetic). The two runs fill their buffers with
different sentinel bytes, so an element left unwritten holds a different
pattern in each run (a single sentinel can coincide with a written value,
since a 16-bit output takes only 65536 values).
"""
import numpy as np
import pytest

from exact_scaled_dot_flash_gb300 import synth
from tests.gpu_util import to_device

pytestmark = pytest.mark.gpu
PAD = 4096                 # sentinel bytes on each side of a guarded buffer
SENTINELS = (0xA5, 0x5A)   # byte patterns of the normal and the bounds-checked run


@pytest.fixture(scope="module")
def checked_path():
    """The bounds-checked library, built (or brought up to date) once."""
    from exact_scaled_dot_flash_gb300 import build
    return build.build(checked=True)


def run_both(checked_path, call):
    """``call(sentinel)`` returns {name: (Guarded, fully_written)}; it runs on
    the normal build with one sentinel byte and on the checked build with the
    other. Every guard band and the status word are checked each time; an
    element holding its run's sentinel in both runs was never written; and
    the two runs' outputs must agree bit for bit."""
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    dev = torch.cuda.current_device()
    results = []
    for path, sentinel in zip((None, checked_path), SENTINELS):
        if path is None:
            bufs = call(sentinel)
        else:
            with attn.use_library(path):
                bufs = call(sentinel)
                torch.cuda.synchronize()
                flags = attn.device_status(dev, clear=True)
            assert flags == 0, f"bounds-checked build: status flags {flags:#x}"
        for name, (g, full) in bufs.items():
            g.check_bands(name)
        results.append({name: (g.words(), g.pattern()) for name, (g, full) in bufs.items() if full})
    for name in results[0]:
        (w0, p0), (w1, p1) = results[0][name], results[1][name]
        unwritten = int(((w0 == p0) & (w1 == p1)).sum())
        assert unwritten == 0, f"{name}: {unwritten} elements left unwritten"
        assert np.array_equal(w0, w1), f"{name}: checked build differs"


@pytest.fixture(scope="module", autouse=True)
def _clean_status():
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    torch.cuda.synchronize()
    attn.device_status(torch.cuda.current_device(), clear=True)
    yield
    torch.cuda.synchronize()
    assert attn.device_status(torch.cuda.current_device(), clear=True) == 0, "a kernel wait timed out"


class Guarded:
    """A contiguous tensor of ``shape``/``dtype`` at byte offset PAD of a
    device buffer filled with the byte ``sentinel``, PAD sentinel bytes after it."""

    def __init__(self, shape, dtype, sentinel):
        import torch
        self.sentinel = sentinel
        self.nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((2 * PAD + self.nbytes,), sentinel, dtype=torch.uint8, device="cuda")
        self.t = self.buf[PAD:PAD + self.nbytes].view(dtype).view(*shape)

    def check_bands(self, name):
        import torch
        torch.cuda.synchronize()
        head = self.buf[:PAD]
        tail = self.buf[PAD + self.nbytes:]
        assert bool((head == self.sentinel).all()), f"{name}: bytes before the buffer were overwritten"
        assert bool((tail == self.sentinel).all()), f"{name}: bytes after the buffer were overwritten"

    def words(self):
        """The buffer's elements as integers of the element size."""
        es = self.t.element_size()
        return self.buf[PAD:PAD + self.nbytes].cpu().numpy().view({1: np.uint8, 2: np.uint16, 4: np.uint32}[es])

    def pattern(self):
        """An element that still holds the sentinel bytes."""
        es = self.t.element_size()
        return int.from_bytes(bytes([self.sentinel] * es), "little")


def guarded_like(t, sentinel):
    return Guarded(tuple(t.shape), t.dtype, sentinel)


def guarded_ws(nbytes, sentinel):
    import torch
    return Guarded((max(int(nbytes), 1),), torch.uint8, sentinel)


def _dense_inputs(w):
    x = synth.make_inputs(w)
    q, k, v = (to_device(x[n], w.dtype) for n in ("q", "k", "v"))
    lens = to_device(x["kv_lens"], "i32") if x["kv_lens"] is not None else None
    bias = to_device(x["bias"], "f32") if x["bias"] is not None else None
    return x, q, k, v, lens, bias


DENSE = [
    synth.Workload("gb_bf16_causal", "bf16", 2, 4, 2, 300, 700, 128, mask=synth.MASK_CAUSAL, seed=201),
    synth.Workload("gb_f16_pad_bias", "f16", 3, 4, 4, 260, 333, 64, mask=synth.MASK_KEY_PADDING, bias=True,
                   bias_b=1, bias_h=4, seed=202, kv_len_range=(1, 333)),
    synth.Workload("gb_f32", "f32", 2, 4, 2, 150, 170, 32, mask=synth.MASK_CAUSAL | synth.MASK_KEY_PADDING,
                   seed=203, kv_len_range=(1, 170)),
]


@pytest.mark.parametrize("w", DENSE, ids=lambda w: w.name)
def test_split_forward_guard_bands(w, checked_path):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    x, q, k, v, lens, bias = _dense_inputs(w)
    ns = 3
    shape = attn.Shape(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, *(x["bias"].shape[:2] if w.bias else (1, 1)))

    def call(sentinel):
        out, lse = guarded_like(q, sentinel), Guarded((w.B, w.Hq, w.Sq), torch.float32, sentinel)
        ws = guarded_ws(attn.split_workspace_bytes(shape, ns), sentinel)
        attn.fwd(q, k, v, causal=w.causal, kv_lens=lens, bias=bias, scale=x["scale"], out=out.t, num_splits=ns,
                 return_lse=True, workspace=ws.t, lse_out=lse.t)
        return {"out": (out, True), "lse": (lse, True), "split workspace": (ws, False)}
    run_both(checked_path, call)


@pytest.mark.parametrize("w", DENSE, ids=lambda w: w.name)
def test_backward_guard_bands(w, checked_path):
    from exact_scaled_dot_flash_gb300 import attn
    x, q, k, v, lens, bias = _dense_inputs(w)
    g = to_device(synth.to_storage(synth.normal_f32(w.seed, 7, (w.B, w.Hq, w.Sq, w.D)), w.dtype), w.dtype)
    o, lse = attn.fwd(q, k, v, causal=w.causal, kv_lens=lens, bias=bias, scale=x["scale"], return_lse=True)
    shape = attn.Shape(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, *(x["bias"].shape[:2] if w.bias else (1, 1)))

    def call(sentinel):
        dq, dk, dv = guarded_like(q, sentinel), guarded_like(k, sentinel), guarded_like(v, sentinel)
        ws = guarded_ws(attn.bwd_workspace_bytes(shape), sentinel)
        attn.bwd(q, k, v, o, g, lse, causal=w.causal, kv_lens=lens, bias=bias, scale=x["scale"], workspace=ws.t,
                 dq=dq.t, dk=dk.t, dv=dv.t)
        return {"dq": (dq, True), "dk": (dk, True), "dv": (dv, True), "backward workspace": (ws, False)}
    run_both(checked_path, call)


def _paged_inputs(pw, share=False):
    x = synth.make_paged_inputs(pw)
    if share:  # sequence 1 reads sequence 0's first physical page too
        x["block_table"] = x["block_table"].copy()
        x["block_table"][1, 0] = x["block_table"][0, 0]
    t = [to_device(x[n], pw.dtype) for n in ("q", "k_cache", "v_cache")]
    meta = [to_device(x[n], "i32") for n in ("block_table", "seq_lens", "q_offsets")]
    pos = to_device(x["positions"], "i32") if x["positions"] is not None else None
    return x, t, meta, pos


PAGED = [  # (workload, key splits of the forward)
    (synth.PagedWorkload("gb_paged_decode_tc", "bf16", 5, 8, 2, 128, 64, (70, 900), (1, 1), seed=211), 3),
    (synth.PagedWorkload("gb_paged_prefill_tc", "f16", 4, 8, 2, 64, 16, (40, 400), (5, 90), seed=212), 1),
    (synth.PagedWorkload("gb_paged_prefill_pos", "bf16", 3, 4, 4, 128, 32, (50, 300), (3, 40), seed=213,
                         explicit_positions=True), 1),
    (synth.PagedWorkload("gb_paged_f32", "f32", 4, 4, 2, 32, 8, (20, 200), (1, 30), seed=214), 2),
]


@pytest.mark.parametrize("pw,ns", PAGED, ids=lambda a: getattr(a, "name", str(a)))
def test_paged_forward_guard_bands(pw, ns, checked_path):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    x, (q, kc, vc), meta, pos = _paged_inputs(pw)
    nq = q.shape[0]
    mq = int(np.diff(x["q_offsets"]).max())
    shape = attn.PagedShape(pw.num_seqs, nq, pw.Hq, pw.Hkv, pw.D, pw.page_size, kc.shape[0], meta[0].shape[1], mq)

    def call(sentinel):
        out, lse = guarded_like(q, sentinel), Guarded((nq, pw.Hq), torch.float32, sentinel)
        ws = guarded_ws(attn.paged_workspace_bytes(shape, ns), sentinel)
        attn.paged_fwd(q, kc, vc, *meta, positions=pos, causal=True, scale=x["scale"], max_queries=mq, out=out.t,
                       return_lse=True, lse_out=lse.t, num_splits=ns, workspace=ws.t)
        return {"out": (out, True), "lse": (lse, True), "paged workspace": (ws, False)}
    run_both(checked_path, call)


@pytest.mark.parametrize("pw,ns", PAGED, ids=lambda a: getattr(a, "name", str(a)))
def test_paged_backward_guard_bands(pw, ns, checked_path):
    from exact_scaled_dot_flash_gb300 import attn
    x, (q, kc, vc), meta, pos = _paged_inputs(pw, share=True)
    nq = q.shape[0]
    mq = int(np.diff(x["q_offsets"]).max())
    g = to_device(synth.to_storage(synth.normal_f32(pw.seed, 9, x["q"].shape), pw.dtype), pw.dtype)
    shape = attn.PagedShape(pw.num_seqs, nq, pw.Hq, pw.Hkv, pw.D, pw.page_size, kc.shape[0], meta[0].shape[1], mq)
    o, lse = attn.paged_fwd(q, kc, vc, *meta, positions=pos, causal=True, scale=x["scale"], max_queries=mq,
                            return_lse=True)

    def call(sentinel):
        dq, dk, dv = guarded_like(q, sentinel), guarded_like(kc, sentinel), guarded_like(vc, sentinel)
        ws = guarded_ws(attn.paged_bwd_workspace_bytes(shape), sentinel)
        attn.paged_bwd(q, kc, vc, *meta, g, out=o, lse=lse, positions=pos, causal=True, scale=x["scale"],
                       max_queries=mq, workspace=ws.t, dq=dq.t, dk=dk.t, dv=dv.t)
        return {"dq": (dq, True), "dk": (dk, True), "dv": (dv, True), "paged backward workspace": (ws, False)}
    run_both(checked_path, call)


MLA = [
    (synth.MlaWorkload("gb_mla_decode_tc", "bf16", 4, 32, 512, 64, 64, (70, 700), (1, 1), seed=221), 2),
    (synth.MlaWorkload("gb_mla_prefill_tc", "f16", 3, 16, 256, 0, 32, (40, 300), (2, 12), seed=222), 1),
    (synth.MlaWorkload("gb_mla_f32", "f32", 3, 8, 128, 16, 16, (20, 150), (1, 6), seed=223), 2),
]


def _mla_inputs(mw, share=False):
    x = synth.make_mla_inputs(mw)
    if share:
        x["block_table"] = x["block_table"].copy()
        x["block_table"][1, 0] = x["block_table"][0, 0]
    t = [to_device(x[n], mw.dtype) for n in ("q", "qp", "latent", "kpos")]
    meta = [to_device(x[n], "i32") for n in ("block_table", "seq_lens", "q_offsets")]
    pos = to_device(x["positions"], "i32") if x["positions"] is not None else None
    return x, t, meta, pos


@pytest.mark.parametrize("mw,ns", MLA, ids=lambda a: getattr(a, "name", str(a)))
def test_mla_forward_guard_bands(mw, ns, checked_path):
    import torch
    from exact_scaled_dot_flash_gb300 import attn
    x, (q, qp, lat, kp), meta, pos = _mla_inputs(mw)
    nq = q.shape[0]
    mq = int(np.diff(x["q_offsets"]).max())
    shape = attn.MlaShape(mw.num_seqs, nq, mw.H, mw.R, mw.Pd, mw.page_size, lat.shape[0], meta[0].shape[1], mq)

    def call(sentinel):
        out, lse = guarded_like(q, sentinel), Guarded((nq, mw.H), torch.float32, sentinel)
        ws = guarded_ws(attn.mla_workspace_bytes(shape, ns), sentinel)
        attn.paged_mla(q, qp, lat, kp, *meta, positions=pos, causal=True, scale=x["scale"], max_queries=mq,
                       out=out.t, return_lse=True, lse_out=lse.t, num_splits=ns, workspace=ws.t)
        return {"out": (out, True), "lse": (lse, True), "MLA workspace": (ws, False)}
    run_both(checked_path, call)


@pytest.mark.parametrize("mw,ns", MLA, ids=lambda a: getattr(a, "name", str(a)))
def test_mla_backward_guard_bands(mw, ns, checked_path):
    from exact_scaled_dot_flash_gb300 import attn
    x, (q, qp, lat, kp), meta, pos = _mla_inputs(mw, share=True)
    nq = q.shape[0]
    mq = int(np.diff(x["q_offsets"]).max())
    g = to_device(synth.to_storage(synth.normal_f32(mw.seed, 9, x["q"].shape), mw.dtype), mw.dtype)
    shape = attn.MlaShape(mw.num_seqs, nq, mw.H, mw.R, mw.Pd, mw.page_size, lat.shape[0], meta[0].shape[1], mq)
    o, lse = attn.paged_mla(q, qp, lat, kp, *meta, positions=pos, causal=True, scale=x["scale"], max_queries=mq,
                            return_lse=True)

    def call(sentinel):
        dq, dlat = guarded_like(q, sentinel), guarded_like(lat, sentinel)
        dqp = guarded_like(qp, sentinel) if mw.Pd else None
        dkp = guarded_like(kp, sentinel) if mw.Pd else None
        ws = guarded_ws(attn.mla_bwd_workspace_bytes(shape), sentinel)
        attn.paged_mla_bwd(q, qp, lat, kp, *meta, g, out=o, lse=lse, positions=pos, causal=True, scale=x["scale"],
                           max_queries=mq, workspace=ws.t, dq=dq.t, dqp=dqp.t if dqp else None, dlatent=dlat.t,
                           dkpos=dkp.t if dkp else None)
        bufs = {"dq": (dq, True), "dlatent": (dlat, True), "MLA backward workspace": (ws, False)}
        if mw.Pd:
            bufs.update({"dqp": (dqp, True), "dkpos": (dkp, True)})
        return bufs
    run_both(checked_path, call)
