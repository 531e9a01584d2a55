"""Device parity of the checked mode and of the device-content checks.

Checked mode must not change a result: every call on valid inputs gives bit-identical
outputs with and without it.  Each broken array below must be caught (status
GCS_ERR_INVALID_ARG, outputs untouched where the header says no kernel writes them).  Every
broken case is chosen so that a kernel fed the broken array anyway would still stay inside
its buffers: lengths that go negative give no tiles, a page-table entry one past num_blocks
names a block that exists in memory (the caches carry one extra zero block that the call is
not told about), and a seq_len above max_seq_len stays within the page-table row."""
import ctypes

import pytest
import torch

import oracle
from synth import make_decode, make_prefill
from helpers import decode_dev, to_dev

pytestmark = pytest.mark.gpu

INVALID = 1
SENTINEL = 3.0


@pytest.fixture
def checked(gcs_lib):
    gcs_lib.get_device_status(clear=True)
    gcs_lib.set_device_checks(True)
    yield gcs_lib
    gcs_lib.set_device_checks(False)
    gcs_lib.get_device_status(clear=True)


def prefill_all(gcs, case, d, cu=None, deterministic=False):
    cu = d["cu"] if cu is None else cu
    ms = max(case.seqlens)
    o, lse = gcs.attn_fwd(d["q"], d["k"], d["v"], cu, ms, case.scale, case.window, d["g"], d["s"])
    g = gcs.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], cu, ms, case.scale, case.window, d["g"], d["s"],
                     deterministic=deterministic)
    torch.cuda.synchronize()
    return [o, lse] + [t for t in g if t is not None]


@pytest.mark.parametrize("dims,det", [((128, 128), True), ((128, 128), False), ((64, 64), False), ((256, 512), True)])
def test_checked_mode_leaves_prefill_results_unchanged(gcs_lib, dims, det):
    case = make_prefill([300, 1, 129], 4, 2, dims[0], dims[1], seed=700 + dims[0], gate=True, sink=True, window=0)
    d = to_dev(case)
    gcs_lib.set_device_checks(False)
    ref = prefill_all(gcs_lib, case, d, deterministic=det)
    assert gcs_lib.get_device_status() == 0
    gcs_lib.set_device_checks(True)
    try:
        got = prefill_all(gcs_lib, case, d, deterministic=det)
        assert gcs_lib.get_device_status() == 0
    finally:
        gcs_lib.set_device_checks(False)
    # o, lse, dq, dk, dv, dlog_gate, dsink: the single-pass route (128 without deterministic)
    # reduce-adds dq and the dS row sums in fp32, whose low bits may vary from call to call
    loose = {2, 5, 6} if (dims == (128, 128) and not det) else set()
    for i, (a, b) in enumerate(zip(ref, got)):
        if i in loose:
            assert oracle.rel_rms(a.double().cpu().numpy(), b.double().cpu().numpy()) <= 1e-4, i
        else:
            assert torch.equal(a, b), i


def paged_calls(gcs, dc, d, segment_len):
    """Decode (workspace and allocation-free) when every q_len <= 4, and the paged prefill."""
    maxl = int(dc.seq_lens.max())
    kw = dict(g_cache=d["g"], sink=d["sink"], window=dc.window)
    args = (d["q"], d["kc"], d["vc"], d["ks"], d["vs"], d["bt"], d["sl"], d["cq"], max(dc.q_lens), maxl, dc.scale)
    outs = [gcs.attn_prefill_paged(*args, segment_len, **kw)]
    if max(dc.q_lens) <= 4:
        outs.append(gcs.attn_decode_paged(*args, 128, **kw))
        outs.append(gcs.attn_decode_paged_noalloc(*args, 2048, **kw))
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("feat", [False, True])
@pytest.mark.parametrize("seg", [0, 128])
def test_checked_mode_leaves_paged_results_unchanged(gcs_lib, feat, seg):
    for sl, ql in (([300, 1000, 17], [1, 3, 4]), ([300, 1000], [100, 57])):
        dc = make_decode(sl, ql, 16, 1, 128, seed=710 + seg, features=feat, window=200 if feat else 0)
        d = decode_dev(dc)
        gcs_lib.set_device_checks(False)
        ref = paged_calls(gcs_lib, dc, d, seg)
        assert gcs_lib.get_device_status() == 0
        gcs_lib.set_device_checks(True)
        try:
            got = paged_calls(gcs_lib, dc, d, seg)
            assert gcs_lib.get_device_status() == 0
        finally:
            gcs_lib.set_device_checks(False)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)


BAD_CU = {
    # seqlens [200, -100, 200]: the middle length is negative
    "not_monotone": [0, 200, 100, 300],
    # ends at 250 but total_tokens is 300
    "end_not_total": [0, 100, 250],
    # one 300-token sequence with max_seqlen 200
    "longer_than_max": [0, 300],
}


@pytest.mark.parametrize("name", list(BAD_CU))
def test_broken_cu_seqlens_is_caught(checked, name):
    gcs = checked
    case = make_prefill([100, 200], 4, 2, 128, 128, seed=720, gate=True, sink=True)
    d = to_dev(case)
    ok = prefill_all(gcs, case, d)  # o, lse of a valid call for the backward's inputs
    assert gcs.get_device_status() == 0
    bad = torch.tensor(BAD_CU[name], dtype=torch.int32, device="cuda:0")
    # the stand-alone check
    gcs.check_prefill_inputs(d["q"], d["k"], d["v"], bad, 200, case.scale, 0, d["g"], d["s"])
    torch.cuda.synchronize()
    assert gcs.get_device_status() == INVALID
    gcs.check_prefill_inputs(d["q"], d["k"], d["v"], d["cu"], 200, case.scale, 0, d["g"], d["s"])
    torch.cuda.synchronize()
    assert gcs.get_device_status() == 0
    # a checked forward: nothing written
    o = torch.full_like(ok[0], SENTINEL)
    lse = torch.full_like(ok[1], SENTINEL)
    gcs.attn_fwd(d["q"], d["k"], d["v"], bad, 200, case.scale, 0, d["g"], d["s"], out=o, lse=lse)
    torch.cuda.synchronize()
    assert gcs.get_device_status() == INVALID
    assert bool((o == SENTINEL).all()) and bool((lse == SENTINEL).all())
    # a checked backward: dQ (two-pass route), dK, dV and d log_gate untouched; the single
    # pass converts its zeroed dQ accumulator, so there dQ holds zeros
    for det in (True, False):
        dq, dk, dv = (torch.full_like(t, SENTINEL) for t in (d["q"], d["k"], d["v"]))
        dg = torch.full_like(d["g"], SENTINEL)
        gcs.attn_bwd(d["q"], d["k"], d["v"], ok[0], ok[1], d["do"], bad, 200, case.scale, 0, d["g"], d["s"], dq=dq,
                     dk=dk, dv=dv, dlog_gate=dg, deterministic=det)
        torch.cuda.synchronize()
        assert gcs.get_device_status() == INVALID
        for t in (dk, dv, dg):
            assert bool((t == SENTINEL).all())
        assert bool((dq == SENTINEL).all()) if det else bool((dq == 0).all())


def padded_paged(gcs, dc, d, max_q_len, max_seq_len, segment_len, bt=None, sl=None, cq=None):
    """DecodeArgs over caches that carry one extra zero block the call is not told about
    (num_blocks stays the case's)."""
    nb = dc.k_cache.shape[0]
    pad = lambda t: torch.cat([t, torch.zeros_like(t[:1])])
    kc, vc, ks, vs = pad(d["kc"]), pad(d["vc"]), pad(d["ks"]), pad(d["vs"])
    a = gcs.decode_args(d["q"], kc, vc, ks, vs, d["bt"] if bt is None else bt, d["sl"] if sl is None else sl,
                        d["cq"] if cq is None else cq, max_q_len, max_seq_len, dc.scale, segment_len)
    a.num_blocks = nb
    return a, (kc, vc, ks, vs)


def run_paged_raw(gcs, a, kind, q):
    """Calls attn_decode_paged or attn_prefill_paged through the C ABI with a sentinel output."""
    L = gcs.load()
    out = torch.full_like(q, SENTINEL)
    size = L.attn_decode_workspace(ctypes.byref(a)) if kind == "decode" else L.attn_prefill_paged_workspace(
        ctypes.byref(a))
    ws = torch.empty(max(size, 1), dtype=torch.uint8, device=q.device)
    fn = L.attn_decode_paged if kind == "decode" else L.attn_prefill_paged
    st = fn(ctypes.byref(a), out.data_ptr(), ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("kind", ["decode", "prefill_paged"])
@pytest.mark.parametrize("name", ["entry_past_num_blocks", "seq_len_above_max", "cu_q_end_not_total"])
def test_broken_paged_arrays_are_caught(checked, kind, name):
    gcs = checked
    ql = [1, 2] if kind == "decode" else [40, 100]
    dc = make_decode([600, 300], ql, 16, 1, 128, seed=730)
    d = decode_dev(dc)
    nb = dc.k_cache.shape[0]
    bt, sl, cq = d["bt"].clone(), d["sl"].clone(), d["cq"].clone()
    max_seq_len = 600
    if name == "entry_past_num_blocks":
        bt[0, 0] = nb  # page 0 of request 0 is read; block nb is the extra zero block
    elif name == "seq_len_above_max":
        max_seq_len = 584  # request 0 holds 600 tokens; its table row has 38 pages
    else:
        cq[2] = cq[1]  # request 1 loses its query rows, so cu_q ends short of total_q
    seg = 128 if kind == "decode" else 0
    a, keep = padded_paged(gcs, dc, d, max(ql), max_seq_len, seg, bt=bt, sl=sl, cq=cq)
    out = run_paged_raw(gcs, a, kind, d["q"])
    assert gcs.get_device_status() == INVALID
    assert bool((out == SENTINEL).all())
    # the stand-alone check agrees, and passes the unbroken arrays
    L = gcs.load()
    s = torch.cuda.current_stream().cuda_stream
    assert L.gcs_check_paged_inputs(ctypes.byref(a), s) == 0
    torch.cuda.synchronize()
    assert gcs.get_device_status() == INVALID
    a_ok, keep2 = padded_paged(gcs, dc, d, max(ql), 600, seg)
    assert L.gcs_check_paged_inputs(ctypes.byref(a_ok), s) == 0
    torch.cuda.synchronize()
    assert gcs.get_device_status() == 0


@pytest.mark.parametrize("kind", ["decode", "prefill_paged"])
def test_window_leaves_unread_pages_unchecked(checked, kind):
    """With a window, pages wholly before the 128-key tile of the earliest visible key are not
    read, so an entry there may name a block outside [0, num_blocks): no error, same result."""
    gcs = checked
    ql = [1, 4] if kind == "decode" else [100, 37]
    dc = make_decode([1000, 1200], ql, 16, 1, 128, seed=740, features=True, window=300)
    d = decode_dev(dc)
    nb = dc.k_cache.shape[0]
    seg = 128 if kind == "decode" else 0
    a_ref, keep = padded_paged(gcs, dc, d, max(ql), 1200, seg)
    a_ref.window = dc.window
    gcs.set_device_checks(False)
    ref = run_paged_raw(gcs, a_ref, kind, d["q"])
    assert gcs.get_device_status() == 0
    gcs.set_device_checks(True)
    bt = d["bt"].clone()
    # keys 48..63 of request 0 and 0..15 of request 1: every key a query row of either shape
    # sees is at least 1000 - 100 - 300 + 1 = 601, in a 128-key tile from key 512 on
    bt[0, 3] = nb
    bt[1, 0] = nb
    a, keep2 = padded_paged(gcs, dc, d, max(ql), 1200, seg, bt=bt)
    a.window = dc.window
    got = run_paged_raw(gcs, a, kind, d["q"])
    assert gcs.get_device_status() == 0
    assert torch.equal(got, ref)


@pytest.mark.parametrize("kind", ["decode", "prefill_paged"])
@pytest.mark.parametrize("name", ["v_scale_at_255", "q_above_f16_max", "per_tensor_v_scale"])
def test_fp8_operand_limits_are_caught(checked, kind, name):
    """With an fp8 cache the tensor cores see f16: a |q| above 65504 or a V scale of 255 or more
    in a slot below seq_len would overflow.  Checked mode refuses both (status
    GCS_ERR_INVALID_ARG, output untouched); the same values where they are not read (slots past
    seq_len hold NaN scales in every case here) pass."""
    gcs = checked
    ql = [1, 3] if kind == "decode" else [40, 100]
    per_tensor = name == "per_tensor_v_scale"
    dc = make_decode([600, 300], ql, 16, 1, 128, seed=750, scale_mode="per_tensor" if per_tensor else "per_token")
    d = decode_dev(dc)
    seg = 128 if kind == "decode" else 0
    q = d["q"].clone()
    vs = d["vs"].clone()
    if name == "v_scale_at_255":
        blk = int(dc.block_table[1, 18])  # request 1 (300 tokens): page 18 holds slots 288..299
        vs[blk, 0, 11] = 255.0
    elif name == "q_above_f16_max":
        q[2, 5, 17] = 65536.0  # bf16-exact, above the f16 range
    else:
        vs.fill_(300.0)
    a = gcs.decode_args(q, d["kc"], d["vc"], d["ks"], vs, d["bt"], d["sl"], d["cq"], max(ql), 600, dc.scale, seg)
    out = run_paged_raw(gcs, a, kind, q)
    assert gcs.get_device_status() == INVALID
    assert bool((out == SENTINEL).all())
    # the limits themselves pass: 254.9 in that slot, 65280 (the largest bf16 below 65504) in q
    if name == "v_scale_at_255":
        vs[blk, 0, 11] = 254.9
    elif name == "q_above_f16_max":
        q[2, 5, 17] = 65280.0
    else:
        vs.fill_(254.9)
    a = gcs.decode_args(q, d["kc"], d["vc"], d["ks"], vs, d["bt"], d["sl"], d["cq"], max(ql), 600, dc.scale, seg)
    L = gcs.load()
    assert L.gcs_check_paged_inputs(ctypes.byref(a), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert gcs.get_device_status() == 0
