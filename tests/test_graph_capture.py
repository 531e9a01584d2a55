"""The library's calls inside a CUDA graph: a captured prefill step (forward + backward) and a
captured decode call, replayed, give the results of the same calls made eagerly.  Every
launch of a call goes to the caller's stream and no call synchronises or allocates, so a
stream capture records the whole call; replays then run without host launch work.

Outputs, workspaces and inputs are allocated before the capture (the replays read and write
those same buffers).  Routes whose results are written once or summed in a fixed order give
the same bits; the single-pass backward reduce-adds dQ and the dS row sums in fp32 in L2, whose
order varies from run to run, so those are compared within a relative RMS of 1e-3."""
import ctypes

import pytest
import torch

import oracle
from synth import make_decode, make_prefill
from helpers import PREFILL_RTOL, assert_close, decode_dev, f64, oracle_decode, DECODE_RTOL, oracle_prefill, to_dev

pytestmark = pytest.mark.gpu


def _capture(fn, warm=2):
    """Warm fn up on a side stream, capture one call into a graph and return it."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warm):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


@pytest.mark.parametrize("deterministic", [False, True])
def test_prefill_step_graph_matches_eager(gcs_lib, deterministic):
    case = make_prefill([300, 1, 517, 129], 8, 2, 128, 128, seed=901, gate=True, sink=True, window=0)
    d = to_dev(case)
    ms = max(case.seqlens)
    dev = d["q"].device
    o = torch.empty((case.total, case.hq, case.dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.hq, case.total), dtype=torch.float32, device=dev)
    grads = dict(dq=torch.empty_like(d["q"]), dk=torch.empty_like(d["k"]), dv=torch.empty_like(d["v"]),
                 dlog_gate=torch.empty_like(d["g"]), dsink=torch.empty_like(d["s"]))
    L = gcs_lib.load()
    a = gcs_lib.prefill_args(d["q"], d["k"], d["v"], d["cu"], ms, case.scale, 0, d["g"], d["s"])
    fws = torch.empty(L.attn_fwd_workspace(ctypes.byref(a)) + 1, dtype=torch.uint8, device=dev)
    a.deterministic = 1 if deterministic else 0
    bws = torch.empty(L.attn_bwd_workspace(ctypes.byref(a)) + 1, dtype=torch.uint8, device=dev)

    def step():
        gcs_lib.attn_fwd(d["q"], d["k"], d["v"], d["cu"], ms, case.scale, 0, d["g"], d["s"], out=o, lse=lse,
                         workspace=fws)
        gcs_lib.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], ms, case.scale, 0, d["g"], d["s"],
                         workspace=bws, deterministic=deterministic, **grads)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, *grads.values())]
    graph = _capture(step)
    for t in (o, lse, *grads.values()):
        t.fill_(float("nan"))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert gcs_lib.get_device_status() == 0
    names = ("o", "lse", "dq", "dk", "dv", "dlog_gate", "dsink")
    for n, got, ref in zip(names, (o, lse, *grads.values()), eager):
        if deterministic or n in ("o", "lse", "dk", "dv"):
            assert torch.equal(got, ref), n
        else:
            assert oracle.rel_rms(f64(got), f64(ref)) <= 1e-3, n
    ro, _, rg = oracle_prefill(case)
    assert_close("o", o, ro, PREFILL_RTOL)
    assert_close("dq", grads["dq"], rg[0], PREFILL_RTOL)


def test_decode_graph_matches_eager(gcs_lib):
    dc = make_decode([1, 700, 4100, 33, 2049], [1, 1, 1, 1, 1], 64, 4, 128, seed=902)
    d = decode_dev(dc)
    out = torch.empty_like(d["q"])
    maxl = int(dc.seq_lens.max())

    def call():
        gcs_lib.attn_decode_paged(d["q"], d["kc"], d["vc"], d["ks"], d["vs"], d["bt"], d["sl"], d["cq"], 1, maxl,
                                  dc.scale, dc.segment_len, out=out)

    call()
    torch.cuda.synchronize()
    eager = out.clone()
    graph = _capture(call)
    out.fill_(float("nan"))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert gcs_lib.get_device_status() == 0
    assert torch.equal(out, eager)
    assert_close("out", out, oracle_decode(dc), DECODE_RTOL)
