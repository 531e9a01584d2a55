"""Workspace poisoning: every call run once with its workspace filled with 0xFF bytes (NaN in
every fp32 slot) and once zero-filled must give bit-identical, finite outputs, so no kernel
reads a workspace byte that the same call did not write first.  The cases take the routes
with the most workspace: split-K decode and paged prefill with short requests and a window
(segments that are skipped or empty), and the prefill backward with gates and a sink."""
import ctypes

import pytest
import torch

from synth import make_decode, make_prefill
from helpers import decode_dev, to_dev

pytestmark = pytest.mark.gpu


def twice(size, run):
    outs = []
    for fill in (0x00, 0xFF):
        ws = torch.full((max(size, 1),), fill, dtype=torch.uint8, device="cuda:0")
        outs.append(run(ws))
        torch.cuda.synchronize()
    return outs


def same(a, b):
    for x, y in zip(a, b):
        if x is None:
            assert y is None
            continue
        assert torch.isfinite(x.float()).all()
        assert torch.equal(x, y)


@pytest.mark.parametrize("feat", [False, True])
def test_paged_calls_ignore_workspace_contents(gcs_lib, feat):
    L = gcs_lib.load()
    for sl, ql, seg in (([3000, 17, 700, 1], [1, 4, 2, 1], 128), ([2000, 300, 40], [100, 60, 40], 128)):
        dc = make_decode(sl, ql, 16, 1, 128, seed=760, features=feat, window=500 if feat else 0)
        d = decode_dev(dc)
        args = (d["q"], d["kc"], d["vc"], d["ks"], d["vs"], d["bt"], d["sl"], d["cq"], max(ql), max(sl), dc.scale,
                seg)
        kw = dict(g_cache=d["g"], sink=d["sink"], window=dc.window)
        a = gcs_lib.decode_args(*args, **kw)
        calls = [(L.attn_prefill_paged_workspace(ctypes.byref(a)),
                  lambda ws: [gcs_lib.attn_prefill_paged(*args, workspace=ws, **kw)])]
        if max(ql) <= 4:
            calls.append((L.attn_decode_workspace(ctypes.byref(a)),
                          lambda ws: [gcs_lib.attn_decode_paged(*args, workspace=ws, **kw)]))
        for size, run in calls:
            assert size > 0
            zero, poisoned = twice(size, run)
            assert gcs_lib.get_device_status() == 0
            same(zero, poisoned)


@pytest.mark.parametrize("dims", [(128, 128), (256, 512)])
def test_prefill_ignores_workspace_contents(gcs_lib, dims):
    L = gcs_lib.load()
    case = make_prefill([300, 1, 129], 4, 2, dims[0], dims[1], seed=770 + dims[0], gate=True, sink=True, window=40)
    d = to_dev(case)
    ms = max(case.seqlens)
    a = gcs_lib.prefill_args(d["q"], d["k"], d["v"], d["cu"], ms, case.scale, case.window, d["g"], d["s"])
    a.deterministic = 1
    fwd = lambda ws: list(gcs_lib.attn_fwd(d["q"], d["k"], d["v"], d["cu"], ms, case.scale, case.window, d["g"],
                                           d["s"], workspace=ws))
    zero, poisoned = twice(L.attn_fwd_workspace(ctypes.byref(a)), fwd)
    same(zero, poisoned)
    o, lse = zero
    bwd = lambda ws: list(gcs_lib.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], ms, case.scale,
                                           case.window, d["g"], d["s"], workspace=ws, deterministic=True))
    zero, poisoned = twice(L.attn_bwd_workspace(ctypes.byref(a)), bwd)
    assert gcs_lib.get_device_status() == 0
    same(zero, poisoned)
