"""The allocation-free decode entry point (attn_decode_paged_noalloc) against the
workspace entry point (attn_decode_paged), through the C ABI.

The no-alloc call exists for callers that cannot allocate device memory (fixed memory
plans, allocator-less C hosts, latency-critical loops where cudaMalloc's possible device
synchronisation is not acceptable); it keeps the split-K partials in a fixed scratch
inside the library.  It runs the same kernels on the same inputs as the workspace call, so
its output must be the same bits.  Before the calls under test, a call of the same shape
with NaN queries fills every partial the scratch will hold with NaN: a partial that a later
call read without first writing it would then show up as NaN or as a changed bit.  Two
calls in a row must both match, and a size whose partials exceed the scratch is rejected
before any launch."""
import ctypes

import pytest
import torch

import oracle
from synth import make_decode
from helpers import DECODE_RTOL, decode_dev, f64, oracle_decode

pytestmark = pytest.mark.gpu


def _args(gcs, dc, d, q=None):
    return gcs.decode_args(d["q"] if q is None else q, d["kc"], d["vc"], d["ks"], d["vs"], d["bt"], d["sl"],
                           d["cq"], max(dc.q_lens), int(dc.seq_lens.max()), dc.scale, dc.segment_len)


def test_noalloc_matches_workspace_entry_point_twice(gcs_lib):
    L = gcs_lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [
        make_decode([1, 40, 2100, 5000], [1, 4, 2, 3], 32, 2, 128, seed=77, scale_reading="B"),
        make_decode([3000, 17, 700], [1, 1, 1], 16, 1, 128, seed=78),
    ]
    for dc in cases:
        d = decode_dev(dc)
        a = _args(gcs_lib, dc, d)
        ws_bytes = L.attn_decode_workspace(ctypes.byref(a))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(d["q"])
        assert L.attn_decode_paged(ctypes.byref(a), ref.data_ptr(), ws.data_ptr(), ws_bytes, stream) == 0
        # poison: the same shape with NaN queries writes NaN into every partial of the scratch
        q_nan = torch.full_like(d["q"], float("nan"))
        poison = torch.empty_like(d["q"])
        a_nan = _args(gcs_lib, dc, d, q=q_nan)
        assert L.attn_decode_paged_noalloc(ctypes.byref(a_nan), poison.data_ptr(), stream) == 0
        torch.cuda.synchronize()
        assert torch.isnan(poison.float()).any()
        expect = oracle_decode(dc)
        for _ in range(2):
            out = torch.full_like(d["q"], float("nan"))
            assert L.attn_decode_paged_noalloc(ctypes.byref(a), out.data_ptr(), stream) == 0
            torch.cuda.synchronize()
            assert gcs_lib.get_device_status() == 0
            assert torch.equal(out, ref)
            assert oracle.rel_rms(f64(out), expect) <= DECODE_RTOL


def test_noalloc_rejects_partials_larger_than_its_scratch(gcs_lib):
    L = gcs_lib.load()
    dc = make_decode([40], [4], 16, 1, 128, seed=79)
    d = decode_dev(dc)
    a = _args(gcs_lib, dc, d)
    # 256 requests x 4 query rows over 1M-token contexts: ~8 GB of partials
    a.num_reqs, a.max_seq_len, a.max_blocks_per_req = 256, 1 << 20, (1 << 20) // 16
    assert L.attn_decode_workspace(ctypes.byref(a)) > 64 << 20
    out = torch.empty_like(d["q"])
    assert L.attn_decode_paged_noalloc(ctypes.byref(a), out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 3
