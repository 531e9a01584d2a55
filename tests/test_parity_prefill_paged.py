"""Device parity: paged chunked prefill (query chunks of any length over the paged fp8 cache)
through the C ABI against the fp64 oracle on the dequantised cache (unused slots NaN-poisoned),
relative RMS <= 1e-2 and |bias| <= 1e-3, as for decode."""
import copy

import numpy as np
import pytest
import torch

from synth import decode_config, make_decode
from helpers import DECODE_BIAS, DECODE_RTOL, assert_close, bias, decode_dev, f64, oracle_decode

pytestmark = pytest.mark.gpu

# segment modes: one segment per request (the kernel writes the output), the library's
# automatic split, and 128-token segments (many split-K partials, some empty)
SEGMENTS = {"direct": 1 << 20, "auto": 0, "seg128": 128}


def run_prefill_paged(gcs, dc, segment_len):
    d = decode_dev(dc)
    max_seq = int(dc.seq_lens.max())
    if segment_len == 1 << 20:
        segment_len = ((max_seq + 127) // 128) * 128
    out = gcs.attn_prefill_paged(d["q"], d["kc"], d["vc"], d["ks"], d["vs"], d["bt"], d["sl"], d["cq"],
                                 max(dc.q_lens), max_seq, dc.scale, segment_len, g_cache=d["g"], sink=d["sink"],
                                 window=dc.window)
    torch.cuda.synchronize()
    assert gcs.get_device_status() == 0
    return out


CASES = {
    # name: (seq_lens, q_lens, hq, hkv, features, window, scale_mode)
    # whole-sequence prefill (q_len == seq_len), a long chunk, a short one, chunks ending
    # mid-page and on page / 128-key tile edges
    "chunks_plain": ([300, 1000, 2049, 129], [300, 57, 5, 128], 32, 2, False, 0, "per_token"),
    # q_len at the 8- and 16-position tile edges and one past them
    "tile_edges": ([17, 40, 1025, 2048, 33], [8, 16, 17, 33, 1], 16, 1, False, 0, "per_token"),
    "gates_sink_window": ([700, 2049, 90], [200, 40, 90], 32, 2, True, 300, "per_token"),
    "gates_sink_no_window": ([520, 1500], [64, 31], 16, 1, True, 0, "per_token"),
    "window_inside_tile": ([400, 260], [150, 260], 16, 1, True, 9, "per_token"),
    "per_tensor": ([1200, 333, 64], [100, 333, 7], 32, 2, False, 0, "per_tensor"),
    "per_tensor_features": ([900, 2100], [77, 300], 16, 1, True, 500, "per_tensor"),
    # a request with no query rows in the middle of the batch is skipped
    "empty_request_in_batch": ([300, 64, 1000], [40, 0, 17], 16, 1, False, 0, "per_token"),
}


@pytest.mark.parametrize("seg", list(SEGMENTS))
@pytest.mark.parametrize("name", list(CASES))
def test_prefill_paged_parity(gcs_lib, name, seg):
    sl, ql, hq, hkv, feat, win, smode = CASES[name]
    dc = make_decode(sl, ql, hq, hkv, 128, seed=500 + len(name), scale_mode=smode, features=feat, window=win)
    out = run_prefill_paged(gcs_lib, dc, SEGMENTS[seg])
    ref = oracle_decode(dc)
    assert np.isfinite(f64(out)).all()
    assert_close("out", out, ref, DECODE_RTOL)
    assert abs(bias(out, ref)) <= DECODE_BIAS


def test_prefill_paged_reading_b_scales(gcs_lib):
    """Dequantised magnitudes that differ 20x between tokens (scale reading B)."""
    dc = make_decode([1500, 600], [300, 600], 32, 2, 128, seed=520, scale_reading="B")
    for seg in (0, 256):
        out = run_prefill_paged(gcs_lib, dc, seg)
        ref = oracle_decode(dc)
        assert_close("out", out, ref, DECODE_RTOL)
        assert abs(bias(out, ref)) <= DECODE_BIAS


def test_prefill_paged_equals_decode_on_short_queries(gcs_lib):
    """On q_len <= 4 the chunked route and the decode route compute the same rows."""
    dc = make_decode([3000, 33, 700], [4, 2, 1], 32, 2, 128, seed=521)
    out = run_prefill_paged(gcs_lib, dc, 0)
    d = decode_dev(dc)
    dec = gcs_lib.attn_decode_paged(d["q"], d["kc"], d["vc"], d["ks"], d["vs"], d["bt"], d["sl"], d["cq"], 4,
                                    int(dc.seq_lens.max()), dc.scale, 2048)
    torch.cuda.synchronize()
    ref = oracle_decode(dc)
    assert_close("out", out, ref, DECODE_RTOL)
    assert oracle_rel(out, dec) < DECODE_RTOL


def oracle_rel(a, b):
    a, b = f64(a), f64(b)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_prefill_paged_gather_order_is_exact(gcs_lib):
    """Each query row has one dominant key (code 448 on a dim only that row's query reads),
    at a chosen visible slot whose value holds the page id in exact e4m3 codes: the output
    names the gathered (block, slot) exactly."""
    sl, ql = [300, 1030], [40, 100]
    dc = make_decode(sl, ql, 16, 1, 128, seed=522)
    kc, vc = dc.k_cache.clone(), dc.v_cache.clone()
    ks, vs = dc.k_scale.clone(), dc.v_scale.clone()
    kc.zero_()
    q = torch.zeros_like(dc.q)
    picks = []
    for r in range(2):
        q0 = int(dc.cu_q[r])
        for t in range(ql[r]):
            pos = sl[r] - ql[r] + t
            slot = (pos * 7919) % (pos + 1)  # some visible key
            picks.append((r, q0 + t, slot))
            blk = int(dc.block_table[r, slot // 16])
            # key code 0x7E (448) on the dim chosen by the row, so only this row's key dominates
            dim = t % 128
            kc[blk, 0, slot % 16, dim] = 0x7E
            ks[blk, 0, slot % 16] = 1.0
            q[q0 + t, :, dim] = 1.0
            vc[blk, 0, slot % 16, 0] = int(torch.tensor(float(blk % 8)).to(torch.float8_e4m3fn).view(torch.uint8))
            vc[blk, 0, slot % 16, 1] = int(torch.tensor(float((blk // 8) % 8)).to(torch.float8_e4m3fn).view(torch.uint8))
            vs[blk, 0, slot % 16] = 1.0
    dc.k_cache, dc.v_cache, dc.k_scale, dc.v_scale, dc.q = kc, vc, ks, vs, q
    dc.scale = 1.0
    out = run_prefill_paged(gcs_lib, dc, 0).float().cpu()
    for r, row, slot in picks:
        blk = int(dc.block_table[r, slot // 16])
        assert out[row, :, 0].eq(float(blk % 8)).all(), (r, row, slot, out[row, :, 0])
        assert out[row, :, 1].eq(float((blk // 8) % 8)).all(), (r, row, slot)


def sampled_rows(dc, picks):
    """One single-row request per picked (request, row t): context ending at that row's
    position, same cache; the oracle of that request is the row's exact result."""
    sub = copy.copy(dc)
    seq, cu, bt, rows = [], [0], [], []
    for r, t in picks:
        L = int(dc.seq_lens[r])
        ql = int(dc.cu_q[r + 1] - dc.cu_q[r])
        rows.append(int(dc.cu_q[r]) + t)
        seq.append(L - ql + t + 1)
        cu.append(cu[-1] + 1)
        bt.append(dc.block_table[r])
    sub.q = dc.q[rows]
    sub.seq_lens = torch.tensor(seq, dtype=torch.int32)
    sub.cu_q = torch.tensor(cu, dtype=torch.int32)
    sub.block_table = torch.stack(bt)
    return sub, rows


@pytest.mark.parametrize("seg", [0, 2048])
def test_prefill_paged_full_size_sampled(gcs_lib, seg):
    """The 4 x 1024-token chunk workload at 8K..32K context, in the launch configuration the
    benchmark times (automatic segments) and in split-K; rows sampled across every request,
    first, last and interior positions."""
    dc = decode_config("paged_fp8_chunked_prefill_4x1024")
    out = run_prefill_paged(gcs_lib, dc, seg)
    picks = [(r, t) for r in range(4) for t in (0, 1, 15, 16, 511, 1000, 1023)]
    sub, rows = sampled_rows(dc, picks)
    ref = oracle_decode(sub)
    got = f64(out)[rows]
    assert_close("out", got, ref, DECODE_RTOL)
    assert abs(bias(got, ref)) <= DECODE_BIAS


@pytest.mark.parametrize("group", [16, 8])
@pytest.mark.parametrize("block", [16, 128])
@pytest.mark.parametrize("features", [False, True])
@pytest.mark.parametrize("seg", ["direct", "seg128"])
def test_prefill_paged_gqa_and_page_matrix(gcs_lib, group, block, features, seg):
    """GQA groups of 16 and 8 (a 128-row tile is 8 positions x 16 heads or 16 positions x 8
    heads, so q_len 16, 17, 33 sit on and past the tile edges of both) over 16- and 128-token
    cache blocks, with and without gates, window and sink."""
    dc = make_decode([17, 300, 1025, 2049], [16, 17, 33, 130], 2 * group, 2, 128, seed=950 + group + block,
                     block_size=block, features=features, window=200 if features else 0)
    out = run_prefill_paged(gcs_lib, dc, SEGMENTS[seg])
    ref = oracle_decode(dc)
    assert np.isfinite(f64(out)).all()
    assert_close("out", out, ref, DECODE_RTOL)
    assert abs(bias(out, ref)) <= DECODE_BIAS
