"""Device parity: paged fp8 decode through the C ABI against the fp64 oracle on the
dequantised cache (unused slots NaN-poisoned), relative RMS <= 1e-2 and |bias| <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from synth import decode_config, make_decode
from helpers import DECODE_BIAS, DECODE_RTOL, assert_close, bias, decode_dev, f64, oracle_decode, run_decode

pytestmark = pytest.mark.gpu


CASES = {
    # name: (seq_lens, q_lens, hq, hkv, reading, segment_len)
    "q1_page_edges": ([1, 15, 16, 17, 100, 2047, 2048, 2049, 5000], [1] * 9, 16, 1, "A", 2048),
    "q1_gqa16_hkv4": ([3000, 33, 700, 4097], [1] * 4, 64, 4, "A", 2048),
    "short_query_tails": ([4, 17, 18, 20, 2049, 4100], [4, 4, 3, 2, 4, 3], 32, 2, "B", 2048),
    "short_query_context_65537": ([65537, 300], [4, 2], 16, 1, "B", 2048),
    "tiny_segments_empty_partials": ([40, 70, 5], [4, 3, 4], 16, 1, "A", 16),
    "mixed_q_lens_reading_A": ([1000, 1001, 1003, 64], [1, 2, 4, 3], 32, 2, "A", 256),
    # a request with no query rows in the middle of the batch is skipped
    "empty_request_in_batch": ([700, 50, 2100], [2, 0, 3], 16, 1, "A", 2048),
}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_parity(gcs_lib, name):
    sl, ql, hq, hkv, reading, seg = CASES[name]
    dc = make_decode(sl, ql, hq, hkv, 128, seed=200 + len(name), scale_reading=reading, segment_len=seg)
    out = run_decode(gcs_lib, dc)
    ref = oracle_decode(dc)
    assert_close("out", out, ref, DECODE_RTOL)
    assert abs(bias(out, ref)) <= DECODE_BIAS


@pytest.mark.parametrize("reading", ["A", "B"])
def test_decode_against_unquantized_reference(gcs_lib, reading):
    """The [AIT] PR's test plan checks the decode against the dequantized reference, the
    unquantized reference and the output bias.  Against the values before fp8 quantization
    the error is the quantization's own: e4m3 keeps 3 mantissa bits (relative rounding error
    at most 2^-4), which the fp64 oracle on the dequantized cache shows as about 3e-2 relative
    RMS in reading A and 9e-2 in reading B (token magnitudes 20x apart sharpen the softmax,
    so score errors weigh more).  The library must add nothing visible on top: its distance
    from the unquantized reference may exceed the dequantized oracle's by at most 5 %, and it
    stays within a fixed 5e-2 (A) / 1.5e-1 (B)."""
    dc = make_decode([1, 17, 100, 2100, 4096, 65537], [1, 4, 2, 3, 1, 4], 16, 1, 128, seed=91,
                     scale_reading=reading, keep_unquantized=True)
    out = run_decode(gcs_lib, dc)
    deq = oracle_decode(dc)
    unq = oracle.decode_paged(f64(dc.q), dc.k_unquant.double().numpy(), dc.v_unquant.double().numpy(), None, None,
                              dc.block_table.numpy(), dc.seq_lens.numpy(), dc.cu_q.numpy(), dc.scale)
    assert_close("out vs dequantized", out, deq, DECODE_RTOL)
    assert abs(bias(out, deq)) <= DECODE_BIAS
    e_q = oracle.rel_rms(deq, unq)
    e_lib = oracle.rel_rms(f64(out), unq)
    assert e_lib <= {"A": 5e-2, "B": 1.5e-1}[reading], e_lib
    assert e_lib <= 1.05 * e_q, (e_lib, e_q)


def test_decode_rejects_prefill_shapes(gcs_lib):
    dc = make_decode([40], [5], 16, 1, 128, seed=3)
    with pytest.raises(NotImplementedError):
        run_decode(gcs_lib, dc)


def test_decode_per_token_scales_matter(gcs_lib):
    """Reading only the first scale of the cache (the bug the per-token path fixed) would be
    far off: the scales span 20x."""
    dc = make_decode([500, 1200], [1, 1], 16, 1, 128, seed=9)
    out = run_decode(gcs_lib, dc)
    ref = oracle_decode(dc)
    vs = dc.v_scale.clone()
    flat = vs.view(-1)
    flat[:] = flat[torch.isfinite(flat)][0]
    ks = dc.k_scale.clone()
    fk = ks.view(-1)
    fk[:] = fk[torch.isfinite(fk)][0]
    wrong = oracle.decode_paged(f64(dc.q), dc.k_cache.numpy(), dc.v_cache.numpy(), ks.numpy(), vs.numpy(),
                                dc.block_table.numpy(), dc.seq_lens.numpy(), dc.cu_q.numpy(), dc.scale)
    assert oracle.rel_rms(wrong, ref) > 0.2
    assert oracle.rel_rms(f64(out), ref) < DECODE_RTOL


def test_decode_gather_order_is_exact(gcs_lib):
    """One dominant key per (request, kv head) at a chosen slot; its value page holds the code
    for the page id, so the output identifies the gathered (block, slot) exactly."""
    sl = [37, 2050, 700]
    dc = make_decode(sl, [1, 1, 1], 16, 1, 128, seed=11)
    kc = dc.k_cache.clone()
    vc = dc.v_cache.clone()
    ks = dc.k_scale.clone()
    vs = dc.v_scale.clone()
    q = torch.zeros_like(dc.q)
    q[:, :, 0] = 1.0
    kc.zero_()  # code 0 = +0
    picks = [5, 2049, 333]
    for r, slot in enumerate(picks):
        blk = int(dc.block_table[r, slot // 16])
        kc[blk, 0, slot % 16, 0] = 0x7E  # 448
        ks[blk, 0, slot % 16] = 1.0
        # integer page identity in e4m3: codes for blk % 8 and (blk // 8) % 8 on dims 0 and 1
        vc[blk, 0, slot % 16, 0] = int(torch.tensor(float(blk % 8)).to(torch.float8_e4m3fn).view(torch.uint8))
        vc[blk, 0, slot % 16, 1] = int(torch.tensor(float((blk // 8) % 8)).to(torch.float8_e4m3fn).view(torch.uint8))
        vs[blk, 0, slot % 16] = 1.0
    dc.k_cache, dc.v_cache, dc.k_scale, dc.v_scale, dc.q = kc, vc, ks, vs, q
    dc.scale = 1.0
    out = run_decode(gcs_lib, dc).float().cpu()
    for r, slot in enumerate(picks):
        blk = int(dc.block_table[r, slot // 16])
        assert out[r, :, 0].eq(float(blk % 8)).all(), (r, out[r, :, 0])
        assert out[r, :, 1].eq(float((blk // 8) % 8)).all()


def test_decode_full_size_64x1_sampled(gcs_lib):
    dc = decode_config("paged_fp8_decode_64x1")
    out = run_decode(gcs_lib, dc)
    pick = [0, 7, 21, 40, 63]
    sub = make_sub(dc, pick)
    ref = oracle_decode(sub)
    got = f64(out)[[int(dc.cu_q[r]) for r in pick]]
    assert_close("out", got, ref, DECODE_RTOL)
    assert abs(bias(got, ref)) <= DECODE_BIAS


def test_decode_full_size_verify_3x4_227k(gcs_lib):
    """Three requests of 4 query positions at ~227K tokens of context: every row of every
    request against the oracle."""
    dc = decode_config("paged_fp8_verify_3x4_227k")
    out = run_decode(gcs_lib, dc)
    for r in range(len(dc.seq_lens)):
        ref = oracle_decode(make_sub(dc, [r]))
        got = f64(out)[int(dc.cu_q[r]) : int(dc.cu_q[r + 1])]
        assert_close(f"out[request {r}]", got, ref, DECODE_RTOL)
        assert abs(bias(got, ref)) <= DECODE_BIAS


def make_sub(dc, reqs):
    """Same cache, only the chosen requests (the oracle is per request)."""
    import copy

    sub = copy.copy(dc)
    rows = []
    cu = [0]
    for r in reqs:
        a, b = int(dc.cu_q[r]), int(dc.cu_q[r + 1])
        rows.extend(range(a, b))
        cu.append(cu[-1] + b - a)
    sub.q = dc.q[rows]
    sub.cu_q = torch.tensor(cu, dtype=torch.int32)
    sub.seq_lens = dc.seq_lens[reqs]
    sub.block_table = dc.block_table[reqs]
    return sub


# ------------------------------------------------- bf16 KV cache and per-tensor fp8 scales
VARIANTS = [("bf16", "per_token"), ("fp8", "per_tensor")]
VARIANT_CASES = {
    # name: (seq_lens, q_lens, hq, hkv, segment_len)
    "page_edges_q1": ([1, 15, 16, 17, 2047, 2048, 2049, 5000], [1] * 8, 16, 1, 2048),
    "short_query_tails_gqa": ([4, 18, 20, 2049, 4100, 65537], [4, 3, 2, 4, 3, 4], 32, 2, 2048),
    "tiny_segments_empty_partials": ([40, 70, 5], [4, 3, 4], 16, 1, 16),
}


@pytest.mark.parametrize("fmt", VARIANTS)
@pytest.mark.parametrize("name", list(VARIANT_CASES))
def test_decode_variant_parity(gcs_lib, fmt, name):
    sl, ql, hq, hkv, seg = VARIANT_CASES[name]
    dc = make_decode(sl, ql, hq, hkv, 128, seed=300 + len(name), segment_len=seg, kv_format=fmt[0],
                     scale_mode=fmt[1])
    out = run_decode(gcs_lib, dc)
    ref = oracle_decode(dc)
    assert np.isfinite(f64(out)).all()
    assert_close("out", out, ref, DECODE_RTOL)
    assert abs(bias(out, ref)) <= DECODE_BIAS


@pytest.mark.parametrize("fmt", VARIANTS)
def test_decode_variant_full_size_64x1_sampled(gcs_lib, fmt):
    dc = decode_config("paged_fp8_decode_64x1", kv_format=fmt[0], scale_mode=fmt[1])
    out = run_decode(gcs_lib, dc)
    pick = [0, 7, 21, 40, 63]
    sub = make_sub(dc, pick)
    ref = oracle_decode(sub)
    got = f64(out)[[int(dc.cu_q[r]) for r in pick]]
    assert_close("out", got, ref, DECODE_RTOL)
    assert abs(bias(got, ref)) <= DECODE_BIAS


def test_decode_bf16_gather_order_is_exact(gcs_lib):
    """bf16 cache: one dominant key per request at a chosen slot whose value row holds the page
    id (exact in bf16), so the output identifies the gathered (block, slot) exactly."""
    sl = [37, 2050, 700]
    dc = make_decode(sl, [1, 1, 1], 16, 1, 128, seed=12, kv_format="bf16")
    kc = torch.zeros_like(dc.k_cache)
    vc = dc.v_cache.clone()
    q = torch.zeros_like(dc.q)
    q[:, :, 0] = 1.0
    picks = [5, 2049, 333]
    for r, slot in enumerate(picks):
        blk = int(dc.block_table[r, slot // 16])
        kc[blk, 0, slot % 16, 0] = 1000.0
        vc[blk, 0, slot % 16, 0] = float(blk % 64)
        vc[blk, 0, slot % 16, 1] = float(blk // 64)
    dc.k_cache, dc.v_cache, dc.q = kc, vc, q
    dc.scale = 1.0
    out = run_decode(gcs_lib, dc).float().cpu()
    for r, slot in enumerate(picks):
        blk = int(dc.block_table[r, slot // 16])
        assert out[r, :, 0].eq(float(blk % 64)).all(), (r, out[r, :, 0])
        assert out[r, :, 1].eq(float(blk // 64)).all()


# ------------------------------------------------------- decode with gates, window and sink
FEATURE_CASES = {
    # name: (seq_lens, q_lens, hq, hkv, segment_len, window, kv_format, scale_mode)
    "gates_sink_no_window": ([1, 17, 700, 2049, 5000], [1, 1, 4, 2, 3], 32, 2, 2048, 0, "fp8", "per_token"),
    "window_skips_segments": ([5000, 4100, 300, 64], [1, 4, 2, 3], 16, 1, 2048, 1000, "fp8", "per_token"),
    "window_inside_page": ([40, 70, 17], [4, 3, 1], 16, 1, 16, 7, "fp8", "per_token"),
    "per_tensor_features": ([3000, 33, 2049], [1, 4, 2], 32, 2, 2048, 500, "fp8", "per_tensor"),
    "bf16_features": ([3000, 33, 2049], [1, 4, 2], 32, 2, 2048, 500, "bf16", "per_token"),
}


@pytest.mark.parametrize("name", list(FEATURE_CASES))
def test_decode_features_parity(gcs_lib, name):
    sl, ql, hq, hkv, seg, win, fmt, smode = FEATURE_CASES[name]
    dc = make_decode(sl, ql, hq, hkv, 128, seed=400 + len(name), segment_len=seg, kv_format=fmt, scale_mode=smode,
                     features=True, window=win)
    out = run_decode(gcs_lib, dc)
    ref = oracle_decode(dc)
    assert np.isfinite(f64(out)).all()
    assert_close("out", out, ref, DECODE_RTOL)
    assert abs(bias(out, ref)) <= DECODE_BIAS


def test_decode_sink_only_and_window_only(gcs_lib):
    """Each feature on its own: the sink alone (split kernel unchanged, combine adds it) and a
    window alone (no gates)."""
    for win, keep_sink in ((0, True), (300, False)):
        dc = make_decode([1000, 2500, 70], [1, 3, 2], 16, 1, 128, seed=41 + win, features=True, window=win)
        dc.g_cache = None
        if not keep_sink:
            dc.sink = None
        out = run_decode(gcs_lib, dc)
        ref = oracle_decode(dc)
        assert_close("out", out, ref, DECODE_RTOL)
        assert abs(bias(out, ref)) <= DECODE_BIAS


@pytest.mark.parametrize("reading", ["A", "B"])
def test_decode_rn_bias_is_far_below_the_limit(gcs_lib, reading):
    """P * vscale is rounded to nearest (not truncated): at full size the relative signed bias
    stays an order of magnitude inside the 1e-3 limit, in both scale readings (32 of the 64
    requests, every query head)."""
    dc = decode_config("paged_fp8_decode_64x1", scale_reading=reading)
    out = run_decode(gcs_lib, dc)
    pick = list(range(0, 64, 2))
    sub = make_sub(dc, pick)
    ref = oracle_decode(sub)
    got = f64(out)[[int(dc.cu_q[r]) for r in pick]]
    assert_close("out", got, ref, DECODE_RTOL)
    assert abs(bias(got, ref)) <= 2e-4


# The aiter PR's test matrix: GQA groups of 16 and 8, head 128, pages of 16 and 128 tokens,
# contexts from 1 to 4096 and 65537, tails that end 1 to 4 tokens into a page.
MATRIX_LENS = [1, 2, 3, 4, 129, 130, 2051, 4096, 65537]
MATRIX_QLENS = [1, 2, 3, 4, 1, 2, 3, 4, 4]


@pytest.mark.parametrize("group", [16, 8])
@pytest.mark.parametrize("block", [16, 128])
@pytest.mark.parametrize("variant", ["A", "B", "bf16", "per_tensor", "features"])
def test_decode_gqa_and_page_matrix(gcs_lib, group, block, variant):
    kw = dict(scale_reading="B") if variant == "B" else dict(kv_format="bf16") if variant == "bf16" else \
        dict(scale_mode="per_tensor") if variant == "per_tensor" else dict(features=True, window=300) \
        if variant == "features" else {}
    dc = make_decode(MATRIX_LENS, MATRIX_QLENS, 2 * group, 2, 128, seed=900 + group + block, block_size=block,
                     segment_len=2048, **kw)
    out = run_decode(gcs_lib, dc)
    ref = oracle_decode(dc)
    assert_close("out", out, ref, DECODE_RTOL)
    assert abs(bias(out, ref)) <= DECODE_BIAS


@pytest.mark.parametrize("group", [16, 8])
def test_decode_gather_is_exact_with_128_token_blocks(gcs_lib, group):
    """One dominant key per request at a chosen slot of a 128-token block; its value codes name
    the block, so the output identifies the gathered (block, slot) exactly."""
    sl = [37, 2050, 700]
    dc = make_decode(sl, [1, 1, 1], group, 1, 128, seed=13, block_size=128)
    kc, vc, ks, vs = dc.k_cache.clone(), dc.v_cache.clone(), dc.k_scale.clone(), dc.v_scale.clone()
    q = torch.zeros_like(dc.q)
    q[:, :, 0] = 1.0
    kc.zero_()  # code 0 = +0
    picks = [5, 2049, 333]
    code = lambda x: int(torch.tensor(float(x)).to(torch.float8_e4m3fn).view(torch.uint8))
    for r, slot in enumerate(picks):
        blk = int(dc.block_table[r, slot // 128])
        kc[blk, 0, slot % 128, 0] = 0x7E  # 448
        ks[blk, 0, slot % 128] = 1.0
        vc[blk, 0, slot % 128, 0] = code(blk % 8)
        vc[blk, 0, slot % 128, 1] = code((blk // 8) % 8)
        vs[blk, 0, slot % 128] = 1.0
    dc.k_cache, dc.v_cache, dc.k_scale, dc.v_scale, dc.q = kc, vc, ks, vs, q
    dc.scale = 1.0
    out = run_decode(gcs_lib, dc).float().cpu()
    for r, slot in enumerate(picks):
        blk = int(dc.block_table[r, slot // 128])
        assert out[r, :, 0].eq(float(blk % 8)).all(), (r, out[r, :, 0])
        assert out[r, :, 1].eq(float((blk // 8) % 8)).all()
