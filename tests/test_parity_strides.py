"""Device parity of strided layouts through the C ABI: the same inputs given in other layouts
must give the same bits as the contiguous call (the kernels compute the same values; only
addresses change), and agree with the fp64 oracle.

Prefill: q, k and v as views of one fused [tokens, (hq + 2 hkv) d] projection; o and the
gradients written into padded or fused buffers; o and dout read back from those layouts.
Paged calls: the caches in the [num_blocks, block_size, hkv, d] layout of vLLM-style engines
(passed as a permuted view), a strided q and a strided output."""
import pytest
import torch

import oracle
from synth import make_decode, make_prefill
from helpers import DECODE_RTOL, PREFILL_RTOL, assert_close, decode_dev, f64, oracle_prefill, oracle_decode, to_dev

pytestmark = pytest.mark.gpu

PREFILL_CASES = {
    # name: (seqlens, hq, hkv, dqk, dv, gate, sink, window)
    "d128_gqa_gate_sink": ([1, 300, 129, 520], 8, 2, 128, 128, True, True, 0),
    "d64_window": ([200, 77], 4, 1, 64, 64, True, False, 50),
    "d256_d512_window": ([300, 140], 4, 2, 256, 512, True, True, 100),
    "d512": ([260, 77], 2, 1, 512, 512, True, True, 0),
}


def fused_views(x_list, pad=0):
    """Copies [T, H_i, D_i] tensors into one [T, sum(H_i (D_i + pad))] buffer and returns views
    of it with the same values (token stride = the fused width, head stride D_i + pad)."""
    T = x_list[0].shape[0]
    widths = [x.shape[1] * (x.shape[2] + pad) for x in x_list]
    buf = torch.zeros(T, sum(widths), dtype=x_list[0].dtype, device=x_list[0].device)
    views, off = [], 0
    for x, w in zip(x_list, widths):
        H, D = x.shape[1], x.shape[2]
        v = buf[:, off:off + w].view(T, H, D + pad)[:, :, :D]
        v.copy_(x)
        views.append(v)
        off += w
    return buf, views


@pytest.mark.parametrize("name", list(PREFILL_CASES))
@pytest.mark.parametrize("deterministic", [False, True])
def test_prefill_strided_layouts_match_contiguous(gcs_lib, name, deterministic):
    lens, hq, hkv, dqk, dv, gate, sink, window = PREFILL_CASES[name]
    if deterministic and dqk == 64:
        pytest.skip("head dim 64 has one backward route")
    case = make_prefill(lens, hq, hkv, dqk, dv, seed=700 + dqk + dv, gate=gate, sink=sink, window=window)
    d = to_dev(case)
    ms = max(case.seqlens)
    # contiguous reference call
    o_ref, lse_ref = gcs_lib.attn_fwd(d["q"], d["k"], d["v"], d["cu"], ms, case.scale, case.window, d["g"], d["s"])
    g_ref = gcs_lib.attn_bwd(d["q"], d["k"], d["v"], o_ref, lse_ref, d["do"], d["cu"], ms, case.scale, case.window,
                             d["g"], d["s"], deterministic=deterministic)
    # strided: q, k, v from one fused projection; o into padded heads; dout padded; gradients
    # into one fused buffer
    _, (q, k, v) = fused_views([d["q"], d["k"], d["v"]])
    assert not q.is_contiguous() and q.stride(0) == (hq + hkv) * dqk + hkv * dv
    obuf = torch.full((case.total, hq, dv + 8), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = obuf[:, :, :dv]
    _, (dout,) = fused_views([d["do"]], pad=16)
    dq0 = torch.full_like(d["q"], float("nan"))
    dk0 = torch.full_like(d["k"], float("nan"))
    dv0 = torch.full_like(d["v"], float("nan"))
    gbuf, (dq, dk, dvv) = fused_views([dq0, dk0, dv0])
    o_out, lse = gcs_lib.attn_fwd(q, k, v, d["cu"], ms, case.scale, case.window, d["g"], d["s"], out=o)
    assert o_out.data_ptr() == o.data_ptr()
    grads = gcs_lib.attn_bwd(q, k, v, o, lse, dout, d["cu"], ms, case.scale, case.window, d["g"], d["s"],
                             dq=dq, dk=dk, dv=dvv, deterministic=deterministic)
    torch.cuda.synchronize()
    assert gcs_lib.get_device_status() == 0
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)
    # the padding between heads is untouched
    assert torch.isnan(obuf[:, :, dv:].float()).all()
    # fp32 reduce-adds of dQ and the dS row sums (single pass at 128, reduce-add route above)
    exact = deterministic or dqk == 64
    for n, got, ref in zip(("dq", "dk", "dv", "dlog_gate", "dsink"), grads, g_ref):
        if ref is None:
            assert got is None
            continue
        if exact:
            assert torch.equal(got, ref), n
        else:  # fp32 reduce-adds: low bits may differ from call to call
            assert oracle.rel_rms(f64(got), f64(ref)) <= 1e-3, n
    assert torch.isfinite(gbuf.float()).all()
    ro, _, rg = oracle_prefill(case)
    assert_close("o", o, ro, PREFILL_RTOL)
    for n, got, ref in zip(("dq", "dk", "dv"), grads[:3], rg[:3]):
        assert_close(n, got, ref, PREFILL_RTOL)


def vllm_view(cache):
    """The same values in the [num_blocks, block_size, hkv, d] layout, returned as a
    [num_blocks, hkv, block_size, d] view of that storage."""
    return cache.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


DECODE_CASES = {
    # name: (seq_lens, q_lens, hq, hkv, make_decode keywords)
    "fp8_per_token": ([1, 40, 2100, 5000], [1, 4, 2, 3], 32, 2, dict(scale_reading="B")),
    "fp8_per_tensor": ([700, 17, 2049], [1, 3, 4], 64, 4, dict(scale_mode="per_tensor")),
    "bf16_kv": ([3000, 33, 700], [2, 1, 4], 32, 2, dict(kv_format="bf16")),
    "fp8_features": ([1500, 64, 300], [4, 1, 2], 32, 2, dict(features=True, window=200)),
}


def _decode_call(gcs, fn, dc, d, kc, vc, q, out, max_q):
    return fn(q, kc, vc, d["ks"], d["vs"], d["bt"], d["sl"], d["cq"], max_q, int(dc.seq_lens.max()), dc.scale,
              dc.segment_len if fn is gcs.attn_decode_paged else 0, out=out, g_cache=d["g"], sink=d["sink"],
              window=dc.window)


@pytest.mark.parametrize("name", list(DECODE_CASES))
def test_decode_vllm_cache_and_strided_q_out(gcs_lib, name):
    sl, ql, hq, hkv, kw = DECODE_CASES[name]
    dc = make_decode(sl, ql, hq, hkv, 128, seed=810 + len(name), **kw)
    d = decode_dev(dc)
    ref = _decode_call(gcs_lib, gcs_lib.attn_decode_paged, dc, d, d["kc"], d["vc"], d["q"], None, max(ql))
    kc, vc = vllm_view(d["kc"]), vllm_view(d["vc"])
    assert kc.stride(1) < kc.stride(2)  # kv head inside the slot
    qbuf = torch.zeros(d["q"].shape[0], hq, 136, dtype=torch.bfloat16, device="cuda")
    q = qbuf[:, :, :128]
    q.copy_(d["q"])
    obuf = torch.full((d["q"].shape[0], hq + 8, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = obuf[:, 4:4 + hq]
    got = _decode_call(gcs_lib, gcs_lib.attn_decode_paged, dc, d, kc, vc, q, out, max(ql))
    torch.cuda.synchronize()
    assert gcs_lib.get_device_status() == 0
    assert got.data_ptr() == out.data_ptr()
    assert torch.equal(out, ref)
    assert torch.isnan(obuf[:, :4].float()).all() and torch.isnan(obuf[:, 4 + hq:].float()).all()
    assert_close("out", out, oracle_decode(dc), DECODE_RTOL)


@pytest.mark.parametrize("features", [False, True])
def test_prefill_paged_vllm_cache_and_strided_q_out(gcs_lib, features):
    dc = make_decode([300, 1000, 70], [40, 130, 3], 32, 2, 128, seed=830 + features, features=features,
                     window=100 if features else 0)
    d = decode_dev(dc)
    ref = _decode_call(gcs_lib, gcs_lib.attn_prefill_paged, dc, d, d["kc"], d["vc"], d["q"], None, 130)
    kc, vc = vllm_view(d["kc"]), vllm_view(d["vc"])
    _, (q,) = fused_views([d["q"]], pad=8)
    obuf = torch.full((d["q"].shape[0], dc.hq, 144), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = obuf[:, :, 8:136]
    _decode_call(gcs_lib, gcs_lib.attn_prefill_paged, dc, d, kc, vc, q, out, 130)
    torch.cuda.synchronize()
    assert gcs_lib.get_device_status() == 0
    assert torch.equal(out, ref)
    assert torch.isnan(obuf[:, :, :8].float()).all() and torch.isnan(obuf[:, :, 136:].float()).all()
    assert_close("out", out, oracle_decode(dc), DECODE_RTOL)


def test_strided_layouts_the_library_refuses_raise(gcs_lib):
    """A layout outside the accepted set is refused before any launch (NotImplementedError from
    GCS_ERR_UNSUPPORTED): heads given head-major ([heads, tokens, dim] viewed as [tokens,
    heads, dim])."""
    case = make_prefill([64, 64], 2, 2, 64, 64, seed=5)
    d = to_dev(case)
    qh = d["q"].transpose(0, 1).contiguous().transpose(0, 1)  # head stride T*D > token stride D
    with pytest.raises(NotImplementedError):
        gcs_lib.attn_fwd(qh, d["k"], d["v"], d["cu"], 64, case.scale)
