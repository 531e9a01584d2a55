"""Pins of the fp64 oracle to things other than itself: library routines (fp64 SDPA,
torch.autograd, torch fp8/bf16 conversions), closed forms, hand-derived values, finite
differences and invariants.  Each test is chosen so that a dropped term, a sign error, a
wrong index or a transposed operand in the oracle fails at least one of them."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from synth import make_prefill, make_decode

HERE = os.path.dirname(os.path.abspath(__file__))


def f64(t):
    return None if t is None else t.double().numpy()


def run_fwd(c, **over):
    kw = dict(log_gate=f64(c.log_gate), sink=f64(c.sink), window=c.window)
    kw.update(over)
    return oracle.prefill_forward(f64(c.q), f64(c.k), f64(c.v), c.cu_seqlens.numpy(), c.scale, **kw)


def run_bwd(c, **over):
    kw = dict(log_gate=f64(c.log_gate), sink=f64(c.sink), window=c.window)
    kw.update(over)
    return oracle.prefill_backward(f64(c.q), f64(c.k), f64(c.v), f64(c.do), c.cu_seqlens.numpy(), c.scale, **kw)


def sdpa_reference(c, use_gate=True, use_sink=True, requires_grad=False):
    """fp64 torch SDPA per sequence; gate as an additive float mask, sink as an extra key
    with zero key/value vectors whose mask entry is sigma; GQA by repeating K/V."""
    group = c.hq // c.hkv
    q = c.q.double().clone().requires_grad_(requires_grad)
    k = c.k.double().clone().requires_grad_(requires_grad)
    v = c.v.double().clone().requires_grad_(requires_grad)
    g = None
    if use_gate and c.log_gate is not None:
        g = c.log_gate.double().clone().requires_grad_(requires_grad)
    s = None
    if use_sink and c.sink is not None:
        s = c.sink.double().clone().requires_grad_(requires_grad)
    outs = []
    cu = c.cu_seqlens.tolist()
    for a, b in zip(cu[:-1], cu[1:]):
        T = b - a
        qs = q[a:b].transpose(0, 1)  # [hq, T, d]
        ks = k[a:b].transpose(0, 1).repeat_interleave(group, 0)
        vs = v[a:b].transpose(0, 1).repeat_interleave(group, 0)
        i = torch.arange(T)[:, None]
        j = torch.arange(T)[None, :]
        allowed = j <= i
        if c.window > 0:
            allowed = allowed & ((i - j) < c.window)
        mask = torch.zeros(c.hq, T, T, dtype=torch.float64)
        if g is not None:
            G = torch.cumsum(g[a:b], 0).transpose(0, 1)  # [hq, T]
            mask = mask + G[:, :, None] - G[:, None, :]
        mask = mask.masked_fill(~allowed, float("-inf"))
        if s is not None:
            ks = torch.cat([ks, torch.zeros(c.hq, 1, c.dqk, dtype=torch.float64)], 1)
            vs = torch.cat([vs, torch.zeros(c.hq, 1, c.dv, dtype=torch.float64)], 1)
            mask = torch.cat([mask, s[:, None, None].expand(c.hq, T, 1)], 2)
        o = F.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=c.scale)
        outs.append(o.transpose(0, 1))
    o = torch.cat(outs, 0)
    return o, dict(q=q, k=k, v=v, g=g, s=s)


# ---------------------------------------------------------------------------- forward
def test_forward_plain_matches_fp64_sdpa_causal():
    c = make_prefill([37, 64], hq=4, hkv=4, dqk=16, dv=8, seed=11)
    o, _ = run_fwd(c)
    cu = c.cu_seqlens.tolist()
    for a, b in zip(cu[:-1], cu[1:]):
        ref = F.scaled_dot_product_attention(
            c.q[a:b].double().transpose(0, 1), c.k[a:b].double().transpose(0, 1),
            c.v[a:b].double().transpose(0, 1), is_causal=True, scale=c.scale).transpose(0, 1)
        np.testing.assert_allclose(o[a:b], ref.numpy(), rtol=0, atol=1e-12)


def test_forward_gate_window_sink_match_sdpa_with_mask():
    c = make_prefill([19, 33], hq=4, hkv=2, dqk=8, dv=12, seed=12, gate=True, sink=True, window=7)
    o, _ = run_fwd(c)
    ref, _ = sdpa_reference(c)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def test_zero_gates_equal_plain_softmax():
    c = make_prefill([40], hq=2, hkv=1, dqk=8, dv=8, seed=13)
    o0, l0 = run_fwd(c)
    o1, l1 = run_fwd(c, log_gate=np.zeros((c.total, c.hq)))
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)


def test_constant_gate_is_alibi_bias():
    c = make_prefill([30], hq=1, hkv=1, dqk=4, dv=4, seed=14)
    cst = -0.3
    o, _ = run_fwd(c, log_gate=np.full((c.total, 1), cst))
    T = c.total
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    bias = ((i - j).double() * cst).masked_fill(j > i, float("-inf"))
    ref = F.scaled_dot_product_attention(c.q.double().transpose(0, 1), c.k.double().transpose(0, 1),
                                         c.v.double().transpose(0, 1), attn_mask=bias, scale=c.scale)
    np.testing.assert_allclose(o, ref.transpose(0, 1).numpy(), atol=1e-12)


def test_sink_closed_form():
    c = make_prefill([25, 9], hq=3, hkv=1, dqk=8, dv=5, seed=15, gate=True, sink=True)
    o_s, l_s = run_fwd(c)
    o_n, l_n = run_fwd(c, sink=None)
    sig = f64(c.sink)
    # O_sink = O_nosink * sigmoid(LSE_nosink - sigma); LSE_sink = logaddexp(LSE_nosink, sigma)
    factor = 1.0 / (1.0 + np.exp(sig[:, None] - l_n))  # [hq, tot]
    np.testing.assert_allclose(o_s, o_n * factor.T[:, :, None], atol=1e-13)
    np.testing.assert_allclose(l_s, np.logaddexp(l_n, sig[:, None]), atol=1e-13)


def test_probabilities_plus_sink_sum_to_one():
    c = make_prefill([31, 17], hq=2, hkv=2, dqk=4, dv=1, seed=16, gate=True, sink=True, window=5)
    ones = np.ones((c.total, c.hkv, 1))
    o, lse = oracle.prefill_forward(f64(c.q), f64(c.k), ones, c.cu_seqlens.numpy(), c.scale,
                                    log_gate=f64(c.log_gate), sink=f64(c.sink), window=c.window)
    p_sink = np.exp(f64(c.sink)[:, None] - lse)  # [hq, tot]
    np.testing.assert_allclose(o[:, :, 0] + p_sink.T, 1.0, atol=1e-14)


def test_window_at_least_T_equals_full_causal_and_window_one_closed_form():
    c = make_prefill([20, 12], hq=2, hkv=1, dqk=4, dv=3, seed=17, gate=True, sink=True)
    o_full, l_full = run_fwd(c, window=0)
    o_big, l_big = run_fwd(c, window=20)
    np.testing.assert_array_equal(o_full, o_big)
    np.testing.assert_array_equal(l_full, l_big)
    o1, l1 = run_fwd(c, window=1)
    p_sink = np.exp(f64(c.sink)[:, None] - l1).T  # [tot, hq]
    v = f64(c.v)
    group = c.hq // c.hkv
    v_rep = np.repeat(v, group, axis=1)
    np.testing.assert_allclose(o1, v_rep * (1.0 - p_sink)[:, :, None], atol=1e-14)
    o2, _ = run_fwd(c, window=2)
    assert not np.allclose(o2, o1)


def test_gqa_equals_mha_on_repeated_kv():
    c = make_prefill([23, 10], hq=6, hkv=2, dqk=8, dv=4, seed=18, gate=True, sink=True, window=9)
    o, lse = run_fwd(c)
    dq, dk, dv, dg, ds = run_bwd(c)
    rep = lambda x: np.repeat(f64(x), 3, axis=1)
    o2, lse2 = oracle.prefill_forward(f64(c.q), rep(c.k), rep(c.v), c.cu_seqlens.numpy(), c.scale,
                                      log_gate=f64(c.log_gate), sink=f64(c.sink), window=c.window)
    dq2, dk2, dv2, dg2, ds2 = oracle.prefill_backward(f64(c.q), rep(c.k), rep(c.v), f64(c.do),
                                                      c.cu_seqlens.numpy(), c.scale, log_gate=f64(c.log_gate),
                                                      sink=f64(c.sink), window=c.window)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(c.total, 2, 3, -1).sum(2), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(c.total, 2, 3, -1).sum(2), atol=1e-13)
    np.testing.assert_allclose(dg, dg2, atol=1e-13)
    np.testing.assert_allclose(ds, ds2, atol=1e-13)


def test_varlen_equals_concatenated_dense():
    c = make_prefill([13, 1, 22, 7], hq=2, hkv=1, dqk=4, dv=6, seed=19, gate=True, sink=True, window=6)
    o, lse = run_fwd(c)
    dq, dk, dv, dg, ds = run_bwd(c)
    cu = c.cu_seqlens.tolist()
    ds_sum = np.zeros_like(ds)
    for a, b in zip(cu[:-1], cu[1:]):
        sl = slice(a, b)
        args = (f64(c.q)[sl], f64(c.k)[sl], f64(c.v)[sl])
        kw = dict(log_gate=f64(c.log_gate)[sl], sink=f64(c.sink), window=c.window)
        o1, l1 = oracle.prefill_forward(*args, np.array([0, b - a]), c.scale, **kw)
        g1 = oracle.prefill_backward(*args, f64(c.do)[sl], np.array([0, b - a]), c.scale, **kw)
        np.testing.assert_array_equal(o[sl], o1)
        np.testing.assert_array_equal(lse[:, sl], l1)
        for full, part in zip((dq, dk, dv, dg), g1[:4]):
            np.testing.assert_allclose(full[sl], part, atol=1e-15)
        ds_sum += g1[4]
    np.testing.assert_allclose(ds, ds_sum, atol=1e-13)


def test_empty_sequences_change_nothing():
    """cu_seqlens with repeated entries (sequences of length 0, first, inside and last) give
    the same outputs and gradients as the same tokens without them."""
    c = make_prefill([9, 6], hq=2, hkv=1, dqk=4, dv=3, seed=23, gate=True, sink=True, window=4)
    args = (f64(c.q), f64(c.k), f64(c.v))
    kw = dict(log_gate=f64(c.log_gate), sink=f64(c.sink), window=4)
    plain, padded = np.array([0, 9, 15]), np.array([0, 0, 9, 9, 15, 15])
    for a, b in zip(oracle.prefill_forward(*args, plain, c.scale, **kw),
                    oracle.prefill_forward(*args, padded, c.scale, **kw)):
        np.testing.assert_array_equal(a, b)
    for a, b in zip(oracle.prefill_backward(*args, f64(c.do), plain, c.scale, **kw),
                    oracle.prefill_backward(*args, f64(c.do), padded, c.scale, **kw)):
        np.testing.assert_array_equal(a, b)


def test_hand_derived_two_token_case():
    with open(os.path.join(HERE, "golden", "tiny_gate_sink.json")) as f:
        fx = json.load(f)
    i, e = fx["inputs"], fx["expected"]
    arr = lambda x: np.array(x, dtype=np.float64)
    cu = np.array(i["cu_seqlens"])
    o, lse = oracle.prefill_forward(arr(i["q"]), arr(i["k"]), arr(i["v"]), cu, i["scale"],
                                    log_gate=arr(i["log_gate"]), sink=arr(i["sink"]))
    dq, dk, dv, dg, ds = oracle.prefill_backward(arr(i["q"]), arr(i["k"]), arr(i["v"]), arr(i["do"]), cu,
                                                 i["scale"], log_gate=arr(i["log_gate"]), sink=arr(i["sink"]))
    for name, got in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv), ("dg", dg), ("dsink", ds)):
        np.testing.assert_allclose(got, arr(e[name]), rtol=0, atol=1e-14, err_msg=name)



def test_hand_derived_paged_decode_case():
    """Gather through a permuted page table, K scales on the score columns, V scales after the
    row sum, bottom-right rows of a short query, NaN slots never read, and split-K with an
    empty partial, against values derived on paper (tests/golden/tiny_paged_decode.json)."""
    with open(os.path.join(HERE, "golden", "tiny_paged_decode.json")) as f:
        fx = json.load(f)
    i, e = fx["inputs"], fx["expected"]
    f32 = lambda x: np.array([[[np.nan if v is None else v for v in s] for s in h] for h in x], dtype=np.float32)
    args = (np.array(i["q"], dtype=np.float64), np.array(i["k_cache"], dtype=np.uint8),
            np.array(i["v_cache"], dtype=np.uint8), f32(i["k_scale"]), f32(i["v_scale"]),
            np.array(i["block_table"]), np.array(i["seq_lens"]), np.array(i["cu_q"]), i["scale"])
    want = np.array(e["out"], dtype=np.float64)
    np.testing.assert_allclose(oracle.decode_paged(*args), want, rtol=0, atol=1e-14)
    parts = oracle.decode_partials(*args, i["segment_len"])
    split = oracle.decode_combine(parts, 2, 1, 1, np.array(i["cu_q"]), 1)
    np.testing.assert_allclose(split, want, rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------- backward
def _loss(c, q, k, v, g, s):
    o, _ = oracle.prefill_forward(q, k, v, c.cu_seqlens.numpy(), c.scale, log_gate=g, sink=s, window=c.window)
    return float((o * f64(c.do)).sum())


def test_backward_central_finite_differences():
    c = make_prefill([5, 3], hq=2, hkv=1, dqk=3, dv=2, seed=20, gate=True, sink=True, window=3)
    dq, dk, dv, dg, ds = run_bwd(c)
    base = dict(q=f64(c.q), k=f64(c.k), v=f64(c.v), g=f64(c.log_gate), s=f64(c.sink))
    grads = dict(q=dq, k=dk, v=dv, g=dg, s=ds)
    eps = 1e-6
    for name, x in base.items():
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = {kk: vv.copy() for kk, vv in base.items()}
            xm = {kk: vv.copy() for kk, vv in base.items()}
            xp[name][idx] += eps
            xm[name][idx] -= eps
            num[idx] = (_loss(c, **xp) - _loss(c, **xm)) / (2 * eps)
        np.testing.assert_allclose(grads[name], num, rtol=1e-6, atol=1e-8, err_msg=name)


def test_backward_matches_torch_autograd_on_sdpa():
    c = make_prefill([11, 6, 15], hq=4, hkv=2, dqk=8, dv=4, seed=21, gate=True, sink=True, window=5)
    dq, dk, dv, dg, ds = run_bwd(c)
    o, leaves = sdpa_reference(c, requires_grad=True)
    (o * c.do.double()).sum().backward()
    np.testing.assert_allclose(dq, leaves["q"].grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, leaves["k"].grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, leaves["v"].grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dg, leaves["g"].grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(ds, leaves["s"].grad.numpy(), atol=1e-12)


def test_sink_gradient_closed_form_and_first_token_gate_gradient():
    c = make_prefill([26, 14, 3], hq=3, hkv=1, dqk=8, dv=6, seed=22, gate=True, sink=True)
    o, lse = run_fwd(c)
    dq, dk, dv, dg, ds = run_bwd(c)
    # dsigma_h = -sum_i p_sink,i (dO_i . O_i): uses the forward output, not P and dP
    p_sink = np.exp(f64(c.sink)[:, None] - lse)  # [hq, tot]
    dot = (f64(c.do) * o).sum(-1).T  # [hq, tot]
    np.testing.assert_allclose(ds, -(p_sink * dot).sum(1), atol=1e-13)
    # each dS entry enters dG once as a row term and once as a column term: the gate of
    # the first token of every sequence never changes a score
    for a in c.cu_seqlens.tolist()[:-1]:
        np.testing.assert_allclose(dg[a], 0.0, atol=1e-13)


# ---------------------------------------------------------------------------- formats
def test_e4m3_table_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    np.testing.assert_array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])
    assert np.nanmax(ours) == 448.0 and np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000), rng.standard_normal(1000) * 1e-30,
                        rng.standard_normal(1000) * 1e30]).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.bf16_round(x), ref)


# ---------------------------------------------------------------------------- decode
def _decode_args(dc):
    return (f64(dc.q), dc.k_cache.numpy(), dc.v_cache.numpy(), dc.k_scale.numpy(), dc.v_scale.numpy(),
            dc.block_table.numpy(), dc.seq_lens.numpy(), dc.cu_q.numpy(), dc.scale)


@pytest.mark.parametrize("reading", ["A", "B"])
def test_splitk_combine_equals_unsplit_with_empty_segments(reading):
    dc = make_decode([1, 17, 40, 70, 33], [1, 2, 4, 3, 4], hq=8, hkv=2, d=16, seed=30, scale_reading=reading,
                     segment_len=2048)
    ref = oracle.decode_paged(*_decode_args(dc))
    for seg in (2048, 32, 16, 3, 2):
        parts = oracle.decode_partials(*_decode_args(dc), seg)
        if seg == 2:
            # a query row that ends before a segment stores an empty partial
            assert any(np.isneginf(p["m"]).any() for p in parts)
        out = oracle.decode_combine(parts, dc.q.shape[0], dc.hq, dc.d, dc.cu_q.numpy(), dc.hkv)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
        assert np.isfinite(out).all()


def test_decode_q1_equals_last_prefill_row_on_dequantized_cache():
    dc = make_decode([45, 16, 1], [1, 1, 1], hq=4, hkv=2, d=8, seed=31)
    out = oracle.decode_paged(*_decode_args(dc))
    for r, L in enumerate(dc.seq_lens.tolist()):
        K = np.stack([oracle.gather_kv(dc.k_cache.numpy(), dc.k_scale.numpy(), dc.block_table[r].numpy(), L, h)
                      for h in range(dc.hkv)], 1)
        V = np.stack([oracle.gather_kv(dc.v_cache.numpy(), dc.v_scale.numpy(), dc.block_table[r].numpy(), L, h)
                      for h in range(dc.hkv)], 1)
        q = np.zeros((L, dc.hq, dc.d))
        q[L - 1] = f64(dc.q)[r]
        o, _ = oracle.prefill_forward(q, K, V, np.array([0, L]), dc.scale)
        np.testing.assert_allclose(out[r], o[L - 1], atol=1e-12)
        # and the same row through torch fp64 SDPA with repeated kv heads
        rep = lambda x: torch.from_numpy(np.repeat(x, dc.hq // dc.hkv, 1)).transpose(0, 1)
        ref = F.scaled_dot_product_attention(torch.from_numpy(f64(dc.q)[r][:, None]), rep(K), rep(V),
                                             scale=dc.scale)
        np.testing.assert_allclose(out[r], ref[:, 0].numpy(), atol=1e-12)


def test_decode_per_token_scales_matter_and_gather_is_exact():
    dc = make_decode([50, 77], [1, 2], hq=4, hkv=1, d=8, seed=32)
    args = list(_decode_args(dc))
    # a dominant key at one chosen slot makes the output equal that slot's dequantized V
    r, slot = 1, 37
    L = int(dc.seq_lens[r])
    blk = int(dc.block_table[r, slot // 16])
    kc = args[1].copy()
    ks = args[3].copy()
    qv = args[0]
    row = int(dc.cu_q[r + 1]) - 1  # last row sees every key
    qv = qv.copy()
    qv[row] = 0.0
    qv[row, :, 0] = 1.0
    kc[:, :, :, :] = 0  # code 0 = +0.0
    kc[blk, 0, slot % 16, 0] = 0x7E  # 448
    ks[blk, 0, slot % 16] = 1.0
    args[0], args[1], args[3] = qv, kc, ks
    args[8] = 1.0
    out = oracle.decode_paged(*args)
    vexp = oracle.e4m3_decode(dc.v_cache[blk, 0, slot % 16].numpy()) * float(dc.v_scale[blk, 0, slot % 16])
    np.testing.assert_allclose(out[row], np.broadcast_to(vexp, out[row].shape), rtol=0, atol=1e-12)
    # per-token scales change the answer (reading only element 0 would be wrong)
    args2 = list(_decode_args(dc))
    vs = args2[4].copy()
    vs[:] = vs.reshape(-1)[0]
    assert not np.allclose(oracle.decode_paged(*args2[:4], vs, *args2[5:]), oracle.decode_paged(*_decode_args(dc)))


def test_decode_never_reads_unused_slots():
    dc = make_decode([19, 3], [1, 3], hq=4, hkv=2, d=8, seed=33)
    out = oracle.decode_paged(*_decode_args(dc))
    assert np.isfinite(out).all()
    # unused slots and spare pages are NaN-poisoned by the generator
    assert np.isnan(dc.k_scale.numpy()).any() and (dc.v_cache.numpy() == 0x7F).any()


# ------------------------------------------------------------- decode variants (bf16 KV, per-tensor scales)
def _variant_args(dc):
    kc = dc.k_cache.float().numpy() if dc.kv_format == "bf16" else dc.k_cache.numpy()
    vc = dc.v_cache.float().numpy() if dc.kv_format == "bf16" else dc.v_cache.numpy()
    ks = None if dc.k_scale is None else dc.k_scale.numpy()
    vs = None if dc.v_scale is None else dc.v_scale.numpy()
    return (f64(dc.q), kc, vc, ks, vs, dc.block_table.numpy(), dc.seq_lens.numpy(), dc.cu_q.numpy(), dc.scale)


def _sdpa_decode(dc):
    """Independent reference: gather each request's pages by indexing the table, dequantize
    with torch's own float8_e4m3fn (or take the bf16 values), and run fp64 SDPA with the
    bottom-right causal mask of a short query (row t of q_len sits at L - q_len + t)."""
    out = torch.zeros(dc.q.shape, dtype=torch.float64)
    group = dc.hq // dc.hkv
    for r, L in enumerate(dc.seq_lens.tolist()):
        q0, q1 = int(dc.cu_q[r]), int(dc.cu_q[r + 1])
        ql = q1 - q0
        npg = (L + dc.block_size - 1) // dc.block_size
        blocks = dc.block_table[r, :npg].long()

        def dequant(cache, sc):
            x = cache[blocks]  # [npg, hkv, bs, d]
            if dc.kv_format == "bf16":
                v = x.double()
            else:
                v = x.view(torch.float8_e4m3fn).double() * float(sc.reshape(-1)[0])
            return v.permute(1, 0, 2, 3).reshape(dc.hkv, npg * dc.block_size, dc.d)[:, :L]

        K, V = dequant(dc.k_cache, dc.k_scale), dequant(dc.v_cache, dc.v_scale)
        K, V = K.repeat_interleave(group, 0), V.repeat_interleave(group, 0)  # [hq, L, d]
        q = dc.q[q0:q1].double().transpose(0, 1)  # [hq, ql, d]
        mask = torch.arange(L)[None, :] <= (L - ql + torch.arange(ql))[:, None]
        out[q0:q1] = F.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=dc.scale).transpose(0, 1)
    return out.numpy()


@pytest.mark.parametrize("fmt", [("bf16", "per_token"), ("fp8", "per_tensor")])
def test_decode_variants_equal_sdpa_and_splitk(fmt):
    kv_format, scale_mode = fmt
    dc = make_decode([1, 17, 40, 70, 33], [1, 2, 4, 3, 4], hq=8, hkv=2, d=16, seed=34, kv_format=kv_format,
                     scale_mode=scale_mode)
    args = _variant_args(dc)
    out = oracle.decode_paged(*args)
    assert np.isfinite(out).all()  # NaN-poisoned unused slots are never read
    np.testing.assert_allclose(out, _sdpa_decode(dc), rtol=0, atol=1e-12)
    for seg in (2048, 16, 3):
        parts = oracle.decode_partials(*args, seg)
        res = oracle.decode_combine(parts, dc.q.shape[0], dc.hq, dc.d, dc.cu_q.numpy(), dc.hkv)
        np.testing.assert_allclose(res, out, rtol=0, atol=1e-12)


def test_decode_per_tensor_scale_is_one_scale_for_every_token():
    # scaling every code by the one K scale: doubling it doubles every score (one scale, not per token)
    dc = make_decode([33, 50], [1, 2], hq=4, hkv=2, d=8, seed=35, scale_mode="per_tensor")
    a = list(_variant_args(dc))
    b = list(a)
    b[3] = a[3] * 2.0
    b[8] = a[8] / 2.0
    np.testing.assert_allclose(oracle.decode_paged(*a), oracle.decode_paged(*b), rtol=0, atol=1e-12)
    c = list(a)
    c[4] = a[4] * 4.0  # the V scale multiplies the output linearly (a power of two keeps the fp32 scale exact)
    np.testing.assert_allclose(oracle.decode_paged(*c), 4.0 * oracle.decode_paged(*a), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------- decode with gate, window and sink
def _feature_kwargs(dc):
    return dict(g_cache=dc.g_cache.numpy(), sink=dc.sink.double().numpy(), window=dc.window)


@pytest.mark.parametrize("window", [0, 5, 23])
def test_decode_features_equal_prefill_rows(window):
    """Decode with gates, window and sink equals the last q_len rows of the prefill oracle
    (itself pinned to fp64 SDPA) over the same dequantized keys and values, with the
    per-token log gates recovered as differences of the cumulative G."""
    dc = make_decode([45, 16, 1, 33], [1, 2, 1, 4], hq=4, hkv=2, d=8, seed=36, features=True, window=window)
    out = oracle.decode_paged(*_decode_args(dc), **_feature_kwargs(dc))
    assert np.isfinite(out).all()
    for r, L in enumerate(dc.seq_lens.tolist()):
        q0, q1 = int(dc.cu_q[r]), int(dc.cu_q[r + 1])
        ql = q1 - q0
        K = np.stack([oracle.gather_kv(dc.k_cache.numpy(), dc.k_scale.numpy(), dc.block_table[r].numpy(), L, h)
                      for h in range(dc.hkv)], 1)
        V = np.stack([oracle.gather_kv(dc.v_cache.numpy(), dc.v_scale.numpy(), dc.block_table[r].numpy(), L, h)
                      for h in range(dc.hkv)], 1)
        npg = (L + 15) // 16
        G = dc.g_cache[dc.block_table[r, :npg].long()].double().permute(0, 2, 1).reshape(npg * 16, dc.hq)[:L]
        g = torch.diff(G, dim=0, prepend=torch.zeros(1, dc.hq, dtype=torch.float64)).numpy()
        q = np.zeros((L, dc.hq, dc.d))
        q[L - ql :] = f64(dc.q)[q0:q1]
        o, _ = oracle.prefill_forward(q, K, V, np.array([0, L]), dc.scale, log_gate=g, sink=dc.sink.double().numpy(),
                                      window=window)
        np.testing.assert_allclose(out[q0:q1], o[L - ql :], rtol=1e-10, atol=1e-12)


def test_decode_features_splitk_equals_unsplit():
    dc = make_decode([1, 17, 40, 70, 33], [1, 2, 4, 3, 4], hq=8, hkv=2, d=16, seed=37, features=True, window=9)
    ref = oracle.decode_paged(*_decode_args(dc), **_feature_kwargs(dc))
    for seg in (2048, 16, 3):
        parts = oracle.decode_partials(*_decode_args(dc), seg, g_cache=dc.g_cache.numpy(), window=dc.window)
        if seg == 3:
            assert any(np.isneginf(p["m"]).any() for p in parts)  # windows and short queries leave empty partials
        out = oracle.decode_combine(parts, dc.q.shape[0], dc.hq, dc.d, dc.cu_q.numpy(), dc.hkv,
                                    sink=dc.sink.double().numpy())
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_decode_window_one_with_sink_closed_form():
    """W = 1: each query sees only its own key, whose gate difference is 0, so
    O = v_pos * e^s / (e^s + e^sigma)."""
    dc = make_decode([20, 9], [1, 3], hq=4, hkv=1, d=8, seed=38, features=True, window=1)
    out = oracle.decode_paged(*_decode_args(dc), **_feature_kwargs(dc))
    for r, L in enumerate(dc.seq_lens.tolist()):
        K = oracle.gather_kv(dc.k_cache.numpy(), dc.k_scale.numpy(), dc.block_table[r].numpy(), L, 0)
        V = oracle.gather_kv(dc.v_cache.numpy(), dc.v_scale.numpy(), dc.block_table[r].numpy(), L, 0)
        q0, q1 = int(dc.cu_q[r]), int(dc.cu_q[r + 1])
        for t in range(q1 - q0):
            pos = L - (q1 - q0) + t
            for h in range(dc.hq):
                s = dc.scale * float(K[pos] @ f64(dc.q)[q0 + t, h])
                w = 1.0 / (1.0 + math.exp(float(dc.sink[h]) - s))
                np.testing.assert_allclose(out[q0 + t, h], V[pos] * w, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("window", [0, 7, 40])
def test_paged_chunks_equal_prefill_rows(window):
    """Query chunks longer than a decode (q_len 5 .. seq_len, the chunked-prefill shape) over
    the paged cache equal the last q_len rows of the prefill oracle (pinned to fp64 SDPA) on
    the dequantized keys and values; a chunk with q_len == seq_len is a whole prefill."""
    dc = make_decode([45, 37, 70, 20], [45, 9, 33, 17], hq=4, hkv=2, d=8, seed=39, features=True, window=window)
    out = oracle.decode_paged(*_decode_args(dc), **_feature_kwargs(dc))
    assert np.isfinite(out).all()
    for r, L in enumerate(dc.seq_lens.tolist()):
        q0, q1 = int(dc.cu_q[r]), int(dc.cu_q[r + 1])
        ql = q1 - q0
        K = np.stack([oracle.gather_kv(dc.k_cache.numpy(), dc.k_scale.numpy(), dc.block_table[r].numpy(), L, h)
                      for h in range(dc.hkv)], 1)
        V = np.stack([oracle.gather_kv(dc.v_cache.numpy(), dc.v_scale.numpy(), dc.block_table[r].numpy(), L, h)
                      for h in range(dc.hkv)], 1)
        npg = (L + 15) // 16
        G = dc.g_cache[dc.block_table[r, :npg].long()].double().permute(0, 2, 1).reshape(npg * 16, dc.hq)[:L]
        g = torch.diff(G, dim=0, prepend=torch.zeros(1, dc.hq, dtype=torch.float64)).numpy()
        q = np.zeros((L, dc.hq, dc.d))
        q[L - ql :] = f64(dc.q)[q0:q1]
        o, _ = oracle.prefill_forward(q, K, V, np.array([0, L]), dc.scale, log_gate=g, sink=dc.sink.double().numpy(),
                                      window=window)
        np.testing.assert_allclose(out[q0:q1], o[L - ql :], rtol=1e-10, atol=1e-12)


def test_paged_chunk_splitk_equals_unsplit_and_rows_are_single_queries():
    """Long chunks in split-K (segments of 16 and 48 tokens leave rows with no visible key in
    a segment: weight 0) equal the unsplit result, and each row equals the single-query
    request that ends at its own position."""
    dc = make_decode([70, 33, 50], [40, 33, 6], hq=8, hkv=2, d=16, seed=40, features=True, window=21)
    ref = oracle.decode_paged(*_decode_args(dc), **_feature_kwargs(dc))
    for seg in (16, 48):
        parts = oracle.decode_partials(*_decode_args(dc), seg, g_cache=dc.g_cache.numpy(), window=dc.window)
        assert any(np.isneginf(p["m"]).any() for p in parts)
        out = oracle.decode_combine(parts, dc.q.shape[0], dc.hq, dc.d, dc.cu_q.numpy(), dc.hkv,
                                    sink=dc.sink.double().numpy())
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # row t of request r == a one-row request whose context ends at position L - q_len + t
    seq, cu = [], [0]
    bt = []
    for r, L in enumerate(dc.seq_lens.tolist()):
        ql = int(dc.cu_q[r + 1] - dc.cu_q[r])
        for t in range(ql):
            seq.append(L - ql + t + 1)
            cu.append(cu[-1] + 1)
            bt.append(dc.block_table[r].numpy())
    one = oracle.decode_paged(f64(dc.q), dc.k_cache.numpy(), dc.v_cache.numpy(), dc.k_scale.numpy(),
                              dc.v_scale.numpy(), np.stack(bt), np.array(seq), np.array(cu), dc.scale,
                              **_feature_kwargs(dc))
    np.testing.assert_allclose(one, ref, rtol=0, atol=1e-12)


def _relayout_blocks(dc, block):
    """The same logical cache with `block` tokens per cache block: every request's tokens are
    copied, in order, into fresh blocks laid out [num_blocks, hkv, block, d] (and the scales and
    gates likewise), with a reversed block order so that no index coincides by accident."""
    bs = dc.k_cache.shape[2]
    L = dc.seq_lens.tolist()
    pages = [(x + block - 1) // block for x in L]
    nb = sum(pages) + 1
    order = list(range(nb))[::-1]
    table = np.zeros((len(L), max(pages)), dtype=np.int32)

    def tokens(arr, r, n):  # [n, heads, ...] token-major values of request r
        old = dc.block_table[r].numpy()
        out = [arr[old[j // bs], :, j % bs] for j in range(n)]
        return np.stack(out)

    def place(arr, fill):
        new = np.full((nb, arr.shape[1], block) + arr.shape[3:], fill, dtype=arr.dtype)
        pos = 0
        for r, n in enumerate(L):
            t = tokens(arr, r, n)
            for j in range(n):
                b = order[pos + j // block]
                new[b, :, j % block] = t[j]
            pos += pages[r]
        return new

    pos = 0
    for r in range(len(L)):
        table[r, : pages[r]] = [order[pos + i] for i in range(pages[r])]
        pos += pages[r]
    kc = place(dc.k_cache.numpy(), 0x7F)
    vc = place(dc.v_cache.numpy(), 0x7F)
    ks = place(dc.k_scale.numpy(), np.nan)
    vs = place(dc.v_scale.numpy(), np.nan)
    g = None if dc.g_cache is None else place(dc.g_cache.numpy(), np.nan)
    return kc, vc, ks, vs, g, table


@pytest.mark.parametrize("window", [0, 30])
def test_decode_oracle_block_size_and_group_of_eight(window):
    """Cache blocks of 128 tokens hold the same attention as blocks of 16 (the same logical
    cache relaid by the test, not by the oracle), and a GQA group of 8 matches the last rows of
    the prefill oracle on the dequantized cache, gates, window and sink included."""
    dc = make_decode([1, 130, 300, 77], [1, 4, 3, 2], 16, 2, 16, seed=61, features=True, window=window)
    kw = dict(sink=f64(dc.sink), window=dc.window)
    args = lambda kc, vc, ks, vs, bt: (f64(dc.q), kc, vc, ks, vs, bt, dc.seq_lens.numpy(), dc.cu_q.numpy(), dc.scale)
    ref = oracle.decode_paged(*args(dc.k_cache.numpy(), dc.v_cache.numpy(), dc.k_scale.numpy(), dc.v_scale.numpy(),
                                    dc.block_table.numpy()), g_cache=dc.g_cache.numpy(), **kw)
    kc, vc, ks, vs, g, bt = _relayout_blocks(dc, 128)
    got = oracle.decode_paged(*args(kc, vc, ks, vs, bt), g_cache=g, **kw)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)
    # group of 8 (hq 16 over hkv 2) against the prefill oracle's last q_len rows, request by request
    cu = dc.cu_q.tolist()
    for r, L in enumerate(dc.seq_lens.tolist()):
        K = np.stack([oracle.gather_kv(dc.k_cache.numpy(), dc.k_scale.numpy(), dc.block_table[r].numpy(), L, h)
                      for h in range(2)], axis=1)
        V = np.stack([oracle.gather_kv(dc.v_cache.numpy(), dc.v_scale.numpy(), dc.block_table[r].numpy(), L, h)
                      for h in range(2)], axis=1)
        G = np.stack([oracle.attention._gate_of(dc.g_cache.numpy(), dc.block_table[r].numpy(), L, h)
                      for h in range(16)], axis=1)
        gates = np.diff(np.concatenate([np.zeros((1, 16)), G]), axis=0)  # per-token log gates
        ql = cu[r + 1] - cu[r]
        q = np.zeros((L, 16, dc.d))
        q[L - ql:] = f64(dc.q)[cu[r]:cu[r + 1]]
        o, _ = oracle.prefill_forward(q, K, V, np.array([0, L]), dc.scale, log_gate=gates, sink=f64(dc.sink),
                                      window=dc.window)
        np.testing.assert_allclose(ref[cu[r]:cu[r + 1]], o[L - ql:], rtol=0, atol=1e-12)
