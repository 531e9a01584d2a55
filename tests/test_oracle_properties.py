"""Property checks of the paged oracle on random small workloads (CPU only).

For any context length L, chunk length 1 <= q_len <= L, GQA ratio, window, gates and sink,
cache format and split-K segment, the paged oracle (decode and chunked prefill) must equal the
last q_len rows of the prefill oracle on the dequantised keys and values (the prefill oracle is
pinned to fp64 SDPA in test_oracle_pins.py), and split-K with the combine must equal the unsplit
result.  hypothesis draws the cases; where it is not installed the module is skipped."""
import numpy as np
import pytest
import torch

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from synth import make_decode  # noqa: E402


def f64(t):
    return t.double().numpy()


@st.composite
def paged_case(draw):
    n = draw(st.integers(1, 3))
    seq = [draw(st.integers(1, 48)) for _ in range(n)]
    ql = [draw(st.integers(1, L)) for L in seq]
    hkv, group = draw(st.sampled_from([(1, 1), (1, 2), (2, 2), (1, 4)]))
    fmt = draw(st.sampled_from([("fp8", "per_token"), ("fp8", "per_tensor"), ("bf16", "per_token")]))
    feat = draw(st.booleans())
    window = draw(st.integers(0, max(seq) + 2)) if feat else 0
    seg = draw(st.sampled_from([1, 3, 16, 2048]))
    seed = draw(st.integers(0, 2**16))
    dc = make_decode(seq, ql, hkv * group, hkv, 8, seed=seed, kv_format=fmt[0], scale_mode=fmt[1], features=feat,
                     window=window)
    return dc, seg


def _args(dc):
    opt = lambda t: None if t is None else t.numpy()
    cache = lambda t: t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()
    return (f64(dc.q), cache(dc.k_cache), cache(dc.v_cache), opt(dc.k_scale), opt(dc.v_scale), dc.block_table.numpy(),
            dc.seq_lens.numpy(), dc.cu_q.numpy(), dc.scale)


@settings(max_examples=40, deadline=None)
@given(paged_case())
def test_paged_oracle_equals_prefill_rows_and_splitk(case):
    dc, seg = case
    g = None if dc.g_cache is None else dc.g_cache.numpy()
    sink = None if dc.sink is None else dc.sink.double().numpy()
    out = oracle.decode_paged(*_args(dc), g_cache=g, sink=sink, window=dc.window)
    assert np.isfinite(out).all()
    args = _args(dc)
    for r, L in enumerate(dc.seq_lens.tolist()):
        q0, q1 = int(dc.cu_q[r]), int(dc.cu_q[r + 1])
        qlen = q1 - q0
        K = np.stack([oracle.gather_kv(args[1], args[3], dc.block_table[r].numpy(), L, h) for h in range(dc.hkv)], 1)
        V = np.stack([oracle.gather_kv(args[2], args[4], dc.block_table[r].numpy(), L, h) for h in range(dc.hkv)], 1)
        lg = None
        if g is not None:
            npg = (L + 15) // 16
            G = dc.g_cache[dc.block_table[r, :npg].long()].double().permute(0, 2, 1).reshape(npg * 16, dc.hq)[:L]
            lg = torch.diff(G, dim=0, prepend=torch.zeros(1, dc.hq, dtype=torch.float64)).numpy()
        q = np.zeros((L, dc.hq, dc.d))
        q[L - qlen :] = f64(dc.q)[q0:q1]
        o, _ = oracle.prefill_forward(q, K, V, np.array([0, L]), dc.scale, log_gate=lg, sink=sink, window=dc.window)
        np.testing.assert_allclose(out[q0:q1], o[L - qlen :], rtol=1e-10, atol=1e-12)
    parts = oracle.decode_partials(*args, seg, g_cache=g, window=dc.window)
    split = oracle.decode_combine(parts, dc.q.shape[0], dc.hq, dc.d, dc.cu_q.numpy(), dc.hkv, sink=sink)
    np.testing.assert_allclose(split, out, rtol=0, atol=1e-12)


@st.composite
def prefill_case(draw):
    from synth import make_prefill

    n = draw(st.integers(1, 3))
    lens = [draw(st.integers(1, 24)) for _ in range(n)]
    hkv, group = draw(st.sampled_from([(1, 1), (1, 2), (2, 2), (1, 3)]))
    dqk, dv = draw(st.sampled_from([(4, 4), (8, 4), (4, 8)]))
    gate, sink = draw(st.booleans()), draw(st.booleans())
    window = draw(st.integers(0, max(lens) + 2))
    seed = draw(st.integers(0, 2**16))
    return make_prefill(lens, hkv * group, hkv, dqk, dv, seed=seed, gate=gate, sink=sink, window=window)


@settings(max_examples=30, deadline=None)
@given(prefill_case())
def test_prefill_oracle_equals_autograd_sdpa(c):
    """Forward and every gradient of the prefill oracle against torch autograd through fp64
    SDPA with the gate as an additive mask and the sink as an extra zero key, on random
    packed shapes, GQA ratios, head dims, windows and feature sets."""
    from test_oracle_pins import run_bwd, run_fwd, sdpa_reference

    o, _ = run_fwd(c)
    ref, leaves = sdpa_reference(c, requires_grad=True)
    np.testing.assert_allclose(o, ref.detach().numpy(), rtol=1e-10, atol=1e-12)
    (ref * c.do.double()).sum().backward()
    dq, dk, dv, dg, ds = run_bwd(c)
    np.testing.assert_allclose(dq, leaves["q"].grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, leaves["k"].grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, leaves["v"].grad.numpy(), atol=1e-11)
    if c.log_gate is not None:
        np.testing.assert_allclose(dg, leaves["g"].grad.numpy(), atol=1e-11)
    if c.sink is not None:
        np.testing.assert_allclose(ds, leaves["s"].grad.numpy(), atol=1e-11)
