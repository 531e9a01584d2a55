"""Device parity: prefill forward and backward through the C ABI against the fp64 oracle on
the same seeded inputs.  Sizes span several 128-row tiles with ragged tails; full-size
configurations are checked on sampled (sequence, kv-head group) blocks."""
import numpy as np
import pytest
import torch

import oracle
from synth import make_prefill, prefill_config
from helpers import PREFILL_RTOL, assert_close, f64, oracle_prefill, run_prefill, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    # name: (seqlens, hq, hkv, dqk, dv, gate, sink, window, backward)
    "dense_mha_t128_d64": ([128], 2, 2, 64, 64, False, False, 0, True),
    "varlen_ragged_gqa_d128_gate_sink": ([1, 100, 128, 129, 300], 8, 2, 128, 128, True, True, 0, True),
    "mqa_d64_window_gate_sink": ([200, 513], 4, 1, 64, 64, True, True, 70, True),
    "mha_d128_window_only": ([385, 64], 2, 2, 128, 128, False, False, 129, True),
    "gqa_d128_sink_only": ([257, 33], 4, 2, 128, 128, False, True, 0, True),
    "gqa_d64_gate_only": ([190, 2, 66], 6, 3, 64, 64, True, False, 0, True),
    "d256_d256": ([190, 130], 2, 2, 256, 256, True, True, 0, True),
    "d256_d512_window": ([300, 140], 4, 2, 256, 512, True, True, 100, True),
    "d512_d512": ([260, 77], 2, 1, 512, 512, True, True, 0, True),
    "d512_d512_window_no_gate": ([200, 129], 4, 2, 512, 512, False, True, 65, True),
    # empty sequences first, in the middle and last: they own no tile and no token
    "empty_seqs_d64_gate_sink": ([0, 130, 0, 70, 0], 4, 2, 64, 64, True, True, 0, True),
    "empty_seqs_d128_window": ([190, 0, 66], 4, 2, 128, 128, True, True, 50, True),
}


# deterministic=True takes the two-pass route at head dim 128 (the single pass otherwise) and the
# query-stationary dQ pass above it
PARITY_RUNS = [(n, False) for n in CASES] + [(n, True) for n in CASES if CASES[n][3] >= 128]


@pytest.mark.parametrize("name,deterministic", PARITY_RUNS)
def test_prefill_parity(gcs_lib, name, deterministic):
    lens, hq, hkv, dqk, dv, gate, sink, window, bwd = CASES[name]
    case = make_prefill(lens, hq, hkv, dqk, dv, seed=100 + len(name), gate=gate, sink=sink, window=window)
    o, lse, grads = run_prefill(gcs_lib, case, backward=bwd, deterministic=deterministic)
    ro, rlse, rg = oracle_prefill(case, backward=bwd)
    assert_close("o", o, ro, PREFILL_RTOL)
    np.testing.assert_allclose(f64(lse), rlse, rtol=0, atol=2e-3)
    if bwd:
        dq, dk, dv_, dg, ds = grads
        rdq, rdk, rdv, rdg, rds = rg
        assert_close("dq", dq, rdq, PREFILL_RTOL)
        assert_close("dk", dk, rdk, PREFILL_RTOL)
        assert_close("dv", dv_, rdv, PREFILL_RTOL)
        if gate:
            assert_close("dlog_gate", dg, rdg, PREFILL_RTOL)
            # the gate of the first token of a sequence never changes a score
            cu = case.cu_seqlens.tolist()
            first = [a for a, b in zip(cu[:-1], cu[1:]) if b > a]
            assert np.abs(f64(dg)[first]).max() <= 1e-3 * np.abs(rdg).max()
        else:
            assert dg is None
        if sink:
            assert_close("dsink", ds, rds, PREFILL_RTOL)
        else:
            assert ds is None


@pytest.mark.parametrize("dims", [(128, 128), (256, 512), (512, 512)])
def test_backward_is_deterministic(gcs_lib, dims):
    """With deterministic=True every gradient is written once or summed in a fixed order:
    repeated backward calls agree bit for bit."""
    dqk, dv = dims
    case = make_prefill([300, 141, 77], 4, 2, dqk, dv, seed=150 + dqk, gate=True, sink=True, window=0)
    d = to_dev(case)
    ms = max(case.seqlens)
    o, lse = gcs_lib.attn_fwd(d["q"], d["k"], d["v"], d["cu"], ms, case.scale, case.window, d["g"], d["s"])
    runs = []
    for _ in range(3):
        g = gcs_lib.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], ms, case.scale, case.window, d["g"],
                             d["s"], deterministic=True)
        torch.cuda.synchronize()
        runs.append([t.clone() for t in g])
    assert gcs_lib.get_device_status() == 0
    for other in runs[1:]:
        for name, a, b in zip(("dq", "dk", "dv", "dlog_gate", "dsink"), runs[0], other):
            assert torch.equal(a, b), name


def test_unsupported_head_dims_raise(gcs_lib):
    case = make_prefill([64], 2, 2, 96, 96, seed=1)
    with pytest.raises(NotImplementedError):
        run_prefill(gcs_lib, case, backward=False)


def test_prefill_gather_order_is_exact(gcs_lib):
    """Keys equal to the queries with a huge diagonal score: every row attends to itself only,
    so O_i must be exactly V_i (integer token ids, bf16-exact), across sequence boundaries."""
    lens = [130, 7, 200]
    tot = sum(lens)
    hq = hkv = 2
    d = 64
    idx = torch.arange(tot)
    q = torch.zeros(tot, hq, d)
    # one-hot on dim (token % 64): q_i . k_j = 900 for j = i and 0 for the other 63 keys of
    # a 64-key window, so P_ii = 1 and every other probability underflows to 0
    q[idx, :, idx % d] = 30.0
    k = q.clone()
    v = torch.zeros(tot, hkv, d)
    v[:, :, 0] = (idx % 256).float()[:, None]
    v[:, :, 1] = (idx // 256).float()[:, None]
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    dev = torch.device("cuda:0")
    o, _ = gcs_lib.attn_fwd(q.bfloat16().to(dev), k.bfloat16().to(dev), v.bfloat16().to(dev), cu.to(dev),
                            max(lens), 1.0, 64)
    torch.cuda.synchronize()
    got = o.float().cpu()
    np.testing.assert_array_equal(got[:, :, 0].numpy(), (idx % 256).float()[:, None].expand(tot, hq).numpy())
    np.testing.assert_array_equal(got[:, :, 1].numpy(), (idx // 256).float()[:, None].expand(tot, hq).numpy())


def _sampled_full_size(gcs_lib, name, kv_group=1, backward=True, seqs=None, deterministic=False):
    case = prefill_config(name)
    o, lse, grads = run_prefill(gcs_lib, case, backward=backward, deterministic=deterministic)
    hq, hkv = case.hq, case.hkv
    group = hq // hkv
    heads = list(range(kv_group * group, (kv_group + 1) * group))
    cu = case.cu_seqlens.tolist()
    seq_ids = seqs if seqs is not None else range(len(cu) - 1)
    for s in seq_ids:
        a, b = cu[s], cu[s + 1]
        sub = dict(q=f64(case.q)[a:b][:, heads], k=f64(case.k)[a:b][:, [kv_group]],
                   v=f64(case.v)[a:b][:, [kv_group]])
        kw = dict(log_gate=None if case.log_gate is None else f64(case.log_gate)[a:b][:, heads],
                  sink=None if case.sink is None else f64(case.sink)[heads], window=case.window)
        ro, rl = oracle.prefill_forward(sub["q"], sub["k"], sub["v"], np.array([0, b - a]), case.scale, **kw)
        assert_close(f"o[seq {s}]", f64(o)[a:b][:, heads], ro, PREFILL_RTOL)
        np.testing.assert_allclose(f64(lse)[heads][:, a:b], rl, rtol=0, atol=2e-3)
        if backward:
            rdq, rdk, rdv, rdg, _ = oracle.prefill_backward(sub["q"], sub["k"], sub["v"],
                                                            f64(case.do)[a:b][:, heads], np.array([0, b - a]),
                                                            case.scale, **kw)
            dq, dk, dv_, dg, _ = grads
            assert_close(f"dq[seq {s}]", f64(dq)[a:b][:, heads], rdq, PREFILL_RTOL)
            assert_close(f"dk[seq {s}]", f64(dk)[a:b][:, [kv_group]], rdk, PREFILL_RTOL)
            assert_close(f"dv[seq {s}]", f64(dv_)[a:b][:, [kv_group]], rdv, PREFILL_RTOL)
            if rdg is not None:
                assert_close(f"dg[seq {s}]", f64(dg)[a:b][:, heads], rdg, PREFILL_RTOL)
    return case, grads


@pytest.mark.parametrize("deterministic,kv_group", [(False, 0), (False, 5), (False, 7), (True, 5)])
def test_full_size_varlen_gqa_d128_sampled(gcs_lib, deterministic, kv_group):
    """Packed 1000/3000/4192, Hq=32, Hkv=8, D=128, gate + sink: every sequence of one kv-head
    group against the oracle; the sink gradient of those heads over the whole batch.  Both
    backward routes: the single pass (the bench's launch configuration: the first, a middle
    and the last group) and the two passes."""
    case, grads = _sampled_full_size(gcs_lib, "varlen_gqa_8192_d128", kv_group=kv_group,
                                     deterministic=deterministic)
    group = case.hq // case.hkv
    heads = list(range(kv_group * group, (kv_group + 1) * group))
    cu = case.cu_seqlens.numpy()
    _, _, _, _, rds = oracle.prefill_backward(
        f64(case.q)[:, heads], f64(case.k)[:, [kv_group]], f64(case.v)[:, [kv_group]], f64(case.do)[:, heads], cu,
        case.scale, log_gate=f64(case.log_gate)[:, heads], sink=f64(case.sink)[heads])
    assert_close("dsink", f64(grads[4])[heads], rds, PREFILL_RTOL)


def test_full_size_dense_mha_t128_d64(gcs_lib):
    case = prefill_config("dense_mha_t128_d64")
    o, lse, grads = run_prefill(gcs_lib, case)
    ro, rl, rg = oracle_prefill(case)
    assert_close("o", o, ro, PREFILL_RTOL)
    for n, got, ref in zip(("dq", "dk", "dv"), grads[:3], rg[:3]):
        assert_close(n, got, ref, PREFILL_RTOL)


@pytest.mark.parametrize("deterministic", [False, True])
def test_full_size_window_dqk256_dv512_sampled(gcs_lib, deterministic):
    _sampled_full_size(gcs_lib, "window_b2_t4096_dqk256_dv512", kv_group=3, backward=True, seqs=[1],
                       deterministic=deterministic)


@pytest.mark.parametrize("deterministic", [False, True])
def test_full_size_varlen_d512_sampled(gcs_lib, deterministic):
    case = prefill_config("varlen_16384_d512")
    shortest = int(np.argmin(case.seqlens))
    _sampled_full_size(gcs_lib, "varlen_16384_d512", kv_group=2, backward=True, seqs=[shortest],
                       deterministic=deterministic)
