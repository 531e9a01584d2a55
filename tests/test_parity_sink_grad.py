"""The sink gradient's precision requirement ([FLA] issue #1322, comment of Oct 3): with bf16
inputs, gates, a sink and packed sequences, a sink gradient formed from the rounded output,
-sum_i p_sink,i (dO_i . bf16(O_i)), missed the 5e-3 relative-RMS budget (both earlier
implementations measured about 5.75e-3); it has to come from the fp32 sum of P * (dO V^T)
taken while P is recomputed.

The exact reference is the closed form of the oracle's sink gradient,
dsigma_h = -sum_i p_sink,i (dO_i . O_i) with O and LSE from the fp64 oracle forward (pinned
against the oracle's analytic backward and finite differences on the CPU).  Each test
measures two errors against it: the library's dsink, and the rounded-output formula evaluated
by the test from the library's own bf16 O and LSE.  The library must sit below the budget
and a clear factor below the rounded-output formula, so a dsink kernel that used the
rounded-output delta alone would fail."""
import numpy as np
import pytest
import torch

import oracle
from synth import make_prefill, prefill_config
from helpers import PREFILL_RTOL, f64, run_prefill

pytestmark = pytest.mark.gpu

# the library's dsink must beat the rounded-output formula by at least this factor
MARGIN = 10.0


def exact_dsink(case, heads):
    """-sum over every sequence and row of p_sink,i (dO_i . O_i) for the given query heads,
    from the fp64 oracle forward (one kv head's group at a time)."""
    group = case.hq // case.hkv
    cu = case.cu_seqlens.tolist()
    out = np.zeros(len(heads))
    for n, h in enumerate(heads):
        kvh = h // group
        for a, b in zip(cu[:-1], cu[1:]):
            if b == a:
                continue
            o, lse = oracle.prefill_forward(
                f64(case.q)[a:b][:, [h]], f64(case.k)[a:b][:, [kvh]], f64(case.v)[a:b][:, [kvh]],
                np.array([0, b - a]), case.scale,
                log_gate=None if case.log_gate is None else f64(case.log_gate)[a:b][:, [h]],
                sink=f64(case.sink)[[h]], window=case.window)
            p_sink = np.exp(float(case.sink[h]) - lse[0])
            out[n] -= float((p_sink * (f64(case.do)[a:b, h] * o[:, 0]).sum(-1)).sum())
    return out


def rounded_output_dsink(case, o_dev, lse_dev, heads):
    """-sum_i p_sink,i (dO_i . O_i) evaluated from the library's bf16 O and fp32 LSE: the
    formula the comment of Oct 3 rules out."""
    o = f64(o_dev)
    lse = f64(lse_dev)
    do = f64(case.do)
    sink = f64(case.sink)
    res = []
    for h in heads:
        p_sink = np.exp(sink[h] - lse[h])
        res.append(-float((p_sink * (do[:, h] * o[:, h]).sum(-1)).sum()))
    return np.array(res)


def check(gcs, case, heads, deterministic=False):
    o, lse, grads = run_prefill(gcs, case, backward=True, deterministic=deterministic)
    ref = exact_dsink(case, heads)
    lib = f64(grads[4])[heads]
    e_lib = oracle.rel_rms(lib, ref)
    e_rounded = oracle.rel_rms(rounded_output_dsink(case, o, lse, heads), ref)
    print(f"dsink relative RMS: library {e_lib:.3e}, rounded-output formula {e_rounded:.3e}")
    assert np.isfinite(lib).all()
    assert e_lib <= PREFILL_RTOL, f"dsink relative RMS {e_lib:.3e} > {PREFILL_RTOL}"
    assert e_lib * MARGIN <= e_rounded, (
        f"dsink relative RMS {e_lib:.3e} is not {MARGIN}x below the rounded-output formula's {e_rounded:.3e}")
    return e_lib, e_rounded


def test_sink_gradient_beats_rounded_output_packed_gqa(gcs_lib):
    """Packed sequences of 700, 2600 and 3100 tokens, GQA 8:2, D = 128, bf16 inputs, gates
    and a sink: every query head."""
    case = make_prefill([700, 2600, 3100], 8, 2, 128, 128, seed=411, gate=True, sink=True)
    check(gcs_lib, case, list(range(8)))


def test_sink_gradient_beats_rounded_output_varlen_gqa_8192_d128(gcs_lib):
    """The full packed 1000/3000/4192, Hq = 32, Hkv = 8, D = 128 workload: every query head."""
    case = prefill_config("varlen_gqa_8192_d128")
    check(gcs_lib, case, list(range(case.hq)))


@pytest.mark.parametrize("deterministic", [False, True])
def test_sink_gradient_window_dqk256_dv512(gcs_lib, deterministic):
    """B = 2 x T = 4096, Dqk = 256, Dv = 512, window 1024, gates and sink: the four query
    heads of kv head 3 over both sequences, in both backward routes."""
    case = prefill_config("window_b2_t4096_dqk256_dv512")
    check(gcs_lib, case, [12, 13, 14, 15], deterministic=deterministic)


def test_sink_gradient_varlen_16384_d512(gcs_lib):
    """Four packed sequences summing to 16384 tokens, Hq = 32, Hkv = 4, D = 512, gates and
    sink: two query heads over all four sequences."""
    case = prefill_config("varlen_16384_d512")
    check(gcs_lib, case, [16, 23])
