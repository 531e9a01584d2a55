"""Device parity over a seeded random sweep of shapes and options, each case against the fp64
oracle on the same inputs:
- prefill forward and backward: every supported (Dqk, Dv) pair, MHA / GQA / MQA, ragged and
  empty sequences, windows, gates and sink in any combination, both backward routes;
- paged decode: 1-4 query positions per request, GQA groups of 16 and 8, cache blocks of 16
  and 128 tokens, fp8 with per-token or per-tensor scales (both scale readings) and bf16 caches,
  the decoding features, segments from one page up;
- paged chunked prefill: query chunks of up to 300 positions, the same cache options (fp8),
  automatic and fixed segments.
The draws are fixed by the seeds below, so a failing case is reproducible from its id."""
import numpy as np
import pytest
import torch

from synth import make_decode, make_prefill
from helpers import (DECODE_BIAS, DECODE_RTOL, PREFILL_RTOL, assert_close, bias, decode_dev, f64, oracle_decode,
                     oracle_prefill, run_decode, run_prefill)

pytestmark = pytest.mark.gpu

DIMS = [(64, 64), (128, 128), (128, 128), (256, 256), (256, 512), (512, 512)]


def prefill_draw(i):
    rng = np.random.default_rng(7000 + i)
    dqk, dv = DIMS[rng.integers(len(DIMS))]
    hkv = int(rng.integers(1, 3))
    hq = hkv * int(rng.choice([1, 2, 4, 8 if dqk <= 128 else 2]))
    top = 420 if dqk <= 128 else 260
    lens = [0 if rng.random() < 0.15 else int(rng.integers(1, top)) for _ in range(int(rng.integers(1, 5)))]
    if sum(lens) == 0:
        lens[-1] = int(rng.integers(1, top))
    gate, sink = bool(rng.random() < 0.6), bool(rng.random() < 0.6)
    window = 0 if rng.random() < 0.5 else int(rng.integers(1, 300))
    det = bool(rng.random() < 0.4)
    return dict(lens=lens, hq=hq, hkv=hkv, dqk=dqk, dv=dv, gate=gate, sink=sink, window=window, det=det,
                seed=7100 + i)


PREFILL_IDS = list(range(24))


@pytest.mark.parametrize("i", PREFILL_IDS)
def test_prefill_sweep(gcs_lib, i):
    c = prefill_draw(i)
    case = make_prefill(c["lens"], c["hq"], c["hkv"], c["dqk"], c["dv"], seed=c["seed"], gate=c["gate"],
                        sink=c["sink"], window=c["window"])
    o, lse, grads = run_prefill(gcs_lib, case, backward=True, deterministic=c["det"])
    ro, rlse, rg = oracle_prefill(case)
    assert_close("o", o, ro, PREFILL_RTOL)
    np.testing.assert_allclose(f64(lse), rlse, rtol=0, atol=2e-3)
    for name, got, ref in zip(("dq", "dk", "dv"), grads[:3], rg[:3]):
        assert_close(name, got, ref, PREFILL_RTOL)
    if c["gate"]:
        assert_close("dlog_gate", grads[3], rg[3], PREFILL_RTOL)
    if c["sink"]:
        assert_close("dsink", grads[4], rg[4], PREFILL_RTOL)


def decode_draw(i, paged_prefill):
    rng = np.random.default_rng((8000 if paged_prefill else 9000) + i)
    G = int(rng.choice([16, 8]))
    hkv = int(rng.choice([1, 2, 4]))
    R = int(rng.integers(1, 5))
    block = int(rng.choice([16, 128]))
    if paged_prefill:
        q_lens = [int(rng.integers(1, 301)) for _ in range(R)]
        fmt, smode = "fp8", str(rng.choice(["per_token", "per_tensor"]))
    else:
        q_lens = [int(rng.integers(1, 5)) for _ in range(R)]
        fmt = str(rng.choice(["fp8", "fp8", "bf16"]))
        smode = "per_token" if fmt == "bf16" else str(rng.choice(["per_token", "per_tensor"]))
    seq_lens = []
    for ql in q_lens:
        # contexts anywhere up to ~3K tokens, or a few tokens around a page / block edge
        if rng.random() < 0.3:
            L = 16 * int(rng.integers(1, 100)) + int(rng.integers(-2, 3))
        else:
            L = int(rng.integers(1, 3000))
        seq_lens.append(max(L, ql))
    feat = bool(rng.random() < 0.4)
    window = int(rng.integers(1, 600)) if feat and rng.random() < 0.6 else 0
    reading = str(rng.choice(["A", "B"])) if (fmt == "fp8" and smode == "per_token") else "A"
    if paged_prefill:
        seg = int(rng.choice([0, 128, 512]))
    else:
        seg = int(rng.choice([16, 64, 256, 2048]))
    return dict(seq_lens=seq_lens, q_lens=q_lens, hq=G * hkv, hkv=hkv, block=block, fmt=fmt, smode=smode, feat=feat,
                window=window, reading=reading, seg=seg, seed=(8100 if paged_prefill else 9100) + i)


def make_case(c, seg):
    return make_decode(c["seq_lens"], c["q_lens"], c["hq"], c["hkv"], 128, seed=c["seed"], block_size=c["block"],
                       scale_reading=c["reading"], segment_len=seg, kv_format=c["fmt"], scale_mode=c["smode"],
                       features=c["feat"], window=c["window"])


@pytest.mark.parametrize("i", list(range(32)))
def test_decode_sweep(gcs_lib, i):
    c = decode_draw(i, paged_prefill=False)
    dc = make_case(c, c["seg"])
    out = run_decode(gcs_lib, dc)
    ref = oracle_decode(dc)
    assert np.isfinite(f64(out)).all()
    assert_close("out", out, ref, DECODE_RTOL)
    assert abs(bias(out, ref)) <= DECODE_BIAS


@pytest.mark.parametrize("i", list(range(12)))
def test_prefill_paged_sweep(gcs_lib, i):
    c = decode_draw(i, paged_prefill=True)
    dc = make_case(c, 2048)
    d = decode_dev(dc)
    out = gcs_lib.attn_prefill_paged(d["q"], d["kc"], d["vc"], d["ks"], d["vs"], d["bt"], d["sl"], d["cq"],
                                     max(dc.q_lens), int(dc.seq_lens.max()), dc.scale, c["seg"], g_cache=d["g"],
                                     sink=d["sink"], window=dc.window)
    torch.cuda.synchronize()
    assert gcs_lib.get_device_status() == 0
    ref = oracle_decode(dc)
    assert np.isfinite(f64(out)).all()
    assert_close("out", out, ref, DECODE_RTOL)
    assert abs(bias(out, ref)) <= DECODE_BIAS
