"""Shared helpers for the device parity tests: run a synthetic case through the C ABI (via
the binding) and compare element by element with the fp64 oracle."""
import numpy as np
import torch

import oracle

# Tolerances: bf16 outputs and all gradients, relative RMS (the pages' budget, 0.005);
# fp8 decode against the dequantised fp64 reference, relative RMS 1e-2 and |bias| 1e-3.
PREFILL_RTOL = 5e-3
DECODE_RTOL = 1e-2
DECODE_BIAS = 1e-3


def f64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def to_dev(case):
    dev = torch.device("cuda:0")
    mv = lambda t: None if t is None else t.to(dev)
    return dict(q=mv(case.q), k=mv(case.k), v=mv(case.v), do=mv(case.do), cu=mv(case.cu_seqlens),
                g=mv(case.log_gate), s=mv(case.sink))


def run_prefill(gcs, case, backward=True, deterministic=False):
    d = to_dev(case)
    ms = max(case.seqlens)
    o, lse = gcs.attn_fwd(d["q"], d["k"], d["v"], d["cu"], ms, case.scale, case.window, d["g"], d["s"])
    grads = None
    if backward:
        grads = gcs.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], ms, case.scale, case.window, d["g"],
                             d["s"], deterministic=deterministic)
    torch.cuda.synchronize()
    assert gcs.get_device_status() == 0
    return o, lse, grads


def oracle_prefill(case, backward=True):
    args = (f64(case.q), f64(case.k), f64(case.v))
    kw = dict(log_gate=f64(case.log_gate), sink=f64(case.sink), window=case.window)
    o, lse = oracle.prefill_forward(*args, case.cu_seqlens.numpy(), case.scale, **kw)
    g = None
    if backward:
        g = oracle.prefill_backward(*args, f64(case.do), case.cu_seqlens.numpy(), case.scale, **kw)
    return o, lse, g


def assert_close(name, got, ref, rtol):
    got = f64(got) if isinstance(got, torch.Tensor) else got
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    e = oracle.rel_rms(got, ref)
    assert e <= rtol, f"{name}: relative RMS {e:.3e} > {rtol:.1e}"
    return e


def bias(got, ref):
    """Relative signed projection sum((got - ref) ref) / sum(ref^2): a multiplicative
    shrink of the output by 0.3% reads as -3e-3."""
    got = f64(got) if isinstance(got, torch.Tensor) else got
    return float(((got - ref) * ref).sum() / (ref * ref).sum())


def decode_dev(dc):
    dev = torch.device("cuda:0")
    opt = lambda t: None if t is None else t.to(dev)
    return dict(q=dc.q.to(dev), kc=dc.k_cache.to(dev), vc=dc.v_cache.to(dev), ks=opt(dc.k_scale),
                vs=opt(dc.v_scale), bt=dc.block_table.to(dev), sl=dc.seq_lens.to(dev), cq=dc.cu_q.to(dev),
                g=opt(dc.g_cache), sink=opt(dc.sink))


def run_decode(gcs, dc, d=None):
    d = d or decode_dev(dc)
    out = gcs.attn_decode_paged(d["q"], d["kc"], d["vc"], d["ks"], d["vs"], d["bt"], d["sl"], d["cq"],
                                max(dc.q_lens), int(dc.seq_lens.max()), dc.scale, dc.segment_len,
                                g_cache=d["g"], sink=d["sink"], window=dc.window)
    torch.cuda.synchronize()
    assert gcs.get_device_status() == 0
    return out


def oracle_decode(dc, rows=None):
    cache = lambda t: t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()
    opt = lambda t: None if t is None else t.numpy()
    return oracle.decode_paged(f64(dc.q), cache(dc.k_cache), cache(dc.v_cache), opt(dc.k_scale), opt(dc.v_scale),
                               dc.block_table.numpy(), dc.seq_lens.numpy(), dc.cu_q.numpy(), dc.scale,
                               g_cache=opt(dc.g_cache), sink=None if dc.sink is None else f64(dc.sink),
                               window=dc.window)
