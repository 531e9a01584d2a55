"""fp64 CPU oracle: gated causal softmax attention, prefill forward/backward and paged
fp8 decode (test infrastructure only).

Sources (page title, section):
  [FLA] fla-org/flash-linear-attention issue #1322, "[Perf] Gluon attention backend with
        large head dimensions": Description (the causal attention contract: dense and
        packed variable-length inputs, MHA/GQA/MQA, unequal query/key and value dims,
        logarithmic gates, sliding windows, sink bias, gradients); comment of Oct 3
        (sink gradient from the backward probabilities, in fp32, not from rounded O).
  [AIT] ROCm/aiter PR #6660 (gfx1250 unified attention): commit messages and "Technical
        details" (per-token K/V scales laid out [num_blocks, num_kv_heads, block_size];
        K scales multiply QK columns, V scales multiply P columns after the row sum,
        slots past seq_len get scale 0; split-K over context segments with an
        LSE-weighted reduce where empty partials, M = -inf, weigh 0).

Readings where the pages leave a step open (each is also listed in the design notes):
  * score s_ij = scale * q_i.k_j + G_i - G_j, G = per-sequence inclusive cumsum of the
    per-token, per-query-head log gates; the gate is not multiplied by the scale.
  * window W > 0 keeps key j for query i iff 0 <= i - j < W; W = 0 means no window.
  * the sink is one logit per query head, present only in the softmax denominator.
  * LSE includes the sink term; the sink gradient is summed over every token of every
    sequence in the batch.
  * decode: query row t of a request with q_len rows sits at position L - q_len + t and
    sees keys 0..L - q_len + t (bottom-right causal alignment).
  * decode with gates keeps the cumulative log gates G of the cached tokens paged like the
    scales, per query head: g_cache [num_blocks, hq, block_size] (natural-log units); a
    query row's own G is the entry at its position.  The window and the sink follow the
    prefill rules; in split-K the sink enters once, in the combine's denominator.

Everything runs in float64 with dense per-(sequence, head) matrices; no blocking, no
online softmax, no fusion.  Inputs are float64 arrays (bf16 / fp32 inputs widened
exactly) and uint8 e4m3 codes for the cache.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

from .formats import e4m3_decode


def _seq_bounds(cu_seqlens):
    """(start, end) token ranges of the packed sequences ([FLA] Description, packed
    variable-length inputs: sequence s owns tokens cu_seqlens[s] .. cu_seqlens[s+1] - 1)."""
    cu = [int(x) for x in np.asarray(cu_seqlens).tolist()]
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


def gate_cumsum(log_gate: np.ndarray, cu_seqlens) -> np.ndarray:
    """G_t = sum of g_u over u = start(seq) .. t, per sequence and head ([FLA] Description,
    the per-token log gates; inclusive cumsum restarted at every sequence start)."""
    g = np.asarray(log_gate, dtype=np.float64)
    G = np.zeros_like(g)
    for a, b in _seq_bounds(cu_seqlens):
        G[a:b] = np.cumsum(g[a:b], axis=0)
    return G


def _allowed(T: int, window: int) -> np.ndarray:
    """Mask of visible (i, j) pairs inside one sequence ([FLA] Description, causal attention
    with sliding windows): causal j <= i, and i - j < W when a window W is set."""
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    m = j <= i
    if window > 0:
        m &= (i - j) < window
    return m


def _scores(qh, kh, scale, Gh, allowed):
    """s_ij = scale q_i . k_j + G_i - G_j for visible pairs, -inf elsewhere ([FLA] Description,
    causal attention with logarithmic gates)."""
    S = scale * (qh @ kh.T)
    if Gh is not None:
        S = S + (Gh[:, None] - Gh[None, :])
    return np.where(allowed, S, -np.inf)


def _softmax_with_sink(S, sink_h):
    """P_ij = e^{s_ij} / Z_i and p_sink,i = e^{sigma} / Z_i with
    Z_i = sum_j e^{s_ij} (+ e^{sigma}); returns P, p_sink (or None), ln Z ([FLA] Description,
    the sink bias: one logit per head in the softmax denominator only)."""
    m = S.max(axis=1)
    if sink_h is not None:
        m = np.maximum(m, sink_h)
    E = np.exp(S - m[:, None])
    Z = E.sum(axis=1)
    ps = None
    if sink_h is not None:
        es = np.exp(sink_h - m)
        Z = Z + es
        ps = es / Z
    P = E / Z[:, None]
    return P, ps, m + np.log(Z)


def prefill_forward(q, k, v, cu_seqlens, scale, log_gate=None, sink=None, window=0):
    """Causal softmax attention forward ([FLA] Description).

    q [tot, hq, dqk], k [tot, hkv, dqk], v [tot, hkv, dv]; query head h reads kv head
    h // (hq // hkv).  Returns o [tot, hq, dv] and lse [hq, tot] (natural log, sink
    included).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    tot, hq, _ = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    group = hq // hkv
    G = gate_cumsum(log_gate, cu_seqlens) if log_gate is not None else None
    sink = None if sink is None else np.asarray(sink, np.float64)
    o = np.zeros((tot, hq, dv))
    lse = np.zeros((hq, tot))
    for a, b in _seq_bounds(cu_seqlens):
        if b == a:
            continue
        allowed = _allowed(b - a, window)
        for h in range(hq):
            kvh = h // group
            S = _scores(q[a:b, h], k[a:b, kvh], scale, None if G is None else G[a:b, h], allowed)
            P, _, L = _softmax_with_sink(S, None if sink is None else sink[h])
            o[a:b, h] = P @ v[a:b, kvh]
            lse[h, a:b] = L
    return o, lse


def prefill_backward(q, k, v, do, cu_seqlens, scale, log_gate=None, sink=None, window=0):
    """Analytic gradients of L = sum(O * dO) ([FLA] Description, the gradient list; Oct 3 comment
    for the sink).

      dP_ij = dO_i . v_j,   D_i = sum_j P_ij dP_ij,   dS_ij = P_ij (dP_ij - D_i)
      dq_i = scale sum_j dS_ij k_j;   dk_j, dv_j summed over the query heads of the group
      dG_t = sum_j dS_tj - sum_i dS_it,   dg_t = sum_{u >= t, same sequence} dG_u
      dsigma_h = - sum over all sequences and rows of p_sink,i * D_i

    Returns dq, dk, dv, dg (or None), dsink (or None).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    tot, hq, dqk = q.shape
    hkv, dv_ = k.shape[1], v.shape[2]
    group = hq // hkv
    G = gate_cumsum(log_gate, cu_seqlens) if log_gate is not None else None
    sink = None if sink is None else np.asarray(sink, np.float64)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dg = np.zeros((tot, hq)) if G is not None else None
    dsink = np.zeros(hq) if sink is not None else None
    for a, b in _seq_bounds(cu_seqlens):
        if b == a:
            continue
        allowed = _allowed(b - a, window)
        for h in range(hq):
            kvh = h // group
            S = _scores(q[a:b, h], k[a:b, kvh], scale, None if G is None else G[a:b, h], allowed)
            P, ps, _ = _softmax_with_sink(S, None if sink is None else sink[h])
            dP = do[a:b, h] @ v[a:b, kvh].T
            D = (P * dP).sum(axis=1)
            dS = P * (dP - D[:, None])
            dq[a:b, h] = scale * (dS @ k[a:b, kvh])
            dk[a:b, kvh] += scale * (dS.T @ q[a:b, h])
            dv[a:b, kvh] += P.T @ do[a:b, h]
            if dg is not None:
                dG = dS.sum(axis=1) - dS.sum(axis=0)
                dg[a:b, h] = np.cumsum(dG[::-1])[::-1]
            if dsink is not None:
                dsink[h] -= float((ps * D).sum())
    return dq, dk, dv, dg, dsink


# ----------------------------------------------------------------------------- decode
def _token_values(cache, scales, blocks, kv_head, L):
    """Stored values and scales of tokens 0..L-1 of one request and kv head, before scaling:
    an e4m3 cache (uint8 codes) with one fp32 scale per token ([AIT] Technical details,
    layout [num_blocks, num_kv_heads, block_size]) or one per tensor (the same section leaves
    per-tensor scaling on the path that existed before); or a bf16 cache
    ([AIT] commit 3, the bf16-KV route) with no scales.  Slots at or past L are never read.
    Returns (values [L, d], scales [L]) in float64."""
    bs = cache.shape[2]
    npages = len(blocks)
    raw = np.asarray(cache[blocks, kv_head])  # [npages, bs, d]
    if raw.dtype == np.uint8:
        vals = e4m3_decode(raw.reshape(npages * bs, -1)[:L])
        sc = np.asarray(scales, dtype=np.float64)
        if sc.size == 1:
            sc = np.full(L, float(sc.reshape(-1)[0]))
        else:
            sc = sc[blocks, kv_head].reshape(-1)[:L]
    else:
        assert scales is None, "a bf16 cache has no scales"
        vals = raw.astype(np.float64).reshape(npages * bs, -1)[:L]
        sc = np.ones(L)
    return vals, sc


def gather_kv(cache, scales, block_table_row, L, kv_head):
    """Dequantized keys (or values) 0..L-1 of one request and kv head: stored value times
    its scale ([AIT] Technical details: key j of a request sits in block table[j / block_size],
    slot j % block_size; see _token_values)."""
    bs = cache.shape[2]
    npages = (L + bs - 1) // bs
    blocks = np.asarray(block_table_row[:npages], dtype=np.int64)
    vals, sc = _token_values(cache, scales, blocks, kv_head, L)
    return vals * sc[:, None]


def _gate_of(g_cache, block_table_row, L, h):
    """G_j, j = 0..L-1, of one request and query head from the paged fp32 array
    [num_blocks, hq, block_size] ([FLA] Description asks for the gates on the decode path and
    gives no layout; read here as the cumulative log gates of the cached tokens kept paged like
    the scales, per query head)."""
    bs = g_cache.shape[2]
    npages = (L + bs - 1) // bs
    blocks = np.asarray(block_table_row[:npages], dtype=np.int64)
    return np.asarray(g_cache[blocks, h], dtype=np.float64).reshape(-1)[:L]


def _visible(pos, window, lo=0, hi=None):
    """Keys visible to a query at position pos: j <= pos (causal) and pos - j < W (window),
    intersected with [lo, hi) ([AIT] commit messages: short queries are the last q_len cached
    tokens, so a query row sees the keys up to its own position; [FLA] Description, windows)."""
    a = max(lo, pos - window + 1) if window > 0 else lo
    b = pos + 1 if hi is None else min(hi, pos + 1)
    return a, b


def decode_paged(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, scale, *, g_cache=None,
                 sink=None, window=0):
    """Paged decode / short-query attention over the dequantized cache, unsplit.

    q [nq, hq, d] (rows of request r are cu_q[r]..cu_q[r+1]); row t of request r sits at
    position L - q_len + t and attends to keys 0..L - q_len + t.  With the decoding
    features of [FLA] Description: s_j = scale q.k_j + G_i - G_j (G from g_cache, the query's
    own G at its position), the window keeps pos - j < W, and the sink adds e^sigma_h to the
    denominator only.  Returns [nq, hq, d].
    """
    q = np.asarray(q, np.float64)
    nq, hq, d = q.shape
    hkv = k_cache.shape[1]
    group = hq // hkv
    seq_lens = np.asarray(seq_lens).tolist()
    cu_q = np.asarray(cu_q).tolist()
    out = np.zeros((nq, hq, d))
    for r, L in enumerate(seq_lens):
        q0, q1 = cu_q[r], cu_q[r + 1]
        ql = q1 - q0
        for kvh in range(hkv):
            K = gather_kv(k_cache, k_scale, block_table[r], L, kvh)
            V = gather_kv(v_cache, v_scale, block_table[r], L, kvh)
            for h in range(kvh * group, (kvh + 1) * group):
                G = None if g_cache is None else _gate_of(g_cache, block_table[r], L, h)
                for t in range(ql):
                    pos = L - ql + t
                    a, b = _visible(pos, window)
                    s = scale * (K[a:b] @ q[q0 + t, h])
                    if G is not None:
                        s = s + (G[pos] - G[a:b])
                    m = s.max() if sink is None else max(s.max(), float(sink[h]))
                    p = np.exp(s - m)
                    den = p.sum() + (0.0 if sink is None else math.exp(float(sink[h]) - m))
                    out[q0 + t, h] = (p @ V[a:b]) / den
    return out


def decode_partials(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, scale, segment_len, *,
                    g_cache=None, window=0):
    """Split-K partials in the pages' order ([AIT] commits and Technical details).

    For each (request, kv head, segment [segment_len*s, segment_len*(s+1)) of the
    context) and each query row: s_j = scale * kscale_j * (q . k8_j) (+ G_i - G_j with
    gates); the running max m and row sum l use the unscaled probabilities p_j = e^{s_j - m};
    the V scales multiply the P columns after the row sum: acc = sum_j (p_j vscale_j) v8_j.
    A row with no visible key in the segment (past its position, or before its window)
    stores (acc, m, l) = (0, -inf, 0).  The sink is not part of any partial.

    Returns a list of dicts {r, kvh, seg, acc [ql, group, d], m [ql, group], l [ql, group]}.
    """
    q = np.asarray(q, np.float64)
    nq, hq, d = q.shape
    hkv = k_cache.shape[1]
    bs = k_cache.shape[2]
    group = hq // hkv
    seq_lens = np.asarray(seq_lens).tolist()
    cu_q = np.asarray(cu_q).tolist()
    parts = []
    for r, L in enumerate(seq_lens):
        q0, q1 = cu_q[r], cu_q[r + 1]
        ql = q1 - q0
        nseg = (L + segment_len - 1) // segment_len
        npages = (L + bs - 1) // bs
        blocks = np.asarray(block_table[r][:npages], dtype=np.int64)
        for kvh in range(hkv):
            k8, ks = _token_values(k_cache, k_scale, blocks, kvh, L)
            v8, vs = _token_values(v_cache, v_scale, blocks, kvh, L)
            Gs = None if g_cache is None else [_gate_of(g_cache, block_table[r], L, h)
                                               for h in range(kvh * group, (kvh + 1) * group)]
            for sg in range(nseg):
                j0, j1 = sg * segment_len, min((sg + 1) * segment_len, L)
                acc = np.zeros((ql, group, d))
                m = np.full((ql, group), -np.inf)
                l = np.zeros((ql, group))
                for t in range(ql):
                    pos = L - ql + t
                    a, b = _visible(pos, window, j0, j1)
                    if b <= a:
                        continue  # empty partial
                    qq = q[q0 + t, kvh * group : (kvh + 1) * group]  # [group, d]
                    s = scale * (qq @ k8[a:b].T) * ks[a:b][None, :]
                    if Gs is not None:
                        s = s + np.stack([G[pos] - G[a:b] for G in Gs])
                    mm = s.max(axis=1)
                    p = np.exp(s - mm[:, None])
                    m[t] = mm
                    l[t] = p.sum(axis=1)
                    acc[t] = (p * vs[a:b][None, :]) @ v8[a:b]
                parts.append(dict(r=r, kvh=kvh, seg=sg, acc=acc, m=m, l=l))
    return parts


def decode_combine(parts, nq, hq, d, cu_q, hkv, *, sink=None):
    """LSE-weighted reduce ([AIT] commit 3 / Technical details): M* = max_s m_s (and the
    sink logit when there is one), w_s = 0 for an empty partial (m_s = -inf) else
    e^{m_s - M*}, O = sum w_s acc_s / (sum w_s l_s + e^{sigma - M*}).  A row whose partials
    are all empty gets 0."""
    group = hq // hkv
    cu_q = np.asarray(cu_q).tolist()
    by_key = {}
    for p in parts:
        by_key.setdefault((p["r"], p["kvh"]), []).append(p)
    out = np.zeros((nq, hq, d))
    for (r, kvh), plist in by_key.items():
        q0 = cu_q[r]
        M = np.max(np.stack([p["m"] for p in plist]), axis=0)  # [ql, group]
        if sink is not None:
            sg = np.asarray(sink, np.float64)[kvh * group : (kvh + 1) * group][None, :]
            M = np.maximum(M, sg)
        num = np.zeros_like(plist[0]["acc"])
        den = np.zeros_like(plist[0]["l"])
        for p in plist:
            w = np.where(np.isneginf(p["m"]), 0.0, np.exp(np.where(np.isneginf(M), 0.0, p["m"] - M)))
            num += w[:, :, None] * p["acc"]
            den += w * p["l"]
        if sink is not None:
            den = den + np.exp(sg - M)
        res = np.where(den[:, :, None] > 0, num / np.where(den > 0, den, 1.0)[:, :, None], 0.0)
        ql = res.shape[0]
        out[q0 : q0 + ql, kvh * group : (kvh + 1) * group] = res
    return out


def decode_paged_splitk(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, scale, segment_len, *,
                        g_cache=None, sink=None, window=0):
    """Split-K decode ([AIT] commits and Technical details): partials per context segment,
    then the LSE-weighted reduce."""
    q = np.asarray(q)
    parts = decode_partials(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, scale, segment_len,
                            g_cache=g_cache, window=window)
    return decode_combine(parts, q.shape[0], q.shape[1], q.shape[2], cu_q, k_cache.shape[1], sink=sink)


def rel_rms(x, ref) -> float:
    """||x - ref||_2 / ||ref||_2 over the whole tensor (the error measure of the [FLA] issue's
    accuracy budget, comment of Oct 3).  A reference that is all zeros gives the absolute
    norm ||x||_2 instead; a NaN in x gives NaN, which fails every tolerance comparison."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = math.sqrt(float((ref * ref).sum()))
    num = math.sqrt(float(((x - ref) ** 2).sum()))
    return num / den if den > 0 else num
