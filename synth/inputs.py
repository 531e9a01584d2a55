"""Seeded synthetic inputs for prefill and paged fp8 decode.

Every array is drawn from ``numpy.random.Generator(PCG64(seed))`` in a fixed order and
encoded to its storage type here: bf16 by round-to-nearest-even (``torch.bfloat16``
conversion), fp8 e4m3 by saturating to +-448 and round-to-nearest-even
(``torch.float8_e4m3fn`` conversion).  The results are CPU tensors; callers copy them to
the device or widen them to float64 for the oracle.

Workload shapes follow the pages' attention contract (dense and packed variable-length
inputs, MHA/GQA/MQA, unequal query/key and value head dims up to 512, log gates, sliding
windows, sink bias) and the paged decode tests (GQA 16, head 128, page 16, per-token
fp8 scales spanning 20x, NaN in unused slots, short queries over long contexts).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

E4M3_MAX = 448.0
E4M3_NAN_CODE = 0x7F


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _e4m3_codes(x: np.ndarray) -> torch.Tensor:
    """float32 -> fp8 e4m3fn codes (uint8), saturating to +-448."""
    x = np.clip(np.asarray(x, dtype=np.float32), -E4M3_MAX, E4M3_MAX)
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn).view(torch.uint8)


def _logsigmoid(x: np.ndarray) -> np.ndarray:
    # log(sigmoid(x)) = -log1p(exp(-x)), evaluated stably in float64
    x = np.asarray(x, dtype=np.float64)
    return np.where(x >= 0, -np.log1p(np.exp(-x)), x - np.log1p(np.exp(x)))


# ----------------------------------------------------------------------------- prefill
@dataclasses.dataclass
class PrefillCase:
    name: str
    cu_seqlens: torch.Tensor  # int32 [num_seqs + 1]
    q: torch.Tensor  # bf16 [tot, hq, dqk]
    k: torch.Tensor  # bf16 [tot, hkv, dqk]
    v: torch.Tensor  # bf16 [tot, hkv, dv]
    do: torch.Tensor  # bf16 [tot, hq, dv]
    log_gate: Optional[torch.Tensor]  # fp32 [tot, hq] or None
    sink: Optional[torch.Tensor]  # fp32 [hq] or None
    scale: float
    window: int  # 0 = no window

    @property
    def seqlens(self) -> list[int]:
        c = self.cu_seqlens.tolist()
        return [c[i + 1] - c[i] for i in range(len(c) - 1)]

    @property
    def total(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def hq(self) -> int:
        return self.q.shape[1]

    @property
    def hkv(self) -> int:
        return self.k.shape[1]

    @property
    def dqk(self) -> int:
        return self.q.shape[2]

    @property
    def dv(self) -> int:
        return self.v.shape[2]


def make_prefill(
    seqlens: Sequence[int],
    hq: int,
    hkv: int,
    dqk: int,
    dv: int,
    *,
    seed: int,
    gate: bool = False,
    sink: bool = False,
    window: int = 0,
    scale: Optional[float] = None,
    name: str = "prefill",
    gate_mean: float = 3.0,
) -> PrefillCase:
    """Draw order: q, k, v, dO (N(0,1) -> bf16), log-gates logsigmoid(N(gate_mean,1)) fp32
    [tot, hq], sink logits N(0,1) fp32 [hq]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    seqlens = [int(s) for s in seqlens]
    tot = sum(seqlens)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    q = _bf16(rng.standard_normal((tot, hq, dqk), dtype=np.float32))
    k = _bf16(rng.standard_normal((tot, hkv, dqk), dtype=np.float32))
    v = _bf16(rng.standard_normal((tot, hkv, dv), dtype=np.float32))
    do = _bf16(rng.standard_normal((tot, hq, dv), dtype=np.float32))
    g = None
    if gate:
        g = torch.from_numpy(_logsigmoid(rng.normal(gate_mean, 1.0, size=(tot, hq))).astype(np.float32))
    s = None
    if sink:
        s = torch.from_numpy(rng.standard_normal(hq).astype(np.float32))
    return PrefillCase(
        name=name,
        cu_seqlens=torch.from_numpy(cu),
        q=q,
        k=k,
        v=v,
        do=do,
        log_gate=g,
        sink=s,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(dqk)),
        window=int(window),
    )


def _c4_lengths(seed: int, total: int = 16384, n: int = 4, lo: int = 512, hi: int = 8192) -> list[int]:
    """Rejection-sample n-1 lengths uniform on {lo..hi} until the remainder is in range."""
    rng = np.random.Generator(np.random.PCG64(seed))
    while True:
        ls = rng.integers(lo, hi + 1, size=n - 1).tolist()
        last = total - sum(ls)
        if lo <= last <= hi:
            return [int(x) for x in ls] + [int(last)]


PREFILL_CONFIGS = {
    # Dense causal MHA, no gate / window / sink, scale 1/sqrt(64), seed 0.
    "dense_mha_t128_d64": dict(seqlens=[128], hq=2, hkv=2, dqk=64, dv=64, seed=0),
    # Packed varlen GQA, 3 sequences 1000/3000/4192, gate + sink, full causal.
    "varlen_gqa_8192_d128": dict(seqlens=[1000, 3000, 4192], hq=32, hkv=8, dqk=128, dv=128, seed=1, gate=True,
                                 sink=True),
    # Unequal head dims with sliding window 1024, B=2 x T=4096 dense.
    "window_b2_t4096_dqk256_dv512": dict(seqlens=[4096, 4096], hq=16, hkv=4, dqk=256, dv=512, seed=2, gate=True,
                                         sink=True, window=1024),
    # Large-head packed prefill: 4 sequences in [512, 8192] summing to 16384, D=512.
    "varlen_16384_d512": dict(seqlens=None, hq=32, hkv=4, dqk=512, dv=512, seed=3, gate=True, sink=True),
}


def prefill_config(name: str) -> PrefillCase:
    cfg = dict(PREFILL_CONFIGS[name])
    if cfg["seqlens"] is None:
        cfg["seqlens"] = _c4_lengths(cfg["seed"])
    return make_prefill(name=name, **cfg)


# ----------------------------------------------------------------------------- decode
@dataclasses.dataclass
class DecodeCase:
    name: str
    q: torch.Tensor  # bf16 [nq, hq, d]
    cu_q: torch.Tensor  # int32 [R + 1]
    seq_lens: torch.Tensor  # int32 [R]
    block_table: torch.Tensor  # int32 [R, max_blocks]
    k_cache: torch.Tensor  # uint8 (fp8 e4m3 codes) or bf16 [num_blocks, hkv, block_size, d]
    v_cache: torch.Tensor  # same
    k_scale: Optional[torch.Tensor]  # fp32 [num_blocks, hkv, block_size] (per token) or [1] (per tensor); None for bf16
    v_scale: Optional[torch.Tensor]
    scale: float
    segment_len: int
    kv_format: str = "fp8"  # "fp8" (e4m3 codes and scales) or "bf16" (values, no scales)
    scale_mode: str = "per_token"  # "per_token" or "per_tensor" (fp8 only)
    g_cache: Optional[torch.Tensor] = None  # fp32 [num_blocks, hq, block_size]: cumulative log gates G
    sink: Optional[torch.Tensor] = None  # fp32 [hq]
    window: int = 0
    # the values before fp8 quantization (fp32, same layout as the caches, NaN where unused);
    # kept only when make_decode is asked to (keep_unquantized), fp8 per-token only
    k_unquant: Optional[torch.Tensor] = None
    v_unquant: Optional[torch.Tensor] = None

    @property
    def num_reqs(self) -> int:
        return self.seq_lens.shape[0]

    @property
    def hq(self) -> int:
        return self.q.shape[1]

    @property
    def hkv(self) -> int:
        return self.k_cache.shape[1]

    @property
    def block_size(self) -> int:
        return self.k_cache.shape[2]

    @property
    def d(self) -> int:
        return self.q.shape[2]

    @property
    def q_lens(self) -> list[int]:
        c = self.cu_q.tolist()
        return [c[i + 1] - c[i] for i in range(len(c) - 1)]


def make_decode(
    seq_lens: Sequence[int],
    q_lens: Sequence[int],
    hq: int,
    hkv: int,
    d: int = 128,
    *,
    seed: int,
    block_size: int = 16,
    spare_blocks: int = 64,
    scale_reading: str = "A",
    scale: Optional[float] = None,
    segment_len: int = 2048,
    name: str = "decode",
    kv_format: str = "fp8",
    scale_mode: str = "per_token",
    features: bool = False,
    window: int = 0,
    keep_unquantized: bool = False,
) -> DecodeCase:
    """Draw order: q N(0,1) -> bf16; a random permutation of the physical blocks (the page
    table); then per request: K scales, V scales (log-uniform over a 20x range), K normals,
    V normals, stored as e4m3 codes of value/scale.

    scale_reading "A": scale ~ logU[1/64, 20/64], code = e4m3(z / scale) (dequantized
    values ~ N(0,1)).  "B": scale ~ logU[1/16, 20/16], code = e4m3(16 z) (dequantized
    magnitudes differ up to 20x between tokens).  Unused slots of used pages and every
    slot of unreferenced pages hold NaN scales and the NaN code 0x7F; unused page-table
    entries point at spare (all-NaN) blocks.

    kv_format "bf16": the cache holds bf16 values z ~ N(0,1) and no scales (NaN in unused
    slots).  scale_mode "per_tensor" (fp8): one K and one V scale for the whole cache, drawn
    once from logU[1/64, 20/64] after the page table, codes e4m3(z / scale).  Both draw
    orders are otherwise those above, so the default cases are unchanged.

    features: after every draw above, per request the log gates g ~ logsigmoid(N(3, 1)) per
    (token, query head), G = their cumulative sum from the request's first token, stored
    in g_cache [num_blocks, hq, block_size] (NaN in unused slots); then sink ~ N(0, 1) [hq].
    window: the sliding window W (0 = none).

    keep_unquantized (fp8 per-token only): also return the values before quantization,
    (code input) x scale in fp32, i.e. z in reading A and 16 z x scale in reading B.  Nothing
    extra is drawn, so the case is otherwise unchanged.
    """
    assert kv_format in ("fp8", "bf16") and scale_mode in ("per_token", "per_tensor")
    assert not (kv_format == "bf16" and scale_mode != "per_token")
    rng = np.random.Generator(np.random.PCG64(seed))
    seq_lens = [int(x) for x in seq_lens]
    q_lens = [int(x) for x in q_lens]
    assert len(seq_lens) == len(q_lens)
    R = len(seq_lens)
    nq = sum(q_lens)
    cu_q = np.zeros(R + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(q_lens)
    q = _bf16(rng.standard_normal((nq, hq, d), dtype=np.float32))

    pages = [(L + block_size - 1) // block_size for L in seq_lens]
    used = sum(pages)
    num_blocks = used + spare_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = max(pages) if pages else 1
    table = np.empty((R, max_blocks), dtype=np.int32)
    spare = perm[used:]
    pos = 0
    for r in range(R):
        table[r, : pages[r]] = perm[pos : pos + pages[r]]
        # unused entries -> spare blocks (never read by a correct kernel)
        fill = spare[np.arange(max_blocks - pages[r]) % max(len(spare), 1)] if len(spare) else perm[:1]
        table[r, pages[r] :] = fill
        pos += pages[r]

    if kv_format == "bf16" or scale_mode == "per_tensor":
        case = _make_decode_variant(rng, seq_lens, q_lens, cu_q, q, table, pages, num_blocks, hkv, d, block_size,
                                    scale, segment_len, name, kv_format, scale_mode)
        return _add_decode_features(rng, case, features, window)
    k_cache = np.full((num_blocks, hkv, block_size, d), E4M3_NAN_CODE, dtype=np.uint8)
    v_cache = np.full((num_blocks, hkv, block_size, d), E4M3_NAN_CODE, dtype=np.uint8)
    k_sc = np.full((num_blocks, hkv, block_size), np.nan, dtype=np.float32)
    v_sc = np.full((num_blocks, hkv, block_size), np.nan, dtype=np.float32)
    unq = {}
    if keep_unquantized:
        unq = {w: np.full((num_blocks, hkv, block_size, d), np.nan, dtype=np.float32) for w in "kv"}
    if scale_reading == "A":
        lo, hi, zmul = 1.0 / 64, 20.0 / 64, None
    elif scale_reading == "B":
        lo, hi, zmul = 1.0 / 16, 20.0 / 16, 16.0
    else:
        raise ValueError(scale_reading)
    for r in range(R):
        L, P = seq_lens[r], pages[r]
        blocks = table[r, :P]
        ks = np.exp(rng.uniform(math.log(lo), math.log(hi), size=(L, hkv))).astype(np.float32)
        vs = np.exp(rng.uniform(math.log(lo), math.log(hi), size=(L, hkv))).astype(np.float32)
        for which, sc, cache, scache in (("k", ks, k_cache, k_sc), ("v", vs, v_cache, v_sc)):
            z = rng.standard_normal((L, hkv, d), dtype=np.float32)
            if zmul is None:
                vals = z / sc[:, :, None]
            else:
                vals = z * np.float32(zmul)
            codes = _e4m3_codes(vals).numpy()  # [L, hkv, d]
            pad = P * block_size - L
            codes = np.concatenate([codes, np.full((pad, hkv, d), E4M3_NAN_CODE, np.uint8)], axis=0)
            scp = np.concatenate([sc, np.full((pad, hkv), np.nan, np.float32)], axis=0)
            cache[blocks] = codes.reshape(P, block_size, hkv, d).transpose(0, 2, 1, 3)
            scache[blocks] = scp.reshape(P, block_size, hkv).transpose(0, 2, 1)
            if unq:
                raw = np.concatenate([vals * sc[:, :, None], np.full((pad, hkv, d), np.nan, np.float32)], axis=0)
                unq[which][blocks] = raw.reshape(P, block_size, hkv, d).transpose(0, 2, 1, 3)
    case = DecodeCase(
        name=name,
        q=q,
        cu_q=torch.from_numpy(cu_q),
        seq_lens=torch.tensor(seq_lens, dtype=torch.int32),
        block_table=torch.from_numpy(table),
        k_cache=torch.from_numpy(k_cache),
        v_cache=torch.from_numpy(v_cache),
        k_scale=torch.from_numpy(k_sc),
        v_scale=torch.from_numpy(v_sc),
        scale=float(scale if scale is not None else 1.0 / math.sqrt(d)),
        segment_len=int(segment_len),
        k_unquant=torch.from_numpy(unq["k"]) if unq else None,
        v_unquant=torch.from_numpy(unq["v"]) if unq else None,
    )
    return _add_decode_features(rng, case, features, window)


def _add_decode_features(rng, case: DecodeCase, features: bool, window: int) -> DecodeCase:
    """Gates (paged cumulative G) and sink, drawn after everything else; see make_decode."""
    case.window = int(window)
    if not features:
        return case
    num_blocks, _, bs, _ = case.k_cache.shape
    hq = case.hq
    g_cache = np.full((num_blocks, hq, bs), np.nan, dtype=np.float32)
    table = case.block_table.numpy()
    for r, L in enumerate(case.seq_lens.tolist()):
        P = (L + bs - 1) // bs
        z = rng.normal(3.0, 1.0, size=(L, hq))
        g = -np.logaddexp(0.0, -z)  # logsigmoid
        G = np.cumsum(g, axis=0).astype(np.float32)  # [L, hq]
        Gp = np.concatenate([G, np.full((P * bs - L, hq), np.nan, np.float32)], axis=0)
        g_cache[table[r, :P]] = Gp.reshape(P, bs, hq).transpose(0, 2, 1)
    case.g_cache = torch.from_numpy(g_cache)
    case.sink = torch.from_numpy(rng.standard_normal(hq).astype(np.float32))
    return case


def _make_decode_variant(rng, seq_lens, q_lens, cu_q, q, table, pages, num_blocks, hkv, d, block_size, scale,
                         segment_len, name, kv_format, scale_mode) -> DecodeCase:
    """bf16 cache, or fp8 codes with one K and one V scale (see make_decode)."""
    R = len(seq_lens)
    if kv_format == "bf16":
        k_cache = np.full((num_blocks, hkv, block_size, d), np.nan, dtype=np.float32)
        v_cache = np.full((num_blocks, hkv, block_size, d), np.nan, dtype=np.float32)
        k_sc = v_sc = None
    else:
        k_cache = np.full((num_blocks, hkv, block_size, d), E4M3_NAN_CODE, dtype=np.uint8)
        v_cache = np.full((num_blocks, hkv, block_size, d), E4M3_NAN_CODE, dtype=np.uint8)
        lo, hi = 1.0 / 64, 20.0 / 64
        k_sc = np.exp(rng.uniform(math.log(lo), math.log(hi), size=1)).astype(np.float32)
        v_sc = np.exp(rng.uniform(math.log(lo), math.log(hi), size=1)).astype(np.float32)
    for r in range(R):
        L, P = seq_lens[r], pages[r]
        blocks = table[r, :P]
        for cache, sc in ((k_cache, k_sc), (v_cache, v_sc)):
            z = rng.standard_normal((L, hkv, d), dtype=np.float32)
            pad = P * block_size - L
            if kv_format == "bf16":
                vals = _bf16(z).float().numpy()
                vals = np.concatenate([vals, np.full((pad, hkv, d), np.nan, np.float32)], axis=0)
            else:
                vals = _e4m3_codes(z / sc[0]).numpy()
                vals = np.concatenate([vals, np.full((pad, hkv, d), E4M3_NAN_CODE, np.uint8)], axis=0)
            cache[blocks] = vals.reshape(P, block_size, hkv, d).transpose(0, 2, 1, 3)
    as_cache = (lambda a: torch.from_numpy(a).to(torch.bfloat16)) if kv_format == "bf16" else torch.from_numpy
    return DecodeCase(
        name=name,
        q=q,
        cu_q=torch.from_numpy(cu_q),
        seq_lens=torch.tensor(seq_lens, dtype=torch.int32),
        block_table=torch.from_numpy(table),
        k_cache=as_cache(k_cache),
        v_cache=as_cache(v_cache),
        k_scale=None if k_sc is None else torch.from_numpy(k_sc),
        v_scale=None if v_sc is None else torch.from_numpy(v_sc),
        scale=float(scale if scale is not None else 1.0 / math.sqrt(d)),
        segment_len=int(segment_len),
        kv_format=kv_format,
        scale_mode=scale_mode,
    )


def _c5a_lengths(seed: int, n: int = 64, max_len: int = 32768) -> list[int]:
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in rng.integers(1, max_len + 1, size=n)]


# 227K context = 227 * 1024 tokens; the three verify requests end 1, 2 and 4 tokens into a page.
CTX_227K = 227 * 1024

DECODE_CONFIGS = {
    # 64 requests x 1 query, context uniform in [1, 32768], Hq=64, Hkv=4, D=128, page 16.
    "paged_fp8_decode_64x1": dict(seq_lens=None, q_lens=[1] * 64, hq=64, hkv=4, d=128, seed=4),
    # Short-query (speculative verify) case: 3 requests x 4 tokens at 227K context.
    "paged_fp8_verify_3x4_227k": dict(seq_lens=[CTX_227K + 1, CTX_227K + 2, CTX_227K + 4], q_lens=[4, 4, 4], hq=64,
                                      hkv=4, d=128, seed=5),
    # Chunked prefill (a batch that is not all-decode): 4 requests, each a 1024-token chunk at
    # the end of its cached context (8K, 16K, 24K, 32K tokens), Hq=64, Hkv=4, D=128, page 16.
    "paged_fp8_chunked_prefill_4x1024": dict(seq_lens=[8192, 16384, 24576, 32768], q_lens=[1024] * 4, hq=64,
                                             hkv=4, d=128, seed=6),
}


def decode_config(name: str, scale_reading: str = "A", kv_format: str = "fp8",
                  scale_mode: str = "per_token", features: bool = False, window: int = 0) -> DecodeCase:
    cfg = dict(DECODE_CONFIGS[name])
    if cfg["seq_lens"] is None:
        cfg["seq_lens"] = _c5a_lengths(cfg["seed"] + 1000)
    return make_decode(name=name, scale_reading=scale_reading, kv_format=kv_format, scale_mode=scale_mode,
                       features=features, window=window, **cfg)
