"""The bench's algorithmic work units (CPU only), the numerators of every rate and roofline
it reports: visible-pair counts against brute force and against the pair counts of the
prefill workloads, the FLOP formulas, and the decode byte model against a per-field sum."""
import itertools
import random

import bench


def brute_pairs(T, W):
    return sum(1 for i, j in itertools.product(range(T), repeat=2) if j <= i and (W == 0 or i - j < W))


def test_pair_counts_match_brute_force():
    rng = random.Random(5)
    for _ in range(60):
        lens = [rng.randint(0, 40) for _ in range(rng.randint(1, 4))]
        W = rng.choice([0, 1, 2, 7, 39, 40, 41, 100])
        hq = rng.randint(1, 3)
        assert bench.prefill_pairs(lens, hq, W) == hq * sum(brute_pairs(T, W) for T in lens), (lens, W)


def test_pair_counts_of_the_prefill_workloads():
    # packed 1000/3000/4192 with 32 query heads, full causal
    assert bench.prefill_pairs([1000, 3000, 4192], 32) == 441_296_896
    # two 4096-token sequences, 16 query heads, window 1024
    assert bench.prefill_pairs([4096, 4096], 16, 1024) == 117_456_896
    # one 128-token sequence, 2 heads
    assert bench.prefill_pairs([128], 2) == 16_512
    fwd, bwd = bench.prefill_flops([1000, 3000, 4192], 32, 128, 128)
    assert fwd == 2 * 256 * 441_296_896 and bwd == 2 * (3 * 128 + 2 * 128) * 441_296_896
    assert round(fwd / 1e9, 1) == 225.9 and round(bwd / 1e9, 1) == 564.9


def test_paged_chunk_flops_match_brute_force():
    rng = random.Random(6)
    for _ in range(40):
        L = [rng.randint(1, 60) for _ in range(rng.randint(1, 3))]
        ql = [rng.randint(1, x) for x in L]
        W = rng.choice([0, 1, 5, 30])
        pairs = 0
        for Lr, qr in zip(L, ql):
            for t in range(qr):
                pos = Lr - qr + t
                pairs += sum(1 for j in range(Lr) if j <= pos and (W == 0 or pos - j < W))
        assert bench.paged_chunk_flops(L, ql, 16, 128, W) == 4 * 128 * pairs * 16


def test_decode_byte_model():
    seq, ql, hq, hkv, d, bs = [1, 16, 17, 1000], [1, 1, 2, 4], 64, 4, 128, 16
    tokens, pages = sum(seq), sum((L + bs - 1) // bs for L in seq)
    q_out = 2 * sum(ql) * hq * d * 2
    fixed = q_out + 4 * pages + 4 * len(seq)
    # fp8 per token: K and V codes (128 B each) and two fp32 scales = 264 B per (token, kv head)
    assert bench.decode_bytes(seq, ql, hq, hkv, d, bs) == tokens * hkv * 264 + fixed
    # fp8 per tensor: the codes only; bf16: 512 B
    assert bench.decode_bytes(seq, ql, hq, hkv, d, bs, "fp8", "per_tensor") == tokens * hkv * 256 + fixed
    assert bench.decode_bytes(seq, ql, hq, hkv, d, bs, "bf16") == tokens * hkv * 512 + fixed
    # gates: one fp32 G per query head of the group (16) = 64 B more, 328 B in all
    assert bench.decode_bytes(seq, ql, hq, hkv, d, bs, gates=True) == tokens * hkv * 328 + fixed


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(10.0, 4, 2.0) == 20.0
