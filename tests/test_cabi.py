"""Host-side tests of the C ABI (no GPU needed): the library builds for sm_103a, loads,
exports every function include/gcs_attn.h declares, and rejects bad arguments on the host
before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gcs_attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\*?\s*([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


@pytest.fixture(scope="module")
def L():
    import gated_causal_softmax_gb300 as gcs

    return gcs.load()


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("attn_fwd", "attn_bwd", "attn_decode_paged", "attn_fwd_workspace", "attn_bwd_workspace",
              "attn_decode_workspace", "gcs_get_device_status", "gcs_status_str", "gcs_version"):
        assert n in names, n


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), f"missing export {n}"
    assert L.gcs_version().startswith(b"gcs_attn")
    assert L.gcs_status_str(2) == b"unsupported shape, dtype or layout"


FAKE = 0x10000  # 16-B aligned, never dereferenced by host validation


def at(k):
    """A fake 16-B aligned address k GiB above 64 GiB: ranges there never meet FAKE's."""
    return (1 << 36) + k * (1 << 30)


OUT, OUT2 = at(0), at(1)  # fake output buffers apart from the inputs


def prefill(**over):
    import gated_causal_softmax_gb300 as gcs

    kw = dict(num_seqs=1, cu_seqlens=FAKE, total_tokens=256, max_seqlen=256, hq=4, hkv=2, dqk=128, dv=128,
              scale=0.088, window=0, q=FAKE, k=FAKE, v=FAKE, log_gate=None, sink=None)
    kw.update(over)
    return gcs.PrefillArgs(**kw)


def decode(**over):
    import gated_causal_softmax_gb300 as gcs

    kw = dict(num_reqs=2, cu_q=FAKE, total_q=2, max_q_len=1, seq_lens=FAKE, max_seq_len=4096, block_table=FAKE,
              max_blocks_per_req=256, k_cache=FAKE, v_cache=FAKE, k_scale=FAKE, v_scale=FAKE, num_blocks=600,
              block_size=16, hq=64, hkv=4, d=128, scale=0.088, segment_len=2048, q=FAKE)
    kw.update(over)
    return gcs.DecodeArgs(**kw)


def test_prefill_validation_on_host(L):
    b = ctypes.byref
    fwd = lambda a: L.attn_fwd(b(a), FAKE, FAKE, FAKE, 1 << 30, None)
    assert fwd(prefill(hq=3, hkv=2)) == 1  # hq % hkv
    assert fwd(prefill(q=None)) == 1
    assert fwd(prefill(q=FAKE + 2)) == 1  # misaligned
    assert fwd(prefill(window=-1)) == 1
    assert fwd(prefill(deterministic=2)) == 1
    assert fwd(prefill(scale=float("nan"))) == 1
    assert fwd(prefill(dqk=96, dv=96)) == 2  # not a compiled head dim
    assert fwd(prefill(dqk=128, dv=256)) == 2
    assert L.attn_fwd(b(prefill()), None, FAKE, FAKE, 0, None) == 1  # no output
    # gated forward needs a workspace
    assert L.attn_fwd(b(prefill(log_gate=FAKE)), OUT, OUT2, None, 0, None) == 3
    bwd = lambda a, **k: L.attn_bwd(b(a), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, k.get("dg"), k.get("ds"), FAKE,
                                    1 << 40, None)
    assert bwd(prefill(log_gate=FAKE)) == 1  # dlog_gate must be given iff log_gate is
    assert bwd(prefill(sink=FAKE)) == 1
    assert bwd(prefill(), dg=FAKE) == 1


def test_workspace_sizes_on_host(L):
    b = ctypes.byref
    assert L.attn_fwd_workspace(b(prefill())) == 0
    assert L.attn_fwd_workspace(b(prefill(log_gate=FAKE))) == 4 * 4 * 256
    ws = L.attn_bwd_workspace(b(prefill(log_gate=FAKE, sink=FAKE, deterministic=1)))
    # G^T, delta, dS row sums, dS column sums, packed per-tile vectors; the single pass at head
    # dim 128 and wider heads on the reduce-add route add the fp32 dQ accumulator, the
    # deterministic routes do not
    n_qtiles = 256 // 64 + 1
    assert ws == 4 * (4 * 256) * 4 + 4 * n_qtiles * 128 * 4
    assert L.attn_bwd_workspace(b(prefill(log_gate=FAKE, sink=FAKE))) == ws + 256 * 4 * 128 * 4
    assert L.attn_bwd_workspace(b(prefill(log_gate=FAKE, sink=FAKE, dqk=64, dv=64))) == ws  # two passes at 64
    ws_wide = L.attn_bwd_workspace(b(prefill(log_gate=FAKE, sink=FAKE, dqk=256, dv=512)))
    assert ws_wide == 4 * (4 * 256) * 4 + 256 * 4 * 256 * 4 + 4 * n_qtiles * 128 * 4
    ws_det = L.attn_bwd_workspace(b(prefill(log_gate=FAKE, sink=FAKE, dqk=256, dv=512, deterministic=1)))
    assert ws_det == ws
    # (512, 512) takes the dQ pass either way: it is the faster route there
    assert L.attn_bwd_workspace(b(prefill(log_gate=FAKE, sink=FAKE, dqk=512, dv=512))) == ws
    units, rows = 2 * 2 * 4, 16
    assert L.attn_decode_workspace(b(decode())) == units * rows * 128 * 4 + units * rows * 2 * 4
    assert L.attn_decode_workspace(b(decode(max_q_len=5))) == 0


def test_decode_validation_on_host(L):
    b = ctypes.byref
    dec = lambda a: L.attn_decode_paged(b(a), FAKE, FAKE, 1 << 40, None)
    # per-token scales on a prefill shape are rejected
    assert dec(decode(max_q_len=5)) == 2
    assert dec(decode(block_size=24)) == 2  # not whole 16-token pages
    assert dec(decode(block_size=48, max_blocks_per_req=128)) == 2  # 3 pages: not a power of two
    assert L.attn_decode_workspace(b(decode(block_size=128, max_blocks_per_req=32))) > 0  # 128-token blocks
    assert dec(decode(d=64)) == 2
    assert dec(decode(hq=48)) == 2  # GQA group must be 16 or 8
    assert L.attn_decode_workspace(b(decode(hq=32))) > 0  # group of 8
    assert dec(decode(segment_len=2040)) == 2
    assert dec(decode(k_scale=None)) == 1
    assert dec(decode(max_blocks_per_req=10)) == 1  # table too short for max_seq_len
    assert L.attn_decode_paged(b(decode()), OUT, None, 0, None) == 3
    assert L.attn_decode_paged(b(decode()), FAKE + 8, FAKE, 1 << 40, None) == 1
    # cache formats and scale modes: a bf16 cache takes no scales; per-tensor scales need
    # 4-byte alignment; unknown formats or modes are invalid
    assert dec(decode(kv_format=1)) == 1
    assert dec(decode(kv_format=1, k_scale=None, v_scale=None, scale_mode=1)) == 1
    assert L.attn_decode_workspace(b(decode(kv_format=1, k_scale=None, v_scale=None))) > 0
    assert dec(decode(scale_mode=1, k_scale=FAKE + 2)) == 1
    assert L.attn_decode_workspace(b(decode(scale_mode=1, k_scale=FAKE + 4, v_scale=FAKE + 8))) > 0
    assert dec(decode(scale_mode=2)) == 1
    assert dec(decode(kv_format=2)) == 1
    # decoding features: a negative window, a misaligned gate array or sink are invalid
    assert dec(decode(window=-1)) == 1
    assert dec(decode(g_cache=FAKE + 4)) == 1
    assert dec(decode(sink=FAKE + 2)) == 1
    assert L.attn_decode_workspace(b(decode(g_cache=FAKE, sink=FAKE + 4, window=1024))) > 0


def test_prefill_paged_validation_and_workspace_on_host(L):
    b = ctypes.byref
    pp = lambda a, ws=1 << 40: L.attn_prefill_paged(b(a), OUT, FAKE, ws, None)
    # any q_len is accepted; the workspace holds the split-K partials of the chosen segments
    a = decode(max_q_len=64, segment_len=256)
    units, rows = 2 * (4096 // 256) * 4, 64 * 16
    assert L.attn_prefill_paged_workspace(b(a)) == units * rows * 128 * 4 + units * rows * 2 * 4
    # one segment per request: the kernel writes the output itself and needs no workspace
    assert L.attn_prefill_paged_workspace(b(decode(max_q_len=64, segment_len=4096))) == 0
    assert pp(a, ws=0) == 3
    assert pp(decode(max_q_len=64, segment_len=200)) == 2  # not a whole number of 128-key tiles
    assert pp(decode(max_q_len=64, kv_format=1, k_scale=None, v_scale=None)) == 2  # fp8 only
    assert pp(decode(max_q_len=5000)) == 1  # more query rows than cached tokens
    assert pp(decode(max_q_len=64, window=-1)) == 1
    assert pp(decode(max_q_len=64, hq=48)) == 2
    assert pp(decode(max_q_len=64, segment_len=-128)) == 1
    assert L.attn_prefill_paged(b(decode(max_q_len=64)), FAKE + 8, FAKE, 1 << 40, None) == 1


def test_device_checks_mode_and_workspace_on_host(L):
    """Checked mode: the switch takes 0 or 1, and while it is on every workspace query adds
    the checked copy of cu_seqlens / cu_q ((n + 1) int32 rounded up to 256 B) at its end.
    The host validation of the stand-alone checks runs before any CUDA call."""
    b = ctypes.byref
    assert L.gcs_set_device_checks(2) == 1
    assert L.gcs_get_device_checks() == 0
    base = dict(fwd=L.attn_fwd_workspace(b(prefill())), fwd_g=L.attn_fwd_workspace(b(prefill(log_gate=FAKE))),
                bwd=L.attn_bwd_workspace(b(prefill(num_seqs=300, log_gate=FAKE))),
                dec=L.attn_decode_workspace(b(decode())),
                pp=L.attn_prefill_paged_workspace(b(decode(max_q_len=64, segment_len=256))),
                pp1=L.attn_prefill_paged_workspace(b(decode(max_q_len=64, segment_len=4096))))
    assert L.gcs_set_device_checks(1) == 0
    try:
        assert L.gcs_get_device_checks() == 1
        assert L.attn_fwd_workspace(b(prefill())) == base["fwd"] + 256
        assert L.attn_fwd_workspace(b(prefill(log_gate=FAKE))) == base["fwd_g"] + 256
        assert L.attn_bwd_workspace(b(prefill(num_seqs=300, log_gate=FAKE))) == base["bwd"] + 1280  # 301 x 4 B
        assert L.attn_decode_workspace(b(decode())) == base["dec"] + 256
        assert L.attn_prefill_paged_workspace(b(decode(max_q_len=64, segment_len=256))) == base["pp"] + 256
        # one segment per request: the copy alone, so the call now needs a workspace
        assert base["pp1"] == 0
        assert L.attn_prefill_paged_workspace(b(decode(max_q_len=64, segment_len=4096))) == 256
        assert L.attn_prefill_paged(b(decode(max_q_len=64, segment_len=4096)), OUT, None, 0, None) == 3
        assert L.attn_fwd(b(prefill()), OUT, OUT2, None, 0, None) == 3
    finally:
        assert L.gcs_set_device_checks(0) == 0
    assert L.attn_fwd_workspace(b(prefill())) == base["fwd"]
    # the stand-alone checks validate their arguments on the host first
    assert L.gcs_check_prefill_inputs(b(prefill(hq=3, hkv=2)), None) == 1
    assert L.gcs_check_prefill_inputs(b(prefill(dqk=96, dv=96)), None) == 2
    assert L.gcs_check_paged_inputs(b(decode(block_size=24)), None) == 2
    assert L.gcs_check_paged_inputs(b(decode(cu_q=None)), None) == 1


def test_size_limits_on_host(L):
    """Sizes the kernels' 32-bit TMA coordinates and element offsets cannot address are
    refused before any launch: a prefill tensor of 2^31 or more elements, and an fp8 cache of
    2^31 or more rows (num_blocks x hkv x block_size); just below both limits is accepted."""
    b = ctypes.byref
    fwd = lambda a: L.attn_fwd(b(a), FAKE, FAKE, FAKE, 1 << 40, None)
    # hq x dqk = 4 x 128 = 512 elements per token: 2^22 tokens reach 2^31 elements
    assert fwd(prefill(total_tokens=1 << 22, max_seqlen=1 << 22)) == 2
    assert L.attn_fwd_workspace(b(prefill(total_tokens=(1 << 22) - 1, max_seqlen=1 << 20))) == 0
    assert L.attn_bwd_workspace(b(prefill(total_tokens=(1 << 22) - 1, max_seqlen=1 << 20))) > 0
    # the larger of dqk and dv counts: dv = 512 with 2^20 tokens and hq = 4 is 2^31 elements
    assert fwd(prefill(total_tokens=1 << 20, max_seqlen=1 << 20, dqk=256, dv=512)) == 2
    # the fp8 pages are fetched by 4-D tensor copies (block coordinate 32-bit), a bf16 cache with
    # 64-bit addressing: 2^25 blocks (2^31 rows of 128 B) are accepted either way
    assert L.attn_decode_workspace(b(decode(num_blocks=1 << 25))) > 0
    assert L.attn_decode_workspace(b(decode(num_blocks=1 << 25, kv_format=1, k_scale=None, v_scale=None))) > 0
    # the table-length check multiplies in 64 bits: (2^28 + 1) x 16 would wrap a 32-bit int to
    # 16 tokens, below max_seq_len, and the valid shape would be refused
    assert L.attn_decode_workspace(b(decode(max_blocks_per_req=(1 << 28) + 1))) > 0
    assert L.attn_decode_workspace(b(decode(max_blocks_per_req=(1 << 31) - 1))) > 0
    assert L.attn_decode_workspace(b(decode(max_blocks_per_req=255))) == 0


def test_degenerate_shapes_on_host(L):
    """Zero or negative counts are invalid arguments; one-token and one-request shapes are
    accepted (their workspace is sized)."""
    b = ctypes.byref
    for bad in (dict(num_seqs=0), dict(total_tokens=0), dict(max_seqlen=0), dict(hq=0), dict(hkv=0)):
        assert L.attn_fwd(b(prefill(**bad)), FAKE, FAKE, FAKE, 1 << 40, None) == 1, bad
        assert L.attn_fwd_workspace(b(prefill(**bad))) == 0, bad
    assert L.attn_bwd_workspace(b(prefill(num_seqs=1, total_tokens=1, max_seqlen=1))) > 0
    for bad in (dict(num_reqs=0), dict(total_q=0), dict(max_q_len=0), dict(max_seq_len=0), dict(num_blocks=0),
                dict(max_blocks_per_req=0), dict(segment_len=0)):
        assert L.attn_decode_paged(b(decode(**bad)), FAKE, FAKE, 1 << 40, None) == 1, bad
    one = decode(num_reqs=1, total_q=1, max_seq_len=1, max_blocks_per_req=1)
    units, rows = 1 * 1 * 4, 16  # one request, one segment, four kv heads
    assert L.attn_decode_workspace(b(one)) == units * rows * 128 * 4 + units * rows * 2 * 4


def test_outputs_overlapping_inputs_are_rejected_on_host(L):
    """An output whose byte range meets an input's or another output's is an invalid
    argument; adjacent ranges are fine.  Accepted calls stop at the missing workspace (3),
    so nothing is launched either way."""
    b = ctypes.byref
    a = prefill(log_gate=FAKE, sink=FAKE)  # inputs may share memory with each other
    qbytes = 256 * 4 * 128 * 2  # q [256, 4, 128] bf16, the largest input
    fwd = lambda o, lse: L.attn_fwd(b(a), o, lse, None, 0, None)
    assert fwd(FAKE, OUT) == 1  # o on q
    assert fwd(FAKE + qbytes - 16, OUT) == 1  # o's first bytes on q's last
    assert fwd(FAKE + qbytes, OUT) == 3  # adjacent
    assert fwd(OUT, OUT + 16) == 1  # lse inside o
    assert fwd(OUT, OUT + 256 * 4 * 128 * 2) == 3  # lse right after o
    bwd = lambda dq, dk, dv, dg, ds, dout=at(5): L.attn_bwd(b(a), at(3), at(4), dout, dq, dk, dv, dg, ds, None, 0,
                                                         None)
    outs = [at(6), at(7), at(8), at(9), at(10)]
    assert bwd(*outs) == 3
    for i in range(5):
        bad = list(outs)
        bad[i] = FAKE  # each output on the inputs
        assert bwd(*bad) == 1, i
    assert bwd(at(6), at(6) + 64, at(8), at(9), at(10)) == 1  # dk inside dq
    assert bwd(*outs, dout=at(8) + 1024) == 1  # dv on dout
    dec = lambda out, **over: L.attn_decode_paged(b(decode(**over)), out, None, 0, None)
    assert dec(OUT) == 3
    assert dec(FAKE) == 1  # out on every input
    assert dec(OUT, block_table=OUT + 32) == 1
    assert dec(OUT, g_cache=OUT2, sink=OUT + 4096) == 1
    assert dec(OUT, g_cache=OUT2, sink=OUT2 + 600 * 64 * 16 * 4) == 3  # sink right after g_cache, apart from out
    pp = lambda out, **over: L.attn_prefill_paged(b(decode(max_q_len=64, segment_len=256, **over)), out, None, 0,
                                                  None)
    assert pp(OUT) == 3
    assert pp(OUT, k_scale=OUT + 512) == 1


def test_strides_on_host(L):
    """Element strides (token, head) of the [tokens, heads, dim] tensors and (block, kv head,
    slot) of the paged caches: token-major layouts without overlap on the 16-byte granule are
    accepted (the calls then stop at the missing workspace, 3); overlapping heads, a token
    stride below the heads' span, strides off the granule and caches whose slots and heads
    meet are refused (2), negative strides are invalid (1).  Outputs that interleave with each
    other inside one fused buffer without sharing bytes are accepted; a shift that makes two
    of them meet is refused."""
    import gated_causal_softmax_gb300 as gcs

    b = ctypes.byref
    S = gcs.Strides
    fused = (4 + 2 * 2) * 128  # [tokens, (hq + 2 hkv) * d] with hq 4, hkv 2, d 128
    fwd = lambda a: L.attn_fwd(b(a), OUT, OUT2, None, 0, None)
    g = dict(log_gate=FAKE)  # a gated forward needs a workspace, so accepted calls return 3
    assert fwd(prefill(q_stride=S(fused, 128), k_stride=S(fused, 128), v_stride=S(fused, 128), **g)) == 3
    assert fwd(prefill(q_stride=S(fused, 136), **g)) == 3  # padded heads
    assert fwd(prefill(q_stride=S(fused, 120), **g)) == 2  # heads overlap
    assert fwd(prefill(q_stride=S(3 * 128, 128), **g)) == 2  # token stride below 4 heads
    assert fwd(prefill(q_stride=S(fused + 4, 128), **g)) == 2  # off the 16-byte granule
    assert fwd(prefill(q_stride=S(-8, 128), **g)) == 1
    assert fwd(prefill(o_stride=S(fused, 264), **g)) == 2  # 4 heads of 264 exceed the token stride
    assert fwd(prefill(o_stride=S(8 * 128, 256), **g)) == 3  # every other head slot
    # dq, dk, dv as interleaved views of one fused gradient buffer: accepted
    a = prefill(log_gate=FAKE, sink=FAKE, dq_stride=S(fused, 128), dk_stride=S(fused, 128),
                dv_stride=S(fused, 128))
    base = OUT
    dq, dk, dv = base, base + 4 * 128 * 2, base + 6 * 128 * 2
    bwd = lambda dq, dk, dv: L.attn_bwd(b(a), at(3), at(4), at(5), dq, dk, dv, at(9), at(10), None, 0, None)
    assert bwd(dq, dk, dv) == 3
    assert bwd(dq, dk - 16, dv) == 1  # dk's first head meets dq's last
    assert bwd(dq, dk, dv + 8 * 128 * 2 * 256) == 3  # dv in another buffer
    assert bwd(dq, dq + fused * 2, dv) == 1  # dk one token later in dq's own slots
    # o given to the backward as a strided input
    a2 = prefill(log_gate=FAKE, sink=FAKE, o_stride=S(fused, 128), do_stride=S(fused, 136))
    assert L.attn_bwd_workspace(b(a2)) == L.attn_bwd_workspace(b(prefill(log_gate=FAKE, sink=FAKE)))
    # paged caches
    dws = L.attn_decode_workspace(b(decode()))
    vllm = dict(kv_stride_block=16 * 4 * 128, kv_stride_head=128, kv_stride_slot=4 * 128)
    assert L.attn_decode_workspace(b(decode(**vllm))) == dws
    assert L.attn_decode_workspace(b(decode(kv_format=1, k_scale=None, v_scale=None, **vllm))) == dws
    assert L.attn_decode_paged(b(decode(**vllm)), OUT, None, 0, None) == 3
    bad = [dict(vllm, kv_stride_slot=2 * 128),  # slots meet the other heads' rows
           dict(vllm, kv_stride_block=16 * 4 * 128 - 16),  # blocks overlap
           dict(vllm, kv_stride_slot=4 * 128 + 8),  # off the granule (fp8: bytes)
           dict(kv_stride_block=16 * 4 * 128, kv_stride_head=16 * 64, kv_stride_slot=128)]  # heads meet
    for over in bad:
        assert L.attn_decode_paged(b(decode(**over)), OUT, None, 0, None) == 2, over
    assert L.attn_decode_paged(b(decode(kv_stride_block=-1, kv_stride_head=128, kv_stride_slot=512)), OUT, None, 0,
                               None) == 1
    # q and out of the paged calls
    assert L.attn_decode_paged(b(decode(q_stride=S(64 * 128 + 256, 128))), OUT, None, 0, None) == 3
    assert L.attn_decode_paged(b(decode(out_stride=S(64 * 128, 64))), OUT, None, 0, None) == 2
    assert L.attn_prefill_paged(b(decode(max_q_len=64, segment_len=256, **vllm)), OUT, None, 0, None) == 3
