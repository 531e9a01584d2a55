"""Host validation under random arguments (CPU only, nothing launched): the workspace
queries of every call accept or refuse any combination of counts, sizes, formats and flags
without crashing, refuse every negative or zero count, and size an accepted workspace in
whole 256-byte regions that grow with the number of requests.  Only the size queries run,
so no device memory is ever addressed."""
import ctypes

import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

FAKE = 0x10000
ints = st.one_of(st.integers(-4, 40), st.integers(-(1 << 31), (1 << 31) - 1), st.sampled_from([0, 1, 16, 64, 128, 2048]))


@pytest.fixture(scope="module")
def L():
    import gated_causal_softmax_gb300 as gcs

    return gcs.load()


@settings(max_examples=300, deadline=None)
@given(num_seqs=ints, total=ints, max_seqlen=ints, hq=ints, hkv=ints, dims=st.sampled_from(
    [(64, 64), (128, 128), (256, 256), (256, 512), (512, 512), (96, 96), (128, 256), (0, 0)]), window=ints,
       det=st.integers(-1, 2), gate=st.booleans(), sink=st.booleans())
def test_prefill_workspace_queries_never_crash(L, num_seqs, total, max_seqlen, hq, hkv, dims, window, det, gate, sink):
    import gated_causal_softmax_gb300 as gcs

    a = gcs.PrefillArgs(num_seqs=num_seqs, cu_seqlens=FAKE, total_tokens=total, max_seqlen=max_seqlen, hq=hq,
                        hkv=hkv, dqk=dims[0], dv=dims[1], scale=0.1, window=window, q=FAKE, k=FAKE, v=FAKE,
                        log_gate=FAKE if gate else None, sink=FAKE if sink else None, deterministic=det)
    fw = L.attn_fwd_workspace(ctypes.byref(a))
    bw = L.attn_bwd_workspace(ctypes.byref(a))
    assert fw % 256 == 0 and bw % 256 == 0
    valid = (num_seqs >= 1 and total >= 1 and max_seqlen >= 1 and hq >= 1 and hkv >= 1 and hq % hkv == 0
             and window >= 0 and det in (0, 1) and dims in ((64, 64), (128, 128), (256, 256), (256, 512), (512, 512))
             and total * hq * max(dims) <= (1 << 31) - 1)
    if not valid:
        assert fw == 0 and bw == 0
    else:
        assert bw > 0
        assert (fw > 0) == gate


@settings(max_examples=300, deadline=None)
@given(num_reqs=ints, total_q=ints, max_q_len=st.integers(-1, 6), max_seq_len=ints, max_blocks=ints,
       num_blocks=ints, hkv=st.sampled_from([-1, 0, 1, 2, 4]), group=st.sampled_from([4, 8, 16]),
       block=st.sampled_from([8, 16, 24, 128]),
       seg=st.sampled_from([-16, 0, 16, 100, 2048]), fmt=st.sampled_from([(0, 0), (0, 1), (1, 0), (2, 0), (0, 2)]),
       window=ints)
def test_decode_workspace_queries_never_crash(L, num_reqs, total_q, max_q_len, max_seq_len, max_blocks, num_blocks,
                                              hkv, group, block, seg, fmt, window):
    import gated_causal_softmax_gb300 as gcs

    kvf, mode = fmt
    scales = None if kvf == 1 else FAKE
    a = gcs.DecodeArgs(num_reqs=num_reqs, cu_q=FAKE, total_q=total_q, max_q_len=max_q_len, seq_lens=FAKE,
                       max_seq_len=max_seq_len, block_table=FAKE, max_blocks_per_req=max_blocks, k_cache=FAKE,
                       v_cache=FAKE, k_scale=scales, v_scale=scales, num_blocks=num_blocks, block_size=block,
                       hq=hkv * group, hkv=hkv, d=128, scale=0.1, segment_len=seg, q=FAKE, kv_format=kvf,
                       scale_mode=mode, window=window)
    dw = L.attn_decode_workspace(ctypes.byref(a))
    pw = L.attn_prefill_paged_workspace(ctypes.byref(a)) if seg != 0 else 0  # 0 asks the device for its SM count
    assert dw % 256 == 0 and pw % 256 == 0
    if min(num_reqs, total_q, max_q_len, max_seq_len, max_blocks, num_blocks, hkv) < 1 or window < 0:
        assert dw == 0 and pw == 0
    if group == 4 or block % 16 != 0:  # GQA groups of 16 or 8, whole 16-token pages
        assert dw == 0 and pw == 0
    if dw > 0 and num_reqs < (1 << 31) - 1:
        # one more request never needs less workspace
        a.num_reqs += 1
        assert L.attn_decode_workspace(ctypes.byref(a)) >= dw
