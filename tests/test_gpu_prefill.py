"""Layer-major prefill on the GPU: parity with the oracle on a small BF16 model over
several ragged chunks, chunk-size invariance, truncate + suffix == scratch prefill
(bit for bit), decode after prefill, error codes.  The full-width 8-layer,
4096-token prefill is checked in test_gpu_stack.py."""
import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_BF16, LazyOracleModel, gpu_model, kv_to_f64, rel_err, to_np

pytestmark = pytest.mark.gpu

# Two small BF16 shapes: the first takes the SIMT GEMMs (head_dim 64, 32 experts),
# the second the tensor-core GEMMs (every weight piece a multiple of 128 rows).
SMALL = synth.LAYER.with_(name="small_bf16", n_layers=2, hidden=512, n_heads=8, head_dim=64,
                          q_rank=128, kv_rank=64, window=16, n_experts=32, top_k=4,
                          expert_inter=128, vocab=1000, gain_sigma=0.1)
SMALL_TC = synth.LAYER.with_(name="small_bf16_tc", n_layers=2, hidden=512, n_heads=8, head_dim=128,
                             q_rank=256, kv_rank=128, window=16, n_experts=128, top_k=4,
                             expert_inter=128, vocab=1000, gain_sigma=0.1)


# The tcgen05 attention (head_dim 128, 64 or 128 heads): 128 heads (one token per
# 128-row block) with a 40-key window, and 64 heads (two tokens a block) with the
# full 128-key window.
SMALL_TCA128 = SMALL_TC.with_(name="small_bf16_tc_attn128", n_heads=128, window=40)
SMALL_TCA64 = SMALL_TC.with_(name="small_bf16_tc_attn64", n_heads=64, window=128)


# (shape, prefill_kernel): 0 the default GEMM form for the shape, 2 the tensor-core
# GEMMs with every activation as a BF16 hi/lo pair
@pytest.fixture(scope="module", params=[(SMALL, 0), (SMALL_TC, 0), (SMALL_TC, 2), (SMALL_TCA128, 0),
                                        (SMALL_TCA64, 0)],
                ids=["simt", "tensor_core", "tensor_core_hilo", "tensor_core_attn128",
                     "tensor_core_attn64"])
def small(request):
    import torch
    torch.cuda.init()
    shape, kernel = request.param
    return (gpu_model(shape, prefill_chunk=32, prefill_kernel=kernel), LazyOracleModel(shape).full(),
            shape)


def kv_np(sess, layer, n):
    k, v = sess.kv(layer)
    return to_np(k[:n]), to_np(v[:n])


def test_small_prefill_ragged_chunks_match_oracle(small):
    import torch
    import prefill_decode_layer_gb300 as pdl
    gm, om, SMALL = small
    toks = synth.host_tokens(100, SMALL.vocab, stream=21)   # chunks 32, 32, 32, 4
    sess = pdl.Session(gm, 160)
    assert sess.prefill(toks) == 0
    torch.cuda.synchronize()
    osess = oracle.OracleSession(om, 160)
    rc, ologits, ohidden = osess.prefill(toks, want_hidden=True)
    assert rc == 0
    assert rel_err(to_np(sess.logits()), ologits) <= TOL_BF16
    px = to_np(sess.debug("prefill_x", 4 * SMALL.hidden)).reshape(4, SMALL.hidden)
    assert rel_err(px, ohidden[96:100]) <= TOL_BF16
    for l in range(SMALL.n_layers):
        gk, gv = kv_np(sess, l, 100)
        ok, ov = oracle.kv_views(osess, l, 160)
        assert rel_err(gk, kv_to_f64(SMALL, ok[:100])) <= TOL_BF16
        assert rel_err(gv, kv_to_f64(SMALL, ov[:100])) <= TOL_BF16
    # decode after prefill
    for t in synth.host_tokens(3, SMALL.vocab, stream=22):
        assert sess.decode(int(t)) == 0
        rc, ologits, _ = osess.decode(int(t))
        torch.cuda.synchronize()
        assert rel_err(to_np(sess.logits()), ologits) <= TOL_BF16


def test_chunk_size_invariance_bitwise(small):
    import torch
    import prefill_decode_layer_gb300 as pdl
    gm, _, SMALL = small
    big = pdl.Model(SMALL, *gm._keep, prefill_chunk=0, prefill_kernel=gm.cfg.prefill_kernel)
    toks = synth.host_tokens(77, SMALL.vocab, stream=23)
    a = pdl.Session(gm, 128)
    b = pdl.Session(big, 128)
    assert a.prefill(toks) == 0 and b.prefill(toks) == 0
    torch.cuda.synchronize()
    assert torch.equal(a.logits(), b.logits())
    for l in range(SMALL.n_layers):
        assert torch.equal(a.kv(l)[0][:77], b.kv(l)[0][:77])
        assert torch.equal(a.kv(l)[1][:77], b.kv(l)[1][:77])


def test_truncate_then_suffix_equals_scratch_bitwise(small):
    import torch
    import prefill_decode_layer_gb300 as pdl
    gm, _, SMALL = small
    common = synth.host_tokens(70, SMALL.vocab, stream=24)
    live_tail = synth.host_tokens(20, SMALL.vocab, stream=25)
    new_tail = synth.host_tokens(9, SMALL.vocab, stream=26)
    new_tail[0] = (live_tail[0] + 1) % SMALL.vocab
    live = pdl.Session(gm, 128)
    assert live.prefill(np.concatenate([common, live_tail])) == 0
    for t in (5, 6):
        assert live.decode(t) == 0
    prompt = np.concatenate([common, new_tail])
    cp = live.common_prefix(prompt)
    assert cp == 70
    assert live.truncate(cp) == 0 and live.len == 70
    assert live.prefill(prompt[cp:]) == 0
    scratch = pdl.Session(gm, 128)
    assert scratch.prefill(prompt) == 0
    torch.cuda.synchronize()
    assert torch.equal(live.logits(), scratch.logits())
    for l in range(SMALL.n_layers):
        assert torch.equal(live.kv(l)[0][:79], scratch.kv(l)[0][:79])
        assert torch.equal(live.kv(l)[1][:79], scratch.kv(l)[1][:79])
    ws = torch.empty(pdl.sample_workspace_bytes(SMALL.vocab), dtype=torch.uint8, device="cuda")
    for _ in range(4):   # greedy continuation is identical
        a, _ = pdl.sample(live.logits(), 0.0, 1.0, None, ws)
        b, _ = pdl.sample(scratch.logits(), 0.0, 1.0, None, ws)
        assert a == b
        assert live.decode(a) == 0 and scratch.decode(b) == 0


def test_sync_and_rewrite_equal_scratch_bitwise(small):
    """ds4g_session_sync and ds4g_session_rewrite_from_common leave the session
    exactly as a scratch prefill of the prompt: K/V of every position and the
    logits, bit for bit, in each case the calls distinguish."""
    import torch
    import prefill_decode_layer_gb300 as pdl
    gm, _, SMALL = small
    hist = synth.host_tokens(90, SMALL.vocab, stream=27)
    fresh = synth.host_tokens(12, SMALL.vocab, stream=28)
    fresh[0] = (hist[60] + 1) % SMALL.vocab

    def same_as_scratch(sess, prompt):
        scratch = pdl.Session(gm, 128)
        assert scratch.prefill(prompt) == 0
        torch.cuda.synchronize()
        assert sess.len == len(prompt)
        assert torch.equal(sess.logits(), scratch.logits())
        for l in range(SMALL.n_layers):
            assert torch.equal(sess.kv(l)[0][:len(prompt)], scratch.kv(l)[0][:len(prompt)])
            assert torch.equal(sess.kv(l)[1][:len(prompt)], scratch.kv(l)[1][:len(prompt)])

    def live():
        s = pdl.Session(gm, 128)
        assert s.prefill(hist[:88]) == 0
        assert s.decode(int(hist[88])) == 0 and s.decode(int(hist[89])) == 0
        return s

    # a prompt that leaves the history after 60 tokens: the suffix only
    s = live()
    prompt = np.concatenate([hist[:60], fresh])
    assert s.sync(prompt) == (0, 12)
    same_as_scratch(s, prompt)
    # a prompt the history holds as a prefix, then the same prompt again: the last
    # token runs again, since its logits were not kept
    s = live()
    assert s.sync(hist[:50]) == (0, 1)
    same_as_scratch(s, hist[:50])
    assert s.sync(hist[:50]) == (0, 1)
    same_as_scratch(s, hist[:50])
    # empty prompt; errors leave the session as it was
    assert s.sync([]) == (0, 0) and s.len == 0
    s = live()
    bad = np.concatenate([hist[:30], [SMALL.vocab]])
    assert s.sync(bad)[0] == pdl.ds4g.ETOKEN and s.len == 90
    assert s.sync(synth.host_tokens(128, SMALL.vocab, stream=29))[0] == pdl.ds4g.ECONTEXT and s.len == 90

    # rewrite from the caller's common prefix, or from any shorter one
    canonical = np.concatenate([hist[:60], fresh[:10]])
    for common in (60, 41):
        s = live()
        assert s.common_prefix(canonical) == 60
        assert s.rewrite_from_common(canonical, common) == 0
        same_as_scratch(s, canonical)
    s = live()
    assert s.rewrite_from_common(canonical, 61) == pdl.ds4g.EINVAL and s.len == 90
    assert s.rewrite_from_common(hist, 90) == 0 and s.len == 90     # already the prompt
    assert s.rewrite_from_common(hist[:70], 70) == 0 and s.len == 70  # cut, nothing to run


def test_checkpoint_save_load_then_suffix_equals_scratch(small):
    """A checkpoint restores the K/V and the history bit for bit; the suffix
    prefilled after it gives the scratch prefill's K/V and logits.  Damaged or
    short buffers and a context that is too small leave the session as it was."""
    import torch
    import prefill_decode_layer_gb300 as pdl
    gm, _, SMALL = small
    hist = synth.host_tokens(72, SMALL.vocab, stream=30)
    suffix = synth.host_tokens(8, SMALL.vocab, stream=31)
    a = pdl.Session(gm, 128)
    assert a.prefill(hist) == 0   # (decode steps would write K/V rows a prefill does not reproduce bitwise)
    buf = bytearray(a.checkpoint_bytes())
    assert a.save(bytearray(len(buf) - 1)) == pdl.ds4g.ESIZE
    assert a.save(buf) == 0
    b = pdl.Session(gm, 128)
    assert b.load(buf) == 0 and b.len == 72
    assert b.common_prefix(hist) == 72
    torch.cuda.synchronize()
    for l in range(SMALL.n_layers):
        assert torch.equal(a.kv(l)[0][:72], b.kv(l)[0][:72])
        assert torch.equal(a.kv(l)[1][:72], b.kv(l)[1][:72])
    prompt = np.concatenate([hist, suffix])
    assert b.sync(prompt) == (0, 8)
    scratch = pdl.Session(gm, 128)
    assert scratch.prefill(prompt) == 0
    torch.cuda.synchronize()
    assert torch.equal(b.logits(), scratch.logits())
    for l in range(SMALL.n_layers):
        assert torch.equal(b.kv(l)[0][:80], scratch.kv(l)[0][:80])
        assert torch.equal(b.kv(l)[1][:80], scratch.kv(l)[1][:80])
    c = pdl.Session(gm, 128)
    assert c.prefill(suffix) == 0
    assert c.load(buf[:len(buf) - 16]) == pdl.ds4g.ESIZE and c.len == 8
    bad = bytearray(buf)
    bad[0] ^= 1                       # magic
    assert c.load(bad) == pdl.ds4g.EINVAL and c.len == 8
    bad = bytearray(buf)
    bad[32] ^= 1                      # configuration digest
    assert c.load(bad) == pdl.ds4g.EINVAL and c.len == 8
    small_ctx = pdl.Session(gm, 72)
    assert small_ctx.load(buf) == pdl.ds4g.ECONTEXT and small_ctx.len == 0


def test_session_errors(small):
    import prefill_decode_layer_gb300 as pdl
    gm, _, SMALL = small
    s = pdl.Session(gm, 16)
    assert s.prefill([1, 2, SMALL.vocab]) == pdl.ds4g.ETOKEN and s.len == 0
    assert s.prefill(list(range(16))) == pdl.ds4g.ECONTEXT and s.len == 0
    assert s.prefill([]) == 0 and s.len == 0
    assert s.prefill(list(range(15))) == 0 and s.len == 15
    assert s.decode(1) == pdl.ds4g.ECONTEXT
    assert s.decode(-1) == pdl.ds4g.ETOKEN
    assert s.truncate(16) == pdl.ds4g.EINVAL and s.truncate(15) == 0 and s.len == 15
    assert s.truncate(0) == 0 and s.len == 0


def test_tensor_core_and_simt_prefill_agree():
    """The two GEMM forms of the prefill on the same BF16 model: hidden states and
    KV within the BF16 tolerance (their activations are rounded differently)."""
    import torch
    import prefill_decode_layer_gb300 as pdl
    tcm = gpu_model(SMALL_TC, prefill_chunk=64)
    simt = pdl.Model(SMALL_TC, *tcm._keep, prefill_chunk=64, prefill_kernel=pdl.ds4g.PREFILL_SIMT)
    toks = synth.host_tokens(150, SMALL_TC.vocab, stream=27)
    a, b = pdl.Session(tcm, 200), pdl.Session(simt, 200)
    assert a.prefill(toks) == 0 and b.prefill(toks) == 0
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert rel_err(to_np(a.logits()), to_np(b.logits())) <= TOL_BF16
    for l in range(SMALL_TC.n_layers):
        assert rel_err(to_np(a.kv(l)[0][:150]), to_np(b.kv(l)[0][:150])) <= TOL_BF16
        assert rel_err(to_np(a.kv(l)[1][:150]), to_np(b.kv(l)[1][:150])) <= TOL_BF16
