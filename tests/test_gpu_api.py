"""The one-call forms of the decode loop against the separate calls they combine:
ds4g_decode_layers_host (decode + the hidden state in host memory) and
ds4g_decode_sample (decode with the lm_head + the next token's draw), bit for bit,
with their error cases leaving the session unchanged."""
import numpy as np
import pytest

import synth
from helpers import gpu_model

pytestmark = pytest.mark.gpu

SHAPE = synth.LAYER.with_(name="api_small", n_layers=2, hidden=512, n_heads=8, head_dim=128,
                          q_rank=256, kv_rank=128, window=16, n_experts=128, top_k=4,
                          expert_inter=128, vocab=1000, gain_sigma=0.1)


@pytest.fixture(scope="module")
def model():
    import torch
    torch.cuda.init()
    return gpu_model(SHAPE)


def test_decode_layers_host_equals_decode_layers(model):
    import torch
    import prefill_decode_layer_gb300 as pdl
    prompt = synth.host_tokens(40, SHAPE.vocab, stream=81)
    a, b = pdl.Session(model, 64), pdl.Session(model, 64)
    assert a.prefill(prompt) == 0 and b.prefill(prompt) == 0
    # pinned memory (written by the kernel through its device view) and pageable
    # memory (copied) take the two routes of the call
    pinned = torch.empty(SHAPE.hidden, dtype=torch.float32, pin_memory=True)
    pageable = torch.empty(SHAPE.hidden, dtype=torch.float32)
    for i, t in enumerate(synth.host_tokens(6, SHAPE.vocab, stream=82)):
        host = pinned if i % 2 == 0 else pageable
        host.fill_(float("nan"))
        assert a.decode_layers(int(t)) == 0
        assert b.decode_layers_host(int(t), host) == 0
        assert torch.equal(b.hidden().cpu(), host)   # complete when the call returns
        torch.cuda.synchronize()
        assert torch.equal(a.hidden().cpu(), host)
    assert a.len == b.len == 46
    for l in range(SHAPE.n_layers):
        for x, y in zip(a.kv(l), b.kv(l)):
            assert torch.equal(x[:45], y[:45])
    # errors: a token out of range leaves the session as it was; NULL host buffer
    assert b.decode_layers_host(SHAPE.vocab, pinned) == pdl.ds4g.ETOKEN and b.len == 46
    assert pdl.ds4g.lib().ds4g_decode_layers_host(b.ptr, 1, None) == pdl.ds4g.EINVAL and b.len == 46


@pytest.mark.parametrize("temperature,top_p", [(0.0, 1.0), (0.7, 0.95), (1.0, 1.0)])
def test_decode_sample_equals_decode_then_sample(model, temperature, top_p):
    import torch
    import prefill_decode_layer_gb300 as pdl
    prompt = synth.host_tokens(30, SHAPE.vocab, stream=83)
    a, b = pdl.Session(model, 80), pdl.Session(model, 80)
    assert a.prefill(prompt) == 0 and b.prefill(prompt) == 0
    ws_a = torch.empty(pdl.sample_workspace_bytes(SHAPE.vocab), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty_like(ws_a)
    sa = sb = 0x9E3779B97F4A7C15
    ta, sa = pdl.sample(a.logits(), temperature, top_p, sa, ws_a)
    tb, sb = pdl.sample(b.logits(), temperature, top_p, sb, ws_b)
    assert ta == tb
    for _ in range(12):
        assert a.decode(ta) == 0
        ta, sa = pdl.sample(a.logits(), temperature, top_p, sa, ws_a)
        tb, sb = b.decode_sample(tb, temperature, top_p, sb, ws_b)
        assert tb >= 0 and ta == tb and sa == sb
        assert torch.equal(a.logits(), b.logits())
    assert a.len == b.len == 42
    # errors before any work: a bad token, a zero RNG state with T > 0
    n = b.len
    assert b.decode_sample(SHAPE.vocab, temperature, top_p, sb, ws_b)[0] == pdl.ds4g.ETOKEN and b.len == n
    if temperature > 0.0:
        assert b.decode_sample(tb, temperature, top_p, 0, ws_b)[0] == pdl.ds4g.EINVAL and b.len == n


def test_prefill_timing_mode_counts_launches_and_keeps_results(model):
    """Timing mode on a tensor-core prefill: every launch is charged to its kind
    (one per layer and chunk for the per-layer GEMMs), the times are positive, and
    the K/V rows and logits are those of a prefill without timing, bit for bit."""
    import torch
    import prefill_decode_layer_gb300 as pdl
    prompt = synth.host_tokens(50, SHAPE.vocab, stream=84)
    a, b = pdl.Session(model, 64), pdl.Session(model, 64)
    b.set_timing(True)
    b.timing()
    assert a.prefill(prompt) == 0 and b.prefill(prompt) == 0
    t = b.timing()
    b.set_timing(False)
    torch.cuda.synchronize()
    assert torch.equal(a.logits(), b.logits())
    for l in range(SHAPE.n_layers):
        for x, y in zip(a.kv(l), b.kv(l)):
            assert torch.equal(x[:50], y[:50])
    chunks = -(-50 // model.cfg.prefill_chunk) if model.cfg.prefill_chunk > 0 else 1
    for kind in ("p_qkv_a", "p_q_b", "p_kv_b", "p_attn", "p_wo", "p_router", "p_topk", "p_group",
                 "p_gate_up", "p_shared_gu", "p_down", "p_shared_down", "p_combine"):
        ms, n = t[kind]
        assert n == SHAPE.n_layers * chunks, (kind, n)
        assert ms > 0.0, kind
    assert t["p_embed"][1] == chunks
