"""The 8-layer full-width model (configs "decode stack", "layer-major prefill" and
"common-prefix resync") against the oracle at full size, where replaying whole
sequences on the CPU would take hours:

- a 4096-token layer-major prefill, checked at its last position layer by layer with
  teacher forcing (the oracle starts each layer from the GPU's input to that layer
  and the GPU's K/V window, and must reproduce the new K/V row and the layer output);
- the decode step that follows (one persistent launch, all 8 layers + lm_head),
  checked from the embedding through the oracle's own layer outputs over the GPU's
  K/V windows: expert ids, new K/V rows, logits, and a T 0.7 / top-p 0.95 draw;
- the resync 16994 -> 16846 -> +91 tokens: truncate + suffix prefill equals a
  from-scratch prefill bit for bit, and greedy continuations agree."""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_sampler import undecidable
from helpers import (TOL_BF16, LazyOracleModel, OracleKV, gpu_model, kv_to_f64, oracle_embed,
                     oracle_layer, oracle_lm_head, rel_err, to_np)

pytestmark = pytest.mark.gpu
SHAPE = synth.STACK


@pytest.fixture(scope="module")
def stack():
    import torch
    torch.cuda.init()
    return gpu_model(SHAPE)


def kv_bits(sess, layer, lo, hi):
    """GPU K and V rows [lo, hi) of a layer as raw BF16 bits (the oracle's storage)."""
    import torch
    k, v = sess.kv(layer)
    return (k[lo:hi].contiguous().view(torch.int16).cpu().numpy().view(np.uint16),
            v[lo:hi].contiguous().view(torch.int16).cpu().numpy().view(np.uint16))


def near_tie(scores, k) -> bool:
    s = np.sort(np.asarray(scores, dtype=np.float64))[::-1]
    return s[k - 1] - s[k] <= 1e-3 * np.max(np.abs(s))


def test_prefill_last_token_and_next_decode_every_layer(stack):
    import torch
    import prefill_decode_layer_gb300 as pdl
    L, H, W, K = SHAPE.n_layers, SHAPE.hidden, SHAPE.window, SHAPE.top_k
    n = 4096
    toks = synth.host_tokens(n + 1, SHAPE.vocab, stream=31)
    sess = pdl.Session(stack, n + 8)
    assert sess.prefill(toks[:n]) == 0
    torch.cuda.synchronize()
    assert sess.status() == 0
    LX = to_np(sess.debug("prefill_layer_x", (L + 1) * H)).reshape(L + 1, H)
    prefill_logits = to_np(sess.logits())
    # the decode step right after the prefill
    assert sess.decode(int(toks[n])) == 0
    torch.cuda.synchronize()
    assert sess.status() == 0
    dec_logits = to_np(sess.logits())
    gpu_ids = [sess.router(l)[0] for l in range(L)]

    om = LazyOracleModel(SHAPE, keep_layers=False)
    p = n - 1
    xd = oracle_embed(om, toks[n])      # the decode step's residual, oracle's own
    dec_valid = True
    checked_prefill = checked_decode = 0
    for l in range(L):
        kv = OracleKV(SHAPE, n + 1)
        kb, vb = kv_bits(sess, l, p - W + 1, n + 1)   # GPU rows p-W+1 .. n
        kv.k[l][p - W + 1:p] = kb[:W - 1]
        kv.v[l][p - W + 1:p] = vb[:W - 1]
        # prefill, last token: from the GPU's input to layer l
        x = LX[l].copy()
        tr = oracle_layer(om, kv, l, p, x, trace=True)
        assert rel_err(kv_to_f64(SHAPE, kb[W - 1]), kv_to_f64(SHAPE, kv.k[l][p])) <= TOL_BF16, f"layer {l}"
        assert rel_err(kv_to_f64(SHAPE, vb[W - 1]), kv_to_f64(SHAPE, kv.v[l][p])) <= TOL_BF16, f"layer {l}"
        if not near_tie(tr["scores"], K):
            assert rel_err(LX[l + 1], x) <= TOL_BF16, f"layer {l} output"
            checked_prefill += 1
        # decode at position n over the GPU's window (rows n-W+1 .. n-1 from the prefill)
        kv.k[l][p] = kb[W - 1]
        kv.v[l][p] = vb[W - 1]
        if dec_valid:
            trd = oracle_layer(om, kv, l, n, xd, trace=True)
            if near_tie(trd["scores"], K):
                dec_valid = False   # everything downstream is undecidable
            else:
                assert list(trd["ids"]) == gpu_ids[l], f"decode layer {l}"
                assert rel_err(kv_to_f64(SHAPE, kb[W]), kv_to_f64(SHAPE, kv.k[l][n])) <= TOL_BF16
                assert rel_err(kv_to_f64(SHAPE, vb[W]), kv_to_f64(SHAPE, kv.v[l][n])) <= TOL_BF16
                checked_decode += 1
    assert checked_prefill >= L - 2
    assert rel_err(prefill_logits, oracle_lm_head(om, LX[L])) <= TOL_BF16
    if dec_valid:
        assert checked_decode == L
        ologits = oracle_lm_head(om, xd)
        assert rel_err(dec_logits, ologits) <= TOL_BF16
    # the sampler on the GPU's logits with the pages' decode settings
    ws = torch.empty(pdl.sample_workspace_bytes(SHAPE.vocab), dtype=torch.uint8, device="cuda")
    state = 0x2545F4914F6CDD1D
    for _ in range(8):
        u = oracle.uniform(state)[0]
        tok, state_next = pdl.sample(sess.logits(), 0.7, 0.95, state, ws)
        otok, info = oracle.sample(dec_logits.astype(np.float32), 0.7, 0.95, u)
        assert tok == otok or undecidable(info, tok)
        state = state_next


def test_resync_full_size_equals_scratch(stack):
    import torch
    import prefill_decode_layer_gb300 as pdl
    live_ids = synth.host_tokens(16994, SHAPE.vocab, stream=51)
    prompt = np.concatenate([live_ids[:16846], synth.host_tokens(91, SHAPE.vocab, stream=52)])
    if prompt[16846] == live_ids[16846]:
        prompt[16846] = (prompt[16846] + 1) % SHAPE.vocab
    live = pdl.Session(stack, 17100)
    assert live.prefill(live_ids) == 0
    cp = live.common_prefix(prompt)
    assert cp == 16846
    assert live.truncate(cp) == 0 and live.prefill(prompt[cp:]) == 0
    scratch = pdl.Session(stack, 17100)
    assert scratch.prefill(prompt) == 0
    torch.cuda.synchronize()
    assert live.status() == 0 and scratch.status() == 0
    assert torch.equal(live.logits(), scratch.logits())
    for l in range(SHAPE.n_layers):
        for a, b in zip(live.kv(l), scratch.kv(l)):
            assert torch.equal(a[:16937], b[:16937]), f"layer {l}"
    ws = torch.empty(pdl.sample_workspace_bytes(SHAPE.vocab), dtype=torch.uint8, device="cuda")
    for _ in range(4):
        a, _ = pdl.sample(live.logits(), 0.0, 1.0, None, ws)
        b, _ = pdl.sample(scratch.logits(), 0.0, 1.0, None, ws)
        assert a == b
        assert live.decode(a) == 0 and scratch.decode(b) == 0
