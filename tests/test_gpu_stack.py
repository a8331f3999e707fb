"""The 8-layer full-width model (workloads "decode stack", "layer-major prefill" and
"common-prefix resync") and the same layers at depth 43, against the oracle at
full size.  Replaying whole sequences on the CPU would take hours, so every check
is teacher-forced: the session records the GPU's residual entering each layer at
chosen positions (ds4g_session_set_probe), and the oracle starts each layer from
that input and the GPU's K/V window, and must reproduce the new K/V row, the
router's choice and the layer's output (ds4 page "端到端推理流程", 阶段四 4.2 for
the layer, 4.3 for lm_head and sampling, 阶段三 for the layer-major prefill;
page "ds4.c を読み解く" section 3 for the common-prefix resync).

- a 4096-token layer-major prefill, at the window edges (127, 128), at 128-token
  tile boundaries, at seeded random interior positions and at its last token;
  then the decode step that follows (ids, K/V rows, outputs, logits, draws);
- the sampled chain of the stack workload: a 512-token prompt, then 256 tokens at
  T 0.7 / top-p 0.95 with the seeded xorshift generator, checked at five steps
  (layers, logits, and each draw given the same uniform);
- the resync 16994 -> 16846 -> +91 tokens: truncate + suffix prefill equals a
  from-scratch prefill bit for bit, and the suffix (RoPE and K/V at p ~ 16.9k)
  and the first decode step after it agree with the oracle;
- 43 layers (the pages' depth; the 8 generated weight sets used in turn, each
  layer with its own K/V cache): prefill and decode checked at layers 0, 21, 42.
"""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_sampler import undecided_band, within_band
from helpers import (TOL_BF16, LazyOracleModel, check_probes, gpu_model, oracle_embed,
                     oracle_lm_head, rel_err, to_np)

pytestmark = pytest.mark.gpu
SHAPE = synth.STACK


@pytest.fixture(scope="module")
def stack():
    import torch
    torch.cuda.init()
    return gpu_model(SHAPE)


def probe_rows(sess, buf):
    import torch
    torch.cuda.synchronize()
    assert sess.status() == 0
    rec = buf.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(rec)), "a probed position was not recorded"
    return rec


def assert_embedding_rows(om, toks_at, rec):
    """Row 0 of each record is the token's widened f16 embedding, bit for bit."""
    for i, t in enumerate(toks_at):
        assert np.array_equal(rec[i][0], oracle_embed(om, t))


def test_prefill_4096_interior_positions_and_next_decode(stack):
    import torch
    import prefill_decode_layer_gb300 as pdl
    L, K = SHAPE.n_layers, SHAPE.top_k
    n = 4096
    toks = synth.host_tokens(n + 1, SHAPE.vocab, stream=31)
    rng = np.random.default_rng(4096)
    fixed = [0, 1, 2, 127, 128, 129, 255, 256, 1023, 1024, 2047, 2048, 3967, 4094, 4095]
    extra = sorted(set(int(p) for p in rng.integers(3, n - 1, 5)) - set(fixed))
    positions = sorted(fixed + extra) + [n]           # n: the decode step after the prefill
    sess = pdl.Session(stack, n + 8)
    buf = sess.set_probe(positions)
    assert sess.prefill(toks[:n]) == 0
    torch.cuda.synchronize()
    prefill_logits = to_np(sess.logits())
    last_x = to_np(sess.debug("prefill_layer_x", (L + 1) * SHAPE.hidden)).reshape(L + 1, -1)
    assert sess.decode(int(toks[n])) == 0
    torch.cuda.synchronize()
    dec_logits = to_np(sess.logits())
    rec = probe_rows(sess, buf)
    gpu_ids = {n: [sess.router(l)[0] for l in range(L)]}
    assert np.array_equal(rec[positions.index(n - 1)], last_x)   # the two records agree

    om = LazyOracleModel(SHAPE, keep_layers=False)
    assert_embedding_rows(om, [toks[p] for p in positions], rec)
    checked, ties = check_probes(om, sess, positions, rec, router_ids=gpu_ids)
    print(f"prefill 4096 + decode: {checked} position-layers checked, "
          f"{len(ties)} of them in the router tie band: {ties}")
    assert checked == len(positions) * L
    # logits: lm_head of the GPU's final hidden state (no final norm)
    assert rel_err(prefill_logits, oracle_lm_head(om, rec[positions.index(n - 1)][L])) <= TOL_BF16
    assert rel_err(dec_logits, oracle_lm_head(om, rec[positions.index(n)][L])) <= TOL_BF16
    # the sampler on the GPU's logits with the stack workload's settings
    ws = torch.empty(pdl.sample_workspace_bytes(SHAPE.vocab), dtype=torch.uint8, device="cuda")
    state = 0x2545F4914F6CDD1D
    host = dec_logits.astype(np.float32)
    for i in range(8):
        u = oracle.uniform(state)[0]
        tok, state_next = pdl.sample(sess.logits(), 0.7, 0.95, state, ws)
        otok, info = oracle.sample(host, 0.7, 0.95, u)
        band = undecided_band(info, otok)
        if band > 0.0:
            assert within_band(host, 0.7, 0.95, u, band, tok, info), f"draw {i}"
        else:
            assert tok == otok, f"draw {i}: {tok} vs {otok}"
        state = state_next


def test_sampled_chain_512_prompt_256_tokens(stack):
    """The stack workload itself: 512 prompt tokens, then 256 tokens drawn at T 0.7,
    top-p 0.95 from a seeded xorshift64* state.  At five steps the oracle checks
    every layer (teacher-forced), the logits, and the draw given the same uniform."""
    import torch
    import prefill_decode_layer_gb300 as pdl
    L, n_prompt, n_gen = SHAPE.n_layers, 512, 256
    prompt = synth.host_tokens(n_prompt, SHAPE.vocab, stream=61)
    steps = [0, 63, 127, 191, 255]
    positions = [n_prompt + s for s in steps]
    sess = pdl.Session(stack, n_prompt + n_gen + 8)
    buf = sess.set_probe(positions)
    ws = torch.empty(pdl.sample_workspace_bytes(SHAPE.vocab), dtype=torch.uint8, device="cuda")
    assert sess.prefill(prompt) == 0
    state = 0x9E3779B97F4A7C15
    tok, state = pdl.sample(sess.logits(), 0.7, 0.95, state, ws)
    toks, ids, logits, draws = [], {}, {}, []
    for s in range(n_gen):
        assert sess.decode(tok) == 0
        toks.append(tok)
        if s in steps:
            p = n_prompt + s
            ids[p] = [sess.router(l)[0] for l in range(L)]
            logits[p] = to_np(sess.logits())
            before = state
            tok, state = pdl.sample(sess.logits(), 0.7, 0.95, state, ws)
            draws.append((p, before, tok))
        else:
            tok, state = pdl.sample(sess.logits(), 0.7, 0.95, state, ws)
    rec = probe_rows(sess, buf)
    assert sess.len == n_prompt + n_gen
    om = LazyOracleModel(SHAPE, keep_layers=False)
    assert_embedding_rows(om, [toks[s] for s in steps], rec)
    checked, ties = check_probes(om, sess, positions, rec, router_ids=ids)
    print(f"sampled chain: {checked} position-layers checked, "
          f"{len(ties)} of them in the router tie band: {ties}")
    assert checked == len(positions) * L
    undecided = 0
    for i, (p, before, gtok) in enumerate(draws):
        assert rel_err(logits[p], oracle_lm_head(om, rec[i][L])) <= TOL_BF16, f"logits at {p}"
        u, after = oracle.uniform(before)
        host = logits[p].astype(np.float32)
        otok, info = oracle.sample(host, 0.7, 0.95, u)
        band = undecided_band(info, otok)
        if band > 0.0:
            undecided += 1
            assert within_band(host, 0.7, 0.95, u, band, gtok, info), f"draw at {p}"
        else:
            assert gtok == otok, f"draw at {p}: {gtok} vs {otok}"
    assert undecided <= 1


def test_resync_full_size_equals_scratch_and_oracle(stack):
    import torch
    import prefill_decode_layer_gb300 as pdl
    L = SHAPE.n_layers
    live_ids = synth.host_tokens(16994, SHAPE.vocab, stream=51)
    prompt = np.concatenate([live_ids[:16846], synth.host_tokens(91, SHAPE.vocab, stream=52)])
    if prompt[16846] == live_ids[16846]:
        prompt[16846] = (prompt[16846] + 1) % SHAPE.vocab
    live = pdl.Session(stack, 17100)
    assert live.prefill(live_ids) == 0
    cp = live.common_prefix(prompt)
    assert cp == 16846
    positions = [16846, 16847, 16890, 16935, 16936, 16937]   # suffix, then the first decode
    buf = live.set_probe(positions)
    assert live.truncate(cp) == 0 and live.prefill(prompt[cp:]) == 0
    scratch = pdl.Session(stack, 17100)
    assert scratch.prefill(prompt) == 0
    torch.cuda.synchronize()
    assert live.status() == 0 and scratch.status() == 0
    assert torch.equal(live.logits(), scratch.logits())
    for l in range(L):
        for a, b in zip(live.kv(l), scratch.kv(l)):
            assert torch.equal(a[:16937], b[:16937]), f"layer {l}"
    suffix_logits = to_np(live.logits())
    ws = torch.empty(pdl.sample_workspace_bytes(SHAPE.vocab), dtype=torch.uint8, device="cuda")
    first = None
    for i in range(4):
        a, _ = pdl.sample(live.logits(), 0.0, 1.0, None, ws)
        b, _ = pdl.sample(scratch.logits(), 0.0, 1.0, None, ws)
        assert a == b
        first = a if i == 0 else first
        assert live.decode(a) == 0 and scratch.decode(b) == 0
        if i == 0:
            ids = {16937: [live.router(l)[0] for l in range(L)]}
            dec_logits = to_np(live.logits())
    rec = probe_rows(live, buf)
    om = LazyOracleModel(SHAPE, keep_layers=False)
    assert_embedding_rows(om, [int(prompt[p]) for p in positions[:-1]] + [first], rec)
    checked, ties = check_probes(om, live, positions, rec, router_ids=ids)
    print(f"resync: {checked} position-layers checked, "
          f"{len(ties)} of them in the router tie band: {ties}")
    assert checked == len(positions) * L
    assert rel_err(suffix_logits, oracle_lm_head(om, rec[positions.index(16936)][L])) <= TOL_BF16
    assert rel_err(dec_logits, oracle_lm_head(om, rec[positions.index(16937)][L])) <= TOL_BF16
    assert int(np.argmax(suffix_logits)) == first


DEPTH = 43


def test_depth_43_prefill_and_decode(stack):
    """43 layers, as many as the pages' decode loop runs: the stack's 8 generated
    weight sets are used in turn (layer l uses set l mod 8: each layer still streams
    its own 275 MB per token, more than L2 holds, so the aliasing gives no cache
    advantage); every layer has its own K/V cache.  A 300-token prefill and two
    decode steps, teacher-forced at layers 0, 21 and 42."""
    import torch
    import prefill_decode_layer_gb300 as pdl
    shape = SHAPE.with_(name="depth43", n_layers=DEPTH)
    emb, lm, layers = stack._keep
    deep = pdl.Model(shape, emb, lm, [layers[l % SHAPE.n_layers] for l in range(DEPTH)])
    n = 300
    toks = synth.host_tokens(n + 2, SHAPE.vocab, stream=71)
    positions = [0, 127, 128, n - 1, n, n + 1]
    sess = pdl.Session(deep, n + 8)
    buf = sess.set_probe(positions)
    assert sess.prefill(toks[:n]) == 0
    ids = {}
    for p in (n, n + 1):
        assert sess.decode(int(toks[p])) == 0
        ids[p] = [sess.router(l)[0] for l in range(DEPTH)]
    rec = probe_rows(sess, buf)
    assert sess.len == n + 2
    om = LazyOracleModel(shape, keep_layers=False, weight_layer=lambda l: l % SHAPE.n_layers)
    assert_embedding_rows(om, [toks[p] for p in positions], rec)
    layers_checked = [0, 21, DEPTH - 1]
    checked, ties = check_probes(om, sess, positions, rec, layers=layers_checked,
                                 router_ids=ids)
    print(f"depth 43: {checked} position-layers checked, "
          f"{len(ties)} of them in the router tie band: {ties}")
    assert checked == len(positions) * len(layers_checked)
    assert rel_err(to_np(sess.logits()), oracle_lm_head(om, rec[-1][DEPTH])) <= TOL_BF16
