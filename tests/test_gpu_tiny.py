"""Tiny FP32 model end to end on the GPU against the oracle: prefill 64 prompt
tokens (layer-major), then greedy-decode 8 tokens, every intermediate checked at
the FP32 tolerance (1e-4) and every id exactly."""
import numpy as np
import pytest

import oracle
import synth
from helpers import (DECODE_KERNELS, TOL_F32, LazyOracleModel, OracleKV, gpu_model, kv_to_f64,
                     oracle_embed, oracle_layer, oracle_lm_head, rel_err, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=DECODE_KERNELS, ids=["persistent", "staged"])
def tiny(request):
    import torch
    torch.cuda.init()
    shape = synth.TINY
    return shape, gpu_model(shape, decode_kernel=request.param), LazyOracleModel(shape)


def test_tiny_prefill_then_greedy_decode(tiny):
    import torch
    import prefill_decode_layer_gb300 as pdl
    shape, gm, om = tiny
    n_ctx = 128
    prompt = synth.host_tokens(64, shape.vocab, seed=0, stream=0)
    sess = pdl.Session(gm, n_ctx)
    assert sess.prefill(prompt) == 0 and sess.len == 64
    torch.cuda.synchronize()

    # oracle: layer-major prefill through its session API
    osess = oracle.OracleSession(om.full(), n_ctx)
    rc, ologits, _ = osess.prefill(prompt)
    assert rc == 0
    assert rel_err(to_np(sess.logits()), ologits) <= TOL_F32
    k, v = sess.kv(0)
    ok, ov = oracle.kv_views(osess, 0, n_ctx)
    assert rel_err(to_np(k[:64]), kv_to_f64(shape, ok[:64])) <= TOL_F32
    assert rel_err(to_np(v[:64]), kv_to_f64(shape, ov[:64])) <= TOL_F32

    ws = torch.empty(pdl.sample_workspace_bytes(shape.vocab), dtype=torch.uint8, device="cuda")
    gl = to_np(sess.logits())
    for step in range(8):
        tok, _ = pdl.sample(sess.logits(), 0.0, 1.0, None, ws)
        otok = oracle.argmax(ologits.astype(np.float32))
        top2 = np.sort(ologits)[-2:]
        if top2[1] - top2[0] > 2 * TOL_F32 * np.max(np.abs(ologits)):
            assert tok == otok, f"step {step}: greedy id {tok} != oracle {otok}"
        else:
            tok = otok   # near-tie: follow the oracle's choice on both sides
        assert tok == int(np.argmax(gl))  # the sampler's argmax equals the logits' argmax
        assert sess.decode(tok) == 0
        rc, ologits, _ = osess.decode(tok)
        assert rc == 0
        torch.cuda.synchronize()
        gl = to_np(sess.logits())
        assert rel_err(gl, ologits) <= TOL_F32, f"step {step}"
    assert sess.len == 72
    k, v = sess.kv(0)
    ok, ov = oracle.kv_views(osess, 0, n_ctx)
    assert rel_err(to_np(k[:72]), kv_to_f64(shape, ok[:72])) <= TOL_F32


def test_tiny_decode_intermediates(tiny):
    """Each stage of one decode step (latents, RoPE'd queries, attention, residuals,
    router scores and ids, SwiGLU hiddens) against the oracle's trace."""
    import torch
    import prefill_decode_layer_gb300 as pdl
    shape, gm, om = tiny
    n_ctx = 64
    toks = synth.host_tokens(40, shape.vocab, seed=0, stream=7)
    sess = pdl.Session(gm, n_ctx)
    kv = OracleKV(shape, n_ctx)
    H, QD, K, I = shape.hidden, shape.n_heads * shape.head_dim, shape.top_k, shape.expert_inter
    for pos, t in enumerate(toks):
        assert sess.decode(int(t)) == 0
        x = oracle_embed(om, t)
        tr = oracle_layer(om, kv, 0, pos, x, trace=True)
        if pos not in (0, 1, 15, 16, 17, 39):   # window edges: 16 keys
            continue
        torch.cuda.synchronize()
        c = to_np(sess.debug("cqkv", shape.q_rank + shape.kv_rank))
        assert rel_err(c[:shape.q_rank], tr["cq"]) <= TOL_F32
        assert rel_err(c[shape.q_rank:], tr["ckv"]) <= TOL_F32
        assert rel_err(to_np(sess.debug("q", QD)), tr["q"]) <= TOL_F32
        assert rel_err(to_np(sess.debug("attn", QD)), tr["attn"]) <= TOL_F32
        assert rel_err(to_np(sess.debug("xmid", H)), tr["x_mid"]) <= TOL_F32
        assert rel_err(to_np(sess.debug("xn2", H)), tr["xn2"]) <= TOL_F32
        assert rel_err(to_np(sess.debug("scores", shape.n_experts)), tr["scores"]) <= TOL_F32
        ids, w = sess.router(0)
        assert ids == list(tr["ids"]), f"pos {pos}"
        assert rel_err(w, tr["weights"]) <= TOL_F32
        assert rel_err(to_np(sess.debug("h", (K + 1) * I)), tr["h"]) <= TOL_F32
        assert rel_err(to_np(sess.debug("x", H)), x) <= TOL_F32
        assert rel_err(to_np(sess.logits()), oracle_lm_head(om, x)) <= TOL_F32
