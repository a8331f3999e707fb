"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a closed form,
an invariant, a library routine (numpy / scipy / torch) on a special case, a
hand-derived fixture under tests/golden/, or brute force on tiny inputs.  The
cases are chosen so that a dropped term, a wrong sign or index, or a transposed
operand fails at least one of them.
"""
import ctypes as C
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
L = oracle.lib()


def p(a):
    return a.ctypes.data


def tiny_cfg(**kw):
    shape = synth.ModelShape("pin", n_layers=1, hidden=16, n_heads=2, head_dim=4, q_rank=8,
                             kv_rank=6, window=3, n_experts=5, top_k=2, expert_inter=6,
                             vocab=11, weight_dtype="f32", kv_dtype="f32")
    return shape.with_(**kw)


def random_layer(shape, rng, scale=0.3):
    w = {}
    for name, kind, shp, sigma in synth.layer_tensors(shape):
        if sigma is None:
            w[name] = (1.0 + 0.2 * rng.standard_normal(shp)).astype(np.float32)
        else:
            w[name] = (scale * rng.standard_normal(shp)).astype(np.float32)
    return w


# ----------------------------------------------------------------------------- formats

def test_f16_widening_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([L.orc_f16_value(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_widening_and_rounding_match_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 65536, 20000).astype(np.uint16)
    t = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([L.orc_bf16_value(int(b)) for b in bits])
    ok = np.isfinite(t)
    assert np.array_equal(got[ok], t[ok].astype(np.float64))
    # rounding: float32 inputs (exact in double) rounded by torch's round-to-nearest-even
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000)).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0]    # exact ties
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([L.orc_round_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_embed_gathers_the_token_row():
    """orc_embed (ds4 page "端到端推理流程", 4.1 embed_token_f16) against numpy
    indexing of a [V][H] float16 table whose rows are all different; the first,
    last and interior tokens are checked, and hidden != vocab, so a wrong stride,
    a transposed table or an off-by-one row fails."""
    V, H = 11, 16
    rng = np.random.default_rng(21)
    vals = rng.standard_normal((V, H)) * 4.0
    vals[:, 0] = np.arange(V)                     # row t starts with t: rows are distinct
    table = np.ascontiguousarray(vals.astype(np.float16))
    cfg = oracle.config_from(tiny_cfg(hidden=H, vocab=V))
    for tok in (0, 1, 5, V - 2, V - 1):
        x = np.full(H, np.nan)
        L.orc_embed(C.byref(cfg), p(table.view(np.uint16)), tok, p(x))
        assert np.array_equal(x, table[tok].astype(np.float64))
        if tok > 0:
            assert not np.array_equal(x, table[tok - 1].astype(np.float64))


# ----------------------------------------------------------------------------- rmsnorm

def rmsnorm(x, g, eps):
    y = np.zeros_like(x)
    L.orc_rmsnorm(len(x), p(x), p(g), eps, p(y))
    return y


def test_rmsnorm_closed_forms():
    g = np.linspace(0.5, 1.5, 32).astype(np.float32)
    g64 = g.astype(np.float64)
    for c in (3.0, -0.25, 1e-3):
        x = np.full(32, c)
        eps = 1e-6
        # constant vector: y = g * c / sqrt(c^2 + eps); at c = 1e-3 eps is half the mean square
        assert np.allclose(rmsnorm(x, g, eps), g64 * c / math.sqrt(c * c + eps), rtol=1e-14)
    rng = np.random.default_rng(0)
    x = rng.standard_normal(64)
    ones = np.ones(64, dtype=np.float32)
    y = rmsnorm(x, ones, 0.0)
    assert abs(np.sqrt(np.mean(y * y)) - 1.0) < 1e-14          # unit RMS at eps = 0
    assert np.allclose(rmsnorm(7.5 * x, ones, 0.0), y, rtol=1e-14)  # scale invariance
    g2 = rng.standard_normal(64).astype(np.float32)
    assert np.allclose(rmsnorm(x, g2, 0.0), g2.astype(np.float64) * y, rtol=1e-13)     # gain is elementwise


# ----------------------------------------------------------------------------- matvec

@pytest.mark.parametrize("dtype", [oracle.F32, oracle.BF16])
def test_matvec_matches_numpy(dtype):
    rng = np.random.default_rng(2)
    W = rng.standard_normal((13, 37)).astype(np.float32)
    if dtype == oracle.BF16:
        Wb = torch.from_numpy(W).to(torch.bfloat16)
        store = Wb.view(torch.int16).numpy().astype(np.uint16)
        Wd = Wb.double().numpy()
    else:
        store, Wd = W, W.astype(np.float64)
    x = rng.standard_normal(37)
    y = np.zeros(13)
    L.orc_matvec(dtype, p(store), 13, 37, p(x), p(y))
    assert np.allclose(y, Wd @ x, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------- rope

def rope(v, pos, base):
    v = np.array(v, dtype=np.float64)
    L.orc_rope(len(v), pos, base, p(v))
    return v


def test_rope_golden_fixture():
    f = {}
    for line in open(os.path.join(GOLD, "rope_hd4.txt")):
        if line.strip() and not line.startswith("#"):
            k, *vals = line.split()
            f[k] = [float(x) for x in vals]
    got = rope(f["input"], int(f["pos"][0]), f["base"][0])
    assert np.allclose(got, f["expected"], rtol=0, atol=1e-15)


def test_rope_invariants():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    assert np.array_equal(rope(q, 0, 10000.0), q)                            # p = 0 identity
    assert abs(np.linalg.norm(rope(q, 977, 1e4)) - np.linalg.norm(q)) < 1e-12  # isometry
    for (pq, pk, d) in [(10, 3, 5), (200, 199, 1000), (4095, 3968, 17)]:
        a = rope(q, pq, 1e4) @ rope(k, pk, 1e4)
        b = rope(q, pq + d, 1e4) @ rope(k, pk + d, 1e4)
        assert abs(a - b) < 1e-9 * (1 + abs(a))                               # relative position


# ----------------------------------------------------------------------------- attention

def make_kv(cfg, K, V):
    kvs = oracle.KV(K.ctypes.data, V.ctypes.data)
    return kvs


def attention(shape, K, V, pos, q):
    cfg = oracle.config_from(shape)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    o = np.zeros(shape.n_heads * shape.head_dim)
    kv = make_kv(cfg, K, V)
    L.orc_attention(C.byref(cfg), C.byref(kv), pos, p(np.ascontiguousarray(q)), p(o))
    return o.reshape(shape.n_heads, shape.head_dim)


def library_attention(K, V, q, lo, pos, hd):
    """Full causal softmax attention via scipy.special.softmax."""
    s = (q @ K[lo:pos + 1].astype(np.float64).T) / math.sqrt(hd)
    return scipy.special.softmax(s, axis=-1) @ V[lo:pos + 1].astype(np.float64)


def test_attention_special_cases():
    rng = np.random.default_rng(4)
    shape = tiny_cfg(n_heads=3, head_dim=8, window=4)
    K = rng.standard_normal((10, 8)).astype(np.float32)
    V = rng.standard_normal((10, 8)).astype(np.float32)
    q = rng.standard_normal(24)
    # one key: every head returns V_0
    assert np.allclose(attention(shape, K, V, 0, q), np.tile(V[0].astype(np.float64), (3, 1)), rtol=1e-14)
    # softmax rows sum to one: V = 1 everywhere gives o = 1
    assert np.allclose(attention(shape, K, np.ones_like(V), 7, q), 1.0, rtol=1e-14)
    # identical keys: o = mean of the window's values
    Ku = np.tile(K[0], (10, 1))
    assert np.allclose(attention(shape, Ku, V, 7, q), np.tile(V[4:8].astype(np.float64).mean(0), (3, 1)),
                       rtol=1e-12)


def test_sliding_window_equals_full_attention_within_window():
    rng = np.random.default_rng(5)
    shape = tiny_cfg(n_heads=2, head_dim=8, window=6)
    K = rng.standard_normal((12, 8)).astype(np.float32)
    V = rng.standard_normal((12, 8)).astype(np.float32)
    q = rng.standard_normal(16)
    for pos in range(6):      # pos + 1 <= window: the window is the whole causal context
        ref = library_attention(K, V, q.reshape(2, 8), 0, pos, 8)
        assert np.allclose(attention(shape, K, V, pos, q), ref, rtol=1e-12)
    for pos in range(6, 12):  # beyond: exactly the last `window` keys, including the current one
        ref = library_attention(K, V, q.reshape(2, 8), pos - 5, pos, 8)
        assert np.allclose(attention(shape, K, V, pos, q), ref, rtol=1e-12)
    # keys that fall out of the window must have no effect even when they would dominate
    K2 = K.copy()
    K2[:6] = 50.0 * q[:8]
    assert np.allclose(attention(shape, K2, V, 11, q), attention(shape, K, V, 11, q), rtol=1e-14)


def test_attention_score_scale_two_keys():
    # two keys with q.K0 = 0 and q.K1 = a: P1 = 1 / (1 + exp(-a / sqrt(hd))); V0 = 0, V1 = 1
    shape = tiny_cfg(n_heads=1, head_dim=4, window=8)
    q = np.array([1.0, 0.0, 0.0, 0.0])
    a = 2.0
    K = np.array([[0, 0, 0, 0], [a, 0, 0, 0]], dtype=np.float32)
    V = np.array([[0, 0, 0, 0], [1, 1, 1, 1]], dtype=np.float32)
    o = attention(shape, K, V, 1, q)
    assert np.allclose(o, 1.0 / (1.0 + math.exp(-a / 2.0)), rtol=1e-14)


# ----------------------------------------------------------------------------- router

def test_topk_equals_stable_full_sort():
    rng = np.random.default_rng(6)
    for trial in range(50):
        n, k = int(rng.integers(2, 300)), 0
        k = int(rng.integers(1, min(n, 8) + 1))
        s = rng.standard_normal(n).astype(np.float32)
        if trial % 3 == 0:                      # plant ties
            s = np.round(s * 2) / 2
        ids = np.zeros(k, dtype=np.int32)
        L.orc_topk(p(s), n, k, p(ids))
        ref = np.argsort(-s, kind="stable")[:k]
        assert np.array_equal(ids, ref)


def router(shape, w, xn2):
    cfg = oracle.config_from(shape)
    lay = oracle.layer_struct(w)
    sc = np.zeros(shape.n_experts, dtype=np.float32)
    ids = np.zeros(shape.top_k, dtype=np.int32)
    wt = np.zeros(shape.top_k)
    L.orc_router(C.byref(cfg), C.byref(lay), p(xn2), p(sc), p(ids), p(wt))
    return sc, ids, wt


def test_router_weights():
    rng = np.random.default_rng(7)
    shape = tiny_cfg(n_experts=9, top_k=3)
    w = random_layer(shape, rng)
    x = rng.standard_normal(shape.hidden)
    sc, ids, wt = router(shape, w, x)
    assert np.allclose(sc, (w["w_router"].astype(np.float64) @ x).astype(np.float32), rtol=1e-6)
    assert abs(wt.sum() - 1.0) < 1e-14 and np.all(np.diff(wt) <= 0)
    assert np.allclose(wt, scipy.special.softmax(sc[ids].astype(np.float64)), rtol=1e-13)
    # k = E: the weights are the full softmax over all experts (in descending order)
    shape2 = shape.with_(top_k=9)
    sc, ids, wt = router(shape2, w, x)
    assert np.allclose(wt, scipy.special.softmax(sc.astype(np.float64))[ids], rtol=1e-13)


def test_swiglu_expert_matches_torch():
    rng = np.random.default_rng(8)
    shape = tiny_cfg()
    cfg = oracle.config_from(shape)
    H, I = shape.hidden, shape.expert_inter
    wg = rng.standard_normal((I, H)).astype(np.float32)
    wu = rng.standard_normal((I, H)).astype(np.float32)
    wd = rng.standard_normal((H, I)).astype(np.float32)
    x = rng.standard_normal(H)
    h, y = np.zeros(I), np.zeros(H)
    L.orc_swiglu_expert(C.byref(cfg), p(wg), p(wu), p(wd), p(x), p(h), p(y))
    xt = torch.from_numpy(x)
    ref_h = torch.nn.functional.silu(torch.from_numpy(wg).double() @ xt) * \
        (torch.from_numpy(wu).double() @ xt)
    assert np.allclose(h, ref_h.numpy(), rtol=1e-12)
    assert np.allclose(y, (torch.from_numpy(wd).double() @ ref_h).numpy(), rtol=1e-12)


# ----------------------------------------------------------------------------- layer step

def run_layer(shape, w, x, pos, K, V):
    cfg = oracle.config_from(shape)
    lay = oracle.layer_struct(w)
    kv = oracle.KV(K.ctypes.data, V.ctypes.data)
    tr, bufs = oracle.make_trace(cfg)
    x = x.copy()
    oracle.layer_step(cfg, lay, kv, pos, x, tr)
    return x, bufs


def test_layer_step_wiring_against_library_routines():
    """Every intermediate of one layer step equals the library computation of the
    pages' formula applied to the previous intermediate (4.2 pseudocode order)."""
    rng = np.random.default_rng(9)
    shape = tiny_cfg(window=3)
    w = random_layer(shape, rng)
    H, NH, HD = shape.hidden, shape.n_heads, shape.head_dim
    n_ctx, pos = 8, 5
    K = rng.standard_normal((n_ctx, HD)).astype(np.float32)
    V = rng.standard_normal((n_ctx, HD)).astype(np.float32)
    x0 = rng.standard_normal(H)
    x1, t = run_layer(shape, w, x0, pos, K, V)
    W = {k: v.astype(np.float64) for k, v in w.items()}
    t64 = torch.from_numpy

    def norm(v, g):
        return (t64(v) * torch.rsqrt((t64(v) ** 2).mean() + shape.rms_eps) * t64(g)).numpy()

    assert np.allclose(t["xn1"], norm(x0, W["attn_norm"]), rtol=1e-12)
    assert np.allclose(t["cq"], W["wq_a"] @ t["xn1"], rtol=1e-12)
    assert np.allclose(t["ckv"], W["wkv_a"] @ t["xn1"], rtol=1e-12)
    q_pre = W["wq_b"] @ t["cq"]
    k_pre = W["wk_b"] @ t["ckv"]
    assert np.allclose(t["q"], np.concatenate([rope(q_pre[h * HD:(h + 1) * HD], pos,
                                                    shape.rope_base) for h in range(NH)]),
                       rtol=1e-12)
    assert np.allclose(t["k"], rope(k_pre, pos, shape.rope_base), rtol=1e-12)
    assert np.allclose(t["v"], W["wv_b"] @ t["ckv"], rtol=1e-12)
    # the new K/V are stored at pos (f32 storage) and attended to
    assert np.array_equal(K[pos], t["k"].astype(np.float32))
    assert np.array_equal(V[pos], t["v"].astype(np.float32))
    o = library_attention(K, V, t["q"].reshape(NH, HD), pos - shape.window + 1, pos, HD)
    assert np.allclose(t["attn"], o.reshape(-1), rtol=1e-12)
    assert np.allclose(t["x_mid"], x0 + W["wo"] @ t["attn"], rtol=1e-12)
    assert np.allclose(t["xn2"], norm(t["x_mid"], W["ffn_norm"]), rtol=1e-12)
    sc = (W["w_router"] @ t["xn2"]).astype(np.float32)
    ids = np.argsort(-sc, kind="stable")[:shape.top_k]
    assert np.array_equal(t["ids"], ids)
    wt = scipy.special.softmax(sc[ids].astype(np.float64))
    assert np.allclose(t["weights"], wt, rtol=1e-12)

    def expert(wg, wu, wd):
        g, u = wg @ t["xn2"], wu @ t["xn2"]
        return wd @ (torch.nn.functional.silu(t64(g)).numpy() * u)

    moe = sum(wt[s] * expert(W["w_gate"][e], W["w_up"][e], W["w_down"][e])
              for s, e in enumerate(ids))
    moe = moe + expert(W["ws_gate"], W["ws_up"], W["ws_down"])
    assert np.allclose(t["moe"], moe, rtol=1e-12)
    assert np.allclose(x1, t["x_mid"] + moe, rtol=1e-12)


def test_layer_step_with_given_router_choice():
    """orc_layer_step_ids: with the oracle's own top-k (or NULL) it is orc_layer_step
    bit for bit; with another choice of experts (the k-th swapped for the (k+1)-th,
    combined in the given order) the MoE output is the library computation of
    sum_s softmax(scores[ids])_s * expert_s(xn2) + shared(xn2)."""
    rng = np.random.default_rng(19)
    shape = tiny_cfg(window=3)
    w = random_layer(shape, rng)
    H, HD, Kk = shape.hidden, shape.head_dim, shape.top_k
    n_ctx, pos = 8, 5
    K0 = rng.standard_normal((n_ctx, HD)).astype(np.float32)
    V0 = rng.standard_normal((n_ctx, HD)).astype(np.float32)
    x0 = rng.standard_normal(H)
    x_ref, t_ref = run_layer(shape, w, x0, pos, K0.copy(), V0.copy())
    cfg = oracle.config_from(shape)
    lay = oracle.layer_struct(w)

    def run_ids(ids):
        K, V = K0.copy(), V0.copy()
        kv = oracle.KV(K.ctypes.data, V.ctypes.data)
        tr, bufs = oracle.make_trace(cfg)
        x = x0.copy()
        if ids is None:
            L.orc_layer_step_ids(C.byref(cfg), C.byref(lay), C.byref(kv), pos, p(x), C.byref(tr),
                                 None)
        else:
            oracle.layer_step_ids(cfg, lay, kv, pos, x, ids, tr)
        return x, bufs

    for ids in (None, t_ref["ids"].copy()):
        x, t = run_ids(ids)
        assert np.array_equal(x, x_ref) and np.array_equal(t["weights"], t_ref["weights"])
    order = np.argsort(-t_ref["scores"], kind="stable")
    alt = np.concatenate([order[:Kk - 1], order[Kk:Kk + 1]])[::-1].astype(np.int32)
    x, t = run_ids(alt)
    assert np.array_equal(t["ids"], alt)
    W = {k: v.astype(np.float64) for k, v in w.items()}
    wt = scipy.special.softmax(t_ref["scores"][alt].astype(np.float64))
    assert np.allclose(t["weights"], wt, rtol=1e-12)

    def expert(wg, wu, wd):
        g, u = wg @ t["xn2"], wu @ t["xn2"]
        return wd @ (torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u)

    moe = sum(wt[s] * expert(W["w_gate"][e], W["w_up"][e], W["w_down"][e])
              for s, e in enumerate(alt))
    moe = moe + expert(W["ws_gate"], W["ws_up"], W["ws_down"])
    assert np.allclose(t["moe"], moe, rtol=1e-12)
    assert np.allclose(x, t_ref["x_mid"] + moe, rtol=1e-12)
    assert not np.allclose(x, x_ref, rtol=1e-6)


def test_layer_step_with_zero_outputs_is_identity():
    rng = np.random.default_rng(10)
    shape = tiny_cfg()
    w = random_layer(shape, rng)
    for k in ("wo", "w_down", "ws_down"):
        w[k][:] = 0.0
    K = np.zeros((8, shape.head_dim), dtype=np.float32)
    V = np.zeros_like(K)
    x0 = rng.standard_normal(shape.hidden)
    x1, _ = run_layer(shape, w, x0, 3, K, V)
    assert np.array_equal(x1, x0)


def test_single_expert_with_unit_weight_is_plain_swiglu_mlp():
    rng = np.random.default_rng(11)
    shape = tiny_cfg(n_experts=1, top_k=1)
    w = random_layer(shape, rng)
    for k in ("ws_down", "wo"):
        w[k][:] = 0.0
    K = np.zeros((8, shape.head_dim), dtype=np.float32)
    x0 = rng.standard_normal(shape.hidden)
    x1, t = run_layer(shape, w, x0, 0, K, K.copy())
    assert t["weights"][0] == 1.0
    W = {k: v.astype(np.float64) for k, v in w.items()}
    g, u = W["w_gate"][0] @ t["xn2"], W["w_up"][0] @ t["xn2"]
    mlp = W["w_down"][0] @ (scipy.special.expit(g) * g * u)
    assert np.allclose(x1 - x0, mlp, rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------------------- sampler

def load_sampler_fixture():
    cases, logits = [], None
    for line in open(os.path.join(GOLD, "sampler_tiny.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        if line.startswith("logits"):
            logits = np.array([float(v) for v in line.split()[1:]], dtype=np.float32)
        else:
            T, tp, u, e = line.split()
            cases.append((float(T), float(tp), float(u), int(e)))
    return logits, cases


def test_sampler_hand_derived_cases():
    logits, cases = load_sampler_fixture()
    for T, tp, u, expect in cases:
        tok, info = oracle.sample(logits, T, tp, u)
        assert tok == expect, (T, tp, u)


def test_sampler_limits():
    rng = np.random.default_rng(12)
    lg = rng.standard_normal(500).astype(np.float32)
    am = int(np.argmax(lg))
    assert oracle.argmax(lg) == am
    # temperature -> 0 concentrates on the argmax; T <= 0 is argmax
    for u in (0.0, 0.3, 0.999):
        assert oracle.sample(lg, 1e-6, 1.0, u)[0] == am
        assert oracle.sample(lg, 0.0, 0.9, u)[0] == am
    # a tiny top_p keeps only the most probable token
    assert oracle.sample(lg, 0.8, 1e-9, 0.77)[0] == am
    # u = 0 returns the first kept token in index order
    tok, info = oracle.sample(lg, 1.0, 1.0, 0.0)
    assert tok == 0
    # argmax ties go to the lowest index
    lg2 = np.zeros(10, dtype=np.float32)
    lg2[[3, 7]] = 1.0
    assert oracle.argmax(lg2) == 3


def test_sampler_top_p_kept_set_brute_force():
    rng = np.random.default_rng(13)
    for _ in range(40):
        n = int(rng.integers(2, 9))
        lg = (rng.standard_normal(n) * 2).astype(np.float32)
        T, tp = float(rng.uniform(0.3, 2.0)), float(rng.uniform(0.05, 0.999))
        pr = np.exp(lg.astype(np.float64) / T - (lg.astype(np.float64) / T).max())
        order = sorted(range(n), key=lambda i: (-pr[i], i))
        cum, kept = 0.0, []
        for i in order:
            cum += pr[i]
            kept.append(i)
            if cum >= tp * pr.sum():
                break
        kept = sorted(kept)
        # brute force: the CDF interval of each kept token in index order
        S = pr[kept].sum()
        edges = np.cumsum(pr[kept]) / S
        for u in rng.uniform(0, 1, 20):
            expect = kept[int(np.searchsorted(edges, u, side="left"))]
            tok, info = oracle.sample(lg, T, tp, float(u))
            if info.cdf_margin > 1e-12:
                assert tok == expect
            assert info.n_kept == len(kept)


def test_sampler_min_p_hand_derived_cases():
    # Relative probabilities 1, 1/2, 1/4, 1/8 and ~8e-4 at T = 1 (logits ln 8, ln 4,
    # ln 2, 0, -5).  Reading of the pages' sample_top_p_min_p (the two filters are
    # named only): a token of the top-p set stays if p >= min_p * max p.
    lg = np.array([np.log(8.0), np.log(4.0), np.log(2.0), 0.0, -5.0], dtype=np.float32)
    cases = [
        # min_p, top_p, u, expected: kept set and CDF worked out by hand
        (0.3, 1.0, 0.5, 0),    # kept {0, 1}, sum 1.5: u*sum = 0.75 lies in token 0's [0, 1)
        (0.3, 1.0, 0.9, 1),    # 1.35 lies in token 1's [1, 1.5)
        (0.2, 1.0, 0.95, 2),   # kept {0, 1, 2}, sum 1.75: 1.6625 lies in token 2's [1.5, 1.75)
        (0.1, 0.6, 0.9, 1),    # top-p target 0.6 * 1.8758 = 1.1255 keeps {0, 1}: 1.35 -> 1
        (0.1, 1.0, 0.99, 3),   # kept {0, 1, 2, 3}, sum 1.875: 1.856 lies in token 3's [1.75, 1.875)
        (1.0, 1.0, 0.999, 0),  # only the largest survives min_p = 1
        (0.0005, 1.0, 0.9999, 4),  # min_p below 8.4e-4 keeps token 4: 1.8757 in [1.875, 1.8758)
        (0.001, 1.0, 0.9999, 3),   # above it drops token 4: sum 1.875, 1.8748 in [1.75, 1.875)
    ]
    for mp, tp, u, expect in cases:
        tok, info = oracle.sample(lg, 1.0, tp, u, min_p=mp)
        assert tok == expect, (mp, tp, u, tok)


def test_sampler_min_p_kept_set_brute_force():
    rng = np.random.default_rng(15)
    for _ in range(40):
        n = int(rng.integers(2, 9))
        lg = (rng.standard_normal(n) * 2).astype(np.float32)
        T, tp = float(rng.uniform(0.3, 2.0)), float(rng.choice([1.0, rng.uniform(0.05, 0.999)]))
        mp = float(rng.uniform(0.01, 0.9))
        pr = np.exp(lg.astype(np.float64) / T - (lg.astype(np.float64) / T).max())
        order = sorted(range(n), key=lambda i: (-pr[i], i))
        cum, nucleus = 0.0, []
        for i in order:
            cum += pr[i]
            nucleus.append(i)
            if tp < 1.0 and cum >= tp * pr.sum():
                break
        kept = sorted(i for i in nucleus if pr[i] >= mp * pr.max())
        S = pr[kept].sum()
        edges = np.cumsum(pr[kept]) / S
        for u in rng.uniform(0, 1, 20):
            expect = kept[int(np.searchsorted(edges, u, side="left"))]
            tok, info = oracle.sample(lg, T, tp, float(u), min_p=mp)
            if info.cdf_margin > 1e-12 and info.minp_margin > 1e-12:
                assert tok == expect
                assert info.n_kept == len(kept)


def test_sampler_frequencies_chi_square():
    rng = np.random.default_rng(14)
    lg = rng.standard_normal(8).astype(np.float32)
    pr = scipy.special.softmax(lg.astype(np.float64) / 0.9)
    state = 0x9E3779B97F4A7C15
    counts = np.zeros(8)
    for _ in range(100000):
        u, state = oracle.uniform(state)
        counts[oracle.sample(lg, 0.9, 1.0, u)[0]] += 1
    stat, pval = scipy.stats.chisquare(counts, pr * counts.sum())
    assert pval > 1e-4


def read_xorshift_golden():
    start, steps = None, []
    for line in open(os.path.join(GOLD, "xorshift64s.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        k, v = line.split()
        if k == "start":
            start = int(v)
        elif k == "state":
            steps.append({"state": int(v)})
        else:
            steps[-1][k] = int(v, 0)
    return start, steps


def test_xorshift_golden_states_draws_and_uniforms():
    """State sequence, scrambled draws and uniforms against the hand-derived fixture
    (Vigna 2016; the workloads' seeded xorshift generator).  A wrong shift fails the
    states, a wrong multiplier the draws, a wrong bit selection the uniforms."""
    start, steps = read_xorshift_golden()
    assert len(steps) == 2 and all(len(st) == 3 for st in steps)
    s = C.c_uint64(start)
    for st in steps:
        draw = L.orc_xorshift64s(C.byref(s))
        assert s.value == st["state"]
        assert draw == st["output"]
    s = C.c_uint64(start)
    for st in steps:
        u = L.orc_uniform(C.byref(s))
        assert s.value == st["state"]
        assert u == st["unum"] / 16777216.0


def test_xorshift_uniformity():
    state = 12345
    us = []
    for _ in range(20000):
        u, state = oracle.uniform(state)
        us.append(u)
    us = np.array(us)
    assert us.min() >= 0.0 and us.max() < 1.0
    assert scipy.stats.kstest(us, "uniform").pvalue > 1e-4
    # 24-bit resolution: every draw is a whole multiple of 2^-24
    assert np.all(us * 16777216.0 == np.floor(us * 16777216.0))


# ----------------------------------------------------------------------------- session

def tiny_model(shape, seed=0, n_layers=None):
    layers = [synth.host_layer(shape, l, seed) for l in range(shape.n_layers)]
    return oracle.OracleModel(shape, layers, synth.host_embedding(shape, seed),
                              synth.host_lm_head(shape, seed))


def small_shape():
    return synth.TINY.with_(name="small", n_layers=2, hidden=64, n_heads=2, head_dim=8,
                            q_rank=16, kv_rank=16, window=4, n_experts=6, top_k=2,
                            expert_inter=32, vocab=50, gain_sigma=0.1)


def test_layer_major_prefill_equals_sequential_decode():
    shape = small_shape()
    om = tiny_model(shape)
    toks = synth.host_tokens(11, shape.vocab, stream=1)
    a = oracle.OracleSession(om, 32)
    rc, la, ha = a.prefill(toks, want_hidden=True)
    assert rc == 0
    b = oracle.OracleSession(om, 32)
    for i, t in enumerate(toks):
        rc, lb, hb = b.decode(int(t), want_hidden=True)
        assert rc == 0
        assert np.array_equal(hb, ha[i])
    assert np.array_equal(la, lb)
    for layer in range(shape.n_layers):
        ka, va = oracle.kv_views(a, layer, 32)
        kb, vb = oracle.kv_views(b, layer, 32)
        assert np.array_equal(ka[:11], kb[:11]) and np.array_equal(va[:11], vb[:11])


@pytest.mark.parametrize("wdtype", ["f32", "bf16"])
def test_prefill_logits_are_lm_head_of_the_last_token(wdtype):
    """orc_prefill's logits (page "端到端推理流程", 4.3: the last layer's output goes
    to lm_head) equal W_lm @ hidden[n-1] computed by numpy from the prefill's own
    final hidden states: the last token, not the first, and no final norm.  The
    same holds for one decode step after the prefill."""
    shape = small_shape().with_(weight_dtype=wdtype)
    om = tiny_model(shape)
    lm = synth.host_lm_head(shape)
    W = lm.astype(np.float64) if wdtype == "f32" else \
        torch.from_numpy(lm.astype(np.int16)).view(torch.bfloat16).double().numpy()
    toks = synth.host_tokens(7, shape.vocab, stream=5)
    s = oracle.OracleSession(om, 16)
    rc, logits, hidden = s.prefill(toks, want_hidden=True)
    assert rc == 0 and hidden.shape == (7, shape.hidden)
    ref = W @ hidden[-1]
    assert np.allclose(logits, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert not np.allclose(logits, W @ hidden[0], rtol=1e-3)
    rc, logits2, h2 = s.decode(int(toks[0]), want_hidden=True)
    assert rc == 0
    ref2 = W @ h2
    assert np.allclose(logits2, ref2, rtol=1e-12, atol=1e-12 * np.abs(ref2).max())


def test_truncate_then_suffix_equals_scratch_prefill():
    shape = small_shape()
    om = tiny_model(shape)
    common = synth.host_tokens(9, shape.vocab, stream=2)
    live_tail = synth.host_tokens(5, shape.vocab, stream=3)
    new_tail = synth.host_tokens(4, shape.vocab, stream=4)
    new_tail[0] = (live_tail[0] + 1) % shape.vocab
    live = oracle.OracleSession(om, 40)
    assert live.prefill(np.concatenate([common, live_tail]))[0] == 0
    prompt = np.concatenate([common, new_tail])
    cp = live.common_prefix(prompt)
    assert cp == 9
    assert live.truncate(cp) == 0 and live.len == 9
    rc, l1, h1 = live.prefill(prompt[cp:], want_hidden=True)
    scratch = oracle.OracleSession(om, 40)
    rc, l2, h2 = scratch.prefill(prompt, want_hidden=True)
    assert np.array_equal(l1, l2) and np.array_equal(h1, h2[cp:])
    # window 4 < common prefix 9: the suffix attends to positions kept by the truncation
    for layer in range(shape.n_layers):
        ka, _ = oracle.kv_views(live, layer, 40)
        kb, _ = oracle.kv_views(scratch, layer, 40)
        assert np.array_equal(ka[:13], kb[:13])


def test_session_errors():
    shape = small_shape()
    om = tiny_model(shape)
    s = oracle.OracleSession(om, 8)
    assert s.prefill([1, 2, 99])[0] == oracle.ETOKEN and s.len == 0
    assert s.prefill([-1])[0] == oracle.ETOKEN
    assert s.prefill(list(range(8)))[0] == oracle.ECONTEXT        # tokens >= context
    assert s.prefill(list(range(7)))[0] == 0 and s.len == 7
    assert s.decode(3)[0] == oracle.ECONTEXT
    assert s.truncate(8) == oracle.EINVAL and s.truncate(-1) == oracle.EINVAL
    assert s.truncate(7) == 0 and s.len == 7                        # no-op
    assert s.common_prefix(list(range(5)) + [9, 9]) == 5
    assert s.truncate(2) == 0 and s.len == 2
