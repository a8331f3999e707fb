"""Shared set-up for the parity tests: the same seeded inputs on the GPU (through
the C ABI) and on the host (for the oracle), and the comparison rules."""
from __future__ import annotations

import ctypes as C

import numpy as np

import oracle
import synth

# Tolerances: max |gpu - ref| / max |ref| per tensor (normwise relative).
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def tol_for(shape) -> float:
    return TOL_F32 if shape.weight_dtype == "f32" else TOL_BF16


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    scale = np.max(np.abs(ref))
    if scale == 0.0:
        return float(np.max(np.abs(gpu)))
    return float(np.max(np.abs(gpu - ref)) / scale)


def to_np(t) -> np.ndarray:
    """Device tensor (f32 / bf16 / int) -> float64 numpy on the host."""
    import torch
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy().astype(np.float64)


def kv_to_f64(shape, arr: np.ndarray) -> np.ndarray:
    """Oracle KV storage (uint16 bf16 bits or float32) -> float64."""
    if shape.kv_dtype == "f32":
        return arr.astype(np.float64)
    return (arr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------- GPU side

def gpu_model(shape, seed=0, prefill_chunk=0, decode_kernel=0, prefill_kernel=0):
    import prefill_decode_layer_gb300 as pdl
    from synth import torch_weights as tw
    emb, lm, layers = tw.dev_model(shape, seed)
    return pdl.Model(shape, emb, lm, layers, prefill_chunk=prefill_chunk,
                     decode_kernel=decode_kernel, prefill_kernel=prefill_kernel)


DECODE_KERNELS = [0, 1]   # persistent single launch (when available), one kernel per stage


# ----------------------------------------------------------------------------- oracle side

class LazyOracleModel:
    """Host weights of a model, generated one layer at a time (large models do not
    fit in host memory all at once)."""

    def __init__(self, shape, seed=0, keep_layers=True, weight_layer=None):
        self.shape = shape
        self.seed = seed
        # layer -> index of the generated weight set it uses (a deep model may alias
        # the weights of a few generated layers)
        self.weight_layer = weight_layer or (lambda l: l)
        self.cfg = oracle.config_from(shape)
        self.emb = synth.host_embedding(shape, seed)
        self.lm = synth.host_lm_head(shape, seed)
        self.keep = keep_layers
        self._layers = {}

    def layer(self, l):
        if l in self._layers:
            return self._layers[l]
        w = synth.host_layer(self.shape, self.weight_layer(l), self.seed)
        st = oracle.layer_struct(w)
        if self.keep:
            self._layers[l] = (w, st)
        return (w, st)

    def full(self) -> oracle.OracleModel:
        layers = [self.layer(l)[0] for l in range(self.shape.n_layers)]
        return oracle.OracleModel(self.shape, layers, self.emb, self.lm)


def oracle_embed(om: LazyOracleModel, token: int) -> np.ndarray:
    x = np.zeros(om.shape.hidden)
    oracle.lib().orc_embed(C.byref(om.cfg), om.emb.ctypes.data, int(token), x.ctypes.data)
    return x


def oracle_lm_head(om: LazyOracleModel, x: np.ndarray) -> np.ndarray:
    out = np.zeros(om.shape.vocab)
    oracle.lib().orc_lm_head(C.byref(om.cfg), om.lm.ctypes.data, x.ctypes.data, out.ctypes.data)
    return out


class OracleKV:
    """Per-layer host KV caches in the storage format, for direct layer stepping."""

    def __init__(self, shape, n_ctx):
        dt = np.float32 if shape.kv_dtype == "f32" else np.uint16
        self.k = [np.zeros((n_ctx, shape.head_dim), dtype=dt) for _ in range(shape.n_layers)]
        self.v = [np.zeros((n_ctx, shape.head_dim), dtype=dt) for _ in range(shape.n_layers)]

    def struct(self, l):
        return oracle.KV(self.k[l].ctypes.data, self.v[l].ctypes.data)


def oracle_layer(om: LazyOracleModel, kv: OracleKV, l: int, pos: int, x: np.ndarray,
                 trace=False):
    """One layer step at pos on x (updated in place); returns the trace dict or None."""
    w, st = om.layer(l)
    kvs = kv.struct(l)
    if trace:
        tr, bufs = oracle.make_trace(om.cfg)
        oracle.layer_step(om.cfg, st, kvs, pos, x, tr)
        return bufs
    oracle.layer_step(om.cfg, st, kvs, pos, x, None)
    return None


# ----------------------------------------------------------------------------- teacher forcing

def near_tie(scores, k) -> bool:
    """The k-th and (k+1)-th router scores are within the tie band (1e-3 of the
    largest magnitude): the GPU may then choose either expert."""
    s = np.sort(np.asarray(scores, dtype=np.float64))[::-1]
    return s[k - 1] - s[k] <= 1e-3 * np.max(np.abs(s))


def gpu_kv_rows(sess, layer, lo, hi):
    """GPU K and V rows [lo, hi) of a layer in the oracle's storage format (raw BF16
    bits as uint16, or float32)."""
    import torch
    k, v = sess.kv(layer)
    if k.dtype == torch.bfloat16:
        return (k[lo:hi].contiguous().view(torch.int16).cpu().numpy().view(np.uint16),
                v[lo:hi].contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
    return k[lo:hi].cpu().numpy(), v[lo:hi].cpu().numpy()


def teacher_forced_layer(om: LazyOracleModel, l: int, p: int, x_in: np.ndarray, k_win, v_win,
                         ids=None):
    """Oracle layer l at position p, started from the GPU's input x_in and the GPU's
    K/V rows of the window before p (k_win, v_win: rows max(0, p-W+1) .. p-1); with
    ids, the router's choice is given instead of the top-k.
    Returns (x_out, trace, k_new, v_new); k_new/v_new in the storage format."""
    shape = om.shape
    dt = np.float32 if shape.kv_dtype == "f32" else np.uint16
    k = np.zeros((p + 1, shape.head_dim), dtype=dt)
    v = np.zeros((p + 1, shape.head_dim), dtype=dt)
    lo = p - len(k_win)
    k[lo:p] = k_win
    v[lo:p] = v_win
    w, st = om.layer(l)
    tr, bufs = oracle.make_trace(om.cfg)
    x = np.array(x_in, dtype=np.float64)
    kv = oracle.KV(k.ctypes.data, v.ctypes.data)
    if ids is None:
        oracle.layer_step(om.cfg, st, kv, p, x, tr)
    else:
        oracle.layer_step_ids(om.cfg, st, kv, p, x, ids, tr)
    return x, bufs, k[p].copy(), v[p].copy()


def tie_choices(scores, k, limit=20):
    """Every choice of k experts that the tie band allows: experts whose score is
    more than the band above the (k+1)-th score are certainly chosen, and the rest
    come from those within the band of the k-th score.  Each choice is in
    descending score order (ties to the lower id)."""
    import itertools
    s = np.asarray(scores, dtype=np.float64)
    order = np.argsort(-s, kind="stable")
    band = 1e-3 * np.max(np.abs(s))
    kth, next_ = s[order[k - 1]], s[order[k]]
    sure = [int(i) for i in order if s[i] > next_ + band]
    cand = [int(i) for i in order if i not in sure and s[i] >= kth - band]
    need = k - len(sure)
    out = []
    for comb in itertools.combinations(cand, need):
        chosen = sorted(sure + list(comb), key=lambda i: (-s[i], i))
        out.append(chosen)
        if len(out) >= limit:
            break
    return out


def check_probes(om: LazyOracleModel, sess, positions, rec: np.ndarray, layers=None,
                 router_ids=None):
    """Teacher-forced parity at recorded positions: for every layer l and position p,
    the oracle starts from the GPU's residual entering layer l at p (rec[i][l]) and
    the GPU's K/V window, and must reproduce the GPU's new K/V row at p and the
    GPU's residual entering layer l + 1 (rec[i][l + 1]).  router_ids: {p: [ids of
    layer 0..L-1]} for decoded positions, compared with the oracle's choice.

    Where the router's k-th and (k+1)-th scores lie within the tie band, either
    expert is a correct choice: the GPU's ids (when known) must be one of the
    choices the band allows and the output must match the oracle run with them;
    otherwise the output must match the oracle run with one of those choices.
    Returns (checked, ties): every position-layer is checked; ties lists those
    decided through the tie band."""
    shape = om.shape
    W, K = shape.window, shape.top_k
    layers = range(shape.n_layers) if layers is None else layers
    checked, ties = 0, []
    for l in layers:
        for i, p in enumerate(positions):
            lo = max(0, p - W + 1)
            kb, vb = gpu_kv_rows(sess, l, lo, p + 1)
            x, tr, kn, vn = teacher_forced_layer(om, l, p, rec[i][l], kb[:-1], vb[:-1])
            assert rel_err(kv_to_f64(shape, kb[-1]), kv_to_f64(shape, kn)) <= TOL_BF16, \
                f"K row: layer {l} position {p}"
            assert rel_err(kv_to_f64(shape, vb[-1]), kv_to_f64(shape, vn)) <= TOL_BF16, \
                f"V row: layer {l} position {p}"
            gids = None if router_ids is None or p not in router_ids else list(router_ids[p][l])
            if not near_tie(tr["scores"], K):
                if gids is not None:
                    assert list(tr["ids"]) == gids, f"ids: layer {l} position {p}"
                assert rel_err(rec[i][l + 1], x) <= TOL_BF16, f"output: layer {l} position {p}"
            else:
                choices = tie_choices(tr["scores"], K)
                if gids is not None:
                    assert sorted(gids) in [sorted(c) for c in choices], \
                        f"ids outside the tie band: layer {l} position {p}"
                    choices = [gids]
                errs = []
                for c in choices:
                    xc = teacher_forced_layer(om, l, p, rec[i][l], kb[:-1], vb[:-1], ids=c)[0]
                    errs.append(rel_err(rec[i][l + 1], xc))
                assert min(errs) <= TOL_BF16, f"output at a tie: layer {l} position {p}: {errs}"
                ties.append((p, l))
            checked += 1
        om._layers.pop(l, None)
    return checked, ties
