"""ctypes wrapper of the plain C oracle (ds4_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline / reference legs may import this module; the product library never does.
It shares no code with the CUDA library; both only read inputs made by ``synth``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libds4_oracle.so")
SRC = os.path.join(HERE, "ds4_oracle.c")
HDR = os.path.join(HERE, "ds4_oracle.h")

F32, BF16 = 0, 1
OK, EINVAL, ECONTEXT, ETOKEN = 0, -1, -2, -3


def build(force: bool = False) -> None:
    if force or not os.path.exists(LIB) or max(os.path.getmtime(SRC), os.path.getmtime(HDR)) > \
            os.path.getmtime(LIB):
        # ISO C, no contraction of a*b+c into fused multiply-adds, no fast-math.
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", LIB, SRC, "-lm"], cwd=HERE)


class Config(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("n_layers", "hidden", "n_heads", "head_dim", "q_rank",
                                       "kv_rank", "window", "n_experts", "top_k",
                                       "expert_inter", "vocab")] + \
               [("rope_base", C.c_double), ("rms_eps", C.c_double),
                ("weight_dtype", C.c_int), ("kv_dtype", C.c_int)]


class Layer(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("attn_norm", "wq_a", "wq_b", "wkv_a", "wk_b", "wv_b",
                                          "wo", "ffn_norm", "w_router", "w_gate", "w_up",
                                          "w_down", "ws_gate", "ws_up", "ws_down")]


class Model(C.Structure):
    _fields_ = [("tok_embd", C.c_void_p), ("lm_head", C.c_void_p),
                ("layers", C.POINTER(Layer))]


class KV(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p)]


class Trace(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("xn1", "cq", "ckv", "q", "k", "v", "attn", "x_mid",
                                          "xn2", "scores", "ids", "weights", "h", "moe")]


class SampleInfo(C.Structure):
    _fields_ = [("n_kept", C.c_int), ("sum_all", C.c_double), ("sum_kept", C.c_double),
                ("cut_sum_margin", C.c_double), ("cut_gap_margin", C.c_double),
                ("cdf_margin", C.c_double), ("cut_index", C.c_int), ("cut_next_index", C.c_int),
                ("cut_p", C.c_double),
                ("p_rms", C.c_double), ("minp_margin", C.c_double)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(LIB)
        vp, i32, d = C.c_void_p, C.c_int, C.c_double
        sig = {
            "orc_f16_value": ([C.c_uint16], d),
            "orc_bf16_value": ([C.c_uint16], d),
            "orc_round_bf16": ([d], C.c_uint16),
            "orc_embed": ([vp, vp, C.c_int32, vp], None),
            "orc_rmsnorm": ([i32, vp, vp, d, vp], None),
            "orc_matvec": ([i32, vp, i32, i32, vp, vp], None),
            "orc_rope": ([i32, i32, d, vp], None),
            "orc_kv_store": ([vp, vp, i32, vp, vp], None),
            "orc_attention": ([vp, vp, i32, vp, vp], None),
            "orc_topk": ([vp, i32, i32, vp], None),
            "orc_router": ([vp, vp, vp, vp, vp, vp], None),
            "orc_swiglu_expert": ([vp, vp, vp, vp, vp, vp, vp], None),
            "orc_layer_step": ([vp, vp, vp, i32, vp, vp], None),
            "orc_layer_step_ids": ([vp, vp, vp, i32, vp, vp, vp], None),
            "orc_lm_head": ([vp, vp, vp, vp], None),
            "orc_argmax": ([vp, i32], C.c_int32),
            "orc_sample": ([vp, i32, d, d, d, vp], C.c_int32),
            "orc_sample_min_p": ([vp, i32, d, d, d, d, vp], C.c_int32),
            "orc_xorshift64s": ([vp], C.c_uint64),
            "orc_uniform": ([vp], d),
            "orc_session_new": ([vp, i32], vp),
            "orc_session_free": ([vp], None),
            "orc_session_len": ([vp], i32),
            "orc_session_kv": ([vp, i32], C.POINTER(KV)),
            "orc_session_tokens": ([vp], C.POINTER(C.c_int32)),
            "orc_session_restore": ([vp, vp, i32], i32),
            "orc_prefill": ([vp, vp, vp, i32, vp, vp], i32),
            "orc_decode_step": ([vp, vp, C.c_int32, vp, vp], i32),
            "orc_common_prefix": ([vp, vp, i32], i32),
            "orc_truncate": ([vp, i32], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def config_from(shape) -> Config:
    """Config from a synth.ModelShape (or any object with the same attributes)."""
    c = Config()
    for n in ("n_layers", "hidden", "n_heads", "head_dim", "q_rank", "kv_rank", "window",
              "n_experts", "top_k", "expert_inter", "vocab"):
        setattr(c, n, int(getattr(shape, n)))
    c.rope_base = float(shape.rope_base)
    c.rms_eps = float(shape.rms_eps)
    c.weight_dtype = F32 if shape.weight_dtype == "f32" else BF16
    c.kv_dtype = F32 if shape.kv_dtype == "f32" else BF16
    return c


def layer_struct(w: dict) -> Layer:
    """Layer struct over a dict of contiguous numpy arrays (kept alive by the caller)."""
    L = Layer()
    for name, _ in Layer._fields_:
        a = w[name]
        assert a.flags["C_CONTIGUOUS"]
        setattr(L, name, a.ctypes.data)
    return L


class OracleModel:
    """Weights of a whole model held on the host, plus the C model struct."""

    def __init__(self, shape, layers: list, tok_embd: np.ndarray, lm_head: np.ndarray):
        self.shape = shape
        self.cfg = config_from(shape)
        self._layers = layers
        self._tok = np.ascontiguousarray(tok_embd)
        self._lm = np.ascontiguousarray(lm_head)
        self._arr = (Layer * len(layers))(*[layer_struct(w) for w in layers])
        self.model = Model(self._tok.ctypes.data, self._lm.ctypes.data, self._arr)


class OracleSession:
    def __init__(self, om: OracleModel, n_ctx: int):
        self.om = om
        self.cfg = om.cfg
        self.ptr = lib().orc_session_new(C.byref(om.cfg), n_ctx)
        if not self.ptr:
            raise ValueError("orc_session_new failed")

    def __del__(self):
        if getattr(self, "ptr", None):
            lib().orc_session_free(self.ptr)
            self.ptr = None

    @property
    def len(self) -> int:
        return lib().orc_session_len(self.ptr)

    def prefill(self, tokens, want_logits=True, want_hidden=False):
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = len(t)
        logits = np.empty(self.cfg.vocab, dtype=np.float64) if want_logits else None
        hidden = np.empty((n, self.cfg.hidden), dtype=np.float64) if want_hidden else None
        rc = lib().orc_prefill(self.ptr, C.byref(self.om.model), _p(t), n, _p(logits),
                               _p(hidden))
        return rc, logits, hidden

    def decode(self, token: int, want_hidden=False):
        logits = np.empty(self.cfg.vocab, dtype=np.float64)
        hidden = np.empty(self.cfg.hidden, dtype=np.float64) if want_hidden else None
        rc = lib().orc_decode_step(self.ptr, C.byref(self.om.model), int(token), _p(logits),
                                   _p(hidden))
        return rc, logits, hidden

    def truncate(self, cp: int) -> int:
        return lib().orc_truncate(self.ptr, cp)

    def common_prefix(self, tokens) -> int:
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        return lib().orc_common_prefix(self.ptr, _p(t), len(t))

    def kv(self, layer: int):
        """numpy views (n_ctx, head_dim) of the layer's K and V caches (storage format)."""
        kvp = lib().orc_session_kv(self.ptr, layer).contents
        return kvp

    def restore(self, tokens) -> int:
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        return lib().orc_session_restore(self.ptr, _p(t), len(t))


def kv_views(sess: OracleSession, layer: int, n_ctx: int):
    kvp = sess.kv(layer)
    dt = np.uint16 if sess.cfg.kv_dtype == BF16 else np.float32
    hd = sess.cfg.head_dim
    nbytes = n_ctx * hd * np.dtype(dt).itemsize
    k = np.frombuffer((C.c_char * nbytes).from_address(kvp.k), dtype=dt).reshape(n_ctx, hd)
    v = np.frombuffer((C.c_char * nbytes).from_address(kvp.v), dtype=dt).reshape(n_ctx, hd)
    return k, v


def make_trace(cfg: Config) -> tuple[Trace, dict]:
    H, QD, K, I, E = cfg.hidden, cfg.n_heads * cfg.head_dim, cfg.top_k, cfg.expert_inter, \
        cfg.n_experts
    bufs = {
        "xn1": np.zeros(H), "cq": np.zeros(cfg.q_rank), "ckv": np.zeros(cfg.kv_rank),
        "q": np.zeros(QD), "k": np.zeros(cfg.head_dim), "v": np.zeros(cfg.head_dim),
        "attn": np.zeros(QD), "x_mid": np.zeros(H), "xn2": np.zeros(H),
        "scores": np.zeros(E, dtype=np.float32), "ids": np.zeros(K, dtype=np.int32),
        "weights": np.zeros(K), "h": np.zeros((K + 1) * I), "moe": np.zeros(H),
    }
    t = Trace(**{k: v.ctypes.data for k, v in bufs.items()})
    return t, bufs


def layer_step(cfg: Config, layer: Layer, kv: KV, pos: int, x: np.ndarray, trace=None):
    """x (float64, [H]) is updated in place; kv is appended at pos."""
    assert x.dtype == np.float64 and x.flags["C_CONTIGUOUS"]
    lib().orc_layer_step(C.byref(cfg), C.byref(layer), C.byref(kv), pos, x.ctypes.data,
                         C.byref(trace) if trace is not None else None)


def layer_step_ids(cfg: Config, layer: Layer, kv: KV, pos: int, x: np.ndarray, ids, trace=None):
    """layer_step with the router's choice given (K expert ids in combine order)."""
    assert x.dtype == np.float64 and x.flags["C_CONTIGUOUS"]
    a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    assert a.shape == (cfg.top_k,)
    lib().orc_layer_step_ids(C.byref(cfg), C.byref(layer), C.byref(kv), pos, x.ctypes.data,
                             C.byref(trace) if trace is not None else None, a.ctypes.data)


def sample(logits: np.ndarray, temperature: float, top_p: float, u: float, min_p: float = 0.0):
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    info = SampleInfo()
    if min_p > 0.0:
        tok = lib().orc_sample_min_p(lg.ctypes.data, len(lg), temperature, top_p, min_p, u,
                                     C.byref(info))
    else:
        tok = lib().orc_sample(lg.ctypes.data, len(lg), temperature, top_p, u, C.byref(info))
    return tok, info


def argmax(logits: np.ndarray) -> int:
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    return lib().orc_argmax(lg.ctypes.data, len(lg))


def uniform(state: int):
    """One uniform draw; returns (u, new_state)."""
    s = C.c_uint64(state)
    u = lib().orc_uniform(C.byref(s))
    return u, s.value
