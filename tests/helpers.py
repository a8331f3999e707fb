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

    def __init__(self, shape, seed=0, keep_layers=True):
        self.shape = shape
        self.seed = seed
        self.cfg = oracle.config_from(shape)
        self.emb = synth.host_embedding(shape, seed)
        self.lm = synth.host_lm_head(shape, seed)
        self.keep = keep_layers
        self._layers = {}

    def layer(self, l):
        if l in self._layers:
            return self._layers[l]
        w = synth.host_layer(self.shape, l, self.seed)
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
