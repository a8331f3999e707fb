"""Seeded synthetic inputs shared by the oracle checks, the GPU tests and the benchmark.

This package generates inputs only: model shapes of the five workloads, weights,
KV-cache contents, token ids and logits, from a counter-based generator
(``ds4g_synth.h``) that gives bit-identical values on the host and the device.
It holds none of the layer's arithmetic.

Workload shapes follow the ds4 pages ("ds4.c 学习笔记 -- 端到端推理流程", 阶段四 4.2:
64-head MQA, window 128, 256 experts top-6 plus a shared expert; 4.3: 129280-token
vocabulary) with the low ranks and sizes of the synthetic workloads listed below.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, replace

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "libds4g_synth_host.so")
DEV_LIB = os.path.join(HERE, "libds4g_synth_dev.so")

# tensor kinds (must match ds4g_synth.h)
ATTN_NORM, WQ_A, WQ_B, WKV_A, WK_B, WV_B, WO, FFN_NORM, W_ROUTER = 1, 2, 3, 4, 5, 6, 7, 8, 9
W_GATE, W_UP, W_DOWN, WS_GATE, WS_UP, WS_DOWN = 10, 11, 12, 13, 14, 15
TOK_EMBD, LM_HEAD, KV_K, KV_V, TOKENS, LOGITS, MISC = 16, 17, 18, 19, 20, 21, 22
GLOBAL_LAYER = 0xFFFF

F32, BF16, F16, TOK = 0, 1, 2, 3


def tensor_id(layer: int, kind: int, expert: int = 0) -> int:
    return (layer << 32) | (kind << 24) | (expert & 0xFFFFFF)


def scale_for(sigma: float) -> float:
    """float32 multiplier that turns a centred Irwin-Hall(4) integer into N(0, sigma^2)."""
    return float(np.float32(sigma * math.sqrt(3.0) / 65536.0))


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    hidden: int
    n_heads: int
    head_dim: int
    q_rank: int
    kv_rank: int
    window: int
    n_experts: int
    top_k: int
    expert_inter: int
    vocab: int
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    weight_dtype: str = "bf16"      # "bf16" or "f32"
    kv_dtype: str = "bf16"          # "bf16" or "f32"
    w_sigma: float = 0.02
    embd_sigma: float = 1.0
    gain_sigma: float = 0.0         # RMSNorm gains are 1 + N(0, gain_sigma^2)

    def with_(self, **kw) -> "ModelShape":
        return replace(self, **kw)


# Tiny decode: FP32 throughout, seed 0.
TINY = ModelShape("tiny", n_layers=1, hidden=256, n_heads=8, head_dim=32, q_rank=64,
                  kv_rank=64, window=16, n_experts=16, top_k=2, expert_inter=128,
                  vocab=1000, weight_dtype="f32", kv_dtype="f32")
# Single full-width decode layer (BF16 weights, BF16 KV).
LAYER = ModelShape("decode_layer", n_layers=1, hidden=4096, n_heads=64, head_dim=128,
                   q_rank=1024, kv_rank=512, window=128, n_experts=256, top_k=6,
                   expert_inter=1024, vocab=129280)
# Eight layers of the full-width shapes (stack, prefill and resync workloads).
STACK = LAYER.with_(name="stack8", n_layers=8)


def layer_tensors(m: ModelShape):
    """(name, kind, shape, sigma) of one layer's tensors, in the ABI's layout."""
    H, NH, HD, RQ, RKV = m.hidden, m.n_heads, m.head_dim, m.q_rank, m.kv_rank
    E, I = m.n_experts, m.expert_inter
    return [
        ("attn_norm", ATTN_NORM, (H,), None),
        ("wq_a", WQ_A, (RQ, H), m.w_sigma),
        ("wq_b", WQ_B, (NH * HD, RQ), m.w_sigma),
        ("wkv_a", WKV_A, (RKV, H), m.w_sigma),
        ("wk_b", WK_B, (HD, RKV), m.w_sigma),
        ("wv_b", WV_B, (HD, RKV), m.w_sigma),
        ("wo", WO, (H, NH * HD), m.w_sigma),
        ("ffn_norm", FFN_NORM, (H,), None),
        ("w_router", W_ROUTER, (E, H), m.w_sigma),
        ("w_gate", W_GATE, (E, I, H), m.w_sigma),
        ("w_up", W_UP, (E, I, H), m.w_sigma),
        ("w_down", W_DOWN, (E, H, I), m.w_sigma),
        ("ws_gate", WS_GATE, (I, H), m.w_sigma),
        ("ws_up", WS_UP, (I, H), m.w_sigma),
        ("ws_down", WS_DOWN, (H, I), m.w_sigma),
    ]


EXPERT_KINDS = (W_GATE, W_UP, W_DOWN)


# --------------------------------------------------------------------------- build

def _newer(target: str, *srcs: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in srcs)


def build(cuda: bool = True, force: bool = False) -> None:
    hdr = os.path.join(HERE, "ds4g_synth.h")
    src = os.path.join(HERE, "synth_host.c")
    if force or _newer(HOST_LIB, src, hdr):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", HOST_LIB, src], cwd=HERE)
    if cuda:
        dsrc = os.path.join(HERE, "synth_dev.cu")
        if force or _newer(DEV_LIB, dsrc, hdr):
            subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                                   "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-o", DEV_LIB,
                                   dsrc], cwd=HERE)


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            build(cuda=False)
        lib = ctypes.CDLL(HOST_LIB)
        u64, sz = ctypes.c_uint64, ctypes.c_size_t
        vp = ctypes.c_void_p
        lib.synth_fill_f32.argtypes = [vp, sz, u64, u64, ctypes.c_float, ctypes.c_float, u64]
        lib.synth_fill_bf16.argtypes = [vp, sz, u64, u64, ctypes.c_float, u64]
        lib.synth_fill_f16.argtypes = [vp, sz, u64, u64, ctypes.c_float, u64]
        lib.synth_fill_tokens.argtypes = [vp, sz, u64, u64, ctypes.c_uint32, u64]
        lib.synth_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.synth_f32_to_bf16.restype = ctypes.c_uint16
        lib.synth_f32_to_f16.argtypes = [ctypes.c_float]
        lib.synth_f32_to_f16.restype = ctypes.c_uint16
        lib.synth_ih4.argtypes = [u64, u64, u64]
        lib.synth_ih4.restype = ctypes.c_int32
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError(f"{DEV_LIB} is not built; call synth.build()")
        lib = ctypes.CDLL(DEV_LIB)
        lib.synth_fill_dev.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t,
                                       ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                                       ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32,
                                       ctypes.c_void_p]
        lib.synth_fill_dev.restype = ctypes.c_int
        _dev = lib
    return _dev


# --------------------------------------------------------------------------- host fills

def host_fill(fmt: int, n: int, seed: int, tid: int, sigma: float = 1.0, offset: float = 0.0,
              index0: int = 0, vocab: int = 0) -> np.ndarray:
    lib = _host_lib()
    if fmt == F32:
        a = np.empty(n, dtype=np.float32)
        lib.synth_fill_f32(a.ctypes.data, n, seed, tid, scale_for(sigma), offset, index0)
    elif fmt == BF16:
        a = np.empty(n, dtype=np.uint16)
        lib.synth_fill_bf16(a.ctypes.data, n, seed, tid, scale_for(sigma), index0)
    elif fmt == F16:
        a = np.empty(n, dtype=np.uint16)
        lib.synth_fill_f16(a.ctypes.data, n, seed, tid, scale_for(sigma), index0)
    elif fmt == TOK:
        a = np.empty(n, dtype=np.int32)
        lib.synth_fill_tokens(a.ctypes.data, n, seed, tid, vocab, index0)
    else:
        raise ValueError(fmt)
    return a


def wfmt(m: ModelShape) -> int:
    return F32 if m.weight_dtype == "f32" else BF16


def kvfmt(m: ModelShape) -> int:
    return F32 if m.kv_dtype == "f32" else BF16


def host_layer(m: ModelShape, layer: int, seed: int = 0) -> dict:
    """All tensors of one layer as numpy arrays (uint16 bits for bf16, float32 for f32)."""
    out = {}
    for name, kind, shape, sigma in layer_tensors(m):
        n = int(np.prod(shape))
        if sigma is None:   # RMSNorm gain
            a = host_fill(F32, n, seed, tensor_id(layer, kind), m.gain_sigma, 1.0)
        elif kind in EXPERT_KINDS:
            per = n // m.n_experts
            a = np.empty(n, dtype=np.float32 if wfmt(m) == F32 else np.uint16)
            for e in range(m.n_experts):
                a[e * per:(e + 1) * per] = host_fill(wfmt(m), per, seed, tensor_id(layer, kind, e),
                                                     sigma)
        else:
            a = host_fill(wfmt(m), n, seed, tensor_id(layer, kind), sigma)
        out[name] = a.reshape(shape)
    return out


def host_embedding(m: ModelShape, seed: int = 0) -> np.ndarray:
    n = m.vocab * m.hidden
    return host_fill(F16, n, seed, tensor_id(GLOBAL_LAYER, TOK_EMBD), m.embd_sigma).reshape(
        m.vocab, m.hidden)


def host_lm_head(m: ModelShape, seed: int = 0) -> np.ndarray:
    n = m.vocab * m.hidden
    return host_fill(wfmt(m), n, seed, tensor_id(GLOBAL_LAYER, LM_HEAD), m.w_sigma).reshape(
        m.vocab, m.hidden)


def host_tokens(n: int, vocab: int, seed: int = 0, stream: int = 0, index0: int = 0) -> np.ndarray:
    return host_fill(TOK, n, seed, tensor_id(GLOBAL_LAYER, TOKENS, stream), index0=index0,
                     vocab=vocab)


def host_kv(m: ModelShape, layer: int, n_pos: int, seed: int = 0, sigma: float = 1.0):
    """Seeded K and V cache contents for positions [0, n_pos), in the KV storage format."""
    n = n_pos * m.head_dim
    k = host_fill(kvfmt(m), n, seed, tensor_id(layer, KV_K), sigma).reshape(n_pos, m.head_dim)
    v = host_fill(kvfmt(m), n, seed, tensor_id(layer, KV_V), sigma).reshape(n_pos, m.head_dim)
    return k, v


def host_logits(n: int, sigma: float, seed: int = 0, stream: int = 0) -> np.ndarray:
    return host_fill(F32, n, seed, tensor_id(GLOBAL_LAYER, LOGITS, stream), sigma)


# --------------------------------------------------------------------------- device fills

def dev_fill(ptr: int, fmt: int, n: int, seed: int, tid: int, sigma: float = 1.0,
             offset: float = 0.0, index0: int = 0, vocab: int = 0, stream: int = 0) -> None:
    rc = _dev_lib().synth_fill_dev(ptr, fmt, n, seed, tid, scale_for(sigma), offset, index0,
                                   vocab, stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_dev failed with CUDA error {rc}")
