"""Device-resident synthetic weights and inputs (torch tensors filled by the
counter-based generator on the GPU, bit-identical to the host fills)."""
from __future__ import annotations

import torch

from . import (BF16, EXPERT_KINDS, F16, F32, GLOBAL_LAYER, KV_K, KV_V, LM_HEAD, LOGITS, TOK,
               TOK_EMBD, TOKENS, ModelShape, dev_fill, layer_tensors, tensor_id, wfmt, kvfmt)


def _empty(shape, fmt, device):
    dt = {F32: torch.float32, BF16: torch.bfloat16, F16: torch.float16, TOK: torch.int32}[fmt]
    return torch.empty(shape, dtype=dt, device=device)


def _stream():
    return torch.cuda.current_stream().cuda_stream


def dev_layer(m: ModelShape, layer: int, seed: int = 0, device="cuda") -> dict:
    out = {}
    for name, kind, shape, sigma in layer_tensors(m):
        if sigma is None:
            t = _empty(shape, F32, device)
            dev_fill(t.data_ptr(), F32, t.numel(), seed, tensor_id(layer, kind), m.gain_sigma,
                     offset=1.0, stream=_stream())
        elif kind in EXPERT_KINDS:
            t = _empty(shape, wfmt(m), device)
            per = t.numel() // m.n_experts
            esz = t.element_size()
            for e in range(m.n_experts):
                dev_fill(t.data_ptr() + e * per * esz, wfmt(m), per, seed,
                         tensor_id(layer, kind, e), sigma, stream=_stream())
        else:
            t = _empty(shape, wfmt(m), device)
            dev_fill(t.data_ptr(), wfmt(m), t.numel(), seed, tensor_id(layer, kind), sigma,
                     stream=_stream())
        out[name] = t
    return out


def dev_embedding(m: ModelShape, seed: int = 0, device="cuda") -> torch.Tensor:
    t = _empty((m.vocab, m.hidden), F16, device)
    dev_fill(t.data_ptr(), F16, t.numel(), seed, tensor_id(GLOBAL_LAYER, TOK_EMBD), m.embd_sigma,
             stream=_stream())
    return t


def dev_lm_head(m: ModelShape, seed: int = 0, device="cuda") -> torch.Tensor:
    t = _empty((m.vocab, m.hidden), wfmt(m), device)
    dev_fill(t.data_ptr(), wfmt(m), t.numel(), seed, tensor_id(GLOBAL_LAYER, LM_HEAD), m.w_sigma,
             stream=_stream())
    return t


def dev_model(m: ModelShape, seed: int = 0, device="cuda"):
    layers = [dev_layer(m, l, seed, device) for l in range(m.n_layers)]
    return dev_embedding(m, seed, device), dev_lm_head(m, seed, device), layers


def fill_kv(m: ModelShape, layer: int, k: torch.Tensor, v: torch.Tensor, n_pos: int, seed: int = 0,
            sigma: float = 1.0) -> None:
    """Seeded K/V contents for positions [0, n_pos) written into cache views [n_ctx][HD]."""
    n = n_pos * m.head_dim
    dev_fill(k.data_ptr(), kvfmt(m), n, seed, tensor_id(layer, KV_K), sigma, stream=_stream())
    dev_fill(v.data_ptr(), kvfmt(m), n, seed, tensor_id(layer, KV_V), sigma, stream=_stream())


def dev_logits(n: int, sigma: float, seed: int = 0, stream_id: int = 0, device="cuda"):
    t = _empty((n,), F32, device)
    dev_fill(t.data_ptr(), F32, n, seed, tensor_id(GLOBAL_LAYER, LOGITS, stream_id), sigma,
             stream=_stream())
    return t
