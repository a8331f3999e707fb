"""ctypes binding of libds4g.so (include/ds4g.h): argument marshalling only.

Device memory and streams come from PyTorch; pointers and sizes cross the C ABI.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libds4g.so")

F32, BF16 = 0, 1
OK, EINVAL, ECONTEXT, ETOKEN, ECUDA, ETIMEOUT, ESIZE, ENONFINITE = 0, -1, -2, -3, -4, -5, -6, -7
DEBUG = {"x": 0, "cqkv": 1, "q": 2, "attn": 3, "xmid": 4, "xn2": 5, "scores": 6, "h": 7,
         "hidden": 8, "prefill_x": 9, "status": 10, "prefill_layer_x": 11}


KERNEL_KINDS = ("qkv_a", "qkv_b", "attn", "wo", "router", "expert_gu", "expert_down", "lm_head",
                "p_embed", "p_norm", "p_qkv_a", "p_q_b", "p_kv_b", "p_attn", "p_wo", "p_router", "p_topk",
                "p_group", "p_gate_up", "p_shared_gu", "p_down", "p_shared_down", "p_combine")


class Ds4gError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {lib().ds4g_strerror(code).decode()} ({code})")
        self.code = code


class Config(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("n_layers", "hidden", "n_heads", "head_dim", "q_rank",
                                       "kv_rank", "window", "n_experts", "top_k",
                                       "expert_inter", "vocab")] + \
               [("rope_base", C.c_float), ("rms_eps", C.c_float), ("weight_dtype", C.c_int),
                ("kv_dtype", C.c_int), ("prefill_chunk", C.c_int), ("decode_kernel", C.c_int),
                ("prefill_kernel", C.c_int)]


LAYER_FIELDS = ("attn_norm", "wq_a", "wq_b", "wkv_a", "wk_b", "wv_b", "wo", "ffn_norm",
                "w_router", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in LAYER_FIELDS]


class Weights(C.Structure):
    _fields_ = [("tok_embd", C.c_void_p), ("lm_head", C.c_void_p),
                ("layers", C.POINTER(LayerWeights))]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                              "(there is no fallback implementation)")
        L = C.CDLL(LIB_PATH)
        vp, i32, sz = C.c_void_p, C.c_int, C.c_size_t
        sig = {
            "ds4g_model_create": ([vp, vp, vp], i32),
            "ds4g_model_destroy": ([vp], None),
            "ds4g_session_bytes": ([vp, i32], sz),
            "ds4g_session_create": ([vp, i32, vp, sz, vp, vp], i32),
            "ds4g_session_destroy": ([vp], None),
            "ds4g_prefill": ([vp, vp, i32], i32),
            "ds4g_decode_step": ([vp, C.c_int32], i32),
            "ds4g_decode_layers": ([vp, C.c_int32], i32),
            "ds4g_sample_static": ([vp, i32, C.c_float, C.c_float, vp, vp], C.c_int32),
            "ds4g_session_hidden": ([vp], vp),
            "ds4g_session_common_prefix": ([vp, vp, i32], i32),
            "ds4g_session_truncate": ([vp, i32], i32),
            "ds4g_session_sync": ([vp, vp, i32, vp], i32),
            "ds4g_checkpoint_bytes": ([vp, i32], sz),
            "ds4g_session_save": ([vp, vp, sz], i32),
            "ds4g_session_load": ([vp, vp, sz], i32),
            "ds4g_session_rewrite_from_common": ([vp, vp, i32, i32], i32),
            "ds4g_session_len": ([vp], i32),
            "ds4g_session_logits": ([vp], vp),
            "ds4g_session_kv": ([vp, i32, vp, vp], i32),
            "ds4g_session_restore": ([vp, vp, i32], i32),
            "ds4g_session_router": ([vp, i32, vp, vp], i32),
            "ds4g_session_debug": ([vp, i32], vp),
            "ds4g_sample_workspace_bytes": ([i32], sz),
            "ds4g_session_launches": ([vp], C.c_uint64),
            "ds4g_session_status": ([vp], i32),
            "ds4g_session_set_trace": ([vp, vp, sz], i32),
            "ds4g_session_set_probe": ([vp, vp, i32, vp], i32),
            "ds4g_decode_layers_host": ([vp, C.c_int32, vp], i32),
            "ds4g_decode_sample": ([vp, C.c_int32, C.c_float, C.c_float, vp, vp, sz], C.c_int32),
            "ds4g_session_set_timing": ([vp, i32], i32),
            "ds4g_session_timing": ([vp, vp, vp, i32], i32),
            "ds4g_sample": ([vp, i32, C.c_float, C.c_float, vp, vp, sz, vp], C.c_int32),
            "ds4g_sample_u": ([vp, i32, C.c_float, C.c_float, C.c_uint32, vp, sz, vp], C.c_int32),
            "ds4g_sample_min_p": ([vp, i32, C.c_float, C.c_float, C.c_float, vp, vp, sz, vp], C.c_int32),
            "ds4g_sample_u_min_p": ([vp, i32, C.c_float, C.c_float, C.c_float, C.c_uint32, vp, sz, vp],
                                    C.c_int32),
            "ds4g_strerror": ([i32], C.c_char_p),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(rc: int, what: str) -> int:
    if rc < 0:
        raise Ds4gError(rc, what)
    return rc


DECODE_AUTO, DECODE_STAGED = 0, 1
PREFILL_AUTO, PREFILL_SIMT, PREFILL_HILO = 0, 1, 2


def config_struct(shape, prefill_chunk: int = 0, decode_kernel: int = DECODE_AUTO,
                  prefill_kernel: int = PREFILL_AUTO) -> Config:
    c = Config()
    for n in ("n_layers", "hidden", "n_heads", "head_dim", "q_rank", "kv_rank", "window",
              "n_experts", "top_k", "expert_inter", "vocab"):
        setattr(c, n, int(getattr(shape, n)))
    c.rope_base = float(shape.rope_base)
    c.rms_eps = float(shape.rms_eps)
    c.weight_dtype = F32 if shape.weight_dtype == "f32" else BF16
    c.kv_dtype = F32 if shape.kv_dtype == "f32" else BF16
    c.prefill_chunk = int(prefill_chunk)
    c.decode_kernel = int(decode_kernel)
    c.prefill_kernel = int(prefill_kernel)
    return c


def session_bytes(shape, n_ctx: int, prefill_chunk: int = 0) -> int:
    c = config_struct(shape, prefill_chunk)
    return lib().ds4g_session_bytes(C.byref(c), n_ctx)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


class Model:
    """Weights are device tensors owned by the caller (kept referenced here)."""

    def __init__(self, shape, tok_embd: torch.Tensor, lm_head: torch.Tensor, layers: list,
                 prefill_chunk: int = 0, decode_kernel: int = DECODE_AUTO,
                 prefill_kernel: int = PREFILL_AUTO):
        self.shape = shape
        self.cfg = config_struct(shape, prefill_chunk, decode_kernel, prefill_kernel)
        self._keep = (tok_embd, lm_head, layers)
        arr = (LayerWeights * len(layers))()
        for i, w in enumerate(layers):
            for n in LAYER_FIELDS:
                setattr(arr[i], n, w[n].data_ptr())
        self._arr = arr
        wts = Weights(tok_embd.data_ptr(), lm_head.data_ptr(), arr)
        h = C.c_void_p()
        _check(lib().ds4g_model_create(C.byref(self.cfg), C.byref(wts), C.byref(h)),
               "ds4g_model_create")
        self.ptr = h.value

    def __del__(self):
        if getattr(self, "ptr", None) and _lib is not None:
            _lib.ds4g_model_destroy(self.ptr)
            self.ptr = None


class Session:
    def __init__(self, model: Model, n_ctx: int, stream=None, device="cuda"):
        self.model = model
        self.n_ctx = n_ctx
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        nbytes = lib().ds4g_session_bytes(C.byref(model.cfg), n_ctx)
        if nbytes == 0:
            raise Ds4gError(EINVAL, "ds4g_session_bytes")
        self.mem = torch.empty(nbytes, dtype=torch.uint8, device=device)
        h = C.c_void_p()
        _check(lib().ds4g_session_create(model.ptr, n_ctx, self.mem.data_ptr(), nbytes,
                                         _stream_ptr(self.stream), C.byref(h)),
               "ds4g_session_create")
        self.ptr = h.value

    def __del__(self):
        if getattr(self, "ptr", None) and _lib is not None:
            _lib.ds4g_session_destroy(self.ptr)
            self.ptr = None

    # -- calls ---------------------------------------------------------------
    def prefill(self, tokens) -> int:
        t = (C.c_int32 * len(tokens))(*[int(x) for x in tokens])
        return lib().ds4g_prefill(self.ptr, t, len(tokens))

    def decode(self, token: int) -> int:
        return lib().ds4g_decode_step(self.ptr, int(token))

    def decode_layers(self, token: int) -> int:
        """One token through every layer without the lm_head."""
        return lib().ds4g_decode_layers(self.ptr, int(token))

    def decode_layers_host(self, token: int, hidden_host: torch.Tensor) -> int:
        """ds4g_decode_layers with the final hidden state copied into hidden_host (a
        host float32 tensor of hidden elements, pinned for speed)."""
        assert hidden_host.dtype == torch.float32 and not hidden_host.is_cuda
        assert hidden_host.numel() == self.model.shape.hidden and hidden_host.is_contiguous()
        return lib().ds4g_decode_layers_host(self.ptr, int(token), hidden_host.data_ptr())

    def decode_sample(self, token: int, temperature: float, top_p: float, rng_state, ws: torch.Tensor):
        """ds4g_decode_sample: one decode step and the next token's draw; returns
        (token or negative code, new rng state)."""
        st = C.c_uint64(rng_state if rng_state is not None else 0)
        tok = lib().ds4g_decode_sample(self.ptr, int(token), float(temperature), float(top_p), C.byref(st),
                                       ws.data_ptr(), ws.numel() * ws.element_size())
        return tok, st.value

    def hidden(self) -> torch.Tensor:
        return self._view(lib().ds4g_session_hidden(self.ptr), self.model.shape.hidden,
                          torch.float32)

    def truncate(self, cp: int) -> int:
        return lib().ds4g_session_truncate(self.ptr, int(cp))

    def sync(self, tokens):
        """Bring the session to the prompt `tokens`: (status, tokens prefilled)."""
        t = (C.c_int32 * max(1, len(tokens)))(*[int(x) for x in tokens])
        n = C.c_int(0)
        rc = lib().ds4g_session_sync(self.ptr, t, len(tokens), C.byref(n))
        return rc, n.value

    def checkpoint_bytes(self) -> int:
        return int(lib().ds4g_checkpoint_bytes(C.byref(self.model.cfg), self.len))

    def save(self, buf: bytearray) -> int:
        """Write the session's checkpoint into the host buffer `buf`."""
        b = (C.c_char * len(buf)).from_buffer(buf)
        return lib().ds4g_session_save(self.ptr, b, len(buf))

    def load(self, buf) -> int:
        b = (C.c_char * len(buf)).from_buffer_copy(bytes(buf))
        return lib().ds4g_session_load(self.ptr, b, len(buf))

    def rewrite_from_common(self, tokens, common: int) -> int:
        t = (C.c_int32 * max(1, len(tokens)))(*[int(x) for x in tokens])
        return lib().ds4g_session_rewrite_from_common(self.ptr, t, len(tokens), int(common))

    def common_prefix(self, tokens) -> int:
        t = (C.c_int32 * len(tokens))(*[int(x) for x in tokens])
        return lib().ds4g_session_common_prefix(self.ptr, t, len(tokens))

    def restore(self, tokens) -> int:
        t = (C.c_int32 * len(tokens))(*[int(x) for x in tokens])
        return lib().ds4g_session_restore(self.ptr, t, len(tokens))

    @property
    def len(self) -> int:
        return lib().ds4g_session_len(self.ptr)

    # -- views of device buffers -----------------------------------------------
    def _view(self, ptr: int, n: int, dtype) -> torch.Tensor:
        off = ptr - self.mem.data_ptr()
        esz = torch.empty((), dtype=dtype).element_size()
        assert 0 <= off and off + n * esz <= self.mem.numel()
        return self.mem[off:off + n * esz].view(dtype)

    def logits(self) -> torch.Tensor:
        return self._view(lib().ds4g_session_logits(self.ptr), self.model.shape.vocab,
                          torch.float32)

    def debug(self, name: str, n: int) -> torch.Tensor:
        return self._view(lib().ds4g_session_debug(self.ptr, DEBUG[name]), n, torch.float32)

    def kv(self, layer: int):
        k, v = C.c_void_p(), C.c_void_p()
        _check(lib().ds4g_session_kv(self.ptr, layer, C.byref(k), C.byref(v)), "ds4g_session_kv")
        s = self.model.shape
        dt = torch.float32 if s.kv_dtype == "f32" else torch.bfloat16
        n = self.n_ctx * s.head_dim
        return (self._view(k.value, n, dt).view(self.n_ctx, s.head_dim),
                self._view(v.value, n, dt).view(self.n_ctx, s.head_dim))

    def set_trace(self, buf) -> None:
        """buf: a device tensor receiving per-CTA stage start times (or None)."""
        _check(lib().ds4g_session_set_trace(self.ptr, buf.data_ptr() if buf is not None else None,
                                            buf.numel() * buf.element_size() if buf is not None
                                            else 0), "ds4g_session_set_trace")

    def set_probe(self, positions) -> torch.Tensor | None:
        """Record the residual entering every layer (then the final hidden state) at
        the given session positions during later prefills and decode steps.  Returns
        the device buffer [n][L+1][H] (f32) the rows go to; an empty list stops it."""
        pos = (C.c_int32 * len(positions))(*[int(p) for p in positions])
        s = self.model.shape
        buf = torch.full((len(positions), s.n_layers + 1, s.hidden), float("nan"),
                         dtype=torch.float32, device="cuda") if len(positions) else None
        _check(lib().ds4g_session_set_probe(self.ptr, pos, len(positions),
                                            buf.data_ptr() if buf is not None else None),
               "ds4g_session_set_probe")
        self._probe = buf   # kept alive while the setting holds
        return buf

    def status(self) -> int:
        return lib().ds4g_session_status(self.ptr)

    @property
    def launches(self) -> int:
        return lib().ds4g_session_launches(self.ptr)

    def set_timing(self, on: bool) -> None:
        _check(lib().ds4g_session_set_timing(self.ptr, int(on)), "ds4g_session_set_timing")

    def timing(self):
        """{kernel kind: (total ms, launches)} since the last call (timing mode)."""
        n = len(KERNEL_KINDS)
        ms = (C.c_double * n)()
        cnt = (C.c_uint64 * n)()
        _check(lib().ds4g_session_timing(self.ptr, ms, cnt, n), "ds4g_session_timing")
        return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}

    def router(self, layer: int):
        K = self.model.shape.top_k
        ids = (C.c_int32 * K)()
        w = (C.c_float * K)()
        _check(lib().ds4g_session_router(self.ptr, layer, ids, w), "ds4g_session_router")
        return list(ids), list(w)


def sample_workspace_bytes(n_vocab: int) -> int:
    return lib().ds4g_sample_workspace_bytes(n_vocab)


def sample(logits: torch.Tensor, temperature: float, top_p: float, rng_state: int | None,
           workspace: torch.Tensor, stream=None, min_p: float = 0.0):
    """Returns (token, new_rng_state); min_p > 0 calls ds4g_sample_min_p."""
    st = C.c_uint64(rng_state or 0)
    if min_p > 0.0:
        tok = lib().ds4g_sample_min_p(logits.data_ptr(), logits.numel(), float(temperature),
                                      float(top_p), float(min_p), C.byref(st), workspace.data_ptr(),
                                      workspace.numel(), _stream_ptr(stream))
    else:
        tok = lib().ds4g_sample(logits.data_ptr(), logits.numel(), float(temperature), float(top_p),
                                C.byref(st), workspace.data_ptr(), workspace.numel(),
                                _stream_ptr(stream))
    return tok, st.value


def sample_static(logits: torch.Tensor, temperature: float, top_p: float,
                  rng_state: int | None, stream=None):
    """ds4g_sample_static: no workspace argument; returns (token, new_rng_state)."""
    st = C.c_uint64(rng_state or 0)
    tok = lib().ds4g_sample_static(logits.data_ptr(), logits.numel(), float(temperature),
                                   float(top_p), C.byref(st), _stream_ptr(stream))
    return tok, st.value


def sample_u(logits: torch.Tensor, temperature: float, top_p: float, u24: int,
             workspace: torch.Tensor, stream=None, min_p: float = 0.0) -> int:
    """Sample with a caller-given uniform draw u = u24 / 2^24."""
    if min_p > 0.0:
        return lib().ds4g_sample_u_min_p(logits.data_ptr(), logits.numel(), float(temperature),
                                         float(top_p), float(min_p), int(u24), workspace.data_ptr(),
                                         workspace.numel(), _stream_ptr(stream))
    return lib().ds4g_sample_u(logits.data_ptr(), logits.numel(), float(temperature),
                               float(top_p), int(u24), workspace.data_ptr(), workspace.numel(),
                               _stream_ptr(stream))
