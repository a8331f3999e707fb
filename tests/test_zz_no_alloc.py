"""ds4g_sample_static (sampler without a caller workspace; scratch is a fixed
device array of the library) against ds4g_sample with a caller workspace, through
the C ABI: two calls in a row on the same logits and RNG state, for greedy,
plain temperature and top-p sampling, and the size limit."""
import ctypes as C

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

DS4G_ESIZE = -6
MAX_VOCAB = 262144


def _logits(n, seed):
    import torch
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(n, generator=g, dtype=torch.float32) * 3.0
    return x.cuda()


@pytest.mark.parametrize("n_vocab", [1000, 129280, MAX_VOCAB])
@pytest.mark.parametrize("temperature,top_p", [(0.0, 1.0), (1.0, 1.0), (0.7, 0.95), (0.7, 0.3)])
def test_static_sampler_matches_workspace_sampler(n_vocab, temperature, top_p):
    import torch
    from prefill_decode_layer_gb300 import ds4g
    L = ds4g.lib()
    logits = _logits(n_vocab, seed=n_vocab + int(temperature * 10))
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = torch.empty(L.ds4g_sample_workspace_bytes(n_vocab), dtype=torch.uint8, device="cuda")
    st_ref, st_new = C.c_uint64(0x9E3779B97F4A7C15), C.c_uint64(0x9E3779B97F4A7C15)
    ref, got = [], []
    for _ in range(2):   # twice in a row: the fixed scratch must come back clean
        ref.append(L.ds4g_sample(C.c_void_p(logits.data_ptr()), n_vocab, temperature, top_p,
                                 C.byref(st_ref), C.c_void_p(ws.data_ptr()), ws.numel(), stream))
        got.append(L.ds4g_sample_static(C.c_void_p(logits.data_ptr()), n_vocab, temperature,
                                        top_p, C.byref(st_new), stream))
    assert min(ref) >= 0, ref
    assert got == ref
    assert st_new.value == st_ref.value
    if temperature == 0.0:
        assert got[0] == int(np.argmax(logits.cpu().numpy()))


def test_static_sampler_rejects_vocab_above_limit():
    import torch
    from prefill_decode_layer_gb300 import ds4g
    L = ds4g.lib()
    logits = torch.zeros(MAX_VOCAB + 1, dtype=torch.float32, device="cuda")
    st = C.c_uint64(1)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.ds4g_sample_static(C.c_void_p(logits.data_ptr()), MAX_VOCAB + 1, 0.7, 0.9,
                                C.byref(st), stream) == DS4G_ESIZE
    assert st.value == 1   # rejected before the draw


def test_static_sampler_allocates_no_device_memory():
    """After one warm-up call per sampler path (which loads the library's kernels
    and its fixed scratch, lazily, on first use), further calls at the largest
    vocabulary leave the device's free memory unchanged."""
    import torch
    from prefill_decode_layer_gb300 import ds4g
    L = ds4g.lib()
    logits = _logits(MAX_VOCAB, seed=7)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = C.c_uint64(0x9E3779B97F4A7C15)
    cases = [(0.0, 1.0), (1.0, 1.0), (0.7, 0.95)]
    for temperature, top_p in cases:   # warm-up: every kernel of the path is loaded
        assert L.ds4g_sample_static(C.c_void_p(logits.data_ptr()), MAX_VOCAB, temperature, top_p,
                                    C.byref(st), stream) >= 0
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for temperature, top_p in cases:
            assert L.ds4g_sample_static(C.c_void_p(logits.data_ptr()), MAX_VOCAB, temperature,
                                        top_p, C.byref(st), stream) >= 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
