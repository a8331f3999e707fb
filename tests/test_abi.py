"""CPU checks of the boundary: the library builds, loads, and exports every entry
point that include/ds4g.h declares (no compute calls: there is no GPU here)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds4g.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ds4g_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib_path():
    from prefill_decode_layer_gb300 import build
    return build.build()


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for required in ("ds4g_decode_step", "ds4g_prefill", "ds4g_session_truncate", "ds4g_sample",
                     "ds4g_session_common_prefix", "ds4g_model_create", "ds4g_session_create"):
        assert required in names


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\S+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def test_library_loads_and_validates_without_gpu(lib_path):
    import ctypes as C
    import prefill_decode_layer_gb300 as pdl
    import synth
    L = pdl.lib()
    for name in declared_functions():
        assert hasattr(L, name)
    assert L.ds4g_strerror(-2).decode().startswith("tokens do not fit")
    # shape validation and sizes are host-only
    c = pdl.config_struct(synth.LAYER)
    assert L.ds4g_session_bytes(C.byref(c), 5000) > 0
    bad = pdl.config_struct(synth.LAYER.with_(head_dim=12))
    assert L.ds4g_session_bytes(C.byref(bad), 5000) == 0
    bad = pdl.config_struct(synth.LAYER.with_(top_k=9))
    assert L.ds4g_session_bytes(C.byref(bad), 5000) == 0
    h = C.c_void_p()
    assert L.ds4g_model_create(C.byref(c), None, C.byref(h)) == pdl.ds4g.EINVAL
    # a null session is rejected before any device work
    assert L.ds4g_decode_step(None, 1) == pdl.ds4g.EINVAL
    assert L.ds4g_session_truncate(None, 0) == pdl.ds4g.EINVAL
    assert L.ds4g_session_sync(None, None, 0, None) == pdl.ds4g.EINVAL
    assert L.ds4g_session_save(None, None, 0) == pdl.ds4g.EINVAL
    assert L.ds4g_session_load(None, None, 0) == pdl.ds4g.EINVAL
    # checkpoint size: 64-byte header, tokens padded to 16 bytes, K and V rows per layer
    sh = synth.LAYER.with_(n_layers=3)
    c3 = pdl.config_struct(sh)
    for n in (0, 1, 5, 4096):
        want = 64 + (4 * n + 15) // 16 * 16 + 3 * 2 * n * sh.head_dim * 2
        assert L.ds4g_checkpoint_bytes(C.byref(c3), n) == want
    assert L.ds4g_checkpoint_bytes(C.byref(c3), -1) == 0
    assert L.ds4g_session_rewrite_from_common(None, None, 0, 0) == pdl.ds4g.EINVAL
    assert L.ds4g_sample_workspace_bytes(129280) > 0


def test_timing_kinds_match_the_header():
    """The binding's kernel-kind names follow the header's DS4G_K_* enumeration, in
    order, and cover DS4G_K_COUNT entries."""
    import prefill_decode_layer_gb300 as pdl
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    kinds = {name: int(v) for name, v in re.findall(r"\bDS4G_K_([A-Z_0-9]+)\s*=\s*(\d+)", src)}
    count = kinds.pop("COUNT")
    assert sorted(kinds.values()) == list(range(count))
    names = [n.lower() for n, _ in sorted(kinds.items(), key=lambda kv: kv[1])]
    assert list(pdl.ds4g.KERNEL_KINDS) == names
