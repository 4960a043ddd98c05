"""The C ABI without a GPU: the library loads, exports every function that
include/dflash.h declares, and its host-side validation answers before any
device work (no CUDA call is made on these paths)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from block_diffusion_speculative_hidden_gb300 import build_lib, _lib
    build_lib.build()
    return _lib.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "dflash.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_\w+)\s*\(", src)))


def test_exports_every_declared_function(L):
    names = header_functions()
    assert len(names) >= 12
    from block_diffusion_speculative_hidden_gb300 import _lib
    assert sorted(_lib.EXPORTED) == names
    for n in names:
        assert hasattr(L, n), n


def _cfg(**kw):
    from block_diffusion_speculative_hidden_gb300 import _lib
    c = _lib.DflashConfig()
    base = dict(n_layers=2, hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn=1320, vocab=5000,
                mask_id=4999, n_taps=3, tap_width=448, block_k=16, page_size=16, max_batch=3,
                max_pages_per_seq=24, n_pages=80, max_rows=300, max_inject_rows=900, rope_theta=1e6,
                rms_eps=1e-6, dtype=1)
    base.update(kw)
    for k, v in base.items():
        setattr(c, k, v)
    return c


def test_sizes_and_config_validation(L):
    c = _cfg()
    pool = L.dflash_kv_pool_size(ctypes.byref(c))
    assert pool == 2 * 2 * (80 + 3) * 2 * 16 * 128 * 2     # K and V, fp16, 3 block pages
    assert L.dflash_workspace_size(ctypes.byref(c)) > 0
    for bad in (dict(block_k=8), dict(page_size=32), dict(head_dim=96), dict(n_q_heads=6),
                dict(hidden=500), dict(dtype=7), dict(mask_id=5000), dict(max_inject_rows=10)):
        cb = _cfg(**bad)
        assert L.dflash_workspace_size(ctypes.byref(cb)) == 0, bad
        assert L.dflash_kv_pool_size(ctypes.byref(cb)) == 0, bad
    f32 = _cfg(dtype=0, hidden=500)
    assert L.dflash_kv_pool_size(ctypes.byref(f32)) == 2 * 2 * (80 + 3) * 2 * 16 * 128 * 4


def test_null_arguments_rejected_before_device_work(L):
    from block_diffusion_speculative_hidden_gb300 import _lib
    c = _cfg()
    out = ctypes.c_void_p()
    w = _lib.DflashWeights()
    assert L.dflash_create(None, None, None, 0, None, None, None, 0, ctypes.byref(out)) == 1
    assert L.dflash_create(ctypes.byref(c), ctypes.byref(w), ctypes.c_void_p(256), 1 << 30, ctypes.c_void_p(256),
                           ctypes.c_void_p(256), ctypes.c_void_p(256), 1 << 30, ctypes.byref(out)) == 1
    assert L.dflash_inject_kv(None, None, None, 0, 1, 1, None) == 1
    assert L.dflash_draft_block(None, 1, 1, None, None, None, None, None) == 1
    assert L.dflash_accept(None, 0, 1, None, None, None, None, 1.0, 0, 0, None, None, None, None) == 1
    assert L.dflash_destroy(None) == 1
    assert L.dflash_status_string(3) == b"KV page pool exhausted"


def test_graph_calls_validate_on_the_host(L):
    out = ctypes.c_void_p(1)
    assert L.dflash_graph_begin(None, None) == 1
    assert L.dflash_graph_end(None, None, ctypes.byref(out)) == 1
    assert L.dflash_graph_launch(None, None) == 1
    assert L.dflash_graph_destroy(None) == 1
    assert L.dflash_status_string(8) == b"not allowed in the context's capture state"
