"""The C ABI library without a GPU: it loads, exports every function include/gva.h declares,
and rejects bad arguments on the host before touching CUDA."""
import ctypes as C
import os
import re
import subprocess

import pytest
import torch

from compact_kv_cache_gva_b300 import gva

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gva.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b((?:gva|gqa)_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(gva.LIB_PATH):
        from compact_kv_cache_gva_b300 import build
        build.build()
    return gva.load()


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ["gva_absorb_query", "gva_cache_append", "gva_decode_attention", "gva_create", "gva_destroy",
              "gva_decode_workspace_size", "gva_get_device_error", "gqa_decode_attention"]:
        assert n in names


def test_library_exports_every_declared_function(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", gva.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT ((?:gva|gqa)_\w+)$", out, flags=re.M))
    declared = set(declared_functions())
    assert declared <= exported, declared - exported
    for n in declared:
        assert hasattr(lib, n)
    assert set(gva.EXPORTS) <= declared


def test_status_strings_and_version(lib):
    assert gva.status_string(gva.GVA_OK) == "ok"
    assert "workspace" in gva.status_string(gva.GVA_ERR_WORKSPACE)
    assert gva.gva_version() >= 100


@pytest.mark.parametrize("bad", [
    dict(H=6, G=4),            # H % G != 0
    dict(d_r=3),               # odd positional width
    dict(d_v=48),              # value width not a multiple of 32
    dict(block_size=32),       # blocks are 64 tokens
    dict(cache_dtype=7),       # unknown dtype
    dict(d_n=30),              # content width not a multiple of 4
])
def test_create_rejects_bad_dims_on_host(lib, bad):
    d = dict(H=16, G=4, d_v=64, d_n=64, d_r=16, block_size=64, cache_dtype=gva.GVA_BF16, rope_base=1e4, scale=0.0)
    d.update(bad)
    dims = gva.gva_dims(**d)
    h = C.c_void_p()
    assert lib.gva_create(C.byref(dims), C.byref(h)) == gva.GVA_ERR_INVALID_ARG
    assert not h.value


def test_null_context_and_sizes_rejected(lib):
    assert lib.gva_absorb_query(None, 1, None, None, None, None, None, None, None) == gva.GVA_ERR_INVALID_ARG
    assert lib.gva_cache_append(None, 1, 1, None, None, None, None, 1, 1, None, None, None) == gva.GVA_ERR_INVALID_ARG
    assert lib.gva_decode_attention(None, 1, None, None, None, None, None, 1, 1, None, 1, None, None, 0,
                                    None) == gva.GVA_ERR_INVALID_ARG
    assert lib.gva_decode_workspace_size(None, 1, 1) == 0
    assert lib.gva_set_split_tokens(None, 64) == gva.GVA_ERR_INVALID_ARG
    # the one-call step and its helpers
    assert lib.gva_decode_step(None, 1, None, None, None, None, None, None, None, None, 1, 1, None, 1, None, None,
                               0, None) == gva.GVA_ERR_INVALID_ARG
    assert lib.gva_decode_step_partial(None, 1, None, None, None, None, None, None, None, None, 1, 1, None, 1, None,
                                       0, None) == gva.GVA_ERR_INVALID_ARG
    assert lib.gva_decode_step_workspace_size(None, 1, 1) == 0
    assert lib.gva_step_is_fused(None, 1, 1) == -1
    assert lib.gva_set_step_mode(None, gva.GVA_STEP_FUSED) == gva.GVA_ERR_INVALID_ARG
    assert lib.gva_decode_attention_multi(None, 1, 2, None, None, None, None, None, 1, 1, None, 2, None, None, 0,
                                          None) == gva.GVA_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_create_without_gpu_reports_cuda_error(lib):
    dims = gva.gva_dims(16, 4, 64, 64, 16, 64, gva.GVA_BF16, 1e4, 0.0)
    h = C.c_void_p()
    assert lib.gva_create(C.byref(dims), C.byref(h)) == gva.GVA_ERR_CUDA


def test_binding_takes_pinned_host_tensors_only_where_the_step_allows():
    t = torch.zeros(1, 4, 32)  # ordinary pageable host memory is never accepted
    with pytest.raises(ValueError, match="pinned"):
        gva._ptr(t, torch.float32, "q_c", allow_pinned=True)
    with pytest.raises(ValueError, match="CUDA"):
        gva._ptr(t, torch.float32, "M")


def test_binding_refuses_host_tensors():
    class Fake:
        dims = gva.gva_dims(4, 2, 32, 32, 16, 64, gva.GVA_F32, 1e4, 0.0)
        cache_torch_dtype = torch.float32
        handle = None
    with pytest.raises(ValueError, match="CUDA"):
        gva.gva_absorb_query(Fake(), torch.zeros(1, 4, 32), torch.zeros(1, 4, 16), torch.zeros(1, dtype=torch.int32),
                             torch.zeros(4, 32, 32), torch.zeros(1, 4, 32), torch.zeros(1, 4, 16))
