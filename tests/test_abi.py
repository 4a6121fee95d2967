"""The C-ABI library loads and behaves on the host side (no GPU needed).

No compute call is made: config validation, NULL handling and error strings
all run before any CUDA call.
"""
import ctypes

import pytest

import __graft_entry__ as entry
import fp8_routed_expert_gb300 as moe
from fp8_routed_expert_gb300._lib import MoEConfig


@pytest.fixture(scope="module")
def L():
    entry.build()
    return moe.lib()


def test_exports_every_declared_function(L):
    names = moe.exported_functions()
    assert {"moe_init", "moe_layer_forward", "moe_free", "moe_get_routing", "moe_status",
            "moe_strerror", "moe_layer_forward_host"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def _init(L, **kw):
    cfg = dict(max_tokens=8, hidden=256, n_experts=8, inter=128, max_top_k=2, device=0)
    cfg.update(kw)
    h = ctypes.c_void_p(1234)
    rc = L.moe_init(ctypes.byref(h), ctypes.byref(MoEConfig(**cfg)))
    return rc, h


@pytest.mark.parametrize("kw", [dict(hidden=200), dict(inter=100), dict(hidden=0),
                                dict(n_experts=0), dict(n_experts=2000), dict(max_top_k=0),
                                dict(max_top_k=9), dict(max_top_k=33, n_experts=64),
                                dict(max_tokens=0), dict(hidden=65536 + 128),
                                dict(max_tokens=1 << 40)])
def test_bad_configs_rejected_before_cuda(L, kw):
    rc, h = _init(L, **kw)
    assert rc == moe.C["MOE_ERR_SHAPE"]
    assert h.value is None  # *out cleared


def test_null_arguments(L):
    assert L.moe_init(None, None) == moe.C["MOE_ERR_ARG"]
    h = ctypes.c_void_p()
    assert L.moe_init(ctypes.byref(h), None) == moe.C["MOE_ERR_ARG"]
    L.moe_free(None)  # no-op
    assert L.moe_layer_forward(None, None, 0, None, None, None, None, None, None, 1, None,
                               None) == moe.C["MOE_ERR_ARG"]
    assert L.moe_status(None) == moe.C["MOE_ERR_ARG"]
    assert L.moe_set_path(None, 0) == moe.C["MOE_ERR_ARG"]
    assert L.moe_resolve_path(None, 1) == moe.C["MOE_ERR_ARG"]
    assert L.moe_selftest_wait_timeout(None, 1000, None, None) == moe.C["MOE_ERR_ARG"]
    assert L.moe_cache_init(None, None, None, None, 1) == moe.C["MOE_ERR_ARG"]
    h = ctypes.c_void_p(99)
    assert L.moe_cache_init(ctypes.byref(h), None, None, None, 1) == moe.C["MOE_ERR_ARG"]
    assert h.value is None
    assert L.moe_cache_forward(None, None, 1, None, None, None, None, 1, None, None) == moe.C["MOE_ERR_ARG"]
    assert L.moe_cache_prefetch(None, None, 0) == moe.C["MOE_ERR_ARG"]
    assert L.moe_cache_stats(None, None, 0) == moe.C["MOE_ERR_ARG"]
    L.moe_cache_free(None)


def test_error_strings(L):
    for name, code in moe.C.items():
        if name.startswith("MOE_ERR_") or name == "MOE_OK":
            s = L.moe_strerror(code).decode()
            assert s and s != "unknown error", name
    assert L.moe_strerror(12345).decode() == "unknown error"
    for k in range(moe.C["MOE_K_COUNT"]):
        assert L.moe_kernel_name(k).decode() != "unknown"


def test_init_without_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = _init(L)
    assert rc in (moe.C["MOE_ERR_CUDA"], moe.C["MOE_ERR_UNSUPPORTED"])
    assert h.value is None
