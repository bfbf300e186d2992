"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import k3moe, native
from mxfp4_routed_expert_k3_gb300.dims import K3, TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    native.build_k3moe()
    return k3moe.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "k3moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(k3moe_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = header_functions()
    for f in ("k3moe_create", "k3moe_load_weights", "k3moe_forward", "k3moe_status", "k3moe_last_error",
              "k3moe_destroy"):
        assert f in names


def test_library_exports_every_declared_symbol(L):
    for f in header_functions():
        assert hasattr(L, f), f"{f} declared in include/k3moe.h but not exported"
    assert set(header_functions()) == set(k3moe.EXPORTS)


def test_create_rejects_bad_config(L):
    bad = [
        K3.with_(hidden=7000),
        K3.with_(top_k=40),
        K3.with_(group=16),
        TINY.with_(n_experts=4, top_k=8),
    ]
    for d in bad:
        h = C.c_void_p()
        rc = L.k3moe_create(C.byref(k3moe.make_config(d, 64)), 0, C.byref(h))
        assert rc == k3moe.EINVAL, (d, rc)
        assert h.value is None
        assert len(k3moe.last_error()) > 0
    h = C.c_void_p()
    rc = L.k3moe_create(C.byref(k3moe.make_config(TINY, 0)), 0, C.byref(h))
    assert rc == k3moe.EINVAL and "max_tokens" in k3moe.last_error()
    # shared experts: both fields or neither, a 128-multiple total, tensor-core paths only
    for d, path, word in [(TINY.with_(n_shared=2, shared_inter=100), 0, "multiple of 128"),
                          (TINY.with_(n_shared=2, shared_inter=0), 0, "both"),
                          (TINY.with_(n_shared=2, shared_inter=384), 1, "force_path"),
                          (TINY.with_(n_shared=2, shared_inter=384), 3, "force_path")]:
        h = C.c_void_p()
        rc = L.k3moe_create(C.byref(k3moe.make_config(d, 16, force_path=path)), 0, C.byref(h))
        assert rc == k3moe.EINVAL and word in k3moe.last_error(), (d, path, k3moe.last_error())
    # kernel paths: 0 (the library's choice), 1 (CUDA cores) and 4 only
    for path in (-1, 2, 3, 5):
        h = C.c_void_p()
        rc = L.k3moe_create(C.byref(k3moe.make_config(TINY, 16, force_path=path)), 0, C.byref(h))
        assert rc == k3moe.EINVAL and "force_path" in k3moe.last_error(), (path, k3moe.last_error())
        assert h.value is None


def test_create_without_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = C.c_void_p()
    rc = L.k3moe_create(C.byref(k3moe.make_config(TINY, 16)), 0, C.byref(h))
    assert rc in (k3moe.ECUDA, k3moe.EINVAL)
    assert h.value is None


def test_step_entry_points_validate_on_host(L):
    buf = np.zeros(1024, np.uint8)
    p = buf.ctypes.data
    assert L.k3moe_mxfp4_dequant(None, p, 4, 64, p, 0, None) == k3moe.EINVAL
    assert L.k3moe_mxfp4_dequant(p, p, 4, 48, p, 0, None) == k3moe.EINVAL  # cols % 64
    assert L.k3moe_mxfp4_dequant(p, p, 4, 64, p, 2, None) == k3moe.EINVAL  # kind
    assert L.k3moe_mxfp4_dequant(p, p, 4, 64, p + 1, 0, None) == k3moe.EINVAL  # alignment
    assert L.k3moe_route(p, 1, p, p, 64, 100, 8, 1, C.c_float(1.0), p, p, p, None) == k3moe.EINVAL
    assert L.k3moe_route(p, 1, p, p, 64, 128, 65, 1, C.c_float(1.0), p, p, p, None) == k3moe.EINVAL
    assert L.k3moe_route(p, 0, None, None, 64, 128, 8, 1, C.c_float(1.0), None, None, None, None) == k3moe.OK
    assert L.k3moe_forward(None, p, 1, p, p, p, None) == k3moe.EINVAL
    assert L.k3moe_load_weights(None, None) == k3moe.EINVAL


def test_last_error_never_null(L):
    assert isinstance(k3moe.last_error(None), str)
