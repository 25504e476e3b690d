"""CPU-only checks of the C-ABI library: it builds, loads without a GPU, exports
every function include/moe.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def built():
    from mxfp4_routed_expert_router_gb300 import build
    return build.build()


def declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(moe_[a-z_0-9]+)\s*\(", src, re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("moe_load_weights", "moe_workspace_bytes", "moe_forward", "moe_dense_sliced_forward",
              "moe_last_error", "moe_free"):
        assert f in names


def test_library_exports_every_declared_symbol(built):
    out = subprocess.run(["nm", "-D", "--defined-only", built], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = declared_functions() - exported
    assert not missing, missing
    lib = ctypes.CDLL(built)
    for name in declared_functions():
        assert hasattr(lib, name)


def test_binding_lists_every_symbol(built):
    from mxfp4_routed_expert_router_gb300 import binding
    assert set(binding.EXPORTED) == declared_functions()


def test_host_side_argument_checks_without_gpu(built):
    from mxfp4_routed_expert_router_gb300 import binding as b
    L = b.lib
    assert L.moe_workspace_bytes(None, 16, 2) == 0
    # NULL config
    h = ctypes.c_void_p()
    assert L.moe_load_weights(None, None, None, None, ctypes.byref(h)) == b.MOE_EINVAL
    assert b"NULL" in L.moe_last_error()
    fake = (b.MoeMx * 2)(b.MoeMx(16, 16), b.MoeMx(16, 16))
    # hidden not a multiple of 32 -> MOE_EDIMS before any CUDA call
    cfg = b.MoeConfig(hidden=100, inter=64, n_experts=2, n_shared=0, k_max=1, n_slices=0, fmt=b.MOE_W_MXFP4)
    assert L.moe_load_weights(ctypes.byref(cfg), fake, fake, None, ctypes.byref(h)) == b.MOE_EDIMS
    # dense slice width cutting a 32-value block
    cfg = b.MoeConfig(hidden=64, inter=96, n_experts=2, n_shared=0, k_max=1, n_slices=2, fmt=b.MOE_W_MXFP4)
    assert L.moe_load_weights(ctypes.byref(cfg), fake, fake, None, ctypes.byref(h)) == b.MOE_EDIMS
    # k_max outside [1, 32] (k_max above n_experts is allowed: caller routing may
    # repeat an expert or leave slots empty)
    for km in (0, 33):
        cfg = b.MoeConfig(hidden=64, inter=64, n_experts=2, n_shared=0, k_max=km, n_slices=0, fmt=b.MOE_W_MXFP4)
        assert L.moe_load_weights(ctypes.byref(cfg), fake, fake, None, ctypes.byref(h)) == b.MOE_EINVAL
    # NULL weight pointer
    cfg = b.MoeConfig(hidden=64, inter=64, n_experts=2, n_shared=0, k_max=1, n_slices=0, fmt=b.MOE_W_MXFP4)
    nul = (b.MoeMx * 2)(b.MoeMx(16, 16), b.MoeMx(16, None))
    assert L.moe_load_weights(ctypes.byref(cfg), nul, fake, None, ctypes.byref(h)) == b.MOE_EINVAL
    # unknown format
    cfg = b.MoeConfig(hidden=64, inter=64, n_experts=2, n_shared=0, k_max=1, n_slices=0, fmt=7)
    assert L.moe_load_weights(ctypes.byref(cfg), fake, fake, None, ctypes.byref(h)) == b.MOE_EINVAL
    # group-32 INT4: scales are FP16, so their pointer must be 2-byte aligned; zero points may be NULL
    cfg = b.MoeConfig(hidden=64, inter=64, n_experts=2, n_shared=0, k_max=1, n_slices=0, fmt=b.MOE_W_INT4G32)
    odd = (b.MoeMx * 2)(b.MoeMx(16, 16, None), b.MoeMx(16, 17, 16))
    assert L.moe_load_weights(ctypes.byref(cfg), fake, odd, None, ctypes.byref(h)) == b.MOE_EINVAL
    assert b"2-byte aligned" in L.moe_last_error()
    assert L.moe_load_weights(ctypes.byref(cfg), nul, fake, None, ctypes.byref(h)) == b.MOE_EINVAL
    assert b"NULL" in L.moe_last_error()
    # forward / dense forward / sync on a NULL handle
    assert L.moe_forward(None, None, None, 1, 1, None, 0, None, 0, None, None) == b.MOE_EINVAL
    assert L.moe_dense_sliced_forward(None, None, 1, None, 0, None, 0, None) == b.MOE_EINVAL
    assert L.moe_sync_status(None, None) == b.MOE_EINVAL
    assert L.moe_forward_routed(None, None, None, None, 1, 1, None, 0, None, 0, None, None) == b.MOE_EINVAL
    assert L.moe_set_expert_range(None, 0, 8) == b.MOE_EINVAL
    # sigmoid routing: sizes and pointers are checked before any CUDA call
    assert L.moe_route_sigmoid(None, None, 4, 0, 1, 1.0, None, None, None) == b.MOE_EINVAL
    assert L.moe_route_sigmoid(None, None, 4, 1025, 1, 1.0, None, None, None) == b.MOE_EINVAL
    assert L.moe_route_sigmoid(None, None, 4, 8, 9, 1.0, None, None, None) == b.MOE_EINVAL
    assert L.moe_route_sigmoid(None, None, 4, 64, 33, 1.0, None, None, None) == b.MOE_EINVAL
    assert L.moe_route_sigmoid(None, None, -1, 8, 2, 1.0, None, None, None) == b.MOE_EINVAL
    assert L.moe_route_sigmoid(None, None, 4, 8, 2, 1.0, None, None, None) == b.MOE_EINVAL
    assert b"NULL" in L.moe_last_error()
    assert L.moe_route_sigmoid(None, None, 0, 8, 2, 1.0, None, None, None) == b.MOE_OK
    g = ctypes.c_void_p()
    assert L.moe_graph_create(None, None, None, None, None, 1, 1, None, 0, None, 0, None, ctypes.byref(g)) == \
        b.MOE_EINVAL
    assert L.moe_graph_create(None, None, None, None, None, 1, 1, None, 0, None, 0, None, None) == b.MOE_EINVAL
    assert L.moe_graph_launch(None, None) == b.MOE_EINVAL
    L.moe_graph_free(None)  # no-op
    # the wait-limit test hook checks its handle before anything else
    assert L.moe_debug_expire_next_wait(None, 1000) == b.MOE_EINVAL
    assert b"NULL handle" in L.moe_last_error()
    L.moe_free(None)  # no-op


def test_oracle_and_library_share_no_source():
    """The oracle and the CUDA path are independent: neither includes or
    imports the other."""
    csrc = os.path.join(ROOT, "mxfp4_routed_expert_router_gb300")
    for dirpath, _, files in os.walk(csrc):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.findall(r"^\s*(?:import|from|#include)\s+\S*", text, re.M).__str__(), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "mxfp4_routed_expert_router_gb300" not in text and "moe.h" not in text, f
