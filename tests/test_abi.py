"""The C-ABI library builds for sm_103a, loads, and exports every symbol that
include/lora_delta.h declares (CPU only: no kernel is launched here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "lora_delta.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(lora_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def library():
    from lora_delta_gb300.build import build
    path = build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("lora_pool_pack", "lora_shrink", "lora_expand", "lora_delta_fused",
                 "lora_moe_fc1_delta", "lora_route", "lora_get_error"):
        assert want in names


def test_every_declared_symbol_is_exported(library):
    missing = [n for n in declared_functions() if not hasattr(library, n)]
    assert not missing, f"not exported: {missing}"


def test_binding_signatures_cover_the_header():
    from lora_delta_gb300._lib import SIGNATURES
    assert sorted(SIGNATURES) == declared_functions()


def test_host_only_calls(library):
    import lora_delta_gb300 as ld
    assert ld.lib().lora_abi_version() >= 1
    assert ld.status_string(0) == "LORA_OK"
    assert ld.status_string(3) == "LORA_ERR_ALIGN"
    # the scale rule of "Module lora_delta", LoraPair: alpha / r or alpha / sqrt(r)
    assert ld.lora_scale(32.0, 16) == 2.0
    assert ld.lora_scale(32.0, 16, use_rslora=True) == 8.0
    assert ld.lora_scale(16.0, 0) == 0.0
    assert ld.lora_workspace_size(8192, 2, 32, 8) >= 8192 * 4 + 10 * 4 + 8192 * 64 * 4
    assert ld.lora_moe_workspace_size(2048, 8, 64, 8, 16, False) >= 2048 * 8 * 4


def test_wait_limit_setter_is_process_wide_and_returns_the_previous_value(library):
    """lora_set_wait_limit_ns: default 2 s; the setter returns the previous limit."""
    import lora_delta_gb300 as ld
    prev = ld.lora_set_wait_limit_ns(12345)
    try:
        assert prev == ld.WAIT_LIMIT_DEFAULT_NS
        assert ld.lora_set_wait_limit_ns(0) == 12345
    finally:
        ld.lora_set_wait_limit_ns(prev)
    assert ld.lora_set_wait_limit_ns(prev) == prev


def test_host_validation_without_a_gpu(library):
    """Argument errors are caught on the host before anything is launched."""
    import lora_delta_gb300 as ld
    L = ld.lib()
    w = (ctypes.c_int32 * 1)(16)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    # k_in not a multiple of 8 -> LORA_ERR_ALIGN
    assert L.lora_delta_fused(fake, 16, fake, 4, 12, fake, fake, fake, None, w, 1, 16, 4, 0, 1,
                              None, 0, None, None) == 3
    # R not a multiple of 8 -> LORA_ERR_ALIGN; R > 128 -> UNSUPPORTED
    assert L.lora_delta_fused(fake, 16, fake, 4, 16, fake, fake, fake, None, w, 1, 12, 4, 0, 1,
                              None, 0, None, None) == 3
    assert L.lora_delta_fused(fake, 16, fake, 4, 16, fake, fake, fake, None, w, 1, 256, 4, 0,
                              1, None, 0, None, None) == 6
    # ld_out smaller than the slices -> LORA_ERR_SHAPE
    assert L.lora_delta_fused(fake, 8, fake, 4, 16, fake, fake, fake, None, w, 1, 16, 4, 0, 1,
                              None, 0, None, None) == 2
    # n > 1024 rows without a workspace -> LORA_ERR_WORKSPACE
    assert L.lora_delta_fused(fake, 16, fake, 2000, 16, fake, fake, fake, None, w, 1, 16, 4, 0,
                              1, None, 0, None, None) == 5
    # NULL x -> LORA_ERR_ARG; n == 0 is a no-op
    assert L.lora_delta_fused(fake, 16, None, 4, 16, fake, fake, fake, None, w, 1, 16, 4, 0, 1,
                              None, 0, None, None) == 1
    assert L.lora_delta_fused(None, 16, None, 0, 16, None, None, None, None, w, 1, 16, 4, 0, 1,
                              None, 0, None, None) == 0
    # MoE: too many keys
    assert L.lora_moe_fc1_delta(fake, fake, fake, 256, fake, 256, 0, fake, fake, 4, 2, 1024, 64,
                                16, 16, 8, 1.0, None, 0, None, None) == 6


def test_moe_in_place_host_validation_without_a_gpu(library):
    """The in-place MoE calls check their arguments on the host, before any launch."""
    import lora_delta_gb300 as ld
    L = ld.lib()
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    # w13: T = 0 is a no-op
    assert L.lora_moe_w13_delta(None, None, None, 0, None, 0, 0, None, None, None, 0, None, 0,
                                2, 4, 64, 16, 16, 2, 1.0, 1, None, 0, None, None) == 0
    # w13: an expert map without its size -> LORA_ERR_ARG
    assert L.lora_moe_w13_delta(fake, fake, fake, 256, fake, 256, 0, fake, fake, fake, 0, None,
                                4, 2, 4, 64, 16, 16, 2, 1.0, 1, None, 0, None, None) == 1
    # w13: I not a multiple of 8 -> LORA_ERR_ALIGN
    assert L.lora_moe_w13_delta(fake, fake, fake, 256, fake, 256, 0, fake, fake, None, 0, None,
                                4, 2, 4, 64, 12, 16, 2, 1.0, 1, None, 0, None, None) == 3
    # w2: NULL y -> LORA_ERR_ARG
    assert L.lora_moe_w2_delta(None, fake, fake, 256, fake, 256, fake, fake, None, 0, None, None,
                               4, 2, 4, 64, 16, 16, 2, 1.0, 1, None, 0, None, None) == 1
    # w2: H not a multiple of 8 -> LORA_ERR_ALIGN
    assert L.lora_moe_w2_delta(fake, fake, fake, 256, fake, 256, fake, fake, None, 0, None, None,
                               4, 2, 4, 60, 16, 16, 2, 1.0, 1, None, 0, None, None) == 3
    # w2: rank past 128 -> LORA_ERR_UNSUPPORTED; no workspace -> LORA_ERR_WORKSPACE
    assert L.lora_moe_w2_delta(fake, fake, fake, 256, fake, 256, fake, fake, None, 0, None, None,
                               4, 2, 4, 64, 16, 256, 2, 1.0, 1, None, 0, None, None) == 6
    assert L.lora_moe_w2_delta(fake, fake, fake, 256, fake, 256, fake, fake, None, 0, None, None,
                               4, 2, 4, 64, 16, 16, 2, 1.0, 1, None, 0, None, None) == 5
