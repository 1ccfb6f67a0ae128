"""The C ABI library: it builds, loads, exports every declared function, and
rejects bad arguments on the host before anything reaches a GPU.  No test
here launches a kernel, so the file runs on a machine without a GPU."""
import ctypes
import os

import pytest

import bit_expert_ffn_gb300 as m
from bit_expert_ffn_gb300 import build as B


@pytest.fixture(scope="module")
def lib():
    B.build()
    return m.load()


def test_every_declared_function_is_exported(lib):
    names = m.header_functions()
    assert len(names) >= 16
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_python_binding_covers_the_header():
    for n in m.header_functions():
        assert hasattr(m, n), f"binding lacks {n}"


def test_status_names(lib):
    assert m.moe_status_name(0) == "MOE_OK"
    assert m.moe_status_name(7) == "MOE_ERR_BOUNDS"
    assert m.moe_status_name(6) == "MOE_ERR_NONFINITE"
    assert m.moe_status_name(8) == "MOE_ERR_RANGE"


def test_packed_size_census(lib):
    # one 2-bit expert of the pages' model: gate||up [1536][2048] + down [2048][768]
    c1, s1 = m.moe_packed_size(2, 1536, 2048)
    c2, s2 = m.moe_packed_size(2, 2048, 768)
    assert c1 + s1 + c2 + s2 == 1_474_560
    c1, s1 = m.moe_packed_size(3, 1536, 2048)
    c2, s2 = m.moe_packed_size(3, 2048, 768)
    assert c1 + s1 + c2 + s2 == 2_064_384


def _err(fn, *args):
    with pytest.raises(m.MoeError) as e:
        fn(*args)
    return e.value


def test_host_validation(lib):
    assert _err(m.moe_packed_size, 4, 1, 32).status == m.MOE_ERR_INVALID_ARG
    assert _err(m.moe_packed_size, 2, 1, 33).status == m.MOE_ERR_INVALID_ARG
    e = _err(m.moe_pack_experts, 5, 1, 1, 32, 16, 16, 16, 16)
    assert e.status == m.MOE_ERR_INVALID_ARG and "bits" in str(e)
    assert _err(m.moe_permute, 16, 1, 2, 0, 16, 16, 16).status == m.MOE_ERR_INVALID_ARG
    assert _err(m.moe_permute, 16, 1, 17, 8, 16, 16, 16).status == m.MOE_ERR_INVALID_ARG
    assert _err(m.moe_topk_from_logits, 16, 1, 8, 9, 16, 16).status == m.MOE_ERR_INVALID_ARG  # k > E
    assert _err(m.moe_topk_from_logits, 16, 1, 2048, 2, 16, 16).status == m.MOE_ERR_INVALID_ARG  # E > 1024
    # a multiple of 32 is required for H
    assert _err(m.moe_router_topk, 16, 1, 100, 16, None, 8, 2, 16, 16, 16).status == m.MOE_ERR_INVALID_ARG
    # misaligned arena pointer
    bad = m.moe_expert_arena(2, 256, 128, 16, 17, 16, 16, 16)
    assert _err(m.moe_expert_forward_workspace_size, bad, 1, 2).status == m.MOE_ERR_INVALID_ARG


def test_workspace_rules(lib):
    arena = m.moe_expert_arena(2, 2048, 768, 512, 16, 16, 16, 16)
    dec = m.moe_expert_forward_workspace_size(arena, 4, 10, m.MOE_PATH_DECODE)
    assert dec >= 4 * 10 * (768 + 2048) * 4
    pre = m.moe_expert_forward_workspace_size(arena, 32768, 10, m.MOE_PATH_PREFILL)
    assert pre > dec
    # a too-small workspace is reported with the bytes needed, before any launch
    e = _err(m.moe_expert_forward, arena, 16, 4, 16, 16, 10, 16, 16, 16, 16, m.MOE_F32, 0, m.MOE_PATH_DECODE, 16, 8)
    assert e.status == m.MOE_ERR_WORKSPACE and str(dec) in str(e)
    assert m.moe_permute_workspace_size(1, 10, 512) == 0
    assert m.moe_permute_workspace_size(32768, 10, 512) > 0
    assert m.moe_router_workspace_size(8, 256, 16, 1) == 0
    assert m.moe_router_workspace_size(8, 256, 16, 0) >= 8 * 16 * 4
    # larger batches keep the three bf16 pieces of the router weights
    assert m.moe_router_workspace_size(9, 256, 16, 1) >= 16 * 3 * 256 * 2
    assert m.moe_router_workspace_size(9, 256, 16, 0) >= 16 * 3 * 256 * 2 + 9 * 16 * 4
    # the decode path refuses more than 8 tokens
    ws = m.moe_expert_forward_workspace_size(arena, 9, 10, m.MOE_PATH_DECODE)
    e = _err(m.moe_expert_forward, arena, 16, 9, 16, 16, 10, 16, 16, 16, 16, m.MOE_F32, 0, m.MOE_PATH_DECODE, 16, ws)
    assert e.status == m.MOE_ERR_INVALID_ARG


def test_library_has_no_host_fallback_symbols(lib):
    """The product library exports only the C ABI (plus nothing named like a CPU path)."""
    out = os.popen(f"nm -D --defined-only {m.LIB_PATH}").read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {s for s in exported if s.startswith("moe_")}
    assert ours == set(m.header_functions())
