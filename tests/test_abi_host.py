"""C-ABI library: it builds for sm_103a, loads without a GPU, exports every call the public
header declares, and rejects bad arguments on the host before any launch (no GPU needed)."""

import ctypes

import pytest

import moe_prefill_nvfp4_gb300 as moe
from moe_prefill_nvfp4_gb300 import _lib, build


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.load()


def test_exports_every_declared_symbol(L):
    names = _lib.exported_names()
    assert "moe_prefill_forward" in names and "moe_w4a16_grouped_gemm" in names
    for n in names:
        assert hasattr(L, n), n
    # the binding wraps every compute call of the header under the same name
    for n in ("moe_route_topk", "moe_sort_by_expert", "moe_w4a16_grouped_gemm", "moe_swiglu_clamp",
              "moe_combine_indexed", "moe_prefill_forward", "moe_router_logits", "moe_dequant_nvfp4"):
        assert hasattr(moe, n), n


def test_version_and_status_strings(L):
    assert b"sm_103a" in L.moe_version()
    assert L.moe_status_string(0) == b"MOE_OK"
    assert L.moe_status_string(3) == b"MOE_ERR_WORKSPACE_TOO_SMALL"


NULL = None
P = ctypes.c_void_p(16)  # a non-NULL, 16-byte aligned dummy address: never dereferenced on these paths


def test_route_topk_rejects(L):
    assert L.moe_route_topk(NULL, NULL, 4, 8, 2, 1, 1.0, P, P, NULL) == 1
    assert L.moe_route_topk(P, NULL, 4, 8, 9, 1, 1.0, P, P, NULL) == 2  # k > E
    assert L.moe_route_topk(P, NULL, 4, 2000, 2, 1, 1.0, P, P, NULL) == 2  # E > 1024
    assert L.moe_route_topk(P, NULL, 0, 8, 2, 1, 1.0, P, P, NULL) == 2  # T = 0


def test_sort_rejects_and_sizes(L):
    assert L.moe_sort_workspace_bytes(2048, 8, 160) == 161 * 8 * 4
    assert L.moe_sort_workspace_bytes(0, 8, 160) == 0
    assert L.moe_sort_by_expert(P, 4, 2, 8, P, P, P, P, P, 0, NULL) == 3  # workspace too small
    assert L.moe_sort_by_expert(P, 4, 33, 64, P, P, P, P, P, 1 << 20, NULL) == 2  # k > 32
    assert L.moe_sort_by_expert(NULL, 4, 2, 8, P, P, P, P, P, 1 << 20, NULL) == 1


def test_sort_noalloc_rejects_before_any_launch(L):
    assert L.moe_status_string(7) == b"MOE_ERR_SCRATCH_LIMIT"
    assert L.moe_sort_by_expert_noalloc(NULL, 4, 2, 8, P, P, P, P, NULL) == 1
    assert L.moe_sort_by_expert_noalloc(P, 4, 33, 64, P, P, P, P, NULL) == 2  # k > 32
    # (E+1) * ceil(T*k / 2048) int32 counts must fit the fixed 65536-entry scratch:
    # E = 160 allows 407 segments (833,536 slots); one more slot needs 408 segments
    assert _lib.MOE_SORT_NOALLOC_MAX_INTS == 65536
    assert L.moe_sort_by_expert_noalloc(P, 104200, 8, 160, P, P, P, P, NULL) == 7
    assert L.moe_sort_by_expert_noalloc(P, 833537, 1, 160, P, P, P, P, NULL) == 7
    # 1025 * 8 counts fit: checked on the host sizes alone (a call would launch on a GPU machine)
    assert L.moe_sort_workspace_bytes(2048, 8, 1024) <= 4 * _lib.MOE_SORT_NOALLOC_MAX_INTS
    assert L.moe_sort_workspace_bytes(104200, 8, 160) > 4 * _lib.MOE_SORT_NOALLOC_MAX_INTS


def test_gemm_and_elementwise_reject(L):
    assert L.moe_w4a16_grouped_gemm(P, 8, 256, NULL, NULL, P, 8, P, 256, 0, NULL) == 1  # no table
    assert L.moe_swiglu_clamp(P, P, 4, 12, 24, P, 12, 7.0, NULL) == 2  # width % 8
    assert L.moe_swiglu_clamp(P, P, 4, 16, 8, P, 16, 7.0, NULL) == 2  # ld_in < width
    assert L.moe_combine_indexed(P, P, P, NULL, 4, 2, 12, P, NULL) == 2  # H % 8
    assert L.moe_combine_indexed(ctypes.c_void_p(18), P, P, NULL, 4, 2, 16, P, NULL) == 1  # misaligned Y
    assert L.moe_router_logits(P, P, 4, 12, 8, P, NULL) == 2
    assert L.moe_dequant_nvfp4(P, P, 1.0, 4, 96, P, NULL) == 2  # K % 64


def test_expert_table_rejects(L):
    E = 2
    pp = (ctypes.c_void_p * E)(16, 32)
    sp = (ctypes.c_void_p * E)(16, 32)
    s2 = (ctypes.c_float * E)(1.0, 1.0)
    out = ctypes.c_void_p()
    assert L.moe_expert_table_create(pp, sp, s2, E, 256, 200, ctypes.byref(out)) == 2  # K % 256
    assert L.moe_expert_table_create(pp, sp, s2, E, 12, 256, ctypes.byref(out)) == 2  # N % 8
    assert L.moe_expert_table_create(pp, sp, s2, 0, 256, 256, ctypes.byref(out)) == 2
    bad = (ctypes.c_void_p * E)(17, 32)
    assert L.moe_expert_table_create(bad, sp, s2, E, 256, 256, ctypes.byref(out)) == 1  # misaligned
    none = (ctypes.c_void_p * E)(None, None)
    assert L.moe_expert_table_create(none, sp, s2, E, 256, 256, ctypes.byref(out)) == 1  # no expert at all
    assert L.moe_expert_table_destroy(None) == 0


def test_workspace_layout(L):
    cfg = _lib.MoePrefillConfig(hidden=2048, moe_intermediate=768, num_experts=64, top_k=8, swiglu_limit=7.0,
                                renormalize=1, routed_scale=1.0)
    lay = _lib.moe_workspace_layout(cfg, 256)
    R = 256 * 8
    offs = [lay.logits, lay.ids, lay.wts, lay.sorted_token_ids, lay.sorted_expert_ids, lay.expert_offsets,
            lay.token_to_perm, lay.sort_scratch, lay.ready, lay.G, lay.act, lay.Y, lay.x_stage, lay.x_sorted]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lay.G - lay.ready >= (2 * 64 + 1) * 4  # per-expert act and row counters, the tile counter
    assert lay.Y - lay.act >= R * 768 * 2 and lay.x_stage - lay.Y >= R * 2048 * 2
    assert lay.x_sorted - lay.x_stage >= 256 * 2048 * 2 and lay.total - lay.x_sorted >= R * 2048 * 2
    assert _lib.moe_workspace_bytes(cfg, 256) == lay.total
    bad = _lib.MoePrefillConfig(hidden=2000, moe_intermediate=768, num_experts=64, top_k=8)
    assert _lib.moe_workspace_bytes(bad, 256) == 0
    with pytest.raises(moe.MoeError):
        _lib.moe_workspace_layout(bad, 256)


def test_forward_rejects(L):
    cfg = _lib.MoePrefillConfig(hidden=2048, moe_intermediate=768, num_experts=64, top_k=8, swiglu_limit=7.0,
                                renormalize=1, routed_scale=1.0)
    f = L.moe_prefill_forward
    # neither router weight nor logits
    assert f(ctypes.byref(cfg), P, 4, NULL, NULL, NULL, P, P, P, 1 << 30, P, NULL, NULL, NULL, NULL) == 1
    # both
    assert f(ctypes.byref(cfg), P, 4, P, P, NULL, P, P, P, 1 << 30, P, NULL, NULL, NULL, NULL) == 1
    # misaligned shared expert output
    assert f(ctypes.byref(cfg), P, 4, P, NULL, NULL, P, P, ctypes.c_void_p(256), 1 << 30, P, ctypes.c_void_p(18), NULL,
             NULL, NULL) == 1
    # unknown flag bits
    bad = _lib.MoePrefillConfig(hidden=2048, moe_intermediate=768, num_experts=64, top_k=8, swiglu_limit=7.0,
                                renormalize=1, routed_scale=1.0, flags=4)
    assert f(ctypes.byref(bad), P, 4, P, NULL, NULL, P, P, P, 1 << 30, P, NULL, NULL, NULL, NULL) == 1


def test_shared_expert_rejects_and_sizes(L):
    T, H, I = 4, 2048, 768
    need = L.moe_shared_expert_workspace_bytes(T, H, I)
    assert need >= T * 3 * I * 2  # gate|up and act
    assert need < (1 << 20)  # nothing but the two stage buffers
    assert L.moe_shared_expert_workspace_bytes(T, H, 12) == 0  # I % 8
    f = L.moe_shared_expert_forward
    W = ctypes.c_void_p(256)
    assert f(NULL, T, H, I, P, P, P, 7.0, W, need, P, NULL) == 1
    assert f(P, T, H, I, P, P, P, 0.0, W, need, P, NULL) == 1  # limit must be positive
    assert f(P, T, H, 12, P, P, P, 7.0, W, need, P, NULL) == 2
    assert f(P, 0, H, I, P, P, P, 7.0, W, need, P, NULL) == 2
    assert f(P, T, H, I, P, P, P, 7.0, W, need - 1, P, NULL) == 3
    assert f(P, T, H, I, P, P, P, 7.0, P, need, P, NULL) == 1  # workspace not 256-byte aligned
