"""GPU parity of each kernel against the CPU oracle, through the C ABI (sm_103a GPU needed).

Integer and byte results (routing ids, the sort, dequantised BF16 weights) must match
bit-exactly; float results within the tolerances of ``gpu_helpers``.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import moe_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402

import moe_prefill_nvfp4_gb300 as moe  # noqa: E402

from gpu_helpers import fused_act_error, TOL_BF16, TOL_EXACT, bf16_bits, bf16_dev, bf16_host, nerr, upload  # noqa: E402


@pytest.fixture(autouse=True)
def _no_device_error():
    moe.moe_get_device_error()
    yield
    assert moe.moe_get_device_error() == 0


# ---------------------------------------------------------------------------- dequantisation


@pytest.mark.parametrize("N,K", [(64, 512), (130, 256), (8, 1536)])
def test_dequant_bit_exact(N, K):
    packed, scales = S.expert_weights(5, 9, N, N, K)
    s2 = float(S.scale2_vector(5, 9, 3)[1])
    got = moe.moe_dequant_nvfp4(torch.from_numpy(packed).cuda(), torch.from_numpy(scales).cuda(), s2)
    ref = O.dequant_nvfp4(packed, scales, s2, "bf16")
    ref_bits = (ref.view(np.uint32) >> 16).astype(np.uint16)
    np.testing.assert_array_equal(bf16_bits(got), ref_bits)


def test_dequant_all_codes_and_scale_range():
    """Every (code, scale byte) pair: 16 codes x all finite E4M3 scales, two scale2 values."""
    scales_all = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], dtype=np.uint8)
    N = scales_all.size
    K = 64
    packed = np.tile(np.array([0x10 * ((2 * j + 1) % 16) + (2 * j) % 16 for j in range(32)], np.uint8), (N, 1))
    scales = np.repeat(scales_all[:, None], K // 16, axis=1)
    for s2 in (1.0, 0.0030517578125 * 1.37):
        got = moe.moe_dequant_nvfp4(torch.from_numpy(packed).cuda(), torch.from_numpy(scales).cuda(), s2)
        ref = O.dequant_nvfp4(packed, scales, s2, "bf16")
        np.testing.assert_array_equal(bf16_bits(got), (ref.view(np.uint32) >> 16).astype(np.uint16))


# ---------------------------------------------------------------------------- routing


def test_router_logits_c1_shapes():
    c = S.workload("c1", with_weights=False)
    got = moe.moe_router_logits(bf16_dev(c.x), bf16_dev(c.router_w)).cpu().numpy()
    ref = O.router_logits(c.x, c.router_w)
    assert nerr(got, ref) < 1e-5


@pytest.mark.parametrize("T,H,E", [(1, 8, 1), (37, 512, 5), (17, 264, 130), (300, 2048, 160), (33, 5120, 64)])
def test_router_logits_ragged_shapes(T, H, E):
    """Token counts off the 16-row tile, E off the 8- and 64-expert groups, H off the 32-element
    step and split 1, 2 or 8 ways over the cluster."""
    g = np.random.default_rng(T * H + E)
    x = S.bf16_bits_from_f32(g.standard_normal((T, H)).astype(np.float32))
    w = S.bf16_bits_from_f32(g.normal(0.0, 0.02, (E, H)).astype(np.float32))
    got = moe.moe_router_logits(bf16_dev(x), bf16_dev(w)).cpu().numpy()
    assert nerr(got, O.router_logits(x, w)) < 1e-5


@pytest.mark.parametrize("T,E,k,bias,renorm", [(300, 160, 8, False, 1), (257, 64, 8, True, 1),
                                               (33, 16, 8, False, 0), (5, 1000, 32, True, 1), (40, 9, 9, False, 1)])
def test_route_topk_bit_exact(T, E, k, bias, renorm):
    g = np.random.default_rng(T * E)
    logits = g.standard_normal((T, E)).astype(np.float32)
    logits[:, ::7] = np.round(logits[:, ::7])  # exact ties
    b = g.normal(0, 0.1, E).astype(np.float32) if bias else None
    ids, wts = moe.moe_route_topk(torch.from_numpy(logits).cuda(), k,
                                  bias=None if b is None else torch.from_numpy(b).cuda(), renormalize=bool(renorm),
                                  routed_scale=1.5)
    rid, rw = O.route_topk(logits, k, b, renorm, 1.5)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)


def test_route_topk_zipf_and_minus_huge():
    lg = S.zipf_logits(1003, 512, 160)
    ids, wts = moe.moe_route_topk(torch.from_numpy(lg).cuda(), 8)
    rid, rw = O.route_topk(lg, 8)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)


# ---------------------------------------------------------------------------- sort


def _check_sort(ids_np, E):
    got = moe.moe_sort_by_expert(torch.from_numpy(ids_np).cuda(), E)
    ref = O.sort_by_expert(ids_np, E)
    for key in ("sorted_token_ids", "sorted_expert_ids", "expert_offsets", "token_to_perm"):
        np.testing.assert_array_equal(got[key].cpu().numpy().reshape(ref[key].shape), ref[key], err_msg=key)


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (64, 8, 16), (256, 8, 64), (256, 8, 512), (2048, 8, 160),
                                   (8192, 8, 160), (16384, 8, 160), (777, 3, 1000), (100, 32, 40)])
def test_sort_bit_exact(T, k, E):
    g = np.random.default_rng(T + E)
    ids = np.argsort(g.random((T, E)), axis=1)[:, :k].astype(np.int32)
    _check_sort(ids, E)


def test_sort_skewed_and_unfilled():
    lg = S.zipf_logits(1003, 8192, 160)
    ids, _ = O.route_topk(lg, 8)
    _check_sort(ids, 160)
    g = np.random.default_rng(3)
    ids2 = g.integers(0, 12, (333, 4)).astype(np.int32)
    ids2[g.random((333, 4)) < 0.1] = -1
    _check_sort(ids2, 12)


def test_sort_single_block_one_bucket_and_tail():
    """R = 2048 slots (the single-block sort's maximum) all in one expert, then every slot but the
    last in the -1 tail: the per-warp counts reach 64 and the bucket prefix 2048."""
    ids = np.full((256, 8), 3, np.int32)
    _check_sort(ids, 5)
    ids[:] = -1
    ids[-1, -1] = 4
    _check_sort(ids, 5)


def test_sort_flags_out_of_range_id():
    ids = np.array([[0, 1], [5, 2]], np.int32)  # 5 >= E
    moe.moe_sort_by_expert(torch.from_numpy(ids).cuda(), 4)
    assert moe.moe_get_device_error() == 1
    fixed = ids.copy()
    fixed[1, 0] = -1
    _check_sort(fixed, 4)  # the bad id was handled as the sentinel


# ---------------------------------------------------------------------------- SwiGLU, combine


def test_swiglu_clamp():
    g = np.random.default_rng(4)
    R, I = 517, 1536
    G = (g.standard_normal((R, 2 * I)) * 4).astype(np.float32)
    G[0, :8] = [7.0, 8.0, 100.0, -100.0, 0.0, -7.5, 6.99, 1e4]
    Gb = S.bf16_bits_from_f32(G)
    Gd = bf16_dev(Gb)
    act = moe.moe_swiglu_clamp(Gd[:, :I], Gd[:, I:], 7.0)
    Gf = O.bf16_bits_to_f64(Gb)
    ref = O.swiglu_clamp(Gf[:, :I], Gf[:, I:], 7.0)
    got = bf16_host(act)
    assert nerr(got, ref) < TOL_BF16
    # each element within one BF16 rounding (plus fp32 evaluation) of the exact value
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6).all()


def test_combine_indexed():
    g = np.random.default_rng(5)
    T, k, H, R = 301, 8, 2048, 301 * 8
    Yb = S.bf16_bits_from_f32(g.standard_normal((R, H)).astype(np.float32))
    perm = g.permutation(R).astype(np.int32).reshape(T, k)
    perm[3, 2] = -1
    wts = g.random((T, k)).astype(np.float32)
    got = moe.moe_combine_indexed(bf16_dev(Yb), torch.from_numpy(perm).cuda(), torch.from_numpy(wts).cuda())
    ref = O.combine_indexed(O.bf16_bits_to_f64(Yb), perm, wts.astype(np.float64))
    assert nerr(bf16_host(got), ref) < TOL_BF16
    sh = S.bf16_bits_from_f32(g.standard_normal((T, H)).astype(np.float32))
    got2 = moe.moe_combine_indexed(bf16_dev(Yb), torch.from_numpy(perm).cuda(), torch.from_numpy(wts).cuda(),
                                   shared_out=bf16_dev(sh))
    ref2 = O.combine_indexed(O.bf16_bits_to_f64(Yb), perm, wts.astype(np.float64), O.bf16_bits_to_f64(sh))
    assert nerr(bf16_host(got2), ref2) < TOL_BF16


# ---------------------------------------------------------------------------- grouped GEMM


def _gemm_case(c, c_dtype=torch.float32, identity=False):
    """Run the GPU sort + grouped GEMM on a GemmCase; returns (gpu C, sort dict, device proj)."""
    srt = moe.moe_sort_by_expert(torch.from_numpy(c.ids).cuda(), c.E)
    proj = upload(c.w)
    R = c.T * c.k
    if identity:
        # A already in sorted order: gather on the host through the GPU's own sort
        st = srt["sorted_token_ids"].long()
        A = bf16_dev(c.x)[st].contiguous()
        C = moe.moe_w4a16_grouped_gemm(A, proj.table, srt["expert_offsets"], R, c_dtype=c_dtype)
    else:
        C = moe.moe_w4a16_grouped_gemm(bf16_dev(c.x), proj.table, srt["expert_offsets"], R,
                                       gather_ids=srt["sorted_token_ids"], c_dtype=c_dtype)
    torch.cuda.synchronize()
    return C, {k: v.cpu().numpy() for k, v in srt.items()}, proj


def _oracle_gemm(c, srt, variant):
    wfn = lambda e: None if c.w.packed[e] is None else O.dequant_nvfp4(c.w.packed[e], c.w.scales[e], c.w.scale2[e],
                                                                     variant)
    return O.grouped_gemm(O.bf16_bits_to_f64(c.x), srt["expert_offsets"], wfn, srt["sorted_token_ids"])


def test_gemm_exact_dyadic_bit_exact():
    """Scales 1.0, scale2 1, integer activations: every product/sum exact -> FP32 output bit-exact."""
    c = S.make_gemm_case(T=48, E=6, k=3, N=256, K=512, seed=21,
                         x_sampler=lambda g, shp: g.integers(-2, 3, shp).astype(np.float32))
    for e in range(c.E):
        c.w.scales[e][:] = 0x38
    c.w.scale2[:] = 1.0
    C, srt, proj = _gemm_case(c)
    ref = _oracle_gemm(c, srt, "bf16")
    np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), ref)
    proj.close()


@pytest.mark.parametrize("c_dtype", [torch.float32, torch.bfloat16])
def test_gemm_c0(c_dtype):
    """The pages' measured shape: M=64 tokens, top_k=8, 16 experts, N=256, K=512."""
    c = S.workload("c0")
    C, srt, proj = _gemm_case(c, c_dtype)
    got = C.float().cpu().numpy().astype(np.float64)
    rb, re = _oracle_gemm(c, srt, "bf16"), _oracle_gemm(c, srt, "exact")
    if c_dtype == torch.float32:
        assert nerr(got, rb) < 2e-6  # same BF16 operands: only the FP32 summation order differs
    assert nerr(got, rb) < TOL_BF16 and nerr(got, re) < TOL_EXACT
    proj.close()


def test_gemm_ragged_multi_tile_absent_and_identity():
    """N not a multiple of 128, K = 768, a heavy expert (> 256 rows: several token tiles),
    empty experts, an absent expert (zero rows), and the identity (no-gather) A path."""
    g = np.random.default_rng(7)
    T, E, k, N, K = 600, 9, 2, 200, 768
    c = S.make_gemm_case(T=T, E=E, k=k, N=N, K=K, seed=22, absent=(4,))
    ids = np.where(g.random((T, k)) < 0.55, 0, g.integers(1, E, (T, k))).astype(np.int32)
    ids[:, 1] = np.where(ids[:, 1] == ids[:, 0], (ids[:, 0] + 1) % E, ids[:, 1])
    ids[ids == 7] = 6  # expert 7 empty
    ids[ids == 8] = 5  # expert 8 empty
    c.ids = ids
    for identity in (False, True):
        C, srt, proj = _gemm_case(c, torch.float32, identity=identity)
        ref = _oracle_gemm(c, srt, "bf16")
        got = C.cpu().numpy().astype(np.float64)
        assert (np.diff(srt["expert_offsets"])[0]) > 256  # expert 0 spans several token tiles
        o = srt["expert_offsets"]
        assert (got[o[4]:o[5]] == 0).all() and o[5] > o[4]
        assert nerr(got, ref) < 2e-6
        proj.close()


def test_gemm_deterministic_and_bad_offsets():
    c = S.workload("c0")
    C1, srt, proj = _gemm_case(c, torch.bfloat16)
    C2, _, proj2 = _gemm_case(c, torch.bfloat16)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    bad = torch.tensor([0, 10, 5] + [5] * (c.E - 2), dtype=torch.int32, device="cuda")  # decreasing
    x = bf16_dev(c.x)
    out = torch.full((c.T * c.k, c.N), 7.0, dtype=torch.float32, device="cuda")
    moe.moe_w4a16_grouped_gemm(x, proj.table, bad, c.T * c.k, out=out, c_dtype=torch.float32)
    assert moe.moe_get_device_error() == 2
    assert (out == 7.0).all()  # nothing written
    proj.close()
    proj2.close()


@pytest.mark.parametrize("T,E,k,N,identity", [(40, 16, 8, 512, False), (40, 16, 8, 512, True), (80, 16, 8, 512, False),
                                              (80, 16, 8, 512, True), (300, 24, 8, 512, False),
                                              (600, 4, 2, 512, False), (40, 16, 8, 384, False),
                                              (300, 24, 8, 384, False), (600, 4, 2, 384, False),
                                              (90, 12, 4, 2048, False)],
                         ids=["48-row-pairs", "48-row-pairs-contiguous", "64-row-pairs", "64-row-pairs-2acc-contiguous",
                              "128-row-pairs", "128-row-pairs-300-mean", "64-row-odd-blocks", "128-row-odd-blocks",
                              "256-row-odd-blocks", "48-row-pairs-cluster8"])
def test_gemm_each_tile_config(T, E, k, N, identity):
    """Mean rows per expert ~20, ~40, ~100 and ~300 with even and odd numbers of 128-row weight
    blocks select every token-tile configuration: 48-row tiles (pairs, two accumulator buffers;
    ~20 rows per expert, so some experts span two token tiles), 64-row tiles (pairs, pairs with
    two accumulator buffers for contiguous rows, single blocks), 128-row tiles (pairs, single
    blocks), 256-row tiles (single blocks); 16 blocks make clusters of 8."""
    c = S.make_gemm_case(T=T, E=E, k=k, N=N, K=512, seed=23 + T + N)
    C, srt, proj = _gemm_case(c, identity=identity)
    ref = _oracle_gemm(c, srt, "bf16")
    assert nerr(C.cpu().numpy().astype(np.float64), ref) < 2e-6
    proj.close()


@pytest.mark.parametrize("T,E,k,I,big,identity", [(40, 16, 8, 256, False, False), (80, 16, 8, 256, False, False),
                                                  (300, 24, 8, 256, True, False), (600, 4, 2, 128, True, False),
                                                  (90, 12, 4, 768, False, True)],
                         ids=["48-row", "64-row", "128-row-clamped", "256-row-mean-clamped", "48-row-identity"])
def test_gemm_swiglu_fused(T, E, k, I, big, identity):
    """Gate/up GEMM with the clamped SwiGLU in the epilogue: g and u rounded to BF16, then
    act = silu(min(g, L)) * clamp(u, -L, L), L = 7, against the oracle's SwiGLU of its
    BF16-rounded product, element by element (a g or u that lies at a BF16 rounding midpoint
    may round either way under another FP32 summation order).  `big` scales scale2 by 200 so
    |g|, |u| reach past L and both clamps act."""
    c = S.make_gemm_case(T=T, E=E, k=k, N=2 * I, K=512, seed=41 + T + I, absent=(1,))
    if big:
        c.w.scale2[:] = c.w.scale2 * 200.0
    srt = moe.moe_sort_by_expert(torch.from_numpy(c.ids).cuda(), c.E)
    proj = upload(c.w)
    R = c.T * c.k
    if identity:
        A = bf16_dev(c.x)[srt["sorted_token_ids"].long()].contiguous()
        act = moe.moe_w4a16_grouped_gemm_swiglu(A, proj.table, srt["expert_offsets"], R, limit=7.0)
    else:
        act = moe.moe_w4a16_grouped_gemm_swiglu(bf16_dev(c.x), proj.table, srt["expert_offsets"], R, limit=7.0,
                                                gather_ids=srt["sorted_token_ids"])
    torch.cuda.synchronize()
    s = {kk: v.cpu().numpy() for kk, v in srt.items()}
    G = _oracle_gemm(c, s, "bf16")
    got = bf16_host(act)
    if big:
        assert (np.abs(G[:, :I]) > 7.0).mean() > 0.05 and (np.abs(G[:, I:]) > 7.0).mean() > 0.05
    o = s["expert_offsets"]
    assert (got[o[1]:o[2]] == 0).all()  # absent expert: zero rows
    e, ok = fused_act_error(got, G, I, 7.0)
    assert ok and e < TOL_BF16, e
    proj.close()


# ---------------------------------------------------------------------------- small-row products


def _small_case(T, E, k, N, K, seed, absent=()):
    c = S.make_gemm_case(T=T, E=E, k=k, N=N, K=K, seed=seed, absent=absent)
    srt = moe.moe_sort_by_expert(torch.from_numpy(c.ids).cuda(), c.E)
    return c, srt, upload(c.w)


@pytest.mark.parametrize("T,E,k,N,K,identity", [(8, 16, 8, 256, 512, False), (5, 40, 6, 384, 1024, True),
                                                (1, 8, 8, 264, 256, False)],
                         ids=["8-rows", "5-rows-identity", "1-row-ragged-N"])
def test_gemv_vs_exact_oracle(T, E, k, N, K, identity):
    """The small-row product keeps the dequantised weights in FP32 (the pages' decode GEMV), so
    its reference is the exact variant; the only rounding left is C's BF16 rounding."""
    c, srt, proj = _small_case(T, E, k, N, K, seed=51 + T, absent=(3,))
    R = T * k
    if identity:
        A = bf16_dev(c.x)[srt["sorted_token_ids"].long()].contiguous()
        C = moe.moe_w4a16_grouped_gemv(A, proj.table, srt["expert_offsets"], R)
    else:
        C = moe.moe_w4a16_grouped_gemv(bf16_dev(c.x), proj.table, srt["expert_offsets"], R,
                                       gather_ids=srt["sorted_token_ids"])
    torch.cuda.synchronize()
    s = {kk: v.cpu().numpy() for kk, v in srt.items()}
    ref = _oracle_gemm(c, s, "exact")
    got = bf16_host(C)
    o = s["expert_offsets"]
    assert (got[o[3]:o[4]] == 0).all()  # absent expert
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-5 * np.abs(ref).max()).all()
    assert nerr(got, _oracle_gemm(c, s, "bf16")) < TOL_BF16  # and close to the BF16-weight variant
    proj.close()


def test_gemv_swiglu_vs_exact_oracle():
    T, E, k, I, K = 8, 12, 8, 256, 512
    c, srt, proj = _small_case(T, E, k, 2 * I, K, seed=57)
    c.w.scale2[:] = c.w.scale2 * 200.0  # |g|, |u| past the limit: both clamps act
    proj.close()
    proj = upload(c.w)
    act = moe.moe_w4a16_grouped_gemv_swiglu(bf16_dev(c.x), proj.table, srt["expert_offsets"], T * k, limit=7.0,
                                            gather_ids=srt["sorted_token_ids"])
    torch.cuda.synchronize()
    s = {kk: v.cpu().numpy() for kk, v in srt.items()}
    G = _oracle_gemm(c, s, "exact")
    ref = O.swiglu_clamp(G[:, :I], G[:, I:], 7.0)
    assert (np.abs(G[:, :I]) > 7.0).mean() > 0.05 and (np.abs(G[:, I:]) > 7.0).mean() > 0.05
    got = bf16_host(act)
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-4 * np.abs(ref).max()).all()
    proj.close()


def test_gemv_refuses_more_than_8_rows_per_expert():
    c, srt, proj = _small_case(16, 4, 2, 128, 256, seed=58)  # 32 slots on 4 experts
    out = torch.full((32, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    moe.moe_w4a16_grouped_gemv(bf16_dev(c.x), proj.table, srt["expert_offsets"], 32,
                               gather_ids=srt["sorted_token_ids"], out=out)
    assert moe.moe_get_device_error() == 6
    off = srt["expert_offsets"].cpu().numpy()
    big = [e for e in range(4) if off[e + 1] - off[e] > 8]
    assert big and all((out[off[e]:off[e + 1]] == 3.0).all() for e in big)  # not written
    proj.close()
