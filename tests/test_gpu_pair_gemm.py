"""GPU parity of the CTA-pair grouped GEMM (tcgen05 cta_group::2) against the oracle.

The pair kernel is the default wherever N % 256 == 0 and the A rows are contiguous (in the
forward the gate/up launch stores its gathered token rows in expert order itself; a standalone
call with gather_ids takes the single-CTA kernel).  These cases force it (``moe_debug_set_gemm_kernel``) on
A rows in expert order and compare with the oracle's grouped GEMM on the same BF16 operands
(FP32 output: only the FP32 summation order differs, so 2e-6 of max|ref|), with the exact
special case bit for bit, and with the single-CTA kernel.  Shapes cover both tile configurations
(128-token tiles with two accumulator buffers, 384-token tiles with one), ragged experts (1 row,
32k + 1 rows, experts spanning several token tiles), absent and empty experts, and the fused
SwiGLU.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import moe_prefill_nvfp4_gb300 as moe  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402

from gpu_helpers import TOL_BF16, bf16_dev, bf16_host, fused_act_error, nerr, upload  # noqa: E402

PAIR = moe.MOE_GEMM_KERNEL_PAIR
SINGLE = moe.MOE_GEMM_KERNEL_SINGLE


@pytest.fixture(autouse=True)
def _no_device_error():
    moe.moe_get_device_error()
    yield
    moe.moe_debug_set_gemm_kernel(moe.MOE_GEMM_KERNEL_AUTO)
    assert moe.moe_get_device_error() == 0


def _run(c, which, c_dtype=torch.float32, identity=False, swiglu=False, guard=0):
    """GPU sort + grouped GEMM with the chosen kernel.  `guard` extra rows and columns around the
    output hold a sentinel that must survive."""
    srt = moe.moe_sort_by_expert(torch.from_numpy(c.ids).cuda(), c.E)
    proj = upload(c.w)
    R = c.T * c.k
    cols = c.N // 2 if swiglu else c.N
    dt = torch.bfloat16 if swiglu else c_dtype
    buf = torch.full((R + 2 * guard, cols + 8 * guard), 3.0, dtype=dt, device="cuda")
    out = buf[guard:guard + R, :cols]
    if identity or which == PAIR:  # the pair kernel reads A rows in expert order
        A = bf16_dev(c.x)[srt["sorted_token_ids"].long()].contiguous()
        gather = None
    else:
        A = bf16_dev(c.x)
        gather = srt["sorted_token_ids"]
    with moe.gemm_kernel(which):
        if swiglu:
            moe.moe_w4a16_grouped_gemm_swiglu(A, proj.table, srt["expert_offsets"], R, limit=7.0, gather_ids=gather,
                                              out=out)
        else:
            moe.moe_w4a16_grouped_gemm(A, proj.table, srt["expert_offsets"], R, gather_ids=gather, out=out,
                                       c_dtype=c_dtype)
        torch.cuda.synchronize()
    if guard:
        g = buf.float()
        assert (g[:guard] == 3.0).all() and (g[guard + R:] == 3.0).all() and (g[:, cols:] == 3.0).all(), "guard band"
    proj.close()
    return out, {k: v.cpu().numpy() for k, v in srt.items()}


def _oracle(c, srt, variant="bf16"):
    wfn = lambda e: None if c.w.packed[e] is None else O.dequant_nvfp4(c.w.packed[e], c.w.scales[e], c.w.scale2[e],
                                                                     variant)
    return O.grouped_gemm(O.bf16_bits_to_f64(c.x), srt["expert_offsets"], wfn, srt["sorted_token_ids"])


def test_pair_exact_dyadic_bit_exact():
    """Unit scales, scale2 = 1, integer activations: every product and partial sum is exact, so the
    FP32 output equals the oracle bit for bit in any summation order."""
    c = S.make_gemm_case(T=48, E=6, k=3, N=512, K=512, seed=121,
                         x_sampler=lambda g, shp: g.integers(-2, 3, shp).astype(np.float32))
    for e in range(c.E):
        c.w.scales[e][:] = 0x38
    c.w.scale2[:] = 1.0
    C, srt = _run(c, PAIR)
    np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), _oracle(c, srt))


@pytest.mark.parametrize("T,E,k,N,K,identity", [
    (40, 16, 8, 256, 512, False),      # ~20 rows per expert: 128-token tiles
    (40, 16, 8, 512, 512, True),       # contiguous rows
    (300, 24, 8, 768, 256, False),     # ~100 rows per expert, K = 256 (one weight stage)
    (600, 4, 2, 512, 768, False),      # ~300 rows per expert: wide (384-token) tiles, both MMA halves
    (600, 4, 2, 256, 512, True),       # wide tiles, contiguous
    (1030, 3, 1, 256, 512, False),     # ~343 rows, ragged 16k+6 tails
], ids=["128tok-gathered", "128tok-contiguous", "100rows-K256", "256tok-gathered", "256tok-contiguous",
        "256tok-ragged"])
def test_pair_vs_oracle(T, E, k, N, K, identity):
    c = S.make_gemm_case(T=T, E=E, k=k, N=N, K=K, seed=131 + T + N + K)
    C, srt = _run(c, PAIR, identity=identity, guard=2)
    assert nerr(C.cpu().numpy().astype(np.float64), _oracle(c, srt)) < 2e-6


def test_pair_ragged_single_rows_absent_and_empty():
    """Experts with 1, 2, 17 and 300+ rows, an absent expert (its rows zero), empty experts."""
    g = np.random.default_rng(11)
    T, E, k, N, K = 400, 9, 1, 256, 512
    c = S.make_gemm_case(T=T, E=E, k=k, N=N, K=K, seed=141, absent=(4,))
    ids = np.zeros((T, k), dtype=np.int32)
    ids[:1] = 1
    ids[1:3] = 2
    ids[3:20] = 3
    ids[20:40] = 4
    ids[40:60] = 5
    ids[60:] = 0  # 340 rows: one 384-token tile
    g.shuffle(ids)
    c.ids = ids
    C, srt = _run(c, PAIR, guard=1)
    got = C.cpu().numpy().astype(np.float64)
    o = srt["expert_offsets"]
    assert o[5] > o[4] and (got[o[4]:o[5]] == 0).all()
    assert nerr(got, _oracle(c, srt)) < 2e-6


@pytest.mark.parametrize("c_dtype", [torch.float32, torch.bfloat16])
def test_pair_equals_single_cta_kernel(c_dtype):
    """Both kernels on the same operands: FP32 outputs within the summation-order difference,
    BF16 outputs within one BF16 rounding."""
    c = S.make_gemm_case(T=200, E=12, k=4, N=512, K=1024, seed=151)
    a, _ = _run(c, PAIR, c_dtype=c_dtype)
    b, _ = _run(c, SINGLE, c_dtype=c_dtype)
    x, y = a.float().cpu().numpy().astype(np.float64), b.float().cpu().numpy().astype(np.float64)
    assert nerr(x, y) < (2e-6 if c_dtype == torch.float32 else 2.0 ** -8)


@pytest.mark.parametrize("T,E,k,I,big,identity", [(40, 16, 8, 256, False, False), (300, 24, 8, 256, True, False),
                                                  (600, 4, 2, 128, True, False), (90, 12, 4, 768, False, True)],
                         ids=["128tok", "100rows-clamped", "256tok-clamped", "identity"])
def test_pair_swiglu_fused(T, E, k, I, big, identity):
    """Gate/up GEMM with the clamped SwiGLU in the epilogue (g and u rounded to BF16, then
    act = silu(min(g, L)) * clamp(u, -L, L)) against the oracle's SwiGLU of its BF16-rounded G,
    element by element.  `big` scales scale2 so that both clamps act."""
    c = S.make_gemm_case(T=T, E=E, k=k, N=2 * I, K=512, seed=161 + T + I, absent=(1,))
    if big:
        c.w.scale2[:] = c.w.scale2 * 200.0
    act, srt = _run(c, PAIR, identity=identity, swiglu=True, guard=1)
    G64 = _oracle(c, srt)
    got = bf16_host(act)
    if big:
        assert (np.abs(G64[:, :I]) > 7.0).mean() > 0.05 and (np.abs(G64[:, I:]) > 7.0).mean() > 0.05
    o = srt["expert_offsets"]
    assert (got[o[1]:o[2]] == 0).all()
    e, ok = fused_act_error(got, G64, I, 7.0)
    assert ok and e < TOL_BF16, e


@pytest.mark.parametrize("counts", [(1, 100, 192, 193, 300, 384, 385, 700, 1000), (17, 191, 383, 769, 1152, 5)],
                         ids=["halves-and-tiles", "ragged"])
def test_pair_swiglu_384_token_tiles(counts):
    """With more than 128 rows per expert the fused gate/up launch takes 384-token tiles: two MMAs
    of N = 192 per k16 step, the second only for tiles with more than 192 rows, and each
    dequantising warpgroup taking half of every weight stage.  Experts whose rows fill one half,
    both halves exactly, several tiles with ragged tails, and an absent expert; every element of
    act within the fused SwiGLU's bound, the absent expert's rows zero."""
    E = len(counts) + 1
    T = sum(counts) + 50
    I = 256
    c = S.make_gemm_case(T=T, E=E, k=1, N=2 * I, K=512, seed=181 + len(counts), absent=(E - 1,))
    ids = np.concatenate([np.full(n, e, dtype=np.int32) for e, n in enumerate(list(counts) + [50])])
    np.random.default_rng(19).shuffle(ids)
    c.ids = ids.reshape(T, 1)
    assert T / E > 128
    act, srt = _run(c, PAIR, swiglu=True, guard=1)
    G64 = _oracle(c, srt)
    got = bf16_host(act)
    o = srt["expert_offsets"]
    assert list(np.diff(o)) == list(counts) + [50]
    assert (got[o[E - 1]:o[E]] == 0).all()
    e, ok = fused_act_error(got, G64, I, 7.0)
    assert ok and e < TOL_BF16, e


def test_pair_refuses_gathered_rows():
    """With gather_ids the pair kernel is not taken: PAIR mode refuses, AUTO takes the single-CTA
    kernel."""
    c = S.make_gemm_case(T=64, E=8, k=2, N=256, K=512, seed=171)
    srt = moe.moe_sort_by_expert(torch.from_numpy(c.ids).cuda(), c.E)
    proj = upload(c.w)
    R = c.T * c.k
    with moe.gemm_kernel(PAIR):
        with pytest.raises(moe.MoeError):
            moe.moe_w4a16_grouped_gemm(bf16_dev(c.x), proj.table, srt["expert_offsets"], R,
                                       gather_ids=srt["sorted_token_ids"])
    C = moe.moe_w4a16_grouped_gemm(bf16_dev(c.x), proj.table, srt["expert_offsets"], R,
                                   gather_ids=srt["sorted_token_ids"], c_dtype=torch.float32)
    s = {kk: v.cpu().numpy() for kk, v in srt.items()}
    assert nerr(C.cpu().numpy().astype(np.float64), _oracle(c, s)) < 2e-6
    proj.close()


@pytest.mark.parametrize("T,H,I,E,k,routing", [(37, 512, 256, 5, 2, "biased"), (256, 2048, 768, 64, 8, "router"),
                                               (600, 512, 256, 4, 2, "biased")],
                         ids=["ragged-small", "256-row-block", "300-rows-per-expert"])
def test_forward_on_the_pair_kernel(T, H, I, E, k, routing):
    """The whole forward with both GEMMs on CTA pairs (the gate/up launch storing its token rows in
    expert order as it runs): routing and sort bit-exact, every float stage within the stage-wise
    bounds."""
    from test_gpu_forward import _check_full

    c = S.make_block_case(T=T, H=H, I=I, E=E, k=k, routing=routing, seed=201 + T)
    with moe.gemm_kernel(PAIR):
        _check_full(c)


@pytest.mark.parametrize("T,E", [(600, 4), (64, 6)], ids=["wide-tiles", "128-token-tiles"])
def test_forward_pair_expert_absent_only_in_gate_up(T, E):
    """An expert the gate/up table lacks: the gate/up launch writes its activation rows as zeros and
    publishes them to the down launch (which otherwise waits out its bound), on both configs."""
    from test_gpu_forward import _check_full

    c = S.make_block_case(T=T, H=512, I=256, E=E, k=2, routing="biased", seed=211 + T)
    c.gate_up.packed[1] = None
    c.gate_up.scales[1] = None
    with moe.gemm_kernel(PAIR):
        _check_full(c)
        assert moe.moe_get_device_error() == 0


@pytest.mark.parametrize("T,E,absent", [(600, 4, None), (600, 4, 1), (2048, 16, 5), (64, 6, 1)],
                         ids=["wide-tiles", "wide-tiles-absent", "2048-rows-absent", "128-token-tiles-absent"])
def test_forward_pair_stores_rows_in_expert_order(T, E, absent):
    """The pair gate/up launch stores its token rows in expert order itself: row p of x_sorted is
    x[sorted_token_ids[p]] bit for bit for every row of an expert present in the gate/up table;
    the rows of an absent expert (no tile reads them) and the rows past expert_offsets[E] keep the
    workspace's previous bytes."""
    from gpu_helpers import DeviceBlock

    c = S.make_block_case(T=T, H=512, I=256, E=E, k=2, routing="biased", seed=221 + T + E)
    if absent is not None:
        c.gate_up.packed[absent] = None
        c.gate_up.scales[absent] = None
    db = DeviceBlock(c)
    db.ws.fill_(0x5A)
    with moe.gemm_kernel(PAIR):
        db.forward()
        torch.cuda.synchronize()
    R = T * c.k
    sti = db.ws_view("sorted_token_ids", torch.int32, (R,)).cpu().long()
    off = db.ws_view("expert_offsets", torch.int32, (E + 1,)).cpu().long()
    xs = db.ws_view("x_sorted", torch.int16, (R, c.H)).cpu()
    x = db.x.cpu().view(torch.int16)
    fill = torch.full((c.H,), 0x5A5A, dtype=torch.int16)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if e == absent:
            assert (xs[lo:hi] == fill).all(), f"rows of absent expert {e} written"
        else:
            assert torch.equal(xs[lo:hi], x[sti[lo:hi]]), f"rows of expert {e}"
    assert (xs[int(off[E]):] == fill).all()
    db.close()
