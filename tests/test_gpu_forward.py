"""GPU parity of the whole routed-MoE prefill path (moe_prefill_forward) against the oracle.

Routing and the sort are compared bit-exactly on shared logits (the GPU's router logits are
fed to the oracle's top-k, so a different summation order cannot flip a near tie).

Float stages (wts, G, act, Y, out):
* against the BF16-rounding oracle, stage by stage: each stage's GPU output against the oracle
  applied to the same BF16 input the GPU stage consumed (G from x, act from the GPU's G, Y from
  the GPU's act, out from the GPU's Y), within 4e-3 of max|ref|.  With the SwiGLU fused into
  the gate/up GEMM (the default) G is never written: act is checked against the oracle's
  SwiGLU of its unrounded G;
* against the exact-FP32 oracle, as one independent chain from x to out, within 1e-2.
A whole independent BF16 chain is not held to 4e-3: when FP32 summation order flips a BF16
rounding of G (about 0.2% of elements), the flip propagates through act and Y, and with
concentrated routing weights it alone can move out by ~2e-3 of max|out| on top of out's own
rounding (up to 2^-8).  Its value is recorded in the assertion message of the exact check.
Full-size workloads are checked on sampled tokens, which the oracle computes one at a time.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import moe_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402

import moe_prefill_nvfp4_gb300 as moe  # noqa: E402

from gpu_helpers import TOL_BF16, TOL_EXACT, DeviceBlock, bf16_host, fused_act_error, nerr  # noqa: E402


@pytest.fixture(autouse=True)
def _no_device_error():
    moe.moe_get_device_error()
    yield
    assert moe.moe_get_device_error() == 0


def _stagewise(case, st, R, wvar="bf16"):
    """Oracle of each float stage on the GPU's own BF16 stage inputs, with the weights the GPU
    path multiplies with (BF16-rounded, or FP32 for the small-row products)."""
    I = case.I
    off = st["expert_offsets"]
    dn = lambda e: (None if case.down.packed[e] is None else
                    O.dequant_nvfp4(case.down.packed[e], case.down.scales[e], case.down.scale2[e], wvar))
    act = O.swiglu_clamp(st["G"][:R, :I], st["G"][:R, I:], case.swiglu_limit)
    Y = O.grouped_gemm(st["act"][:R], off, dn)
    out = O.combine_indexed(st["Y"], st["token_to_perm"], st["wts"].astype(np.float64), st.get("shared"))
    return act, Y, out


def _small_rows(case, separate=False, flags=0) -> bool:
    """With MOE_FWD_SMALL_ROWS, chunks of <= 8 rows take the small-row products (FP32
    dequantised weights, as the pages' decode GEMV): their reference is the exact-weight oracle."""
    return case.T <= 8 and not separate and bool(flags & moe.MOE_FWD_SMALL_ROWS)


def _check_full(case, separate=False):
    db = DeviceBlock(case, separate=separate)
    db.forward()
    torch.cuda.synchronize()
    st = db.stages()
    db.close()
    # without a router the forward routes on the caller's logits and leaves the workspace's
    # logits buffer unwritten
    shared_logits = st["logits"] if case.router_w is not None else case.logits
    if case.router_w is not None:
        assert nerr(st["logits"], O.router_logits(case.x, case.router_w)) < 1e-5
    chains = {v: O.prefill_forward(case, v, logits=shared_logits) for v in ("bf16", "exact")}
    wvar = "exact" if _small_rows(case, separate) else "bf16"  # the weights the GPU path multiplies with
    ref = chains[wvar]
    for key in ("ids", "sorted_token_ids", "sorted_expert_ids", "expert_offsets", "token_to_perm"):
        np.testing.assert_array_equal(st[key], ref[key], err_msg=key)
    np.testing.assert_allclose(st["wts"], ref["wts"], rtol=2e-6, atol=1e-7)
    R = int(ref["expert_offsets"][-1])
    I = case.I
    if separate:
        act, Y, out = _stagewise(case, st, R, wvar)
        errs = {"G": nerr(st["G"][:R], ref["G64"][:R]), "act": nerr(st["act"][:R], act)}
    else:
        G = ref["G64"][:R]
        _, Y, out = _stagewise(case, dict(st, G=np.zeros((R, 2 * I))), R, wvar)
        if _small_rows(case, separate):  # the small-row products apply the SwiGLU to FP32 g and u
            errs = {"act": nerr(st["act"][:R], O.swiglu_clamp(G[:, :I], G[:, I:], case.swiglu_limit))}
        else:  # the fused epilogue rounds g and u to BF16 first
            e_act, ok = fused_act_error(st["act"][:R], G, I, case.swiglu_limit)
            assert ok, "fused SwiGLU element bound"
            errs = {"act": e_act}
    errs.update(Y=nerr(st["Y"][:R], Y), out=nerr(st["out"], out))
    if case.shared is not None:
        errs["shared"] = nerr(st["shared"], ref["shared64"])
    assert all(e < TOL_BF16 for e in errs.values()), ("bf16 stage-wise", errs)
    ex = chains["exact"]
    keys = ("G", "act", "Y", "out") if separate else ("act", "Y", "out")
    chain = {k: nerr(st[k][:R] if k != "out" else st[k], ex[k + "64"][:R] if k != "out" else ex["out64"])
             for k in keys}
    chain_bf16 = nerr(st["out"], ref["out64"])
    assert all(e < TOL_EXACT for e in chain.values()), ("exact chain", chain, "bf16 chain out", chain_bf16)


@pytest.mark.parametrize("separate", [False, True], ids=["fused-swiglu", "separate-swiglu"])
def test_small_ragged_block(separate):
    c = S.make_block_case(T=37, H=512, I=256, E=5, k=2, routing="biased", seed=31)
    _check_full(c, separate)


def test_single_row():
    c = S.make_block_case(T=1, H=256, I=512, E=8, k=8, routing="biased", seed=32)
    _check_full(c)


@pytest.mark.parametrize("separate", [False, True], ids=["fused-swiglu", "separate-swiglu"])
def test_absent_expert_block(separate):
    c = S.make_block_case(T=64, H=256, I=256, E=6, k=2, routing="biased", seed=33, absent=(2,))
    _check_full(c, separate)


def test_expert_absent_only_in_gate_up():
    """The down GEMM starts on an expert once the gate/up GEMM has published all its activation
    rows; for an expert the gate/up table lacks, those rows are the zero rows that launch writes,
    and they must be published too (the down GEMM would otherwise wait out its 2 s bound)."""
    c = S.make_block_case(T=64, H=256, I=256, E=6, k=2, routing="biased", seed=35)
    c.gate_up.packed[3] = None
    c.gate_up.scales[3] = None
    assert (c.logits.argsort(axis=1)[:, -2:] == 3).any()  # expert 3 receives rows
    _check_full(c)
    assert moe.moe_get_device_error() == 0


@pytest.mark.parametrize("flags", [0, 2], ids=["tensor-core-gemms", "small-row-products"])
def test_eight_row_chunk(flags):
    """T = 8 at GLM-like widths: the default tensor-core GEMMs, and the small-row products that
    MOE_FWD_SMALL_ROWS selects."""
    c = S.make_block_case(T=8, H=1024, I=512, E=40, k=8, routing="biased", seed=38)
    db = DeviceBlock(c)
    db.cfg.flags = flags
    db.forward()
    torch.cuda.synchronize()
    st = db.stages()
    db.close()
    wvar = "exact" if flags else "bf16"
    ref = O.prefill_forward(c, wvar, logits=c.logits)
    for key in ("ids", "sorted_token_ids", "expert_offsets", "token_to_perm"):
        np.testing.assert_array_equal(st[key], ref[key], err_msg=key)
    R = c.T * c.k
    G = ref["G64"]
    _, Y, out = _stagewise(c, dict(st, G=np.zeros((R, 2 * c.I))), R, wvar)
    e_act = (nerr(st["act"], O.swiglu_clamp(G[:, :c.I], G[:, c.I:], c.swiglu_limit)) if flags
             else fused_act_error(st["act"], G, c.I, c.swiglu_limit)[0])
    errs = dict(act=e_act, Y=nerr(st["Y"], Y), out=nerr(st["out"], out))
    assert all(e < TOL_BF16 for e in errs.values()), errs
    assert nerr(st["out"], O.prefill_forward(c, "exact", logits=c.logits)["out64"]) < TOL_EXACT


@pytest.mark.parametrize("separate", [False, True], ids=["fused-swiglu", "separate-swiglu"])
def test_c1_full_chunk(separate):
    """Full routed-MoE block on one 256-row chunk, with the router GEMM (H 2048, I 768, E 64)."""
    _check_full(S.workload("c1"), separate)


def _check_sampled(case, tokens, variants=("bf16",)):
    """Sampled tokens at full size.  The sample always contains the tokens holding the largest
    |out|, |G| and |Y| of the GPU tensors, so the denominator max|ref| over the sampled rows is
    the full tensor's ||ref||_inf, as in the tolerance's definition; the numerator is the max
    over the sampled rows."""
    db = DeviceBlock(case)
    db.forward()
    torch.cuda.synchronize()
    T, k, E, H, I = case.T, case.k, case.E, case.H, case.I
    R = T * k
    ids = db.ws_view("ids", torch.int32, (T, k)).cpu().numpy()
    wts = db.ws_view("wts", torch.float32, (T, k)).cpu().numpy()
    t2p = db.ws_view("token_to_perm", torch.int32, (T, k)).cpu().numpy()
    off = db.ws_view("expert_offsets", torch.int32, (E + 1,)).cpu().numpy()
    sti = db.ws_view("sorted_token_ids", torch.int32, (R,))
    Ad = db.ws_view("act", torch.bfloat16, (R, I))
    Yd = db.ws_view("Y", torch.bfloat16, (R, H))
    # routing and the sort at full size, bit-exact
    rid, rw = O.route_topk(case.logits, k)
    np.testing.assert_array_equal(ids, rid)
    np.testing.assert_allclose(wts, rw, rtol=2e-6, atol=1e-7)
    srt = O.sort_by_expert(rid, E)
    np.testing.assert_array_equal(off, srt["expert_offsets"])
    np.testing.assert_array_equal(t2p, srt["token_to_perm"])
    np.testing.assert_array_equal(sti.cpu().numpy(), srt["sorted_token_ids"])
    nvalid = int(off[E])
    extra = [int(db.out.abs().amax(1).argmax()),
             int(sti[int(Ad[:nvalid].abs().amax(1).argmax())]),
             int(sti[int(Yd[:nvalid].abs().amax(1).argmax())])]
    tokens = sorted(set(list(tokens) + extra))
    out = bf16_host(db.out[tokens])
    rows = torch.from_numpy(t2p[tokens].reshape(-1)).long().cuda()
    Y = bf16_host(Yd[rows])
    A = bf16_host(Ad[rows])
    # act against the fused epilogue's reference (the SwiGLU of the oracle's BF16-rounded G),
    # then Y and out stage by stage on the GPU's own stage inputs; weights as the GPU path uses
    # them (BF16-rounded; FP32 for the small-row products, whose SwiGLU takes FP32 g and u)
    dq = {}
    ref = O.token_forward(case, tokens, rid, rw, "exact" if _small_rows(case) else "bf16", dq)
    G64 = ref["G64"].reshape(-1, 2 * I)
    ea = (nerr(A, O.swiglu_clamp(G64[:, :I], G64[:, I:], case.swiglu_limit)) if _small_rows(case)
          else fused_act_error(A, G64, I, case.swiglu_limit)[0])
    ys = np.stack([A[r] @ dq["dn"](int(e)).astype(np.float64).T for r, e in enumerate(rid[tokens].reshape(-1))])
    ey = nerr(Y, ys)
    perm = np.arange(len(tokens) * k, dtype=np.int32).reshape(len(tokens), k)
    eo = nerr(out, O.combine_indexed(Y, perm, rw[tokens]))
    assert max(ea, ey, eo) < TOL_BF16, ("bf16 stage-wise", tokens, ea, ey, eo)
    if "exact" in variants:
        ex = O.token_forward(case, tokens, rid, rw, "exact")
        Gx = ex["G64"].reshape(-1, 2 * I)
        chain = (nerr(A, O.swiglu_clamp(Gx[:, :I], Gx[:, I:], case.swiglu_limit)), nerr(Y, ex["Y64"].reshape(-1, H)),
                 nerr(out, ex["out64"]))
        assert max(chain) < TOL_EXACT, ("exact chain", tokens, chain, "bf16 chain out", nerr(out, ref["out64"]))
    db.close()


def test_c2_glm_chunk_sampled():
    c = S.workload("c2")
    _check_sampled(c, [0, 1023, 2047], variants=("bf16", "exact"))


def test_c3_zipf_skew_sampled():
    c = S.workload("c3")
    _check_sampled(c, [5, 8191], variants=("bf16", "exact"))


@pytest.mark.parametrize("T", [8, 16384])
def test_c4_sweep_points_sampled(T):
    c = S.workload("c4", T=T)
    _check_sampled(c, [0, T - 1])


def test_forward_graph_capture_replay():
    """No host round trip: the forward captures into a CUDA graph and replays bit-identically."""
    c = S.make_block_case(T=96, H=512, I=256, E=12, k=4, routing="biased", seed=34)
    db = DeviceBlock(c)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        db.forward(stream=s)
    torch.cuda.synchronize()
    eager = db.out.clone()
    db.out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        db.forward(stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(db.out.view(torch.int16), eager.view(torch.int16))
    db.close()


@pytest.mark.parametrize("routing,T,E,k", [("biased", 96, 12, 4), ("router", 96, 12, 4), ("router", 96, 80, 4),
                                            ("biased", 600, 4, 2)],
                         ids=["host-logits", "router-fused-topk", "router-e80", "host-logits-rows-in-expert-order"])
def test_host_memory_inputs_and_output(routing, T, E, k):
    """x, logits and out may be page-locked host memory: a host x is staged into the workspace
    (by the router kernel, or without a router by a staging kernel; with ~300 rows per expert the
    CTA-pair gate/up GEMM takes its rows in expert order, and the kernel storing them reads each
    host row once), host logits are read in place, the combine stores into the host out.  Eagerly
    and inside a captured graph the result equals the device-memory run bit for bit."""
    c = S.make_block_case(T=T, H=512, I=256, E=E, k=k, routing=routing, seed=36)
    db = DeviceBlock(c)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        db.forward(stream=s)
    torch.cuda.synchronize()
    ref = db.out.cpu()
    x_host = db.x.cpu().pin_memory()
    lg_host = db.logits.cpu().pin_memory() if db.logits is not None else None
    host = torch.zeros(c.T, c.H, dtype=torch.bfloat16).pin_memory()
    db.ws.zero_()

    def run():
        moe.moe_prefill_forward(db.cfg, x_host, db.gu.table, db.dn.table, db.ws, w_router=db.router_w,
                                logits=lg_host, out=host, stream=s)

    run()
    s.synchronize()
    assert torch.equal(host.view(torch.int16), ref.view(torch.int16))
    R = c.T * c.k
    if R / c.E > 128:  # the rows in expert order, each host row stored to its sorted positions
        sti = db.ws_view("sorted_token_ids", torch.int32, (R,)).cpu().long()
        n = int(db.ws_view("expert_offsets", torch.int32, (c.E + 1,))[c.E].item())
        rows = db.ws_view("x_sorted", torch.bfloat16, (R, c.H))[:n].cpu()
        assert torch.equal(rows.view(torch.int16), x_host[sti[:n]].view(torch.int16))
    else:
        staged = db.ws_view("x_stage", torch.bfloat16, (c.T, c.H))
        assert torch.equal(staged.cpu().view(torch.int16), x_host.view(torch.int16))
    host.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(host.view(torch.int16), ref.view(torch.int16))
    db.close()


def test_stage_events_inside_graph_capture():
    """Stage events recorded during capture become timestamp nodes: each replay records them."""
    c = S.make_block_case(T=96, H=512, I=256, E=12, k=4, routing="biased", seed=35)
    db = DeviceBlock(c)
    s = torch.cuda.Stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_FWD_NUM_EVENTS)]
    for e in evs:
        e.record(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_prefill_forward(db.cfg, db.x, db.gu.table, db.dn.table, db.ws, logits=db.logits, out=db.out,
                                stage_events=evs, stream=s)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        ms = [evs[j].elapsed_time(evs[j + 1]) for j in range(len(evs) - 1)]
        assert all(m >= 0.0 for m in ms) and evs[0].elapsed_time(evs[-1]) > 0.0
    db.close()


# ---------------------------------------------------------------------------- shared expert


def _shared_stagewise(case, T, clamped=False):
    """Shared expert alone against the oracle: gate/up, act and out each on the GPU's own BF16
    stage inputs (read back from the workspace), and the exact-FP32 chain."""
    db = DeviceBlock(case)
    out = db.shared_forward()
    torch.cuda.synchronize()
    I = case.shared.I
    ws = db.shared["ws"]
    gu = ws[:T * 2 * I * 2].view(torch.bfloat16).view(T, 2 * I)
    a_off = (T * 2 * I * 2 + 255) // 256 * 256
    act = ws[a_off:a_off + T * I * 2].view(torch.bfloat16).view(T, I)
    gu_h, act_h, out_h = bf16_host(gu), bf16_host(act), bf16_host(out)
    ref = O.shared_expert_mlp(case.x, case.shared, case.swiglu_limit, "bf16")
    errs = dict(gate=nerr(gu_h[:, :I], ref["gate64"]), up=nerr(gu_h[:, I:], ref["up64"]),
                act=nerr(act_h, O.swiglu_clamp(gu_h[:, :I], gu_h[:, I:], case.swiglu_limit)),
                out=nerr(out_h, act_h @ O.bf16_bits_to_f64(case.shared.down).T))
    assert all(e < TOL_BF16 for e in errs.values()), errs
    ex = O.shared_expert_mlp(case.x, case.shared, case.swiglu_limit, "exact")
    assert nerr(out_h, ex["out64"]) < TOL_EXACT, ("exact chain", nerr(out_h, ex["out64"]))
    if clamped:  # both clamps are exercised
        assert (ref["gate64"] > case.swiglu_limit).any() and (np.abs(ref["up64"]) > case.swiglu_limit).any()
    db.close()


@pytest.mark.parametrize("T,H,I,gain", [(37, 512, 256, 4.0), (256, 2048, 768, 1.0)],
                         ids=["ragged-small-clamped", "c1-size"])
def test_shared_expert_vs_oracle(T, H, I, gain):
    """`gain` scales the gate and up weights (a power of two: exact in BF16) so that |g| and |u|
    pass the SwiGLU limit and both clamps act."""
    c = S.make_block_case(T=T, H=H, I=I, E=2, k=1, routing="biased", seed=36, shared_inter=I)
    scale = lambda w: S.bf16_bits_from_f32((O.bf16_bits_to_f64(w) * gain).astype(np.float32))
    c.shared = S.SharedExpert(I=I, gate=scale(c.shared.gate), up=scale(c.shared.up), down=c.shared.down)
    _shared_stagewise(c, T, clamped=gain > 1.0)


def test_c1_chunk_with_shared_expert():
    """The 256-row chunk with the shared expert in the combine (routed steps stage by stage,
    the shared output against the oracle, the exact chain)."""
    _check_full(S.workload("c1s"))


def test_shared_expert_on_a_second_stream():
    """The shared expert on its own stream, joined by an event before the combine: the same
    bits as the serial forward, eagerly and from a captured graph."""
    c = S.make_block_case(T=96, H=512, I=256, E=12, k=4, routing="biased", seed=37, shared_inter=256)
    db = DeviceBlock(c)
    db.forward()
    torch.cuda.synchronize()
    serial = db.out.clone()
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    ready, fork = torch.cuda.Event(), torch.cuda.Event()

    def run():
        fork.record(main)
        side.wait_event(fork)
        db.shared_forward(stream=side)
        ready.record(side)
        db.forward(stream=main, shared_ready=ready)
        main.wait_stream(side)

    db.out.zero_()
    with torch.cuda.stream(main):
        run()
    torch.cuda.synchronize()
    assert torch.equal(db.out.view(torch.int16), serial.view(torch.int16))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        run()
    db.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(db.out.view(torch.int16), serial.view(torch.int16))
    db.close()


@pytest.mark.gpu
@pytest.mark.parametrize("T,H,E,k,renorm,bias", [(37, 512, 5, 2, True, False), (130, 1024, 40, 8, False, True),
                                                 (66, 512, 72, 4, True, True), (256, 2048, 64, 8, True, True)],
                         ids=["E5-cluster1-ragged", "E40-cluster5-no-renorm-bias", "E72-separate-launches",
                              "c1-shape-cluster8-bias"])
def test_forward_routing_equals_standalone_entry_points(T, H, E, k, renorm, bias):
    """With a router and E <= 64, the forward runs the router GEMM and the top-k as one launch (a
    cluster of ceil(E/8) CTAs per 4 rows); its logits, ids and weights must be the bits of
    moe_router_logits followed by moe_route_topk (the same tile routine and the same per-row
    selection routine).  T % 4 != 0 and E % 8 != 0 exercise the partial tiles; E = 72 takes the
    two separate launches."""
    c = S.make_block_case(T=T, H=H, I=256, E=E, k=k, routing="router", seed=61 + T + E)
    c.renormalize = 1 if renorm else 0
    db = DeviceBlock(c)
    b = torch.linspace(-0.05, 0.05, E, dtype=torch.float32, device="cuda") if bias else None
    moe.moe_prefill_forward(db.cfg, db.x, db.gu.table, db.dn.table, db.ws, w_router=db.router_w, router_bias=b,
                            out=db.out)
    torch.cuda.synchronize()
    st = db.stages()
    lg = moe.moe_router_logits(db.x, db.router_w)
    ids, wts = moe.moe_route_topk(lg, k, bias=b, renormalize=renorm, routed_scale=c.routed_scale)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    np.testing.assert_array_equal(st["logits"].view(np.uint32), lg.cpu().numpy().view(np.uint32))
    np.testing.assert_array_equal(st["ids"], ids.cpu().numpy())
    np.testing.assert_array_equal(st["wts"].view(np.uint32), wts.cpu().numpy().view(np.uint32))
    db.close()
