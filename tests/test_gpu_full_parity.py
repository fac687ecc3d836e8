"""Full-size parity of the forward against the oracle, element by element where the oracle can
afford it, and the guard bands around every output the forward writes.

* 256-row block (router GEMM, 64 experts): the whole BF16 chain (the oracle rounding dequantised
  weights and every inter-stage activation to BF16, run independently from x) against out.
* 2048-row GLM chunk: every element of act, Y and out, stage by stage on the GPU's own stage
  inputs, plus the whole BF16 chain and the exact-weight chain, over the full tensors.
* 8192-row Zipf chunk: every row of the hottest expert (act and Y), and 64 seeded tokens plus the
  tokens holding the largest |act|, |Y| and |out|: out against both chains.
* Row sweep at GLM shapes, all eleven row counts: sampled tokens against both oracle variants.

The oracle's per-expert stages run in worker processes (tests/oracle_pool.py, pinned to the
oracle's own prefill_forward).  Each check prints one ``PARITY_RECORD`` line with the measured
normalised errors (max|gpu - ref| / max|ref|).

Bounds.  Stage by stage against the BF16 variant: 4e-3.  Exact-weight chain: 1e-2.  Whole BF16
chain from x: 5e-3 (BF16_CHAIN_BOUND).  out is BF16 and the oracle's out unrounded, so out's own
rounding alone reaches up to 2^-8 = 3.9e-3 of max|out| (half a unit at the bottom of a binade);
on top of it, FP32 summation order moves about 0.2% of G's BF16 roundings (the fused SwiGLU
rounds its accumulators to BF16 like the oracle's G stage) and those flips reach out through act
and Y.  Measured: 2.2e-3 to 4.7e-3 over the checks below.
"""

import json

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import moe_prefill_nvfp4_gb300 as moe  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402

from gpu_helpers import TOL_BF16, TOL_EXACT, DeviceBlock, bf16_host, fused_act_error, nerr  # noqa: E402
from oracle_pool import OraclePool, run_block, run_rows  # noqa: E402

BF16_CHAIN_BOUND = 5e-3


def record(name, **vals):
    print("PARITY_RECORD", json.dumps({"check": name, **{k: float(v) for k, v in vals.items()}}), flush=True)


@pytest.fixture(scope="module")
def pool():
    with OraclePool() as p:
        yield p


@pytest.fixture(autouse=True)
def _no_device_error():
    moe.moe_get_device_error()
    yield
    assert moe.moe_get_device_error() == 0


def _routing_and_sort_bit_exact(db, case, logits):
    T, k, E = case.T, case.k, case.E
    R = T * k
    ids = db.ws_view("ids", torch.int32, (T, k)).cpu().numpy()
    wts = db.ws_view("wts", torch.float32, (T, k)).cpu().numpy()
    rid, rw = O.route_topk(logits, k)
    np.testing.assert_array_equal(ids, rid)
    np.testing.assert_allclose(wts, rw, rtol=2e-6, atol=1e-7)
    srt = O.sort_by_expert(rid, E)
    for key, shape in (("sorted_token_ids", (R,)), ("sorted_expert_ids", (R,)), ("expert_offsets", (E + 1,)),
                       ("token_to_perm", (T, k))):
        np.testing.assert_array_equal(db.ws_view(key, torch.int32, shape).cpu().numpy(), srt[key], err_msg=key)
    return rid, rw, srt


MODES = pytest.mark.parametrize("separate", [False, True], ids=["fused-swiglu", "separate-swiglu"])


@MODES
def test_whole_bf16_chain_256_row_block(separate):
    c = S.workload("c1")
    db = DeviceBlock(c, separate=separate)
    db.forward()
    torch.cuda.synchronize()
    st = db.stages()
    db.close()
    chains = {v: O.prefill_forward(c, v, logits=st["logits"]) for v in ("bf16", "exact")}
    R = c.T * c.k
    e_bf16 = {k: nerr(st[k][:R], chains["bf16"][k + "64"][:R]) for k in ("act", "Y")}
    e_bf16["out"] = nerr(st["out"], chains["bf16"]["out64"])
    e_ex = nerr(st["out"], chains["exact"]["out64"])
    record(f"c1 whole chain ({'separate' if separate else 'fused'} SwiGLU)",
           **{f"bf16_chain_{k}": v for k, v in e_bf16.items()}, exact_chain_out=e_ex)
    assert e_bf16["out"] < BF16_CHAIN_BOUND and e_ex < TOL_EXACT


@MODES
def test_2048_row_glm_chunk_every_element(pool, separate):
    c = S.workload("c2")
    db = DeviceBlock(c, separate=separate)
    db.forward()
    torch.cuda.synchronize()
    rid, rw, srt = _routing_and_sort_bit_exact(db, c, c.logits)
    st = db.stages()
    db.close()
    R = c.T * c.k
    I = c.I
    act, Y, out = st["act"][:R], st["Y"][:R], st["out"]
    bf = run_block(pool, c, srt, "bf16", act_in=act, keep_g=True)
    ex = run_block(pool, c, srt, "exact", keep_g=False)
    assert not np.isnan(bf["act64"]).any() and not np.isnan(ex["Y64"]).any()
    # stage by stage on the GPU's own inputs: with the SwiGLU fused into the gate/up epilogue act is
    # the SwiGLU of the BF16-rounded FP32 accumulators (no G in memory: its reference is the
    # oracle's BF16 G, either rounding at a midpoint); separately, G and then act of the GPU's G
    G64 = bf.pop("G64")
    if separate:
        G = st["G"][:R]
        stage = {"G": nerr(G, G64), "act": nerr(act, O.swiglu_clamp(G[:, :I], G[:, I:], c.swiglu_limit))}
    else:
        e_act, ok = fused_act_error(act, G64, I, c.swiglu_limit)
        assert ok, "fused SwiGLU element bound"
        stage = {"act": e_act}
    del G64
    stage["Y"] = nerr(Y, bf["Y64_in"])
    stage["out"] = nerr(out, O.combine_indexed(Y, st["token_to_perm"], rw))
    # whole chains from x
    chain_bf16 = {"act": nerr(act, bf["act64"]), "Y": nerr(Y, bf["Y64"]),
                  "out": nerr(out, O.combine_indexed(O._to_stage(bf["Y64"], "bf16"), srt["token_to_perm"], rw))}
    chain_ex = {"act": nerr(act, ex["act64"]), "Y": nerr(Y, ex["Y64"]),
                "out": nerr(out, O.combine_indexed(O._to_stage(ex["Y64"], "exact"), srt["token_to_perm"], rw))}
    record(f"c2 every element ({'separate' if separate else 'fused'} SwiGLU)",
           **{f"stage_{k}": v for k, v in stage.items()}, **{f"bf16_chain_{k}": v for k, v in chain_bf16.items()},
           **{f"exact_chain_{k}": v for k, v in chain_ex.items()})
    assert max(stage.values()) < TOL_BF16
    assert chain_bf16["out"] < BF16_CHAIN_BOUND
    assert max(chain_ex.values()) < TOL_EXACT


def _rows_of(db, name, rows, width):
    t = db.ws_view(name, torch.bfloat16, (db.case.T * db.case.k, width))
    return bf16_host(t[torch.as_tensor(np.asarray(rows), dtype=torch.long, device="cuda")])


def _sampled_check(pool, c, db, tokens, rid, rw, srt, tag):
    """act, Y (stage-wise and whole chain) on the sampled tokens' rows and out on the tokens;
    returns the record."""
    k, I, H = c.k, c.I, c.H
    t2p = srt["token_to_perm"]
    tokens = np.asarray(sorted(set(int(t) for t in tokens)))
    rows = t2p[tokens].reshape(-1)
    act = _rows_of(db, "act", rows, I)
    Y = _rows_of(db, "Y", rows, H)
    out = bf16_host(db.out[torch.as_tensor(tokens, dtype=torch.long, device="cuda")])
    bf = run_rows(pool, c, srt, "bf16", rows, act_in=act, keep_g=True)
    ex = run_rows(pool, c, srt, "exact", rows)
    perm = np.arange(len(tokens) * k).reshape(len(tokens), k)
    G64 = bf["G64"]  # the fused SwiGLU's act: the SwiGLU of the BF16-rounded FP32 accumulators
    e = dict(stage_act=fused_act_error(act, G64, I, c.swiglu_limit)[0],
             stage_Y=nerr(Y, bf["Y64_in"]), bf16_chain_act=nerr(act, bf["act64"]),
             stage_out=nerr(out, O.combine_indexed(Y, perm, rw[tokens])),
             bf16_chain_out=nerr(out, O.combine_indexed(O._to_stage(bf["Y64"], "bf16"), perm, rw[tokens])),
             exact_chain_out=nerr(out, O.combine_indexed(O._to_stage(ex["Y64"], "exact"), perm, rw[tokens])),
             exact_chain_act=nerr(act, ex["act64"]), exact_chain_Y=nerr(Y, ex["Y64"]))
    record(tag, tokens=len(tokens), **e)
    assert max(e["stage_act"], e["stage_Y"], e["stage_out"]) < TOL_BF16, e
    assert e["bf16_chain_out"] < BF16_CHAIN_BOUND, e
    assert max(e["exact_chain_out"], e["exact_chain_act"], e["exact_chain_Y"]) < TOL_EXACT, e


def _argmax_tokens(db, srt, R, I, H):
    sti = srt["sorted_token_ids"]
    a = db.ws_view("act", torch.bfloat16, (R, I))
    y = db.ws_view("Y", torch.bfloat16, (R, H))
    return [int(db.out.abs().amax(1).argmax()), int(sti[int(a.abs().amax(1).argmax())]),
            int(sti[int(y.abs().amax(1).argmax())])]


def test_8192_row_zipf_hot_expert_rows_and_sampled_tokens(pool):
    c = S.workload("c3")
    db = DeviceBlock(c)
    db.forward()
    torch.cuda.synchronize()
    rid, rw, srt = _routing_and_sort_bit_exact(db, c, c.logits)
    off = srt["expert_offsets"]
    counts = np.diff(off)
    hot = int(counts.argmax())
    rows = np.arange(off[hot], off[hot + 1])
    act = _rows_of(db, "act", rows, c.I)
    Y = _rows_of(db, "Y", rows, c.H)
    R = int(off[-1])
    bf = run_rows(pool, c, srt, "bf16", rows, act_in=act, keep_g=True, rows_per_task=256)
    G64 = bf["G64"]
    e_act = fused_act_error(act, G64, c.I, c.swiglu_limit)[0]
    e_y = nerr(Y, bf["Y64_in"])
    record("c3 hottest expert, every row", expert=hot, rows=len(rows), stage_act=e_act, stage_Y=e_y,
           bf16_chain_act=nerr(act, bf["act64"]), bf16_chain_Y=nerr(Y, bf["Y64"]))
    assert len(rows) > 4000 and max(e_act, e_y) < TOL_BF16
    g = np.random.default_rng(2024)
    tokens = list(g.choice(c.T, 64, replace=False)) + _argmax_tokens(db, srt, R, c.I, c.H)
    _sampled_check(pool, c, db, tokens, rid, rw, srt, "c3 sampled tokens")
    db.close()


def test_row_sweep_all_row_counts_sampled(pool):
    base = S.workload("c4", T=8)
    for T in S.SWEEP_ROWS:
        c = S.make_block_case(T=T, H=base.H, I=base.I, E=base.E, k=base.k, routing="biased",
                              seed=S.WORKLOADS["c4"]["seed"], with_weights=False)
        c.gate_up, c.down = base.gate_up, base.down
        db = DeviceBlock(c)
        db.forward()
        torch.cuda.synchronize()
        rid, rw, srt = _routing_and_sort_bit_exact(db, c, c.logits)
        R = T * c.k
        g = np.random.default_rng(T)
        tokens = [0, T - 1] + list(g.choice(T, min(T, 2), replace=False)) + _argmax_tokens(db, srt, R, c.I, c.H)
        _sampled_check(pool, c, db, tokens, rid, rw, srt, f"c4 T={T}")
        db.close()


# ------------------------------------------------------------------------------- guard bands


@pytest.mark.parametrize("pair", [False, True], ids=["auto-kernels", "pair-kernel"])
@pytest.mark.parametrize("routing,T,H,I,E,k", [("router", 256, 2048, 768, 64, 8), ("biased", 300, 1024, 512, 40, 8),
                                               ("biased", 37, 512, 256, 5, 2)],
                         ids=["256-row-block", "300-rows-E40", "ragged-small"])
def test_forward_writes_nothing_outside_its_outputs(routing, T, H, I, E, k, pair):
    """Sentinel margins: two guard rows on each side of out, and the workspace filled with a
    pattern before the forward; afterwards the guard rows and every workspace byte past the used
    part of each buffer (up to the next buffer, and the buffers the path does not use) still hold
    the sentinel."""
    c = S.make_block_case(T=T, H=H, I=I, E=E, k=k, routing=routing, seed=191 + T)
    db = DeviceBlock(c)
    big = torch.full((T + 4, H), -5.0, dtype=torch.bfloat16, device="cuda")
    db.out = big[2:T + 2]
    db.ws.fill_(0x5A)
    with moe.gemm_kernel(moe.MOE_GEMM_KERNEL_PAIR if pair else moe.MOE_GEMM_KERNEL_AUTO):
        db.forward()
        torch.cuda.synchronize()
    assert (big[:2] == -5.0).all() and (big[T + 2:] == -5.0).all()
    L = db.layout
    R = T * k
    used = {"logits": T * E * 4 if routing == "router" else 0, "ids": R * 4, "wts": R * 4, "sorted_token_ids": R * 4,
            "sorted_expert_ids": R * 4, "expert_offsets": (E + 1) * 4, "token_to_perm": R * 4,
            "ready": (2 * E + 1) * 4, "G": 0, "act": R * I * 2, "Y": R * H * 2, "x_stage": 0,
            "x_sorted": R * H * 2 if pair else 0}
    names = ["logits", "ids", "wts", "sorted_token_ids", "sorted_expert_ids", "expert_offsets", "token_to_perm",
             "sort_scratch", "ready", "G", "act", "Y", "x_stage", "x_sorted", "total"]
    ws = db.ws.cpu().numpy()
    for a, b in zip(names[:-1], names[1:]):
        if a not in used:
            continue  # the sort's scratch: its used size depends on the segment count
        lo, hi = getattr(L, a) + used[a], getattr(L, b)
        assert (ws[lo:hi] == 0x5A).all(), f"bytes after {a} changed"
    st = db.stages()
    assert np.isfinite(st["act"][:R]).all() and np.isfinite(st["Y"][:R]).all()
    db.close()
