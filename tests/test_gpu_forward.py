"""GPU parity of the whole routed-MoE prefill path (moe_prefill_forward) against the oracle.

Routing and the sort are compared bit-exactly on shared logits (the GPU's router logits are
fed to the oracle's top-k, so a different summation order cannot flip a near tie); every
float stage (wts, G, act, Y, out) within the tolerances.  Full-size workloads are checked on
sampled tokens, which the oracle computes one token at a time.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import moe_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402

import moe_prefill_nvfp4_gb300 as moe  # noqa: E402

from gpu_helpers import TOL_BF16, TOL_EXACT, DeviceBlock, bf16_host, nerr  # noqa: E402


@pytest.fixture(autouse=True)
def _no_device_error():
    moe.moe_get_device_error()
    yield
    assert moe.moe_get_device_error() == 0


def _check_full(case, variants=("bf16", "exact")):
    db = DeviceBlock(case)
    db.forward()
    torch.cuda.synchronize()
    st = db.stages()
    db.close()
    for v in variants:
        ref = O.prefill_forward(case, v, logits=st["logits"])
        if case.router_w is not None and v == "bf16":
            assert nerr(st["logits"], O.router_logits(case.x, case.router_w)) < 1e-5
        for key in ("ids", "sorted_token_ids", "sorted_expert_ids", "expert_offsets", "token_to_perm"):
            np.testing.assert_array_equal(st[key], ref[key], err_msg=key)
        np.testing.assert_allclose(st["wts"], ref["wts"], rtol=2e-6, atol=1e-7)
        R = int(ref["expert_offsets"][-1])
        tol = TOL_BF16 if v == "bf16" else TOL_EXACT
        for key in ("G", "act", "Y"):
            e = nerr(st[key][:R], ref[key + "64"][:R])
            assert e < tol, (v, key, e)
        e = nerr(st["out"], ref["out64"])
        assert e < tol, (v, "out", e)


def test_small_ragged_block():
    c = S.make_block_case(T=37, H=512, I=256, E=5, k=2, routing="biased", seed=31)
    _check_full(c)


def test_single_row():
    c = S.make_block_case(T=1, H=256, I=512, E=8, k=8, routing="biased", seed=32)
    _check_full(c)


def test_absent_expert_block():
    c = S.make_block_case(T=64, H=256, I=256, E=6, k=2, routing="biased", seed=33, absent=(2,))
    _check_full(c)


def test_c1_full_chunk():
    """Full routed-MoE block on one 256-row chunk, with the router GEMM (H 2048, I 768, E 64)."""
    _check_full(S.workload("c1"))


def _check_sampled(case, tokens, variants=("bf16",)):
    db = DeviceBlock(case)
    db.forward()
    torch.cuda.synchronize()
    T, k, E, H, I = case.T, case.k, case.E, case.H, case.I
    ids = db.ws_view("ids", torch.int32, (T, k)).cpu().numpy()
    wts = db.ws_view("wts", torch.float32, (T, k)).cpu().numpy()
    t2p = db.ws_view("token_to_perm", torch.int32, (T, k)).cpu().numpy()
    off = db.ws_view("expert_offsets", torch.int32, (E + 1,)).cpu().numpy()
    # routing and the sort at full size, bit-exact
    rid, rw = O.route_topk(case.logits, k)
    np.testing.assert_array_equal(ids, rid)
    np.testing.assert_allclose(wts, rw, rtol=2e-6, atol=1e-7)
    srt = O.sort_by_expert(rid, E)
    np.testing.assert_array_equal(off, srt["expert_offsets"])
    np.testing.assert_array_equal(t2p, srt["token_to_perm"])
    out = bf16_host(db.out[tokens])
    rows = t2p[tokens].reshape(-1)
    G = bf16_host(db.ws_view("G", torch.bfloat16, (T * k, 2 * I))[torch.from_numpy(rows).long().cuda()])
    Y = bf16_host(db.ws_view("Y", torch.bfloat16, (T * k, H))[torch.from_numpy(rows).long().cuda()])
    db.close()
    for v in variants:
        ref = O.token_forward(case, tokens, rid, rw, v)
        tol = TOL_BF16 if v == "bf16" else TOL_EXACT
        assert nerr(G, ref["G64"].reshape(-1, 2 * I)) < tol, (v, "G")
        assert nerr(Y, ref["Y64"].reshape(-1, H)) < tol, (v, "Y")
        e = nerr(out, ref["out64"])
        assert e < tol, (v, "out", e)


def test_c2_glm_chunk_sampled():
    c = S.workload("c2")
    _check_sampled(c, [0, 1023, 2047], variants=("bf16", "exact"))


def test_c3_zipf_skew_sampled():
    c = S.workload("c3")
    _check_sampled(c, [5, 8191])


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
