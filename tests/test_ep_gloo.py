"""Expert parallelism's host logic on CPU ranks over gloo.

The expert partition, the per-rank forward over the local experts (every other expert absent),
the shared expert on rank 0 only, and the one all-reduce (sum) of out.  The per-rank compute here
is the oracle's forward over this rank's experts (``ep_prefill_forward``'s `forward` argument; the
library's GPU forward is the per-rank compute in tests/test_gpu_ep.py), so the sum over the ranks
must equal the oracle's forward over all experts up to fp64 summation order: absent experts leave
their rows zero, and every local row is the same computation as in the single-GPU forward.
"""

import copy
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from moe_prefill_nvfp4_gb300.ep import expert_block


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    from synth import inputs as S

    return S.make_block_case(T=24, H=256, I=128, E=7, k=3, routing="biased", seed=77, shared_inter=128)


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    import moe_prefill_nvfp4_gb300 as moe
    from moe_prefill_nvfp4_gb300.ep import ep_prefill_forward
    from oracle import moe_oracle as O

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = _case()
        mine = expert_block(case.E, rank, world)
        local = copy.copy(case)
        for name in ("gate_up", "down"):
            proj = copy.copy(getattr(case, name))
            proj.packed = [p if e in mine else None for e, p in enumerate(proj.packed)]
            proj.scales = [s if e in mine else None for e, s in enumerate(proj.scales)]
            setattr(local, name, proj)
        seen = {}

        def forward(cfg, x, w_gu, w_dn, ws, *, w_router, logits, router_bias, out, stream, shared_out):
            seen["flags"] = cfg.flags
            c = copy.copy(local)
            c.shared = case.shared if shared_out is not None else None
            return torch.from_numpy(O.prefill_forward(c, "bf16")["out64"].copy())

        cfg = moe.MoePrefillConfig(case.H, case.I, case.E, case.k, case.swiglu_limit, case.renormalize,
                                   case.routed_scale, 0)
        marker = torch.zeros(1)  # the shared expert's output (its presence is what the rank sees)
        out = ep_prefill_forward(cfg, torch.zeros(case.T, case.H), None, None, None, forward=forward,
                                 shared_out=marker)
        q.put((rank, seen["flags"], out.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ep_sum_over_ranks_equals_the_single_gpu_forward(world):
    from oracle import moe_oracle as O

    import moe_prefill_nvfp4_gb300 as moe

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ref = O.prefill_forward(_case(), "bf16")["out64"]
    for rank, flags, out in got:
        assert flags & moe.MOE_FWD_NO_MULTICAST  # no cluster-multicast loads in a multi-GPU run
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("E,world", [(160, 8), (64, 3), (7, 7), (5, 2), (1, 1)])
def test_expert_block_partition(E, world):
    blocks = [expert_block(E, r, world) for r in range(world)]
    assert [e for b in blocks for e in b] == list(range(E))  # contiguous, disjoint, covering
    sizes = [len(b) for b in blocks]
    assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        expert_block(E, world, world)
