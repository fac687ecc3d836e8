"""Expert parallelism on one GPU: the per-rank forward of ``moe_prefill_nvfp4_gb300.ep``.

Runs on more than one GPU are not made here (one GPU per run); the ranks are emulated one after
another on the same GPU, with no collective between them (their forwards do not wait on each
other), and their partial outputs are summed on the host in place of the all-reduce, whose host
logic tests/test_ep_gloo.py runs on gloo ranks.

* ``MOE_FWD_NO_MULTICAST`` changes how the single-CTA GEMM loads activation tiles, not what it
  computes: the forward's outputs are bit-identical with and without it.
* Each emulated rank holds one block of experts (``local_projection``: the others absent); its
  act and Y rows of the local experts equal the single-GPU forward's bit for bit and all other
  rows are zero; the sum of the partial outs (rank 0 adding the shared expert) matches the
  single-GPU out within the BF16 roundings of the partials.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import moe_prefill_nvfp4_gb300 as moe  # noqa: E402
from moe_prefill_nvfp4_gb300.ep import expert_block, local_projection  # noqa: E402
from synth import inputs as S  # noqa: E402

from gpu_helpers import DeviceBlock, bf16_host, make_cfg  # noqa: E402

CASES = [(256, 2048, 768, 64, 8, "router", None), (600, 512, 256, 4, 2, "biased", None),
         (96, 512, 256, 12, 4, "biased", 256)]
IDS = ["256-row-block-multicast-clusters", "300-rows-per-expert-pairs", "shared-expert"]


@pytest.fixture(autouse=True)
def _no_device_error():
    moe.moe_get_device_error()
    yield
    assert moe.moe_get_device_error() == 0


def _block(T, H, I, E, k, routing, shared):
    return S.make_block_case(T=T, H=H, I=I, E=E, k=k, routing=routing, seed=301 + T, shared_inter=shared)


@pytest.mark.parametrize("T,H,I,E,k,routing,shared", CASES[:2], ids=IDS[:2])
def test_no_multicast_forward_is_bit_identical(T, H, I, E, k, routing, shared):
    c = _block(T, H, I, E, k, routing, shared)
    db = DeviceBlock(c)
    db.forward()
    torch.cuda.synchronize()
    ref = {n: v.copy() for n, v in db.stages().items() if v is not None}
    db.cfg = make_cfg(c, moe.MOE_FWD_NO_MULTICAST)
    db.out.zero_()
    db.forward()
    torch.cuda.synchronize()
    got = db.stages()
    for n in ("ids", "sorted_token_ids", "expert_offsets", "act", "Y", "out"):
        np.testing.assert_array_equal(got[n], ref[n], err_msg=n)
    db.close()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("T,H,I,E,k,routing,shared", CASES, ids=IDS)
def test_emulated_ranks_sum_to_the_single_gpu_forward(T, H, I, E, k, routing, shared, world):
    c = _block(T, H, I, E, k, routing, shared)
    full = DeviceBlock(c)
    full.forward()
    torch.cuda.synchronize()
    ref = full.stages()
    off = ref["expert_offsets"]
    R = T * k
    total = np.zeros((T, H), dtype=np.float64)
    partial_max = 0.0
    cfg = make_cfg(c, moe.MOE_FWD_NO_MULTICAST)
    for rank in range(world):
        gu = local_projection(c.gate_up.packed, c.gate_up.scales, c.gate_up.scale2, 2 * I, H, rank, world)
        dn = local_projection(c.down.packed, c.down.scales, c.down.scale2, H, I, rank, world)
        full.ws.fill_(0x5A)
        out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        shared_out = full.shared["out"] if (shared and rank == 0) else None
        moe.moe_prefill_forward(cfg, full.x, gu.table, dn.table, full.ws, w_router=full.router_w, logits=full.logits,
                                out=out, shared_out=shared_out)
        torch.cuda.synchronize()
        st = full.stages()
        mine = expert_block(E, rank, world)
        rows = np.zeros(R, dtype=bool)
        for e in mine:
            rows[off[e]:off[e + 1]] = True
        for n in ("act", "Y"):
            np.testing.assert_array_equal(st[n][:R][rows], ref[n][:R][rows], err_msg=f"rank {rank} {n}")
            assert (st[n][:R][~rows] == 0).all(), f"rank {rank} {n}: rows of remote experts"
        part = bf16_host(out).astype(np.float64)
        partial_max += np.abs(part).max()
        total += part
        gu.close()
        dn.close()
    # each partial out and the single-GPU out are rounded to BF16 once (at most half a unit: 2^-8
    # of the magnitude, BF16 having 8 significant bits), and the FP32 sums differ only in their
    # association across the ranks
    ref_out = ref["out"].astype(np.float64)
    bound = 2.0 ** -8 * (partial_max + np.abs(ref_out).max()) + 1e-5 * np.abs(ref_out).max()
    assert np.abs(total - ref_out).max() <= bound, (np.abs(total - ref_out).max(), bound)
    full.close()
