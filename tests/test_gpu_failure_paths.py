"""Failure paths of the GPU kernels, made on the host (no GPU fault, trap or endless loop).

* A pipeline wait that runs out: the grouped GEMM runs as the consumer of the forward's GEMM
  overlap with per-expert counters that nothing publishes, under a short wait bound.  The
  kernel must record MOE_DEVERR_TIMEOUT, drain its copies and MMAs, free its tensor memory and
  return; the device must keep working (a normal GEMM right after it matches the oracle).
* A gather index outside A (host-made): MOE_DEVERR_BAD_GATHER, row 0 read in its place.
* Counters published in time: the same consumer entry with counters already at their final
  value runs to the oracle's result.
"""

import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import moe_prefill_nvfp4_gb300 as moe  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402

from gpu_helpers import bf16_dev, nerr, upload  # noqa: E402


@pytest.fixture(autouse=True)
def _restore():
    moe.moe_get_device_error()
    yield
    moe.moe_debug_set_wait_limit_ns(0)
    moe.moe_debug_set_gemm_kernel(moe.MOE_GEMM_KERNEL_AUTO)
    moe.moe_get_device_error()


def _case(T=96, E=6):
    c = S.make_gemm_case(T=T, E=E, k=2, N=256, K=512, seed=181)
    srt = moe.moe_sort_by_expert(torch.from_numpy(c.ids).cuda(), c.E)
    return c, srt, upload(c.w)


def _oracle(c, s):
    wfn = lambda e: O.dequant_nvfp4(c.w.packed[e], c.w.scales[e], c.w.scale2[e], "bf16")
    return O.grouped_gemm(O.bf16_bits_to_f64(c.x), s["expert_offsets"], wfn, s["sorted_token_ids"])


@pytest.mark.parametrize("T,E", [(96, 6), (600, 4)], ids=["128-token-tiles", "384-token-tiles"])
def test_wait_runs_out_and_the_kernel_returns(T, E):
    """Both CTA-pair configurations: 128-token tiles with two accumulator buffers (16 rows per
    expert) and 384-token tiles with one (300 rows per expert)."""
    c, srt, proj = _case(T, E)
    R = c.T * c.k
    x = bf16_dev(c.x)
    never = torch.zeros(c.E, dtype=torch.int32, device="cuda")  # nothing ever publishes
    prev = moe.moe_debug_set_wait_limit_ns(50_000_000)  # 50 ms
    assert prev == 2_000_000_000
    xs = x[srt["sorted_token_ids"].long()].contiguous()  # rows in expert order (the pair kernel's A)
    with moe.gemm_kernel(moe.MOE_GEMM_KERNEL_PAIR):
        t0 = time.perf_counter()
        moe.moe_debug_grouped_gemm_after(xs, proj.table, srt["expert_offsets"], R, never, 1)
        code = moe.moe_get_device_error()
        dt = time.perf_counter() - t0
    assert code == 3, code  # MOE_DEVERR_TIMEOUT
    assert dt < 5.0  # returned after the short bound, not the default 2 s per wait chain
    moe.moe_debug_set_wait_limit_ns(0)
    # the device keeps answering: the same GEMM, then with counters that are already published
    C = moe.moe_w4a16_grouped_gemm(x, proj.table, srt["expert_offsets"], R, gather_ids=srt["sorted_token_ids"],
                                   c_dtype=torch.float32)
    assert moe.moe_get_device_error() == 0
    s = {k: v.cpu().numpy() for k, v in srt.items()}
    ref = _oracle(c, s)
    assert nerr(C.cpu().numpy().astype(np.float64), ref) < 2e-6
    counts = np.diff(s["expert_offsets"]).astype(np.int64) * 4  # rows x ready_need (1) x 4 warps
    ready = torch.from_numpy(counts.astype(np.int32)).cuda()
    with moe.gemm_kernel(moe.MOE_GEMM_KERNEL_PAIR):
        C2 = moe.moe_debug_grouped_gemm_after(xs, proj.table, srt["expert_offsets"], R, ready, 1)
        assert moe.moe_get_device_error() == 0
    assert nerr(C2.cpu().numpy().astype(np.float64), ref) < 2e-6
    proj.close()


def test_bad_gather_index():
    """The in-kernel A gather (single-CTA kernel: the pair kernel reads rows in expert order)."""
    which = moe.MOE_GEMM_KERNEL_SINGLE
    c, srt, proj = _case()
    R = c.T * c.k
    gather = srt["sorted_token_ids"].clone()
    bad = [0, 7, R - 1]
    gather[bad[0]] = c.T
    gather[bad[1]] = 1 << 30
    gather[bad[2]] = -1
    with moe.gemm_kernel(which):
        C = moe.moe_w4a16_grouped_gemm(bf16_dev(c.x), proj.table, srt["expert_offsets"], R, gather_ids=gather,
                                       c_dtype=torch.float32)
        assert moe.moe_get_device_error() == 5  # MOE_DEVERR_BAD_GATHER
    s = {k: v.cpu().numpy() for k, v in srt.items()}
    s["sorted_token_ids"] = gather.cpu().numpy().copy()
    s["sorted_token_ids"][bad] = 0
    assert nerr(C.cpu().numpy().astype(np.float64), _oracle(c, s)) < 2e-6
    proj.close()
