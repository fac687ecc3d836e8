"""The whole forward on seeded random shapes against the oracle, stage by stage.

Each case draws T, H, I, E, k, the routing recipe, the SwiGLU mode and the GEMM kernel choice
(automatic, single-CTA, CTA pairs where the shapes allow) from a fixed seed, so the sweep is the
same on every run; ``_check_full`` compares routing and the sort bit for bit and every float
stage within the BF16 stage-wise and exact-chain bounds.  The draws cover one-row chunks,
single-expert layers, top-1 routing, ragged token counts that leave partial tiles, and shapes on
both sides of the per-expert row counts where the kernel choice changes.
"""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

import moe_prefill_nvfp4_gb300 as moe  # noqa: E402
from synth import inputs as S  # noqa: E402

from test_gpu_forward import _check_full  # noqa: E402


def _draw(i):
    g = np.random.default_rng(9000 + i)
    H = int(g.choice([256, 512, 768, 1024]))
    I = int(g.choice([256, 512, 768]))  # the expert tables take K (H, and I for down) in multiples of 256
    E = int(g.choice([1, 2, 3, 7, 16, 33, 40]))
    k = int(g.integers(1, min(8, E) + 1))
    T = int(g.choice([1, 2, 7, 31, 96, 257, 600]))
    routing = "router" if (E <= 64 and g.random() < 0.5) else "biased"
    separate = bool(g.random() < 0.25)
    pair_ok = I % 256 == 0 and H % 256 == 0
    # the separate-SwiGLU path's gate/up GEMM gathers its rows inside the kernel: single-CTA only
    mode = g.choice(["auto", "single", "pair"] if pair_ok and not separate else ["auto", "single"])
    return dict(T=T, H=H, I=I, E=E, k=k, routing=routing, separate=separate, mode=str(mode), seed=9100 + i)


CASES = [_draw(i) for i in range(18)]


@pytest.mark.parametrize("p", CASES, ids=[f"T{c['T']}-H{c['H']}-I{c['I']}-E{c['E']}-k{c['k']}-{c['routing']}"
                                          f"-{'sep' if c['separate'] else 'fused'}-{c['mode']}" for c in CASES])
def test_random_shape_forward(p):
    moe.moe_get_device_error()
    c = S.make_block_case(T=p["T"], H=p["H"], I=p["I"], E=p["E"], k=p["k"], routing=p["routing"], seed=p["seed"])
    mode = {"auto": moe.MOE_GEMM_KERNEL_AUTO, "single": moe.MOE_GEMM_KERNEL_SINGLE,
            "pair": moe.MOE_GEMM_KERNEL_PAIR}[p["mode"]]
    with moe.gemm_kernel(mode):
        _check_full(c, separate=p["separate"])
    assert moe.moe_get_device_error() == 0
