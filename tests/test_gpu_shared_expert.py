"""GPU parity of the shared expert's dense tensor-core GEMMs against the oracle.

The shared expert ("glm5next_mlp/forward.rs" (spark), forward_dense) runs as a dense BF16 GEMM
for gate and up (one launch, written as gate | up into the workspace), the SwiGLU, and a dense
BF16 GEMM for down.  Every stage is checked element by element against the oracle on the GPU's
own BF16 stage inputs: a dense product's BF16 output lies within one BF16 unit of the oracle's
fp64 product (its rounding of an FP32 sum, whose order differs from the oracle's) plus the FP32
accumulation's own error (1e-6 of the tensor's max); the SwiGLU within one BF16 unit of the
oracle's SwiGLU of the GPU's gate and up.  Shapes cover k not a multiple of 64, weight rows not a
multiple of 128, a single token, and the 64-, 128- and 256-token tiles (with several tiles per
CTA); sentinels around the output must survive.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import moe_prefill_nvfp4_gb300 as moe  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402

from gpu_helpers import TOL_BF16, bf16_dev, bf16_host, nerr  # noqa: E402


@pytest.fixture(autouse=True)
def _no_device_error():
    moe.moe_get_device_error()
    yield
    assert moe.moe_get_device_error() == 0


def _within_one_bf16_unit(got, ref64, what):
    bound = np.abs(ref64) * 2.0 ** -8 + 1e-6 * np.abs(ref64).max()
    bad = np.abs(got - ref64) > bound
    assert not bad.any(), (what, np.argwhere(bad)[:4], got[bad][:4], ref64[bad][:4])
    assert nerr(got, ref64) < TOL_BF16, (what, nerr(got, ref64))


@pytest.mark.parametrize("T,H,I", [(300, 520, 200), (1, 256, 128), (2048, 512, 768), (4096, 512, 768)],
                         ids=["ragged-k-and-rows", "one-token", "128-token-tiles", "256-token-tiles"])
def test_shared_expert_dense_gemms(T, H, I):
    g = np.random.default_rng(T + H + I)
    x = S.bf16_bits_from_f32(g.standard_normal((T, H)).astype(np.float32))
    sh = S.shared_expert_weights(T + 7, H, I)
    pad = 64
    flat = torch.full((T * H + 2 * pad,), 3.0, dtype=torch.bfloat16, device="cuda")
    out = flat[pad:pad + T * H].view(T, H)
    ws = torch.full((moe.moe_shared_expert_workspace_bytes(T, H, I),), 0x7F, dtype=torch.uint8, device="cuda")
    moe.moe_shared_expert_forward(bf16_dev(x), bf16_dev(sh.gate), bf16_dev(sh.up), bf16_dev(sh.down), 7.0, ws=ws,
                                  out=out)
    torch.cuda.synchronize()
    assert (flat[:pad].float() == 3.0).all() and (flat[pad + T * H:].float() == 3.0).all(), "guard band"
    gu = bf16_host(ws[:T * 2 * I * 2].view(torch.bfloat16).view(T, 2 * I))
    a_off = (T * 2 * I * 2 + 255) // 256 * 256
    act = bf16_host(ws[a_off:a_off + T * I * 2].view(torch.bfloat16).view(T, I))
    got = bf16_host(out)
    ref = O.shared_expert_mlp(x, sh, 7.0, "bf16")
    _within_one_bf16_unit(gu[:, :I], ref["gate64"], "gate")
    _within_one_bf16_unit(gu[:, I:], ref["up64"], "up")
    _within_one_bf16_unit(act, O.swiglu_clamp(gu[:, :I], gu[:, I:], 7.0), "act")
    _within_one_bf16_unit(got, act @ O.bf16_bits_to_f64(sh.down).T, "out")


def test_shared_expert_exact_dyadic():
    """Small integers in x and in the weights (powers of two): every product and FP32 partial sum
    is exact, so gate and up equal the oracle's exactly in any summation order."""
    T, H, I = 130, 384, 256
    g = np.random.default_rng(5)
    x = S.bf16_bits_from_f32(g.integers(-2, 3, (T, H)).astype(np.float32))
    w = lambda r, c: S.bf16_bits_from_f32((2.0 ** g.integers(-4, 0, (r, c)) * g.choice([-1, 0, 1], (r, c)))
                                          .astype(np.float32))
    sh = S.SharedExpert(I=I, gate=w(I, H), up=w(I, H), down=w(H, I))
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(moe.moe_shared_expert_workspace_bytes(T, H, I), dtype=torch.uint8, device="cuda")
    moe.moe_shared_expert_forward(bf16_dev(x), bf16_dev(sh.gate), bf16_dev(sh.up), bf16_dev(sh.down), 7.0, ws=ws,
                                  out=out)
    torch.cuda.synchronize()
    gu = bf16_host(ws[:T * 2 * I * 2].view(torch.bfloat16).view(T, 2 * I))
    ref = O.shared_expert_mlp(x, sh, 7.0, "bf16")
    np.testing.assert_array_equal(gu[:, :I], ref["gate"])
    np.testing.assert_array_equal(gu[:, I:], ref["up"])
