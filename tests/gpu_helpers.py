"""Helpers of the GPU parity tests: move synthetic cases to the device, compare with the oracle."""

from __future__ import annotations

import numpy as np
import torch

import moe_prefill_nvfp4_gb300 as moe
from moe_prefill_nvfp4_gb300.weights import upload_projection

# float outputs vs the oracle, max|gpu - ref| / max|ref|
TOL_BF16 = 4e-3  # against the variant that rounds weights and inter-stage activations to BF16
TOL_EXACT = 1e-2  # against the exact FP32-weight variant


def nerr(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    return float(np.abs(gpu - ref).max() / (den if den > 0 else 1.0))


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_host(t: torch.Tensor) -> np.ndarray:
    """BF16 device tensor -> float64 numpy."""
    return t.float().cpu().numpy().astype(np.float64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def upload(proj):
    return upload_projection(proj.packed, proj.scales, proj.scale2, proj.N, proj.K)


def make_cfg(case, flags: int = 0) -> moe.MoePrefillConfig:
    return moe.MoePrefillConfig(hidden=case.H, moe_intermediate=case.I, num_experts=case.E, top_k=case.k,
                                swiglu_limit=case.swiglu_limit, renormalize=case.renormalize,
                                routed_scale=case.routed_scale, flags=flags)


class DeviceBlock:
    """A routed-MoE block case on the device, with one workspace.  `separate` runs the SwiGLU
    as its own kernel on a materialised G (else it is fused into the gate/up GEMM)."""

    def __init__(self, case, separate: bool = False):
        self.case = case
        self.separate = separate
        self.x = bf16_dev(case.x)
        self.router_w = bf16_dev(case.router_w) if case.router_w is not None else None
        self.logits = torch.from_numpy(case.logits).cuda() if case.logits is not None else None
        self.gu = upload(case.gate_up)
        self.dn = upload(case.down)
        self.cfg = make_cfg(case, moe.MOE_FWD_SEPARATE_SWIGLU if separate else 0)
        self.layout = moe.moe_workspace_layout(self.cfg, case.T)
        self.ws = torch.empty(self.layout.total, dtype=torch.uint8, device="cuda")
        self.out = torch.empty(case.T, case.H, dtype=torch.bfloat16, device="cuda")
        self.shared = None
        if case.shared is not None:
            sh = case.shared
            self.shared = dict(gate=bf16_dev(sh.gate), up=bf16_dev(sh.up), down=bf16_dev(sh.down),
                               out=torch.empty(case.T, case.H, dtype=torch.bfloat16, device="cuda"),
                               ws=torch.empty(moe.moe_shared_expert_workspace_bytes(case.T, case.H, sh.I),
                                              dtype=torch.uint8, device="cuda"))

    def shared_forward(self, stream=None):
        sh = self.shared
        return moe.moe_shared_expert_forward(self.x, sh["gate"], sh["up"], sh["down"], self.case.swiglu_limit,
                                             ws=sh["ws"], out=sh["out"], stream=stream)

    def forward(self, stream=None, shared_ready=None):
        """The routed forward; with a shared expert, its output (computed by shared_forward,
        here on the same stream unless `shared_ready` says it comes from another) joins the
        combine."""
        shared_out = None
        if self.shared is not None:
            if shared_ready is None:
                self.shared_forward(stream)
            shared_out = self.shared["out"]
        return moe.moe_prefill_forward(self.cfg, self.x, self.gu.table, self.dn.table, self.ws, w_router=self.router_w,
                                       logits=self.logits, out=self.out, stream=stream, shared_out=shared_out,
                                       shared_ready=shared_ready)

    def ws_view(self, name: str, dtype: torch.dtype, shape) -> torch.Tensor:
        off = getattr(self.layout, name)
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        return self.ws[off:off + n].view(dtype).view(*shape)

    def stages(self):
        c = self.case
        R = c.T * c.k
        return dict(
            logits=self.ws_view("logits", torch.float32, (c.T, c.E)).cpu().numpy(),
            ids=self.ws_view("ids", torch.int32, (c.T, c.k)).cpu().numpy(),
            wts=self.ws_view("wts", torch.float32, (c.T, c.k)).cpu().numpy(),
            sorted_token_ids=self.ws_view("sorted_token_ids", torch.int32, (R,)).cpu().numpy(),
            sorted_expert_ids=self.ws_view("sorted_expert_ids", torch.int32, (R,)).cpu().numpy(),
            expert_offsets=self.ws_view("expert_offsets", torch.int32, (c.E + 1,)).cpu().numpy(),
            token_to_perm=self.ws_view("token_to_perm", torch.int32, (c.T, c.k)).cpu().numpy(),
            G=bf16_host(self.ws_view("G", torch.bfloat16, (R, 2 * c.I))) if self.separate else None,
            act=bf16_host(self.ws_view("act", torch.bfloat16, (R, c.I))),
            Y=bf16_host(self.ws_view("Y", torch.bfloat16, (R, c.H))),
            out=bf16_host(self.out),
            shared=bf16_host(self.shared["out"]) if self.shared is not None else None,
        )

    def close(self):
        self.gu.close()
        self.dn.close()


def bf16_stage(v64: np.ndarray) -> np.ndarray:
    """The BF16 stage rounding of the oracle's BF16 variant (fp32, then BF16 nearest even)."""
    from oracle import moe_oracle as O

    return O._to_stage(np.asarray(v64, dtype=np.float64), "bf16")


def bf16_bracket(v64: np.ndarray):
    """The two BF16 values around v64: its BF16 stage rounding r, and r's neighbour on v64's other
    side (r itself where v64 is r).  An FP32 sum of v64's terms in any order lies far closer to
    v64 than one BF16 unit, so its BF16 rounding is one of the two."""
    v = np.asarray(v64, dtype=np.float64)
    r = bf16_stage(v)
    b = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.int64)
    away = ((v > r) & (r > 0)) | ((v < r) & (r < 0))  # step away from zero, else toward it
    nb = np.where(away, b + 1, b - 1)
    other = (nb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    other = np.where((v == r) | (r == 0), r, other)
    return r, other


def fused_act_candidates(G64: np.ndarray, I: int, limit: float):
    """References of the fused SwiGLU epilogue, which rounds its FP32 accumulators g and u to BF16
    before the SwiGLU: the SwiGLU over the two BF16 values around g and the two around u (the
    oracle's rounding, and the other one an FP32 summation order may reach).  Returns [4, R, I]."""
    from oracle import moe_oracle as O

    gs = bf16_bracket(G64[:, :I])
    us = bf16_bracket(G64[:, I:])
    return np.stack([O.swiglu_clamp(a, b, limit) for a in gs for b in us])


def fused_act_error(got: np.ndarray, G64: np.ndarray, I: int, limit: float):
    """(normalised error, per-element ok) of a fused SwiGLU output against the closest of its
    references; per element within 2^-8 of it relative (act's BF16 rounding, the FP32 SwiGLU's
    own few ulp included) plus 1e-5 of the tensor's max."""
    cands = fused_act_candidates(G64, I, limit)
    d = np.abs(cands - got[None])
    best = np.take_along_axis(cands, d.argmin(axis=0)[None], axis=0)[0]
    bad = np.abs(got - best) > np.abs(best) * 2.0 ** -8 + 1e-5 * np.abs(best).max()
    if bad.any():
        idx = np.argwhere(bad)[:4]
        for r, j in idx:
            print("fused act element", int(r), int(j), "gpu", got[r, j], "best", best[r, j], "g", G64[r, j],
                  "u", G64[r, I + j], "candidates", cands[:, r, j])
    return nerr(got, best), bool(not bad.any())
