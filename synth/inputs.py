"""Seeded synthetic inputs for the routed-MoE NVFP4 (W4A16) prefill workloads.

Every array here is raw storage, the way the GPU path and the oracle both
receive it:

* activations and router weights: BF16 bit patterns (``np.uint16``);
* NVFP4 weights: packed E2M1 nibbles ``uint8 [N, K/2]`` (two codes per byte,
  the even ``k`` in the low nibble), E4M3 block scales ``uint8 [N, K/16]``,
  and one FP32 ``scale2`` per expert and projection (module docs of
  ``forward_prefill_gemm``, table "Layout compatibility");
* router logits: FP32; expert ids: int32.

Float -> BF16 and float -> E4M3 encodings of the random draws are done by
PyTorch's own dtype conversions (round to nearest even); this module contains
no dequantisation, routing, sort, GEMM, activation or combine arithmetic.

Randomness: numpy ``PCG64`` streams keyed by ``(seed, stream id, index)`` so
that one expert's weights can be regenerated alone (the oracle's sampled
parity checks at full size need that).  The seed of workload ``cN`` is
``1000 + N``.
"""

from __future__ import annotations

import dataclasses
from typing import Callable, Dict, List, Optional, Tuple

import numpy as np
import torch

__all__ = [
    "WORKLOADS",
    "SWEEP_ROWS",
    "GemmCase",
    "BlockCase",
    "ExpertWeights",
    "SharedExpert",
    "shared_expert_weights",
    "make_gemm_case",
    "make_block_case",
    "expert_weights",
    "scale2_vector",
    "bf16_bits_from_f32",
    "e4m3_bits_from_f32",
    "workload",
]

# stream ids of the seeded generators
_S_X = 1
_S_ROUTER_W = 2
_S_LOGITS = 3
_S_BIAS = 4
_S_IDS = 5
_S_SCALE2 = 6
_S_ZIPF = 7
_S_SHARED = 8  # + projection index 0 gate, 1 up, 2 down
_S_W = 100  # + projection id
PROJ_GEMM = 0
PROJ_GATE_UP = 1
PROJ_DOWN = 2

SWEEP_ROWS = (8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096, 16384)

# The five workloads (rows T, hidden H, moe_intermediate I, experts E, top_k k).
WORKLOADS: Dict[str, dict] = {
    # single grouped W4A16 GEMM: 64 tokens, 16 experts, 8 distinct experts per token
    "c0": dict(kind="gemm", T=64, E=16, k=8, N=256, K=512, seed=1000),
    # full routed-MoE block on one 256-row prefill chunk, with the router GEMM
    "c1": dict(kind="block", T=256, H=2048, I=768, E=64, k=8, routing="router", seed=1001),
    # the same chunk with the shared expert (dense BF16 SwiGLU MLP, intermediate 768) in the combine
    "c1s": dict(kind="block", T=256, H=2048, I=768, E=64, k=8, routing="router", seed=1001, shared_inter=768),
    # GLM-scale chunk, synthetic logits N(0,1) plus a per-expert bias N(0, 0.1^2)
    "c2": dict(kind="block", T=2048, H=5120, I=1536, E=160, k=8, routing="biased", seed=1002),
    # skewed routing: Zipf(1.2) popularity, 16 experts never chosen
    "c3": dict(kind="block", T=8192, H=5120, I=1536, E=160, k=8, routing="zipf", seed=1003),
    # row-count sweep at the GLM shapes (T is given per point), balanced routing
    "c4": dict(kind="block", T=None, H=5120, I=1536, E=160, k=8, routing="biased", seed=1004),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of float32 draws (PyTorch's round-to-nearest-even cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def e4m3_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """E4M3 (OCP "FN") bit patterns of float32 draws (PyTorch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


@dataclasses.dataclass
class ExpertWeights:
    """NVFP4 weights of one projection for all experts (GLOBAL expert index)."""

    N: int
    K: int
    packed: List[Optional[np.ndarray]]  # per expert uint8 [N, K/2] or None (absent expert)
    scales: List[Optional[np.ndarray]]  # per expert uint8 [N, K/16] or None
    scale2: np.ndarray  # float32 [E]

    @property
    def E(self) -> int:
        return len(self.packed)

    def nbytes(self) -> int:
        return sum(p.nbytes + s.nbytes for p, s in zip(self.packed, self.scales) if p is not None)


def expert_weights(seed: int, proj: int, e: int, N: int, K: int) -> Tuple[np.ndarray, np.ndarray]:
    """One expert's packed nibbles (uniform over the 16 codes) and E4M3 scales U[0.25, 2]."""
    if K % 32 != 0:
        raise ValueError("K must be a multiple of 32")
    g = _rng(seed, _S_W + proj, e)
    packed = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = e4m3_bits_from_f32(g.uniform(0.25, 2.0, size=(N, K // 16)).astype(np.float32))
    return packed, scales


def scale2_vector(seed: int, proj: int, E: int) -> np.ndarray:
    """Per-expert FP32 scale2, uniform in [0.5/448, 2/448]."""
    return _rng(seed, _S_SCALE2, proj).uniform(0.5 / 448.0, 2.0 / 448.0, size=E).astype(np.float32)


def make_projection(seed: int, proj: int, E: int, N: int, K: int,
                    experts: Optional[List[int]] = None,
                    absent: Tuple[int, ...] = ()) -> ExpertWeights:
    """All experts of one projection; ``experts`` limits which ones are materialised
    (the others are left ``None`` and must not be touched); ``absent`` ones are None too."""
    packed: List[Optional[np.ndarray]] = [None] * E
    scales: List[Optional[np.ndarray]] = [None] * E
    want = range(E) if experts is None else experts
    for e in want:
        if e in absent:
            continue
        packed[e], scales[e] = expert_weights(seed, proj, e, N, K)
    return ExpertWeights(N=N, K=K, packed=packed, scales=scales, scale2=scale2_vector(seed, proj, E))


# ----------------------------------------------------------------------------------------------
# single grouped GEMM case (workload c0 and small variants)


@dataclasses.dataclass
class GemmCase:
    T: int
    E: int
    k: int
    N: int
    K: int
    x: np.ndarray  # uint16 bf16 bits [T, K]
    ids: np.ndarray  # int32 [T, k]
    w: ExpertWeights


def distinct_ids(g: np.random.Generator, T: int, E: int, k: int) -> np.ndarray:
    """k distinct experts per token, uniform (prefix of a random permutation)."""
    return np.argsort(g.random((T, E)), axis=1)[:, :k].astype(np.int32)


def make_gemm_case(T: int = 64, E: int = 16, k: int = 8, N: int = 256, K: int = 512,
                   seed: int = 1000, absent: Tuple[int, ...] = (),
                   x_sampler: Optional[Callable[[np.random.Generator, tuple], np.ndarray]] = None,
                   ) -> GemmCase:
    gx = _rng(seed, _S_X, T)
    xf = gx.standard_normal((T, K), dtype=np.float32) if x_sampler is None else x_sampler(gx, (T, K))
    ids = distinct_ids(_rng(seed, _S_IDS, T), T, E, k)
    w = make_projection(seed, PROJ_GEMM, E, N, K, absent=absent)
    return GemmCase(T=T, E=E, k=k, N=N, K=K, x=bf16_bits_from_f32(xf), ids=ids, w=w)


# ----------------------------------------------------------------------------------------------
# full routed-MoE block (workloads c1-c4)


@dataclasses.dataclass
class SharedExpert:
    """Dense BF16 SwiGLU MLP weights of the shared expert: gate and up [I, H], down [H, I]."""

    I: int
    gate: np.ndarray  # uint16 bf16 bits [I, H]
    up: np.ndarray  # uint16 bf16 bits [I, H]
    down: np.ndarray  # uint16 bf16 bits [H, I]


def shared_expert_weights(seed: int, H: int, I: int) -> SharedExpert:
    """BF16 N(0, 1/H) gate and up rows, so that with x ~ N(0, 1) the gate/up products are
    ~N(0, 1) and the SwiGLU clamps act, and N(0, (0.025)^2/I) down rows, which puts the
    shared output at the scale of the routed sum of the synthetic NVFP4 experts (std ~0.01)."""
    def w(j, rows, cols, sd):
        return bf16_bits_from_f32(_rng(seed, _S_SHARED, j).normal(0.0, sd, size=(rows, cols)).astype(np.float32))
    return SharedExpert(I=I, gate=w(0, I, H, H ** -0.5), up=w(1, I, H, H ** -0.5),
                        down=w(2, H, I, 0.025 * I ** -0.5))


@dataclasses.dataclass
class BlockCase:
    T: int
    H: int
    I: int
    E: int
    k: int
    x: np.ndarray  # uint16 bf16 bits [T, H]
    router_w: Optional[np.ndarray]  # uint16 bf16 bits [E, H] (routing "router")
    logits: Optional[np.ndarray]  # float32 [T, E] (synthetic routings)
    gate_up: ExpertWeights  # N = 2I (rows 0..I-1 gate, I..2I-1 up), K = H
    down: ExpertWeights  # N = H, K = I
    swiglu_limit: float = 7.0
    routed_scale: float = 1.0
    renormalize: int = 1
    shared: Optional[SharedExpert] = None  # the shared expert, added in the combine


def zipf_logits(seed: int, T: int, E: int, s: float = 1.2, n_zero: int = 16) -> np.ndarray:
    """Skewed routing logits: popularity p_e ~ rank^-s over a seeded permutation, n_zero
    seeded experts with p = 0 (logit -1e30), plus Gumbel(0,1) noise per (token, expert) so
    that top-k of the logits samples k distinct experts without replacement by popularity."""
    g = _rng(seed, _S_ZIPF, E)
    perm = g.permutation(E)
    p = np.empty(E, dtype=np.float64)
    p[perm] = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    zero = g.choice(E, size=n_zero, replace=False)
    p[zero] = 0.0
    p /= p.sum()
    gt = _rng(seed, _S_LOGITS, T)
    gumbel = -np.log(-np.log(gt.uniform(np.finfo(np.float64).tiny, 1.0, size=(T, E))))
    with np.errstate(divide="ignore"):
        lp = np.where(p > 0, np.log(np.where(p > 0, p, 1.0)), -1e30)
    out = (lp[None, :] + gumbel).astype(np.float32)
    out[:, p == 0] = np.float32(-1e30)
    return out


def biased_logits(seed: int, T: int, E: int) -> np.ndarray:
    """Near-balanced routing logits N(0,1) plus a fixed per-expert bias N(0, 0.1^2)."""
    b = _rng(seed, _S_BIAS, E).normal(0.0, 0.1, size=E).astype(np.float32)
    z = _rng(seed, _S_LOGITS, T).standard_normal((T, E), dtype=np.float32)
    return z + b[None, :]


def make_block_case(T: int, H: int, I: int, E: int, k: int, routing: str, seed: int,
                    experts: Optional[List[int]] = None, absent: Tuple[int, ...] = (),
                    with_weights: bool = True, shared_inter: Optional[int] = None) -> BlockCase:
    x = bf16_bits_from_f32(_rng(seed, _S_X, T).standard_normal((T, H), dtype=np.float32))
    router_w = None
    logits = None
    if routing == "router":
        router_w = bf16_bits_from_f32(_rng(seed, _S_ROUTER_W, E).normal(0.0, 0.02, size=(E, H)).astype(np.float32))
    elif routing == "biased":
        logits = biased_logits(seed, T, E)
    elif routing == "zipf":
        logits = zipf_logits(seed, T, E)
    else:
        raise ValueError(f"unknown routing {routing!r}")
    if with_weights:
        gu = make_projection(seed, PROJ_GATE_UP, E, 2 * I, H, experts=experts, absent=absent)
        dn = make_projection(seed, PROJ_DOWN, E, H, I, experts=experts, absent=absent)
    else:
        gu = ExpertWeights(N=2 * I, K=H, packed=[None] * E, scales=[None] * E,
                           scale2=scale2_vector(seed, PROJ_GATE_UP, E))
        dn = ExpertWeights(N=H, K=I, packed=[None] * E, scales=[None] * E,
                           scale2=scale2_vector(seed, PROJ_DOWN, E))
    shared = shared_expert_weights(seed, H, shared_inter) if shared_inter else None
    return BlockCase(T=T, H=H, I=I, E=E, k=k, x=x, router_w=router_w, logits=logits,
                     gate_up=gu, down=dn, shared=shared)


def workload(name: str, T: Optional[int] = None, **kw):
    """Build a named workload (``c0`` .. ``c4``); ``T`` overrides the row count."""
    cfg = dict(WORKLOADS[name])
    kind = cfg.pop("kind")
    if kind == "gemm":
        if T is not None:
            cfg["T"] = T
        cfg.update(kw)
        return make_gemm_case(**cfg)
    if T is not None:
        cfg["T"] = T
    if cfg["T"] is None:
        raise ValueError(f"workload {name} needs an explicit row count")
    cfg.update(kw)
    return make_block_case(**cfg)
