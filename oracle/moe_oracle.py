"""Plain fp64 CPU oracle of the routed-MoE NVFP4 (W4A16) prefill path.

TEST INFRASTRUCTURE ONLY -- see the package docstring for who may call it.

Sources (web pages, cited by title and section):

* [fpg-docs] "Module forward_prefill_gemm" (spark_model::layers::glm5next_mlp),
  sections "What this replaces", "Layout compatibility -- VERIFIED, not assumed"
  (the term-by-term table), "What is NOT bit-identical" (items 1-2 and the
  measured error table) and "Buffer discipline".  The source page of the same
  module ("forward_prefill_gemm.rs") repeats this doc comment.
* [fwd-old] "spark_model/layers/glm5next_mlp/forward.rs": ``swiglu`` doc,
  the router/top-k launch in ``forward_moe``, the "-1 is the kernel's slot
  unfilled sentinel" note.
* [fwd-new] "metrale_model_arch/glm5next_mlp/forward.rs": ``swiglu_rows``,
  the ``Glm5NextMlpWorkspace`` field docs (``sorted_token_ids``,
  ``sorted_expert_ids``, ``expert_offsets``, ``token_to_perm``,
  ``expert_out``), and ``forward_moe`` (router, one top-k launch, zeroed
  routed outputs, grouped prefill arm, ``combine_indexed``).

Precision: every contraction accumulates in fp64.  Stage outputs are rounded to
fp32 at each stage boundary; the ``"bf16"`` variant additionally rounds the
dequantised weights and the inter-stage activations G, act and Y to BF16
(round to nearest even), which is what the grouped kernel stages ([fpg-docs],
"What is NOT bit-identical", item 2).  The ``"exact"`` variant keeps them fp32.
Each stage also returns its unrounded fp64 value, which is what a GPU result is
compared against.
"""

from __future__ import annotations

import math
from typing import Callable, Dict, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "E2M1",
    "E4M3",
    "GROUP_SIZE",
    "e2m1_value",
    "e4m3_value",
    "bf16_bits_to_f64",
    "round_to_bf16",
    "dequant_nvfp4",
    "router_logits",
    "route_topk",
    "sort_by_expert",
    "grouped_gemm",
    "swiglu_clamp",
    "combine_indexed",
    "shared_expert_mlp",
    "prefill_forward",
    "token_forward",
    "VARIANTS",
]

VARIANTS = ("bf16", "exact")

# [fpg-docs] "Layout compatibility": block scale index k/16, GROUP_SIZE 16 (not 32).
GROUP_SIZE = 16


# ----------------------------------------------------------------------------------------------
# number formats


def e2m1_value(c: int) -> float:
    """Value of a 4-bit E2M1 code: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.

    The pages name the codebook (``E2M1_LUT`` / ``E2M1_LUT_MOE``, "same 16 values",
    [fpg-docs] "Layout compatibility", row "codebook") but do not print it; this is
    the standard E2M1 element format.  Exponent field 0 is subnormal: 0.5 * m.
    """
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = 0.5 * m if e == 0 else (2.0 ** (e - 1)) * (1.0 + 0.5 * m)
    return -mag if s else mag


def e4m3_value(b: int) -> float:
    """Value of an E4M3 byte (OCP "FN" flavour: bias 7, no infinities, 0x7F/0xFF NaN).

    The block scale is "E4M3" ([fpg-docs] "Layout compatibility", row "block scale");
    the flavour is not stated, FN (max 448) is the one that fits scale2 ~ 1/448.
    """
    s = (b >> 7) & 1
    e = (b >> 3) & 0xF
    m = b & 7
    if e == 0xF and m == 7:
        return math.nan
    mag = (2.0 ** -6) * (m / 8.0) if e == 0 else (2.0 ** (e - 7)) * (1.0 + m / 8.0)
    return -mag if s else mag


E2M1 = np.array([e2m1_value(c) for c in range(16)], dtype=np.float32)
E4M3 = np.array([e4m3_value(b) for b in range(256)], dtype=np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float64 (a BF16 value is the top half of an fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest BF16 value, ties to even; returns float32.

    Written from the definition: keep the top 16 bits of the fp32 pattern, adding half
    a BF16 unit (0x7FFF plus the kept lsb) first.  NaNs stay NaN.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    lsb = (u >> 16) & 1
    r = ((u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)).astype(np.uint32)
    out = r.view(np.float32)
    return np.where(np.isnan(f), f, out)


def _to_stage(x64: np.ndarray, variant: str) -> np.ndarray:
    """Stage boundary: round an fp64 stage output to fp32, then to BF16 for ``"bf16"``."""
    f = x64.astype(np.float32)
    if variant == "bf16":
        f = round_to_bf16(f)
    return f.astype(np.float64)


# ----------------------------------------------------------------------------------------------
# dequantisation


def dequant_nvfp4(packed: np.ndarray, scales: np.ndarray, scale2: float, variant: str = "bf16") -> np.ndarray:
    """Dequantise one expert's NVFP4 weight to a dense float matrix [N, K] (float32 values).

    [fpg-docs] "Layout compatibility":
      * the byte holding logical k of row n is ``packed[n * (K/2) + k/2]`` (N-major [N, K/2]);
      * even k is ``byte & 0xF``, odd k is ``byte >> 4``;
      * the E4M3 block scale of (n, k) is ``scales[n * (K/16) + k/16]``;
      * the per-expert FP32 ``scale2`` multiplies the dequantised value.
    [fpg-docs] "What is NOT bit-identical", item 2: the grouped kernel's value is
    ``E2M1_LUT[nibble] * e4m3 * scale2`` evaluated left to right in FP32 and rounded to
    BF16.  ``lut * e4m3`` is exact in FP32, so only the ``* scale2`` rounds.  The
    ``"exact"`` variant stops at FP32; ``"bf16"`` rounds to BF16.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    N, half_k = packed.shape
    K = 2 * half_k
    if scales.shape != (N, K // GROUP_SIZE):
        raise ValueError(f"scales shape {scales.shape} != {(N, K // GROUP_SIZE)}")
    codes = np.empty((N, K), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF  # even k: low nibble
    codes[:, 1::2] = packed >> 4  # odd k: high nibble
    lut = E2M1[codes]
    blk = np.repeat(E4M3[scales], GROUP_SIZE, axis=1)
    w = (lut * blk).astype(np.float32) * np.float32(scale2)
    if variant == "bf16":
        w = round_to_bf16(w)
    elif variant != "exact":
        raise ValueError(variant)
    return w.astype(np.float32)


# ----------------------------------------------------------------------------------------------
# routing


def router_logits(x_bits: np.ndarray, wr_bits: np.ndarray) -> np.ndarray:
    """FP32 router logits ``x[T, H] @ Wr[E, H]^T`` (BF16 inputs, fp64 sum, rounded to fp32).

    [fwd-new] ``forward_moe``: the router writes ``[rows, num_experts]`` F32 logits from
    BF16 ``x`` and the router weight.
    """
    x = bf16_bits_to_f64(x_bits)
    w = bf16_bits_to_f64(wr_bits)
    return (x @ w.T).astype(np.float32)


def route_topk(logits: np.ndarray, k: int, bias: Optional[np.ndarray] = None, renormalize: int = 1,
               routed_scale: float = 1.0) -> Tuple[np.ndarray, np.ndarray]:
    """Top-k routing of FP32 logits [T, E] -> ids int32 [T, k], weights float64 [T, k].

    [fwd-new]/[fwd-old] ``forward_moe``: one top-k launch for all rows over FP32 logits
    with ``router_bias``, ``routed_scale`` and ``renormalize``; ``n_group`` must be 1.
    Readings where the pages are silent:
      * the selection key is ``logit + bias`` computed in FP32 (bias selects, it does not
        weight); ties go to the lower expert id; slots are ordered by descending key;
      * the weight of a selected expert is its softmax over all E logits, renormalised over
        the k selected (= a softmax over the k selected logits) when ``renormalize``,
        then times ``routed_scale``; without ``renormalize`` it is the full-E softmax.
    NaN logits are rejected.
    """
    lg = np.asarray(logits, dtype=np.float32)
    T, E = lg.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    if np.isnan(lg).any():
        raise ValueError("NaN logit")
    key = lg if bias is None else (lg + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    # stable sort of -key: equal keys keep ascending expert id
    order = np.argsort(-key.astype(np.float64), axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(lg, ids, axis=1).astype(np.float64)
    if renormalize:
        m = sel.max(axis=1, keepdims=True)
        ex = np.exp(sel - m)
        wts = ex / ex.sum(axis=1, keepdims=True)
    else:
        l64 = lg.astype(np.float64)
        m = l64.max(axis=1, keepdims=True)
        wts = np.exp(sel - m) / np.exp(l64 - m).sum(axis=1, keepdims=True)
    return ids, wts * routed_scale


# ----------------------------------------------------------------------------------------------
# expert sort


def sort_by_expert(ids: np.ndarray, E: int) -> Dict[str, np.ndarray]:
    """Stable counting sort of the R = T*k routed slots by expert id.

    [fwd-new] ``Glm5NextMlpWorkspace``: ``sorted_token_ids [rows*top_k]`` maps a sorted
    row to its ORIGINAL TOKEN; ``sorted_expert_ids`` maps it to its expert;
    ``expert_offsets [E+1]`` is the prefix sum over the expert-sorted rows;
    ``token_to_perm [rows, top_k]`` is a slot's row in the sorted output.
    Readings: rows of one expert keep flat slot order i = t*k + s (stable); a slot whose
    id is -1 (the "slot unfilled" sentinel, [fwd-old]) goes to a tail after
    ``expert_offsets[E]`` with expert id -1 and ``token_to_perm = -1``.
    """
    ids = np.asarray(ids, dtype=np.int32)
    T, k = ids.shape
    flat = ids.reshape(-1)
    R = flat.size
    if ((flat < -1) | (flat >= E)).any():
        raise ValueError("expert id out of range")
    valid = flat >= 0
    key = np.where(valid, flat, E)
    perm = np.argsort(key, kind="stable")  # sorted position p -> flat slot index
    counts = np.bincount(flat[valid], minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    sorted_token_ids = (perm // k).astype(np.int32)
    sorted_expert_ids = np.where(valid[perm], flat[perm], -1).astype(np.int32)
    token_to_perm = np.empty(R, dtype=np.int32)
    token_to_perm[perm] = np.arange(R, dtype=np.int32)
    token_to_perm[~valid] = -1
    return dict(sorted_token_ids=sorted_token_ids, sorted_expert_ids=sorted_expert_ids,
                expert_offsets=offsets, token_to_perm=token_to_perm.reshape(T, k))


# ----------------------------------------------------------------------------------------------
# grouped GEMM, activation, combine


WeightFn = Callable[[int], Optional[np.ndarray]]


def grouped_gemm(a: np.ndarray, expert_offsets: np.ndarray, weight: WeightFn,
                 gather: Optional[np.ndarray] = None) -> np.ndarray:
    """Grouped GEMM over all experts in expert-sorted order, fp64, unrounded.

    ``C[p, :] = a[gather[p], :] @ W_e^T`` for every sorted row p in
    ``[expert_offsets[e], expert_offsets[e+1])``; ``gather`` is ``sorted_token_ids`` for
    gate/up (the in-kernel A gather, [fpg-docs] "What this replaces") and the identity
    for down.  ``weight(e)`` returns expert e's dense dequantised [N, K] matrix, or None
    for an absent (remote) expert, whose rows stay zero ([fpg-docs] "Layout
    compatibility", row "remote expert": the caller's zeros stand).
    """
    a = np.asarray(a, dtype=np.float64)
    E = len(expert_offsets) - 1
    R = int(expert_offsets[E])
    out = None
    for e in range(E):
        lo, hi = int(expert_offsets[e]), int(expert_offsets[e + 1])
        w = weight(e)
        if out is None and w is not None:
            out = np.zeros((R, w.shape[0]), dtype=np.float64)
        if hi == lo or w is None:
            continue
        rows = np.arange(lo, hi) if gather is None else np.asarray(gather[lo:hi])
        out[lo:hi] = a[rows] @ w.astype(np.float64).T
    if out is None:
        raise ValueError("no present expert")
    return out


def swiglu_clamp(g: np.ndarray, u: np.ndarray, limit: float) -> np.ndarray:
    """Clamped SwiGLU ``silu(min(g, L)) * clamp(u, -L, L)``, silu(z) = z / (1 + exp(-z)).

    [fwd-old] ``swiglu`` and [fwd-new] ``swiglu_rows`` doc comments.  Only the gate has an
    upper clamp; a negative gate goes through silu unclamped.
    """
    g = np.minimum(np.asarray(g, dtype=np.float64), limit)
    u = np.clip(np.asarray(u, dtype=np.float64), -limit, limit)
    with np.errstate(over="ignore"):
        silu = g / (1.0 + np.exp(-g))
    return silu * u


def combine_indexed(y: np.ndarray, token_to_perm: np.ndarray, wts: np.ndarray,
                    shared_out: Optional[np.ndarray] = None) -> np.ndarray:
    """Routing-weighted combine back to token order, fp64, slot order.

    [fwd-new] ``forward_moe``: ``glm5next_moe_combine_indexed`` finds each slot's row of
    the expert-sorted outputs through ``token_to_perm``; the shared expert's output joins
    the sum.  A slot with ``token_to_perm = -1`` adds zero.
    """
    T, k = token_to_perm.shape
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for s in range(k):
        p = token_to_perm[:, s]
        ok = p >= 0
        out[ok] += np.asarray(wts, dtype=np.float64)[ok, s, None] * y[p[ok]]
    if shared_out is not None:
        out += shared_out
    return out


# ----------------------------------------------------------------------------------------------
# whole path


def shared_expert_mlp(x_bits: np.ndarray, shared, limit: float, variant: str = "bf16") -> Dict[str, np.ndarray]:
    """The shared expert over every row: a dense SwiGLU MLP with BF16 weights.

    [fwd-old] ``forward_dense``: ``a_gate = x @ W_gate^T`` and ``a_up = x @ W_up^T`` (two
    dense GEMMs into the BF16 workspace buffers ``a_gate``, ``a_up``), ``a_act =
    swiglu(a_gate, a_up)`` with the layer's ``swiglu_limit``, then ``shared_out = a_act @
    W_down^T``; [fwd-new] ``forward_moe`` adds ``shared_out`` in the combine.  Stage rounding
    as in ``prefill_forward``: fp32, then BF16 for the ``"bf16"`` variant (the pages' buffers
    are BF16).  Returns each stage unrounded (``gate64`` ...) and rounded (``gate`` ...).
    """
    if variant not in VARIANTS:
        raise ValueError(variant)
    x = bf16_bits_to_f64(x_bits)
    res: Dict[str, np.ndarray] = {}
    res["gate64"] = x @ bf16_bits_to_f64(shared.gate).T
    res["up64"] = x @ bf16_bits_to_f64(shared.up).T
    res["gate"], res["up"] = _to_stage(res["gate64"], variant), _to_stage(res["up64"], variant)
    res["act64"] = swiglu_clamp(res["gate"], res["up"], limit)
    res["act"] = _to_stage(res["act64"], variant)
    res["out64"] = res["act"] @ bf16_bits_to_f64(shared.down).T
    res["out"] = _to_stage(res["out64"], variant)
    return res


class _Dequant:
    """Caches one projection's dequantised experts (built on first use)."""

    def __init__(self, proj, variant: str):
        self.proj = proj
        self.variant = variant
        self.cache: Dict[int, Optional[np.ndarray]] = {}

    def __call__(self, e: int) -> Optional[np.ndarray]:
        if e not in self.cache:
            p = self.proj.packed[e]
            self.cache[e] = None if p is None else dequant_nvfp4(p, self.proj.scales[e], float(self.proj.scale2[e]),
                                                                 self.variant)
        return self.cache[e]


def prefill_forward(case, variant: str = "bf16", logits: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """The routed-MoE prefill path over one chunk of rows, every stage kept.

    Steps ([fwd-new] ``forward_moe``, grouped-prefill arm): router logits (when the case
    has a router weight) -> top-k -> expert sort -> grouped gate/up GEMM with the A
    gather through ``sorted_token_ids`` -> clamped SwiGLU -> grouped down GEMM ->
    ``combine_indexed``.  Gate/up weights are one [2I, H] matrix per expert: rows
    0..I-1 gate, rows I..2I-1 up (reading: concatenation).  When the case has a shared
    expert, its BF16 output (``shared_expert_mlp``) joins the combine.

    ``logits`` overrides the case's routing input (routing bit-exactness is checked on
    shared logits).  Returns a dict: ``logits``, ``ids``, ``wts``, the four sort arrays,
    and for G, act, Y, out both the unrounded fp64 value (``G64`` ...) and the
    stage-rounded value the next stage consumed (``G`` ...).
    """
    if variant not in VARIANTS:
        raise ValueError(variant)
    res: Dict[str, np.ndarray] = {}
    if logits is None:
        logits = router_logits(case.x, case.router_w) if case.router_w is not None else case.logits
    res["logits"] = np.asarray(logits, dtype=np.float32)
    ids, wts = route_topk(res["logits"], case.k, None, case.renormalize, case.routed_scale)
    res["ids"], res["wts"] = ids, wts
    srt = sort_by_expert(ids, case.E)
    res.update(srt)
    x = bf16_bits_to_f64(case.x)
    I = case.I
    g64 = grouped_gemm(x, srt["expert_offsets"], _Dequant(case.gate_up, variant), srt["sorted_token_ids"])
    res["G64"], res["G"] = g64, _to_stage(g64, variant)
    act64 = swiglu_clamp(res["G"][:, :I], res["G"][:, I:], case.swiglu_limit)
    res["act64"], res["act"] = act64, _to_stage(act64, variant)
    y64 = grouped_gemm(res["act"], srt["expert_offsets"], _Dequant(case.down, variant))
    res["Y64"], res["Y"] = y64, _to_stage(y64, variant)
    shared_out = None
    if getattr(case, "shared", None) is not None:
        sh = shared_expert_mlp(case.x, case.shared, case.swiglu_limit, variant)
        res["shared64"], res["shared"] = sh["out64"], sh["out"]
        shared_out = sh["out"]
    out64 = combine_indexed(res["Y"], srt["token_to_perm"], wts, shared_out)
    res["out64"] = out64
    return res


def token_forward(case, tokens: Sequence[int], ids: np.ndarray, wts: np.ndarray, variant: str = "bf16",
                  dq_cache: Optional[dict] = None) -> Dict[str, np.ndarray]:
    """The same path for a few tokens, one token at a time, with no sort.

    For each token t and slot s: ``G = x[t] @ W_gu[ids[t,s]]^T`` -> SwiGLU -> ``Y = act @
    W_d^T``; ``out[t] = sum_s wts[t,s] * Y``.  Used for sampled checks at full size, where
    running every row is too slow; per-row results do not depend on the other rows.
    """
    dq = dq_cache if dq_cache is not None else {}
    if "gu" not in dq:
        dq["gu"] = _Dequant(case.gate_up, variant)
        dq["dn"] = _Dequant(case.down, variant)
    x = bf16_bits_to_f64(case.x)
    I = case.I
    shared = None
    if getattr(case, "shared", None) is not None:
        shared = shared_expert_mlp(case.x[list(tokens)], case.shared, case.swiglu_limit, variant)["out"]
    outs, gs, ys = [], [], []
    for ti, t in enumerate(tokens):
        acc = np.zeros(case.H, dtype=np.float64) if shared is None else shared[ti].copy()
        g_rows, y_rows = [], []
        for s in range(case.k):
            e = int(ids[t, s])
            wgu = dq["gu"](e)
            wdn = dq["dn"](e)
            if wgu is None or wdn is None:
                g_rows.append(np.zeros(2 * I))
                y_rows.append(np.zeros(case.H))
                continue
            g64 = x[t] @ wgu.astype(np.float64).T
            g = _to_stage(g64, variant)
            act = _to_stage(swiglu_clamp(g[:I], g[I:], case.swiglu_limit), variant)
            y64 = act @ wdn.astype(np.float64).T
            y = _to_stage(y64, variant)
            acc += float(wts[t, s]) * y
            g_rows.append(g64)
            y_rows.append(y64)
        outs.append(acc)
        gs.append(np.stack(g_rows))
        ys.append(np.stack(y_rows))
    return dict(out64=np.stack(outs), G64=np.stack(gs), Y64=np.stack(ys))
