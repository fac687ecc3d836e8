"""Expert parallelism over the ranks of a process group.

"Module forward_prefill_gemm", "Layout compatibility": an expert that lives on another GPU has a
NULL entry in the expert table and its rows add zero; the caller all-reduces ``out``
(metrale ``glm5next_mlp/forward.rs``, module doc and ``forward_moe``: the combine, shared
expert included, runs before that all-reduce, so the partial sums of every rank reduce together).

Each rank holds the weights of one contiguous block of experts and runs the whole forward on the
chunk: routing and the sort are replicated (every rank computes the same ids and the same
sorted order), the grouped GEMMs multiply only the local experts' rows (the others stay zero),
and the combine writes this rank's partial ``out``.  One all-reduce (sum) of ``out`` over the
group gives the layer's output.  The shared expert's output joins the combine on rank 0 only, so
it is counted once.  The forward runs with ``MOE_FWD_NO_MULTICAST``: no cluster-multicast loads
in a run that spans GPUs.

Every step of the per-rank compute is the library's forward; this module only partitions the
experts, builds the local expert tables and issues the collective.
"""

from __future__ import annotations

from typing import Callable, Optional, Sequence

import torch
import torch.distributed as dist

from ._lib import MOE_FWD_NO_MULTICAST, MoePrefillConfig, moe_prefill_forward
from .weights import DeviceProjection, upload_projection

__all__ = ["expert_block", "local_projection", "ep_prefill_forward"]


def expert_block(E: int, rank: int, world: int) -> range:
    """The experts rank `rank` of `world` holds: a contiguous block, the first E % world ranks
    one expert more."""
    if world < 1 or not 0 <= rank < world or E < 1:
        raise ValueError(f"bad partition: E={E}, rank={rank}, world={world}")
    base, extra = divmod(E, world)
    lo = rank * base + min(rank, extra)
    return range(lo, lo + base + (1 if rank < extra else 0))


def local_projection(packed: Sequence, scales: Sequence, scale2, N: int, K: int, rank: int, world: int,
                     device: str = "cuda") -> DeviceProjection:
    """One projection's expert table for this rank: the local experts' packed weights and scales
    uploaded, every other expert absent (NULL: its rows stay zero)."""
    E = len(packed)
    mine = expert_block(E, rank, world)
    p = [packed[e] if e in mine else None for e in range(E)]
    s = [scales[e] if e in mine else None for e in range(E)]
    return upload_projection(p, s, scale2, N, K, device=device)


def ep_prefill_forward(cfg: MoePrefillConfig, x: torch.Tensor, w_gate_up, w_down, ws: torch.Tensor, *,
                       group=None, w_router: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                       router_bias: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                       shared_out: Optional[torch.Tensor] = None, stream=None,
                       forward: Optional[Callable] = None) -> torch.Tensor:
    """The layer's output on every rank of `group`: this rank's forward over its local expert
    tables (`w_gate_up`, `w_down` from ``local_projection``), then one all-reduce (sum) of out.

    `shared_out` (the shared expert's output) is added on rank 0 only.  `forward` replaces the
    library's forward (same signature as ``moe_prefill_forward``), e.g. to run the host logic
    without a GPU; it defaults to ``moe_prefill_forward``."""
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    run = forward or moe_prefill_forward
    local_cfg = MoePrefillConfig(cfg.hidden, cfg.moe_intermediate, cfg.num_experts, cfg.top_k, cfg.swiglu_limit,
                                 cfg.renormalize, cfg.routed_scale, cfg.flags | MOE_FWD_NO_MULTICAST)
    out = run(local_cfg, x, w_gate_up, w_down, ws, w_router=w_router, logits=logits, router_bias=router_bias,
              out=out, stream=stream, shared_out=shared_out if rank == 0 else None)
    if dist.is_initialized() and dist.get_world_size(group) > 1:
        if stream is not None:
            torch.cuda.current_stream().wait_stream(stream)
        dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    return out
