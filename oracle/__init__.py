"""CPU oracle for the routed-MoE NVFP4 (W4A16) prefill path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 restatement of what the path computes, written from the
web pages' host-side contracts and prose (module docs and source of
``forward_prefill_gemm``; the two ``glm5next_mlp/forward.rs`` pages).  It shares
no code with the CUDA library and imports nothing from it.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline``
leg (and its ``--impl reference`` arm) may import or run anything here.  The
product path never calls it: there is no CPU fallback.

Parity status of each function (what pins it, see ``tests/test_oracle_pins.py``):

* ``e2m1_value``/``E2M1``: pinned (closed form vs the OCP MX codebook fixture,
  symmetry, max 6).
* ``e4m3_value``/``E4M3``: pinned (closed form vs PyTorch's float8_e4m3fn decode
  of all 256 codes; 0x38 = 1, 0x7E = 448).
* ``round_to_bf16``: pinned (PyTorch's bfloat16 cast on random and edge values).
* ``dequant_nvfp4``: pinned (hand-built bytes for the low-nibble-first order and
  the 16-wide scale block; scale2 multiply order).
* ``router_logits``: pinned (exact small-integer case; library matmul).
* ``route_topk``: pinned (brute-force full sort on tiny inputs; k = E is a full
  softmax permutation; weights sum to routed_scale).
* ``sort_by_expert``: pinned (permutation and offset invariants; brute-force
  Python counting sort).
* ``grouped_gemm``: pinned (exact dyadic special case; brute-force dense
  dequant-then-matmul per (token, slot) with no sort).
* ``swiglu_clamp``: pinned (special values g >= L, g = 0, u clamps).
* ``combine_indexed``: pinned (k = 1 with weight 1 reproduces the rows).
* ``prefill_forward``: pinned (E = 1, k = 1 reduces to a dense SwiGLU MLP).
* The pages' own numeric results for their random data: parity unpinned (their
  data and seeds are not given); the measured error table only fixes a scale.
"""

from .moe_oracle import *  # noqa: F401,F403
