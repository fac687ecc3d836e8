"""The oracle's per-expert stages run in worker processes, for full-size parity tests.

Test infrastructure.  Every number here comes from ``oracle.moe_oracle`` functions, called the
way ``prefill_forward`` calls them, one expert (or one block of an expert's rows) per task:
``dequant_nvfp4`` -> ``grouped_gemm`` over that expert's rows -> stage rounding -> ``swiglu_clamp``
-> stage rounding -> ``grouped_gemm`` (down) -> stage rounding.  Rows are independent in every
one of these steps, so splitting them over processes changes nothing in the arithmetic; the
pinning test ``test_oracle_pins.py::test_pooled_expert_chain_equals_prefill_forward`` checks the
pooled chain against ``prefill_forward`` (equal up to the fp64 summation order of the BLAS
matmul, whose blocking depends on the row count, and bit for bit after each stage rounding).

The pool uses the ``spawn`` start method (never fork a process that has touched the GPU), and
each worker keeps BLAS to one thread.
"""

from __future__ import annotations

import multiprocessing as mp
import os
from typing import Dict, List, Optional, Sequence

import numpy as np


def _init_worker():
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    try:
        from threadpoolctl import threadpool_limits

        threadpool_limits(1)
    except Exception:
        pass


def _to_stage(x64: np.ndarray, variant: str) -> np.ndarray:
    from oracle import moe_oracle as O

    return O._to_stage(x64, variant)


def expert_rows_chain(task: dict) -> dict:
    """One expert's rows through gate/up, SwiGLU and down with the oracle's functions.

    task: gu (packed, scales, scale2), dn (packed, scales, scale2), x_rows (BF16 bits [m, H], the
    gathered tokens), I, limit, variant, and optionally act_in (float64 [m, I]: an external act for
    a stage-wise down product).  Returns G64, act64, Y64 (the chain) and Y64_in (down on act_in).
    """
    from oracle import moe_oracle as O

    variant = task["variant"]
    I = task["I"]
    x = O.bf16_bits_to_f64(task["x_rows"])
    m = x.shape[0]
    off = np.array([0, m], dtype=np.int64)
    res = {}
    if task.get("gu") is not None:
        wgu = O.dequant_nvfp4(*task["gu"], variant)
        g64 = O.grouped_gemm(x, off, lambda _e: wgu)
        del wgu
        g = _to_stage(g64, variant)
        act64 = O.swiglu_clamp(g[:, :I], g[:, I:], task["limit"])
        act = _to_stage(act64, variant)
        res.update(G64=g64 if task.get("keep_g", True) else None, act64=act64)
    else:
        act = None
    if task.get("dn") is not None:
        wdn = O.dequant_nvfp4(*task["dn"], variant)
        if act is not None:
            res["Y64"] = O.grouped_gemm(act, off, lambda _e: wdn)
        if task.get("act_in") is not None:
            res["Y64_in"] = O.grouped_gemm(task["act_in"], off, lambda _e: wdn)
    return res


class OraclePool:
    """A spawn process pool running ``expert_rows_chain`` tasks."""

    def __init__(self, workers: Optional[int] = None):
        n = workers or max(1, min(32, (os.cpu_count() or 2)))
        self.pool = mp.get_context("spawn").Pool(n, initializer=_init_worker)

    def map(self, tasks: List[dict]) -> List[dict]:
        return self.pool.map(expert_rows_chain, tasks, chunksize=1)

    def close(self):
        self.pool.close()
        self.pool.join()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False


def run_rows(pool: OraclePool, case, srt: Dict[str, np.ndarray], variant: str, rows: Sequence[int],
             act_in: Optional[np.ndarray] = None, keep_g: bool = False,
             rows_per_task: int = 512) -> Dict[str, np.ndarray]:
    """The oracle's chain for the given sorted rows (any order), grouped by expert into tasks of at
    most rows_per_task rows.  Returns arrays aligned with `rows`: act64, Y64, G64 (with keep_g)
    and, with act_in (float64 [len(rows), I], aligned with rows), Y64_in = down(act_in).  Rows of
    absent experts stay NaN."""
    rows = np.asarray(rows, dtype=np.int64)
    sti = srt["sorted_token_ids"]
    off = srt["expert_offsets"]
    expert_of = np.searchsorted(off, rows, side="right") - 1
    tasks, where = [], []
    for e in np.unique(expert_of):
        e = int(e)
        if case.gate_up.packed[e] is None or case.down.packed[e] is None:
            continue
        pos = np.nonzero(expert_of == e)[0]
        for b in range(0, pos.size, rows_per_task):
            p = pos[b:b + rows_per_task]
            r = rows[p]
            tasks.append(dict(
                variant=variant, I=case.I, limit=case.swiglu_limit, keep_g=keep_g, x_rows=case.x[sti[r]],
                gu=(case.gate_up.packed[e], case.gate_up.scales[e], float(case.gate_up.scale2[e])),
                dn=(case.down.packed[e], case.down.scales[e], float(case.down.scale2[e])),
                act_in=None if act_in is None else act_in[p]))
            where.append(p)
    outs = pool.map(tasks)
    widths = dict(G64=2 * case.I, act64=case.I, Y64=case.H, Y64_in=case.H)
    res: Dict[str, np.ndarray] = {}
    for p, o in zip(where, outs):
        for k, v in o.items():
            if v is None:
                continue
            if k not in res:
                res[k] = np.full((rows.size, widths[k]), np.nan)
            res[k][p] = v
    return res


def run_block(pool: OraclePool, case, srt: Dict[str, np.ndarray], variant: str, act_in=None, keep_g=True,
              rows_per_task: int = 512) -> Dict[str, np.ndarray]:
    """run_rows over every sorted row [0, R) (act_in, if given, is [R, I])."""
    R = int(srt["expert_offsets"][case.E])
    return run_rows(pool, case, srt, variant, np.arange(R), act_in, keep_g, rows_per_task)
