"""ctypes binding of the C ABI in ``include/moe_prefill.h``.

Argument marshalling only: every function takes torch tensors, passes their device pointers
and the current CUDA stream to the library of the same name, and raises ``MoeError`` on a
non-zero status.  All computation runs in the library's kernels; there is no fallback: if the
library is missing the import of this module's functions fails loudly.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

import torch

from . import build as _build

__all__ = [
    "MoeError", "lib", "load", "HEADER", "exported_names",
    "MoePrefillConfig", "WorkspaceLayout", "ExpertTable",
    "moe_router_logits", "moe_route_topk", "moe_sort_workspace_bytes", "moe_sort_by_expert",
    "moe_sort_by_expert_noalloc", "MOE_SORT_NOALLOC_MAX_INTS",
    "moe_w4a16_grouped_gemm", "moe_w4a16_grouped_gemm_swiglu", "MOE_FWD_SEPARATE_SWIGLU", "moe_dequant_nvfp4",
    "moe_w4a16_grouped_gemv", "moe_w4a16_grouped_gemv_swiglu", "MOE_FWD_SMALL_ROWS", "MOE_FWD_NO_MULTICAST", "moe_swiglu_clamp", "moe_combine_indexed",
    "moe_workspace_bytes", "moe_workspace_layout", "moe_prefill_forward", "moe_get_device_error",
    "moe_shared_expert_workspace_bytes", "moe_shared_expert_forward",
    "MOE_DTYPE_BF16", "MOE_DTYPE_F32", "MOE_FWD_NUM_EVENTS", "DEVERR",
    "moe_debug_set_gemm_kernel", "moe_debug_set_wait_limit_ns", "MOE_GEMM_KERNEL_AUTO", "MOE_GEMM_KERNEL_SINGLE",
    "MOE_GEMM_KERNEL_PAIR", "gemm_kernel", "moe_debug_grouped_gemm_after",
]

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_prefill.h")

MOE_OK = 0
MOE_DTYPE_BF16 = 0
MOE_DTYPE_F32 = 1
MOE_FWD_NUM_EVENTS = 8
MOE_FWD_SEPARATE_SWIGLU = 1  # moe_prefill_config.flags: SwiGLU as its own kernel on a materialised G
MOE_FWD_SMALL_ROWS = 2  # moe_prefill_config.flags: small-row products (FP32 weights) for chunks of <= 8 rows
MOE_FWD_NO_MULTICAST = 4  # moe_prefill_config.flags: no cluster-multicast loads (runs on more than one GPU)
MOE_SORT_NOALLOC_MAX_INTS = 65536  # int32 entries of the library's fixed sort scratch
MOE_GEMM_KERNEL_AUTO = 0  # moe_debug_set_gemm_kernel: CTA-pair kernel where its shapes allow
MOE_GEMM_KERNEL_SINGLE = 1  # the single-CTA kernel
MOE_GEMM_KERNEL_PAIR = 2  # the CTA-pair kernel only (other shapes are refused)
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_WORKSPACE_TOO_SMALL",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE", 6: "MOE_ERR_NOT_BUILT_FOR_DEVICE", 7: "MOE_ERR_SCRATCH_LIMIT"}
DEVERR = {0: "none", 1: "bad expert id", 2: "bad expert offsets", 3: "pipeline wait timeout", 4: "NaN logit",
          5: "bad gather index", 6: "more than 8 rows for the small-row products"}


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class MoePrefillConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("moe_intermediate", ctypes.c_int), ("num_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("swiglu_limit", ctypes.c_float), ("renormalize", ctypes.c_int),
                ("routed_scale", ctypes.c_float), ("flags", ctypes.c_int)]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("logits", "ids", "wts", "sorted_token_ids", "sorted_expert_ids",
                                               "expert_offsets", "token_to_perm", "sort_scratch", "ready", "G", "act", "Y",
                                               "x_stage", "x_sorted", "total")]


_LIB: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "moe_version": (ctypes.c_char_p, []),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_expert_table_create": (_I, [ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_F), _I, _I, _I,
                                     ctypes.POINTER(_P)]),
    "moe_expert_table_destroy": (_I, [_P]),
    "moe_expert_table_shape": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "moe_router_logits": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "moe_route_topk": (_I, [_P, _P, _I, _I, _I, _I, _F, _P, _P, _P]),
    "moe_sort_workspace_bytes": (_SZ, [_I, _I, _I]),
    "moe_sort_by_expert": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_sort_by_expert_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_w4a16_grouped_gemm": (_I, [_P, _I, _I, _P, _P, _P, _I, _P, _I, _I, _P]),
    "moe_w4a16_grouped_gemm_swiglu": (_I, [_P, _I, _I, _P, _P, _P, _I, _P, _I, _F, _P]),
    "moe_w4a16_grouped_gemv": (_I, [_P, _I, _I, _P, _P, _P, _I, _P, _I, _P]),
    "moe_w4a16_grouped_gemv_swiglu": (_I, [_P, _I, _I, _P, _P, _P, _I, _P, _I, _F, _P]),
    "moe_dequant_nvfp4": (_I, [_P, _P, _F, _I, _I, _P, _P]),
    "moe_swiglu_clamp": (_I, [_P, _P, _I64, _I64, _I64, _P, _I64, _F, _P]),
    "moe_combine_indexed": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_workspace_bytes": (_SZ, [ctypes.POINTER(MoePrefillConfig), _I]),
    "moe_workspace_layout": (_I, [ctypes.POINTER(MoePrefillConfig), _I, ctypes.POINTER(WorkspaceLayout)]),
    "moe_prefill_forward": (_I, [ctypes.POINTER(MoePrefillConfig), _P, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P, _P,
                                 ctypes.POINTER(_P), _P]),
    "moe_shared_expert_workspace_bytes": (_SZ, [_I, _I, _I]),
    "moe_shared_expert_forward": (_I, [_P, _I, _I, _I, _P, _P, _P, _F, _P, _SZ, _P, _P]),
    "moe_get_device_error": (_I, [_P, ctypes.POINTER(_I)]),
    "moe_debug_set_gemm_kernel": (_I, [_I]),
    "moe_debug_set_wait_limit_ns": (ctypes.c_ulonglong, [ctypes.c_ulonglong]),
    "moe_debug_grouped_gemm_after": (_I, [_P, _I, _I, _P, _P, _P, _I, _P, _I, _I, _P, _I, _P]),
}


def load(path: Optional[str] = None, build_if_missing: bool = True) -> ctypes.CDLL:
    """Load the shared library (building it in-tree first if it is missing or stale)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if path is None:
        path = _build.lib_path()
        if build_if_missing and not _build.up_to_date():
            _build.build()
    if not os.path.exists(path):
        raise FileNotFoundError(f"CUDA library not built: {path}")
    torch.cuda.is_available()  # make sure torch's libcudart is loaded first (one runtime per process)
    L = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _LIB = L
    return L


def lib() -> ctypes.CDLL:
    return load()


def exported_names(header: str = HEADER) -> list:
    """Function names the public header declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: need a contiguous CUDA {dtype} tensor, got {t.dtype} on {t.device}")


# ------------------------------------------------------------------------------------------ tables


class ExpertTable:
    """One NVFP4 projection of all experts (see ``moe_expert_table_create``).

    ``packed[e]`` uint8 [N, K/2] and ``scales[e]`` uint8 [N, K/16] CUDA tensors (None = absent
    expert); ``scale2`` E floats.  The table keeps references to the tensors it points at.
    """

    def __init__(self, packed: Sequence[Optional[torch.Tensor]], scales: Sequence[Optional[torch.Tensor]],
                 scale2, N: int, K: int):
        E = len(packed)
        pp = (_P * E)(*[None if p is None else p.data_ptr() for p in packed])
        sp = (_P * E)(*[None if s is None else s.data_ptr() for s in scales])
        s2 = (_F * E)(*[float(v) for v in scale2])
        for p, s in zip(packed, scales):
            if p is not None:
                _need(p, torch.uint8, "packed")
                _need(s, torch.uint8, "scales")
        h = _P()
        _check(lib().moe_expert_table_create(pp, sp, s2, E, N, K, ctypes.byref(h)), "moe_expert_table_create")
        self.handle = h
        self.E, self.N, self.K = E, N, K
        self._keep = (list(packed), list(scales))

    def close(self):
        if self.handle is not None and self.handle.value:
            lib().moe_expert_table_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------------------------------ calls


def moe_router_logits(x: torch.Tensor, w_router: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None):
    _need(x, torch.bfloat16, "x")
    _need(w_router, torch.bfloat16, "w_router")
    T, H = x.shape
    E = w_router.shape[0]
    if out is None:
        out = torch.empty(T, E, dtype=torch.float32, device=x.device)
    _check(lib().moe_router_logits(_ptr(x), _ptr(w_router), T, H, E, _ptr(out), _stream(stream)), "moe_router_logits")
    return out


def moe_route_topk(logits: torch.Tensor, k: int, bias: Optional[torch.Tensor] = None, renormalize: bool = True,
                   routed_scale: float = 1.0, ids=None, wts=None, stream=None):
    _need(logits, torch.float32, "logits")
    T, E = logits.shape
    if ids is None:
        ids = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    if wts is None:
        wts = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    _check(lib().moe_route_topk(_ptr(logits), _ptr(bias), T, E, k, int(renormalize), float(routed_scale), _ptr(ids),
                                _ptr(wts), _stream(stream)), "moe_route_topk")
    return ids, wts


def moe_sort_workspace_bytes(T: int, k: int, E: int) -> int:
    return int(lib().moe_sort_workspace_bytes(T, k, E))


def moe_sort_by_expert(ids: torch.Tensor, E: int, ws: Optional[torch.Tensor] = None, stream=None) -> dict:
    _need(ids, torch.int32, "ids")
    T, k = ids.shape
    R = T * k
    dev = ids.device
    out = dict(sorted_token_ids=torch.empty(R, dtype=torch.int32, device=dev),
               sorted_expert_ids=torch.empty(R, dtype=torch.int32, device=dev),
               expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               token_to_perm=torch.empty(T, k, dtype=torch.int32, device=dev))
    need = moe_sort_workspace_bytes(T, k, E)
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check(lib().moe_sort_by_expert(_ptr(ids), T, k, E, _ptr(out["sorted_token_ids"]), _ptr(out["sorted_expert_ids"]),
                                    _ptr(out["expert_offsets"]), _ptr(out["token_to_perm"]), _ptr(ws), ws.numel(),
                                    _stream(stream)), "moe_sort_by_expert")
    return out


def moe_sort_by_expert_noalloc(ids: torch.Tensor, E: int, out: Optional[dict] = None, stream=None) -> dict:
    """moe_sort_by_expert on the library's fixed scratch (no workspace, nothing allocated by the
    library).  `out` may hold preallocated output tensors with the keys of the returned dict."""
    _need(ids, torch.int32, "ids")
    T, k = ids.shape
    R = T * k
    dev = ids.device
    if out is None:
        out = dict(sorted_token_ids=torch.empty(R, dtype=torch.int32, device=dev),
                   sorted_expert_ids=torch.empty(R, dtype=torch.int32, device=dev),
                   expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   token_to_perm=torch.empty(T, k, dtype=torch.int32, device=dev))
    _check(lib().moe_sort_by_expert_noalloc(_ptr(ids), T, k, E, _ptr(out["sorted_token_ids"]),
                                            _ptr(out["sorted_expert_ids"]), _ptr(out["expert_offsets"]),
                                            _ptr(out["token_to_perm"]), _stream(stream)),
           "moe_sort_by_expert_noalloc")
    return out


def moe_w4a16_grouped_gemm_swiglu(A: torch.Tensor, W: ExpertTable, expert_offsets: torch.Tensor, R: int,
                                  limit: float = 7.0, gather_ids: Optional[torch.Tensor] = None,
                                  out: Optional[torch.Tensor] = None, stream=None):
    """Gate/up GEMM over a [2I, K] table with the clamped SwiGLU in its epilogue: BF16 act [R, I]."""
    _need(A, torch.bfloat16, "A")
    _need(expert_offsets, torch.int32, "expert_offsets")
    if gather_ids is not None:
        _need(gather_ids, torch.int32, "gather_ids")
    if out is None:
        out = torch.empty(R, W.N // 2, dtype=torch.bfloat16, device=A.device)
    _check(lib().moe_w4a16_grouped_gemm_swiglu(_ptr(A), A.shape[0], A.stride(0), _ptr(gather_ids), W.handle,
                                               _ptr(expert_offsets), R, _ptr(out), out.stride(0), limit,
                                               _stream(stream)),
           "moe_w4a16_grouped_gemm_swiglu")
    return out


def moe_w4a16_grouped_gemv(A: torch.Tensor, W: ExpertTable, expert_offsets: torch.Tensor, R: int,
                           gather_ids: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None, stream=None):
    """Small-row product (<= 8 rows per expert), FP32 dequantised weights, BF16 [R, N]."""
    _need(A, torch.bfloat16, "A")
    _need(expert_offsets, torch.int32, "expert_offsets")
    if gather_ids is not None:
        _need(gather_ids, torch.int32, "gather_ids")
    if out is None:
        out = torch.empty(R, W.N, dtype=torch.bfloat16, device=A.device)
    _check(lib().moe_w4a16_grouped_gemv(_ptr(A), A.shape[0], A.stride(0), _ptr(gather_ids), W.handle,
                                        _ptr(expert_offsets), R, _ptr(out), out.stride(0), _stream(stream)),
           "moe_w4a16_grouped_gemv")
    return out


def moe_w4a16_grouped_gemv_swiglu(A: torch.Tensor, W: ExpertTable, expert_offsets: torch.Tensor, R: int,
                                  limit: float = 7.0, gather_ids: Optional[torch.Tensor] = None,
                                  out: Optional[torch.Tensor] = None, stream=None):
    """Small-row gate/up product with the clamped SwiGLU: BF16 act [R, I]."""
    _need(A, torch.bfloat16, "A")
    _need(expert_offsets, torch.int32, "expert_offsets")
    if gather_ids is not None:
        _need(gather_ids, torch.int32, "gather_ids")
    if out is None:
        out = torch.empty(R, W.N // 2, dtype=torch.bfloat16, device=A.device)
    _check(lib().moe_w4a16_grouped_gemv_swiglu(_ptr(A), A.shape[0], A.stride(0), _ptr(gather_ids), W.handle,
                                               _ptr(expert_offsets), R, _ptr(out), out.stride(0), limit,
                                               _stream(stream)),
           "moe_w4a16_grouped_gemv_swiglu")
    return out


def moe_w4a16_grouped_gemm(A: torch.Tensor, W: ExpertTable, expert_offsets: torch.Tensor, R: int,
                           gather_ids: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                           c_dtype: torch.dtype = torch.bfloat16, stream=None):
    _need(A, torch.bfloat16, "A")
    _need(expert_offsets, torch.int32, "expert_offsets")
    if gather_ids is not None:
        _need(gather_ids, torch.int32, "gather_ids")
    code = MOE_DTYPE_F32 if c_dtype == torch.float32 else MOE_DTYPE_BF16
    if out is None:
        out = torch.empty(R, W.N, dtype=c_dtype, device=A.device)
    _check(lib().moe_w4a16_grouped_gemm(_ptr(A), A.shape[0], A.stride(0), _ptr(gather_ids), W.handle,
                                        _ptr(expert_offsets), R, _ptr(out), out.stride(0), code, _stream(stream)),
           "moe_w4a16_grouped_gemm")
    return out


def moe_dequant_nvfp4(packed: torch.Tensor, scales: torch.Tensor, scale2: float, stream=None) -> torch.Tensor:
    _need(packed, torch.uint8, "packed")
    _need(scales, torch.uint8, "scales")
    N, half = packed.shape
    out = torch.empty(N, 2 * half, dtype=torch.bfloat16, device=packed.device)
    _check(lib().moe_dequant_nvfp4(_ptr(packed), _ptr(scales), float(scale2), N, 2 * half, _ptr(out), _stream(stream)),
           "moe_dequant_nvfp4")
    return out


def moe_swiglu_clamp(gate: torch.Tensor, up: torch.Tensor, limit: float, out: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """``gate``/``up`` may be column slices of one [R, 2I] tensor (row stride 2I)."""
    rows, width = gate.shape
    if gate.dtype != torch.bfloat16 or up.dtype != torch.bfloat16 or gate.stride(1) != 1 or up.stride(1) != 1:
        raise ValueError("gate/up: BF16 with unit column stride")
    if gate.stride(0) != up.stride(0):
        raise ValueError("gate/up: same row stride")
    if out is None:
        out = torch.empty(rows, width, dtype=torch.bfloat16, device=gate.device)
    _check(lib().moe_swiglu_clamp(_ptr(gate), _ptr(up), rows, width, gate.stride(0), _ptr(out), out.stride(0),
                                  float(limit), _stream(stream)), "moe_swiglu_clamp")
    return out


def moe_combine_indexed(Y: torch.Tensor, token_to_perm: torch.Tensor, wts: torch.Tensor,
                        shared_out: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    _need(Y, torch.bfloat16, "Y")
    _need(token_to_perm, torch.int32, "token_to_perm")
    _need(wts, torch.float32, "wts")
    T, k = token_to_perm.shape
    H = Y.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=Y.device)
    _check(lib().moe_combine_indexed(_ptr(Y), _ptr(token_to_perm), _ptr(wts), _ptr(shared_out), T, k, H, _ptr(out),
                                     _stream(stream)), "moe_combine_indexed")
    return out


def moe_workspace_bytes(cfg: MoePrefillConfig, max_rows: int) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(cfg), max_rows))


def moe_workspace_layout(cfg: MoePrefillConfig, max_rows: int) -> WorkspaceLayout:
    L = WorkspaceLayout()
    _check(lib().moe_workspace_layout(ctypes.byref(cfg), max_rows, ctypes.byref(L)), "moe_workspace_layout")
    return L


def moe_prefill_forward(cfg: MoePrefillConfig, x: torch.Tensor, w_gate_up: ExpertTable, w_down: ExpertTable,
                        ws: torch.Tensor, w_router: Optional[torch.Tensor] = None,
                        logits: Optional[torch.Tensor] = None, router_bias: Optional[torch.Tensor] = None,
                        out: Optional[torch.Tensor] = None, stage_events: Optional[Sequence] = None,
                        stream=None, shared_out: Optional[torch.Tensor] = None, shared_ready=None) -> torch.Tensor:
    """`shared_out`: the shared expert's BF16 [T, H] output, added in the combine; `shared_ready`:
    a torch.cuda.Event the stream waits for before the combine (shared_out made on another stream).
    `x`, `logits` and `out` may also be (pinned) host tensors: the library checks that the device
    can reach them, stages a host x into the workspace on the device, reads host logits in place
    and stores into a host out directly."""
    for t, n, dt in ((x, "x", torch.bfloat16), (logits, "logits", torch.float32), (out, "out", torch.bfloat16)):
        if t is not None and (t.dtype != dt or not t.is_contiguous() or t.device.type not in ("cuda", "cpu")):
            raise ValueError(f"{n}: need a contiguous {dt} tensor (CUDA or host), got {t.dtype} on {t.device}")
    if shared_out is not None:
        _need(shared_out, torch.bfloat16, "shared_out")
    T = x.shape[0]
    if out is None:
        dev = x.device if x.is_cuda else torch.device("cuda", torch.cuda.current_device())
        out = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device=dev)
    ev = None
    if stage_events is not None:
        ev = (_P * MOE_FWD_NUM_EVENTS)(*[e.cuda_event for e in stage_events])
    ready = ctypes.c_void_p(shared_ready.cuda_event) if shared_ready is not None else None
    _check(lib().moe_prefill_forward(ctypes.byref(cfg), _ptr(x), T, _ptr(w_router), _ptr(logits), _ptr(router_bias),
                                     w_gate_up.handle, w_down.handle, _ptr(ws), ws.numel(), _ptr(out),
                                     _ptr(shared_out), ready, ev, _stream(stream)), "moe_prefill_forward")
    return out


def moe_shared_expert_workspace_bytes(T: int, H: int, I: int) -> int:
    return int(lib().moe_shared_expert_workspace_bytes(T, H, I))


def moe_shared_expert_forward(x: torch.Tensor, w_gate: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor,
                              limit: float = 7.0, ws: Optional[torch.Tensor] = None,
                              out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Shared expert (dense BF16 SwiGLU MLP): out = swiglu(x W_gate^T, x W_up^T) W_down^T."""
    for t, n in ((x, "x"), (w_gate, "w_gate"), (w_up, "w_up"), (w_down, "w_down")):
        _need(t, torch.bfloat16, n)
    T, H = x.shape
    I = w_gate.shape[0]
    if ws is None:
        ws = torch.empty(max(moe_shared_expert_workspace_bytes(T, H, I), 1), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_shared_expert_forward(_ptr(x), T, H, I, _ptr(w_gate), _ptr(w_up), _ptr(w_down), limit, _ptr(ws),
                                           ws.numel(), _ptr(out), _stream(stream)), "moe_shared_expert_forward")
    return out


def moe_get_device_error(stream=None) -> int:
    code = _I(0)
    rc = lib().moe_get_device_error(_stream(stream), ctypes.byref(code))
    if rc not in (MOE_OK, 5):
        raise MoeError(rc, "moe_get_device_error")
    return int(code.value)


def moe_debug_set_gemm_kernel(which: int) -> None:
    """Process-wide choice of the grouped GEMM kernel (MOE_GEMM_KERNEL_*), for tests and debugging."""
    _check(lib().moe_debug_set_gemm_kernel(int(which)), "moe_debug_set_gemm_kernel")


def moe_debug_set_wait_limit_ns(ns: int) -> int:
    """Bound of the CTA-pair GEMM's pipeline waits (0 restores 2 s); returns the previous bound."""
    return int(lib().moe_debug_set_wait_limit_ns(int(ns)))


def moe_debug_grouped_gemm_after(A: torch.Tensor, W: ExpertTable, expert_offsets: torch.Tensor, R: int,
                                 ready: torch.Tensor, ready_need: int, gather_ids: Optional[torch.Tensor] = None,
                                 out: Optional[torch.Tensor] = None, c_dtype: torch.dtype = torch.float32,
                                 stream=None) -> torch.Tensor:
    """The grouped GEMM waiting per expert on producer counters ``ready`` (int32 [E])."""
    _need(A, torch.bfloat16, "A")
    _need(ready, torch.int32, "ready")
    code = MOE_DTYPE_F32 if c_dtype == torch.float32 else MOE_DTYPE_BF16
    if out is None:
        out = torch.empty(R, W.N, dtype=c_dtype, device=A.device)
    _check(lib().moe_debug_grouped_gemm_after(_ptr(A), A.shape[0], A.stride(0), _ptr(gather_ids), W.handle,
                                              _ptr(expert_offsets), R, _ptr(out), out.stride(0), code, _ptr(ready),
                                              int(ready_need), _stream(stream)),
           "moe_debug_grouped_gemm_after")
    return out


class gemm_kernel:
    """``with gemm_kernel(MOE_GEMM_KERNEL_PAIR): ...`` runs the block with that kernel choice."""

    def __init__(self, which: int):
        self.which = which

    def __enter__(self):
        moe_debug_set_gemm_kernel(self.which)
        return self

    def __exit__(self, *exc):
        moe_debug_set_gemm_kernel(MOE_GEMM_KERNEL_AUTO)
        return False
