"""Upload NVFP4 expert weights to the GPU and build their expert tables (done once, at load)."""

from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

from ._lib import ExpertTable

__all__ = ["DeviceProjection", "upload_projection"]


class DeviceProjection:
    """One projection's per-expert packed/scales tensors on the device plus its expert table."""

    def __init__(self, packed, scales, scale2, N: int, K: int):
        self.packed = packed
        self.scales = scales
        self.scale2 = np.asarray(scale2, dtype=np.float32)
        self.N, self.K = N, K
        self.table = ExpertTable(packed, scales, self.scale2, N, K)

    @property
    def E(self) -> int:
        return len(self.packed)

    def nbytes(self) -> int:
        return sum(p.numel() + s.numel() for p, s in zip(self.packed, self.scales) if p is not None)

    def close(self):
        self.table.close()


def _to_dev(a, device) -> Optional[torch.Tensor]:
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a)) if isinstance(a, np.ndarray) else a
    return t.to(device=device, dtype=torch.uint8, non_blocking=False).contiguous()


def upload_projection(packed: Sequence, scales: Sequence, scale2, N: int, K: int,
                      device: str = "cuda") -> DeviceProjection:
    """``packed[e]`` uint8 [N, K/2], ``scales[e]`` uint8 [N, K/16] (numpy or torch, None = absent)."""
    p = [_to_dev(a, device) for a in packed]
    s = [_to_dev(a, device) for a in scales]
    return DeviceProjection(p, s, scale2, N, K)
