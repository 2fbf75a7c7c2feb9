"""Checkpoint of the layer's mutable state.

The only state the layer carries from step to step is the routing bias b [E]
fp32 of the auxiliary-loss-free balancing ("DeepSeek-V3技术报告" digest,
mpbf.cn, section 2.2), plus the step counter. It is saved as raw bytes so that
a resumed run continues the bias trajectory bit for bit.
"""
from __future__ import annotations

import struct

import torch

_MAGIC = b"MOEB"


def save_bias(bias: torch.Tensor, step: int) -> bytes:
    """Raw fp32 bias and step counter: magic, step (int64), E (int32), data."""
    b = bias.detach().to("cpu", torch.float32).contiguous()
    return _MAGIC + struct.pack("<qi", int(step), b.numel()) + b.numpy().tobytes()


def load_bias(blob: bytes, device="cpu"):
    """Inverse of save_bias: returns (bias tensor on `device`, step)."""
    if blob[:4] != _MAGIC:
        raise ValueError("not a routing-bias checkpoint")
    step, n = struct.unpack("<qi", blob[4:16])
    data = bytearray(blob[16:16 + 4 * n])
    if len(data) != 4 * n:
        raise ValueError("truncated routing-bias checkpoint")
    b = torch.frombuffer(data, dtype=torch.float32).clone()
    return b.to(device), step
