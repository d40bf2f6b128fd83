"""Device-side plumbing around the C ABI: buffers allocated with PyTorch,
weights uploaded in the prepared layout, and the route + forward call pair.

Nothing here computes any part of the layer; it only allocates, copies and
calls the binding.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import binding as B
from .synth import Workload


def shape_of(wl: Workload, tokens: int | None = None) -> B.Shape:
    return B.make_shape(wl.tokens if tokens is None else tokens, wl.hidden, wl.inter, wl.experts, wl.top_k,
                        wl.group_gate_up, wl.group_down, wl.activation, wl.reduction, wl.format)


@dataclass
class PreparedWeights:
    gate_up: torch.Tensor  # uint8, prepared stream
    down: torch.Tensor

    @property
    def nbytes(self) -> int:
        return self.gate_up.numel() + self.down.numel()


def prepare_host(wl: Workload, w: dict) -> tuple[np.ndarray, np.ndarray]:
    """Canonical numpy weights -> the two prepared streams (host)."""
    sh = shape_of(wl, 1)
    gu = B.moe_w4a16_prepare(sh, B.GATE_UP, w["gate_up_q"], w["gate_up_scale"], w["gate_up_zero"])
    dn = B.moe_w4a16_prepare(sh, B.DOWN, w["down_q"], w["down_scale"], w["down_zero"])
    return gu, dn


def upload_weights(wl: Workload, w: dict, device="cuda") -> PreparedWeights:
    gu, dn = prepare_host(wl, w)
    return PreparedWeights(torch.from_numpy(gu).to(device), torch.from_numpy(dn).to(device))


@dataclass
class Buffers:
    """Per-canvas device buffers: routing, workspace and output."""
    shape: B.Shape
    routing: B.RoutingBuffers
    workspace: torch.Tensor
    out: torch.Tensor


def alloc_buffers(wl: Workload, tokens: int | None = None, device="cuda", stream=None) -> Buffers:
    sh = shape_of(wl, tokens)
    T, k, E = sh.tokens, sh.top_k, sh.experts
    routing = B.RoutingBuffers(
        topk_idx=torch.empty((T, k), dtype=torch.int32, device=device),
        topk_w=torch.empty((T, k), dtype=torch.float32, device=device),
        expert_offsets=torch.empty((E + 1,), dtype=torch.int32, device=device),
        pair_list=torch.empty((max(T * k, 1),), dtype=torch.int32, device=device),
    )
    ws = torch.empty((B.moe_w4a16_workspace_bytes(sh),), dtype=torch.uint8, device=device)
    B.moe_w4a16_workspace_init(ws, stream)
    out = torch.empty((T, wl.hidden), dtype=torch.float16, device=device)
    return Buffers(sh, routing, ws, out)


def run_layer(buf: Buffers, x: torch.Tensor, logits: torch.Tensor, w: PreparedWeights,
              gamma: torch.Tensor | None = None, eps: float = 1e-6, out: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """Route the canvas, then run the experts and the combine; returns the output tensor."""
    o = buf.out if out is None else out
    B.moe_w4a16_route(buf.shape, logits, buf.routing, buf.workspace, stream)
    B.moe_w4a16_forward(buf.shape, x, buf.routing, w.gate_up, w.down, gamma, eps, o, buf.workspace, stream)
    return o


def run_block(buf: Buffers, x: torch.Tensor, gamma_pre: torch.Tensor, router_w: torch.Tensor, w: PreparedWeights,
              eps: float = 1e-6, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The MoE block: pre-norm, router projection, routing, experts, combine plus the residual."""
    o = buf.out if out is None else out
    B.moe_w4a16_block(buf.shape, x, gamma_pre, eps, router_w, buf.routing, w.gate_up, w.down, o, buf.workspace,
                      stream)
    return o


def to_device_u16(a: np.ndarray, device="cuda") -> torch.Tensor:
    """fp16 bit patterns (uint16) as an fp16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).to(device)


def to_device_x(x_bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.float16)).to(device)


def to_device_f32(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
