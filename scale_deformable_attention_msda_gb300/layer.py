"""Multi-scale deformable attention layer: the projections around the operator.

The msda-triton course, ch. 1 ("The idea: attend to a few learned
locations" and "The equation, term by term"), describes the layer: a linear
layer on the query features predicts K sampling offsets per head and level,
another predicts the attention weights (softmax-normalised over levels and
points), the value is projected per head, and W_m projects the heads' output.
The deformops README ("Multi-scale deformable attention") gives the call
shape: layer(query, reference, value, spatial_shapes, level_start_index).

The four projections are ordinary dense matmuls (torch.nn.Linear, i.e.
cuBLAS); the sampling, the softmax over the L*K logits and their backward run
in libmsda's fused-softmax kernels. Offsets are in pixels of each level: the
sampling location of (q, m, l, k) is reference[q, l] + offset / (W_l, H_l).
"""
from __future__ import annotations

import math

import torch
from torch import nn

from . import binding


class MultiScaleDeformableAttention(nn.Module):
    """query (B, Q, dim), reference (B, Q, L, 2) or (B, Q, 2) normalised (x, y),
    value (B, S, dim), spatial_shapes (L, 2) int64 (H, W), level_start_index
    (L,) int64 -> (B, Q, dim). dim = num_heads * head_dim."""

    def __init__(self, dim: int = 256, num_heads: int = 8, num_levels: int = 4,
                 num_points: int = 4, accum: int = binding.MSDA_ACC_FP32_BUFFER):
        super().__init__()
        if dim % num_heads != 0:
            raise ValueError("dim must be divisible by num_heads")
        self.dim, self.num_heads = dim, num_heads
        self.num_levels, self.num_points = num_levels, num_points
        self.head_dim = dim // num_heads
        self.accum = accum
        self.sampling_offsets = nn.Linear(dim, num_heads * num_levels * num_points * 2)
        self.attention_weights = nn.Linear(dim, num_heads * num_levels * num_points)
        self.value_proj = nn.Linear(dim, dim)
        self.output_proj = nn.Linear(dim, dim)
        self.reset_parameters()

    @torch.no_grad()
    def reset_parameters(self):
        # Offsets start on a ring of directions, one per head, growing with the
        # point index; logits start at zero (uniform weights).
        nn.init.zeros_(self.sampling_offsets.weight)
        theta = torch.arange(self.num_heads, dtype=torch.float32) * (2.0 * math.pi / self.num_heads)
        grid = torch.stack([theta.cos(), theta.sin()], -1)
        grid = grid / grid.abs().max(-1, keepdim=True)[0]
        grid = grid.view(self.num_heads, 1, 1, 2).repeat(1, self.num_levels, self.num_points, 1)
        grid = grid * torch.arange(1, self.num_points + 1, dtype=torch.float32).view(1, 1, -1, 1)
        self.sampling_offsets.bias.copy_(grid.reshape(-1))
        nn.init.zeros_(self.attention_weights.weight)
        nn.init.zeros_(self.attention_weights.bias)
        nn.init.xavier_uniform_(self.value_proj.weight)
        nn.init.zeros_(self.value_proj.bias)
        nn.init.xavier_uniform_(self.output_proj.weight)
        nn.init.zeros_(self.output_proj.bias)

    def forward(self, query, reference, value, spatial_shapes, level_start_index):
        B, Q, _ = query.shape
        S = value.shape[1]
        M, L, K, D = self.num_heads, self.num_levels, self.num_points, self.head_dim
        v = self.value_proj(value).view(B, S, M, D)
        off = self.sampling_offsets(query).view(B, Q, M, L, K, 2)
        logits = self.attention_weights(query).view(B, Q, M, L, K)
        wh = spatial_shapes.flip(-1).to(off.dtype)                      # (L, 2) = (W, H)
        if reference.dim() == 3:
            reference = reference[:, :, None, :].expand(B, Q, L, 2)
        loc = reference[:, :, None, :, None, :].to(off.dtype) + off / wh[None, None, None, :, None, :]
        out = binding.multi_scale_deformable_attention(v, spatial_shapes, level_start_index, loc,
                                                       logits, accum=self.accum, softmax=True)
        return self.output_proj(out)
