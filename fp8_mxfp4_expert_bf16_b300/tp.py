"""Tensor-parallel split of the expert middle dimension over a process group.

The pages deploy the layer over 8 H200s (TP8) or 4 MI355X (TP4) (vLLM recipe
"XiaomiMiMo/MiMo-V2.6-Pro-RL", "Overview" hardware line and the TP8 / TP4
launch recipes).  Rank r of G holds, for every expert, gate and up rows
[r I/G, (r+1) I/G) of W13 and the same columns of W2 (``MoELayer(...,
tp_size=G, tp_rank=r)``).  Routing, dispatch and the input quantisation are
the same on every rank; each rank's grouped GEMMs produce the expert outputs
summed over its slice only, and the gate-weighted combine leaves them in
fp32 (``forward_partial``).  One sum all-reduce over the group then gives
the layer's fp32 output, rounded once to bf16 by the library
(``sum_partials_bf16``).  The only exchange is that all-reduce of T x H fp32
values per layer.
"""
from __future__ import annotations

from . import MoELayer, sum_partials_bf16


class TensorParallelMoE:
    """One rank of a tensor-parallel MoE layer.

    ``layer`` is this rank's shard (a ``MoELayer`` made with tp_size = the
    group's size and tp_rank = the rank, weights loaded from the whole
    layer's tensors).  ``round_bf16(y32, y)`` turns the all-reduced fp32 sum
    into the bf16 output; the default is the library's
    ``moe_sum_partials_bf16``.
    """

    def __init__(self, layer, group=None, round_bf16=None):
        self.layer = layer
        self.group = group
        self._round = round_bf16 or (lambda y32, y: sum_partials_bf16([y32], y))
        self._y32 = None   # the partial-output buffer, reused while T stays the same

    def forward(self, x, y=None):
        """x: bf16 [T, H] (the same on every rank) -> y: bf16 [T, H] (the same on every rank)."""
        import torch
        import torch.distributed as dist
        T, H = x.shape
        if self._y32 is None or tuple(self._y32.shape) != (T, H) or self._y32.device != x.device:
            self._y32 = torch.empty((T, H), dtype=torch.float32, device=x.device)
        y32 = self.layer.forward_partial(x, self._y32)
        if dist.is_available() and dist.is_initialized() and dist.get_world_size(self.group) > 1:
            dist.all_reduce(y32, op=dist.ReduceOp.SUM, group=self.group)
        return self._round(y32, y)


def make_shard(hidden, inter, num_experts, top_k, max_tokens, tp_size, tp_rank, score_func=0, device=0,
               act_scale_mode=0) -> MoELayer:
    """This rank's shard of the layer (load the whole layer's weights into it)."""
    if inter % (128 * tp_size):
        raise ValueError(f"inter={inter} must be a multiple of 128 * tp_size={128 * tp_size}")
    return MoELayer(hidden, inter, num_experts, top_k, max_tokens, score_func, device, act_scale_mode,
                    tp_size=tp_size, tp_rank=tp_rank)
