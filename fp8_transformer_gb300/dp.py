"""Data-parallel use of the block across ranks, with torch.distributed collectives.

The block is row-local: with the weights replicated, each rank runs te_layernorm_mlp_fwd /
te_layernorm_mlp_bwd on its own tokens, and two exchanges make the ranks one data-parallel job
(LayerNorm MLP page, Signature: the sharding-axes arguments that place the batch dimension on
a data-parallel mesh axis; LayerNorm Dense page, Description: sharding constraints):

* The gradients of the replicated parameters -- dkernel1, dkernel2, dbias1, dbias2, dgamma,
  dbeta -- are summed over the ranks.  ``GradBuckets`` lays them out in two flat buffers, the
  kernels' gradients in the activation dtype and the vectors in fp32, each reduced by one
  all_reduce(SUM).
* The per-tensor amax of every quantizer is reduced with MAX, so that the scales of the next
  step (delayed scaling) are the same on every rank and every rank's E4M3 codes mean the same
  numbers.  ``QuantizerBank`` keeps the scalars of the five quantizers of a QuantizerSet in
  three contiguous tensors, so the exchange is one all_reduce(MAX) of a 5-float tensor, after
  which ``te_update_scales`` derives every scale on the device (scale = 448 / amax).

Only the collectives run here (torch.distributed, NCCL on GPUs); every step of the block runs in
the library's kernels.  Nothing here is needed on one GPU.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from .binding import Quantizer, QuantizerSet, te_layernorm_mlp_bwd, te_update_scales

NAMES = ("x", "kernel1", "act", "kernel2", "grad")


class QuantizerBank:
    """The quantizers of a QuantizerSet with their scale, scale_inv and amax scalars stored as
    elements of three contiguous fp32 tensors (in the order of NAMES)."""

    def __init__(self, scales=None, modes=None, device="cuda"):
        scales = scales or {}
        modes = modes or {}
        init = [float(scales.get(n, 1.0)) for n in NAMES]
        self.scale = torch.tensor(init, dtype=torch.float32, device=device)
        self.scale_inv = torch.tensor([1.0 / v for v in init], dtype=torch.float32, device=device)
        self.amax = torch.zeros(len(NAMES), dtype=torch.float32, device=device)
        self.quantizers = {}
        for i, n in enumerate(NAMES):
            self.quantizers[n] = Quantizer.from_tensors(self.scale[i:i + 1],
                                                        self.scale_inv[i:i + 1],
                                                        self.amax[i:i + 1],
                                                        modes.get(n, "delayed"))

    def quantizer_set(self) -> QuantizerSet:
        return QuantizerSet(**self.quantizers)

    def allreduce_amax(self, group=None):
        """Every quantizer's amax becomes the maximum over the ranks (one collective)."""
        dist.all_reduce(self.amax, op=dist.ReduceOp.MAX, group=group)

    def update_scales(self, stream=None):
        """scale = 448 / amax, scale_inv = 1 / scale for every quantizer, on the device."""
        te_update_scales([self.quantizers[n] for n in NAMES], stream=stream)


class GradBuckets:
    """Gradients of the replicated parameters of one LayerNorm-MLP block in two flat buffers:
    ``weights`` (dkernel1 [H, F'] then dkernel2 [F, H], in ``dtype``) and ``vectors`` (dbias1
    [F'], dbias2 [H], dgamma [H], dbeta [H], fp32), F' = 2F for a gated activation.  The named
    attributes are views into them, 16-byte aligned when H and F are multiples of 16."""

    def __init__(self, H, F, gated, dtype=torch.bfloat16, device="cuda"):
        F1 = 2 * F if gated else F
        self.weights = torch.empty(H * F1 + F * H, dtype=dtype, device=device)
        self.vectors = torch.empty(F1 + 3 * H, dtype=torch.float32, device=device)
        self.dkernel1 = self.weights[:H * F1].view(H, F1)
        self.dkernel2 = self.weights[H * F1:].view(F, H)
        o = 0
        views = {}
        for name, n in (("dbias1", F1), ("dbias2", H), ("dgamma", H), ("dbeta", H)):
            views[name] = self.vectors[o:o + n]
            o += n
        self.dbias1, self.dbias2 = views["dbias1"], views["dbias2"]
        self.dgamma, self.dbeta = views["dgamma"], views["dbeta"]

    def allreduce(self, group=None):
        """Sum every gradient over the ranks (one collective per buffer)."""
        dist.all_reduce(self.weights, op=dist.ReduceOp.SUM, group=group)
        dist.all_reduce(self.vectors, op=dist.ReduceOp.SUM, group=group)


def layernorm_mlp_bwd_dp(dy, x, gamma, kernel1, kernel2, saved_h, saved_ln_out, mu, rsigma, dx,
                         buckets: GradBuckets, norm_type="layernorm", zero_centered_gamma=False,
                         activation_type=("relu",), quantizer_set=None, group=None, stream=None):
    """te_layernorm_mlp_bwd on this rank's tokens, writing the parameter gradients into
    ``buckets``, then their sum over the ranks.  dx stays local (it belongs to this rank's
    tokens).  RMSNorm writes zeros into ``buckets.dbeta`` (beta is unused)."""
    te_layernorm_mlp_bwd(dy, x, gamma, kernel1, kernel2, saved_h, saved_ln_out, mu, rsigma, dx,
                         buckets.dgamma, buckets.dkernel1, buckets.dkernel2, dbeta=buckets.dbeta,
                         dbias1=buckets.dbias1, dbias2=buckets.dbias2, norm_type=norm_type,
                         zero_centered_gamma=zero_centered_gamma,
                         activation_type=activation_type, quantizer_set=quantizer_set,
                         stream=stream)
    buckets.allreduce(group)
