"""MoeLayer: owns the workspace and the per-call ids/weights buffers of one layer shape."""
from __future__ import annotations

import torch

from . import _lib


class MoeLayer:
    """Routed MoE layer of a fixed shape on one CUDA device.

    __call__ runs the whole layer and returns the BF16 output [T, d]: with the automatic
    kernel choice one moe_layer call (fused router + plan front for moderate T * k), else
    router, plan and experts as three C-ABI calls on the current stream.  Weights are a dict of device tensors:
    w13_codes [E, 2*ffn, d/2] uint8, w13_scales [E, 2*ffn, d/16] uint8 (E4M3),
    w2_codes [E, d, ffn/2] uint8, w2_scales [E, d, ffn/16] uint8, and the FP32 tensor
    scales w13_ts / w2_ts (Python floats).
    """

    def __init__(self, T, d, ffn, E, k, device="cuda", algo=_lib.ALGO_AUTO):
        self.shape = _lib.shape_of(T, d, ffn, E, k)
        rc = _lib.check_shape(self.shape)
        if rc != _lib.MOE_OK:
            raise _lib.MoeError("moe_check_shape", rc)
        self.device = torch.device(device)
        self.algo = algo
        self.ws = _lib.Workspace(self.shape, device=self.device)
        self.ids = torch.empty((T, k), dtype=torch.int32, device=self.device)
        self.weights = torch.empty((T, k), dtype=torch.float32, device=self.device)

    def route(self, logits):
        _lib.route_topk(self.shape, logits, self.ids, self.weights)
        return self.ids, self.weights

    def plan(self):
        _lib.plan(self.shape, self.ids, self.weights, self.ws)

    def experts(self, hidden, w, residual=None, out=None):
        if out is None:
            out = torch.empty((self.shape.T, self.shape.d), dtype=torch.bfloat16, device=self.device)
        _lib.forward(self.shape, hidden, w, residual, out, self.ws, self.algo)
        return out

    def __call__(self, logits, hidden, w, residual=None, out=None):
        if self.algo == _lib.ALGO_AUTO:
            if out is None:
                out = torch.empty((self.shape.T, self.shape.d), dtype=torch.bfloat16, device=self.device)
            _lib.layer(self.shape, logits, hidden, w, residual, out, self.ids, self.weights, self.ws)
            return out
        self.route(logits)
        self.plan()
        return self.experts(hidden, w, residual, out)

    def status(self, clear=True):
        return _lib.read_status(self.ws, clear)
