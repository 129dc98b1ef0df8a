"""Device-memory plumbing around the C ABI: pack a layer's weights once, own the
workspace, and issue moe_step. PyTorch only allocates memory and provides streams; every
computation is a call into libmoestep.so.
"""
from __future__ import annotations

import torch

from . import moestep as ms

WHICH = {"w13": ms.MOE_W13, "w2": ms.MOE_W2, "sh13": ms.MOE_SH13, "sh2": ms.MOE_SH2}


def _dev_bytes(n, device):
    return torch.empty(max(int(n), 16), dtype=torch.uint8, device=device)


class MoELayer:
    """One MoE layer on one GPU: packed weights + workspace.

    `inputs` is a dict in the canonical layouts of synth.make_inputs (weights as
    (codes, scales, global_scale) triples on `device`).
    """

    def __init__(self, cfg, inputs, device="cuda", stream=None):
        self.cfg = cfg
        self.device = torch.device(device)
        self.d = ms.layer_desc(cfg, inputs["gs_a"])
        self.wg = inputs["wg"]
        self.bias = inputs["bias"]
        self.gamma = inputs["gamma"]
        self.packed, self.gs, self.qw = {}, {}, {}
        for name in ("w13", "w2", "sh13", "sh2"):
            if name not in inputs:
                self.qw[name] = ms.QWeight(None, None)
                continue
            codes, scales, gs = inputs[name]
            buf = _dev_bytes(ms.moe_packed_bytes(self.d, WHICH[name]), self.device)
            ms.moe_pack_weights(self.d, WHICH[name], codes, scales, buf, stream)
            self.packed[name] = buf
            self.gs[name] = gs.contiguous()
            self.qw[name] = ms.qweight(buf, self.gs[name])
        self.ws = _dev_bytes(ms.moe_workspace_bytes(self.d), self.device)
        ms.moe_workspace_init(self.d, self.ws, stream)
        self.view = ms.moe_ws_view(self.d, self.ws)

    def args(self, x, residual, out, outq=None, outq_scales=None) -> ms.StepArgs:
        q = self.qw
        return ms.StepArgs(x.data_ptr(), self.wg.data_ptr(), None if self.bias is None else self.bias.data_ptr(),
                           q["w13"], q["w2"], q["sh13"], q["sh2"], residual.data_ptr(), self.gamma.data_ptr(),
                           out.data_ptr(), None if outq is None else outq.data_ptr(),
                           None if outq_scales is None else outq_scales.data_ptr())

    def step(self, x, residual, out, outq=None, outq_scales=None, stream=None, args=None):
        M = x.shape[0]
        a = args if args is not None else self.args(x, residual, out, outq, outq_scales)
        ms.moe_step(self.d, a, M, self.ws, stream)

    def ws_tensor(self, name, dtype, shape):
        """A torch view of one intermediate inside the workspace (see moe_ws_view)."""
        addr = getattr(self.view, name)
        off = addr - self.ws.data_ptr()
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(*shape)

    def status(self, stream=None):
        return ms.moe_get_status(self.ws, stream)

    def weight_bytes(self):
        return sum(t.numel() for t in self.packed.values())
