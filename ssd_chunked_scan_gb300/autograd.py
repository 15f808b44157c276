"""Differentiable entry point over the library's forward and backward calls.

``ssd_scan(q, k, v, log_alpha, h0=None, chunk=64)`` returns out [B,L,H,dv] of
the gated linear-attention scan S_t = exp(log_alpha_t) S_{t-1} + k_t v_t^T,
out_t = S_t^T q_t (q, k [B,L,G,dk]; v [B,L,H,dv]; log_alpha [B,L,H]; h0
[B,H,dk,dv] or None for zeros), as a torch.autograd.Function: the forward is
one ssd_fwd call, the backward one ssd_bwd call, which recomputes what it needs
from the saved inputs (nothing but the inputs is kept between the two).  With
``return_final_state=True`` it returns (out, hT) through ssd_fwd_ex /
ssd_bwd_ex, and hT's gradient flows too.  Tensors must be contiguous float32
CUDA tensors; there is no CPU path.
"""
import torch

from . import ssd


class _Scan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, log_alpha, h0, chunk, final):
        if final:
            out, hT = ssd.ssd_fwd_ex(q, k, v, log_alpha, h0, chunk=chunk)
        else:
            out, hT = ssd.ssd_fwd(q, k, v, log_alpha, h0, chunk=chunk), None
        ctx.save_for_backward(q, k, v, log_alpha, h0)
        ctx.chunk, ctx.final = chunk, final
        return (out, hT) if final else out

    @staticmethod
    def backward(ctx, dout, dhT=None):
        q, k, v, log_alpha, h0 = ctx.saved_tensors
        want_dh0 = h0 is not None and ctx.needs_input_grad[4]
        dout = dout.contiguous()
        if ctx.final:
            g = ssd.ssd_bwd_ex(q, k, v, log_alpha, h0, dout,
                               None if dhT is None else dhT.contiguous(),
                               chunk=ctx.chunk, want_dh0=want_dh0)
        else:
            g = ssd.ssd_bwd(q, k, v, log_alpha, h0, dout, chunk=ctx.chunk, want_dh0=want_dh0)
        return g["dq"], g["dk"], g["dv"], g["dlog_alpha"], g["dh0"], None, None


def ssd_scan(q, k, v, log_alpha, h0=None, chunk=64, return_final_state=False):
    """out (or (out, hT) with return_final_state), differentiable in every tensor input."""
    return _Scan.apply(q, k, v, log_alpha, h0, int(chunk), bool(return_final_state))
