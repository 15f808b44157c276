"""Differentiable entry point over the library's forward and backward calls.

``ssd_scan(q, k, v, log_alpha, h0=None, chunk=64)`` returns out [B,L,H,dv] of
the gated linear-attention scan S_t = exp(log_alpha_t) S_{t-1} + k_t v_t^T,
out_t = S_t^T q_t (q, k [B,L,G,dk]; v [B,L,H,dv]; log_alpha [B,L,H]; h0
[B,H,dk,dv] or None for zeros), as a torch.autograd.Function: the forward is
one ssd_fwd_ex call, the backward one ssd_bwd_ex call, which recomputes what
it needs from the saved inputs (nothing but the inputs is kept between the
two).  With ``save_states=True`` they are ssd_fwd_save / ssd_bwd_saved
instead: the two also keep the final state and, on the tensor-core path, the
states entering each segment (ssd_saved_bytes: B*H*dk*dv*4 bytes per
segment, about one segment per SM in all), which the backward then reads
instead of recomputing.  With ``return_final_state=True`` it returns
(out, hT), and hT's gradient flows too.  Tensors must be contiguous float32
CUDA tensors; there is no CPU path.
"""
import torch

from . import ssd


class _Scan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, log_alpha, h0, chunk, final, save_states):
        if save_states:
            out, hT, saved = ssd.ssd_fwd_save(q, k, v, log_alpha, h0, chunk=chunk)
            ctx.save_for_backward(q, k, v, log_alpha, h0, hT, saved)
        else:
            out, hT = ssd.ssd_fwd_ex(q, k, v, log_alpha, h0, chunk=chunk)
            ctx.save_for_backward(q, k, v, log_alpha, h0)
        ctx.chunk, ctx.final, ctx.save_states = chunk, final, save_states
        return (out, hT) if final else out

    @staticmethod
    def backward(ctx, dout, dhT=None):
        want_dh0 = ctx.needs_input_grad[4] and ctx.saved_tensors[4] is not None
        dout = dout.contiguous()
        dhT = dhT.contiguous() if (ctx.final and dhT is not None) else None
        if ctx.save_states:
            q, k, v, log_alpha, h0, hT, saved = ctx.saved_tensors
            g = ssd.ssd_bwd_saved(q, k, v, log_alpha, h0, dout, dhT, hT, saved, chunk=ctx.chunk,
                                  want_dh0=want_dh0)
        else:
            q, k, v, log_alpha, h0 = ctx.saved_tensors
            g = ssd.ssd_bwd_ex(q, k, v, log_alpha, h0, dout, dhT, chunk=ctx.chunk, want_dh0=want_dh0)
        return g["dq"], g["dk"], g["dv"], g["dlog_alpha"], g["dh0"], None, None, None


def ssd_scan(q, k, v, log_alpha, h0=None, chunk=64, return_final_state=False, save_states=False):
    """out (or (out, hT) with return_final_state), differentiable in every tensor input."""
    return _Scan.apply(q, k, v, log_alpha, h0, int(chunk), bool(return_final_state), bool(save_states))
