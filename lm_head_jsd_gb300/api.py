"""Torch-facing wrapper of the C ABI: allocation of outputs and workspace, and an
autograd Function. PyTorch supplies device memory and streams only; every step
of the loss runs in libfljsd.so."""
from __future__ import annotations

import torch

from . import _lib
from ._lib import fljsd_backward, fljsd_forward, fljsd_plan, make_problem

_DT = {torch.float32: "fp32", torch.bfloat16: "bf16"}


def _check(name, t, dtype, device, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


class FusedLinearJSD:
    """Plans one problem shape and keeps its workspace for repeated calls.

    ``forward`` returns (loss, grad_input, grad_weight) for an upstream gradient
    of 1; ``backward`` scales both gradients in place by a device scalar.
    """

    def __init__(self, bt, h_s, h_t, v, dtype=torch.bfloat16, *, beta=0.5, temperature=1.0,
                 reduction="batchmean", ignore_index=-100, chunk_rows=0, device="cuda",
                 free_hbm_bytes=None, t2_scale=False, accum_fp32=False):
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.dtype = dtype
        self.reduction = reduction
        self.problem = make_problem(bt, h_s, h_t, v, _DT[dtype], reduction, beta, temperature,
                                    ignore_index, chunk_rows, t2_scale, accum_fp32)
        if free_hbm_bytes is None:
            free_hbm_bytes = torch.cuda.mem_get_info(self.device)[0]
        self.plan = fljsd_plan(self.problem, int(free_hbm_bytes))
        self.workspace = torch.empty(self.plan.workspace_bytes, dtype=torch.uint8,
                                     device=self.device)

    @property
    def shape(self):
        p = self.problem
        return p.bt, p.h_s, p.h_t, p.v

    def alloc_outputs(self):
        bt, h_s, _, v = self.shape
        n_loss = bt if self.reduction == "none" else 1
        loss = torch.empty(n_loss, dtype=torch.float32, device=self.device)
        gi = torch.empty(bt, h_s, dtype=self.dtype, device=self.device)
        gw = torch.empty(v, h_s, dtype=self.dtype, device=self.device)
        return loss, gi, gw

    def forward(self, x_s, w_s, x_t, w_t, labels=None, row_grad=None, out=None, stream=None):
        bt, h_s, h_t, v = self.shape
        dev = self.device
        _check("x_s", x_s, self.dtype, dev, (bt, h_s))
        _check("w_s", w_s, self.dtype, dev, (v, h_s))
        _check("x_t", x_t, self.dtype, dev, (bt, h_t))
        _check("w_t", w_t, self.dtype, dev, (v, h_t))
        if labels is not None:
            _check("labels", labels, torch.int64, dev, (bt,))
        if row_grad is not None:
            _check("row_grad", row_grad, torch.float32, dev, (bt,))
        loss, gi, gw = self.alloc_outputs() if out is None else out
        fljsd_forward(self.problem, self.plan, x_s, w_s, x_t, w_t, labels, row_grad, loss, gi,
                      gw, self.workspace, stream=stream)
        return loss, gi, gw

    def backward(self, grad_output, grad_input, grad_weight, stream=None):
        _check("grad_output", grad_output, torch.float32, self.device)
        fljsd_backward(self.problem, grad_output, grad_input, grad_weight, stream=stream)
        return grad_input, grad_weight


class _FusedLinearJSDFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x_s, w_s, x_t, w_t, labels, beta, temperature, reduction, ignore_index,
                chunk_rows):
        bt, h_s = x_s.shape
        runner = FusedLinearJSD(bt, h_s, x_t.shape[1], w_s.shape[0], x_s.dtype, beta=beta,
                                temperature=temperature, reduction=reduction,
                                ignore_index=ignore_index, chunk_rows=chunk_rows,
                                device=x_s.device)
        xs, ws, xt, wt = (t.detach().contiguous() for t in (x_s, w_s, x_t, w_t))
        lab = None if labels is None else labels.contiguous()
        loss, gi, gw = runner.forward(xs, ws, xt, wt, lab)
        ctx.runner = runner
        ctx.inputs = (xs, ws, xt, wt, lab)
        ctx.save_for_backward(gi, gw)
        return loss if reduction == "none" else loss.reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        gi, gw = ctx.saved_tensors
        runner = ctx.runner
        if runner.reduction == "none":
            # a per-row upstream gradient: run the forward again with it
            rg = grad_out.detach().to(torch.float32).contiguous()
            _, gi, gw = runner.forward(*ctx.inputs, row_grad=rg)
        else:
            g = grad_out.detach().to(torch.float32).reshape(1).contiguous()
            runner.backward(g, gi, gw)
        return gi, gw, None, None, None, None, None, None, None, None


def fused_linear_jsd(x_s, w_s, x_t, w_t, labels=None, *, beta=0.5, temperature=1.0,
                     reduction="batchmean", ignore_index=-100, chunk_rows=0):
    """Generalized JSD distillation loss between student logits x_s.w_s^T and
    teacher logits x_t.w_t^T, differentiable in x_s and w_s (the teacher is
    frozen). Tensors are 2-D, contiguous, on one CUDA device, fp32 or bf16."""
    return _FusedLinearJSDFunction.apply(x_s, w_s, x_t, w_t, labels, float(beta),
                                         float(temperature), reduction, int(ignore_index),
                                         int(chunk_rows))


def _dist_call(kind, x, y, labels, reduction, ignore_index, beta=0.5):
    if x.shape != y.shape or x.dim() != 2:
        raise ValueError("expected two [rows x V] tensors of the same shape")
    _check("x", x, None, x.device)
    _check("y", y, x.dtype, x.device)
    if labels is not None:
        _check("labels", labels, torch.int64, x.device, (x.shape[0],))
    rows, v = x.shape
    if reduction == "none":
        loss = torch.empty((rows, v) if kind == "tvd" else (rows,), dtype=torch.float32,
                           device=x.device)
    else:
        loss = torch.empty(1, dtype=torch.float32, device=x.device)
    grad = torch.empty_like(x)
    ws = torch.empty(_lib.fljsd_rows_workspace_bytes(rows), dtype=torch.uint8, device=x.device)
    if kind == "tvd":
        _lib.fljsd_tvd(rows, v, _DT[x.dtype], reduction, ignore_index, x, y, labels, loss, grad, ws)
    else:
        _lib.fljsd_jsd_logspace(rows, v, _DT[x.dtype], beta, reduction, ignore_index, x, y,
                                labels, loss, grad, ws)
    return loss, grad


class _DistFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, kind, x, y, labels, reduction, ignore_index, beta):
        loss, grad = _dist_call(kind, x.detach().contiguous(), y.detach().contiguous(),
                                None if labels is None else labels.contiguous(), reduction,
                                ignore_index, beta)
        ctx.save_for_backward(grad)
        ctx.reduction = reduction
        ctx.dtype = x.dtype
        return loss if reduction == "none" else loss.reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        (grad,) = ctx.saved_tensors
        if ctx.reduction == "none":
            raise NotImplementedError("backward through reduction='none' is not provided")
        g = grad_out.detach().to(torch.float32).reshape(1).contiguous()
        _lib.fljsd_scale(_DT[ctx.dtype], grad, grad.numel(), g)
        return None, grad, None, None, None, None, None


def jsd_logspace(input, target, labels=None, *, beta=0.5, reduction="batchmean",
                 ignore_index=-100):
    """Generalized JSD between given log-probabilities (input = log Q, student;
    target = log P, teacher), differentiable in input."""
    return _DistFunction.apply("jsd", input, target, labels, reduction, int(ignore_index),
                               float(beta))


def tvd(p, q, labels=None, *, reduction="batchmean", ignore_index=-100):
    """Total variation distance 0.5 * sum |p - q| (zero gradient at ties),
    differentiable in p."""
    return _DistFunction.apply("tvd", p, q, labels, reduction, int(ignore_index), 0.0)


class FusedLinearCrossEntropy:
    """Plans one FLCE problem shape and keeps its workspace (see fljsd_ce_forward)."""

    def __init__(self, bt, h, v, dtype=torch.bfloat16, *, reduction="mean", ignore_index=-100,
                 label_smoothing=0.0, lse_square_scale=0.0, softcap=0.0, chunk_rows=0,
                 accum_fp32=False, device="cuda", free_hbm_bytes=None):
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.dtype = dtype
        self.reduction = reduction
        self.problem = _lib.make_ce_problem(bt, h, v, _DT[dtype], reduction, ignore_index,
                                            chunk_rows, label_smoothing, lse_square_scale,
                                            softcap, accum_fp32)
        if free_hbm_bytes is None:
            free_hbm_bytes = torch.cuda.mem_get_info(self.device)[0]
        self.plan = _lib.fljsd_ce_plan(self.problem, int(free_hbm_bytes))
        self.workspace = torch.empty(self.plan.workspace_bytes, dtype=torch.uint8,
                                     device=self.device)

    def alloc_outputs(self):
        p = self.problem
        loss = torch.empty(p.bt if self.reduction == "none" else 1, dtype=torch.float32,
                           device=self.device)
        gi = torch.empty(p.bt, p.h, dtype=self.dtype, device=self.device)
        gw = torch.empty(p.v, p.h, dtype=self.dtype, device=self.device)
        return loss, gi, gw

    def forward(self, x, w, labels, out=None, stream=None):
        p = self.problem
        _check("x", x, self.dtype, self.device, (p.bt, p.h))
        _check("w", w, self.dtype, self.device, (p.v, p.h))
        _check("labels", labels, torch.int64, self.device, (p.bt,))
        loss, gi, gw = self.alloc_outputs() if out is None else out
        _lib.fljsd_ce_forward(p, self.plan, x, w, labels, loss, gi, gw, self.workspace,
                              stream=stream)
        return loss, gi, gw


class _FLCEFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w, labels, reduction, ignore_index, label_smoothing, lse_square_scale,
                softcap, chunk_rows):
        run = FusedLinearCrossEntropy(x.shape[0], x.shape[1], w.shape[0], x.dtype,
                                      reduction=reduction, ignore_index=ignore_index,
                                      label_smoothing=label_smoothing,
                                      lse_square_scale=lse_square_scale, softcap=softcap,
                                      chunk_rows=chunk_rows, device=x.device)
        loss, gi, gw = run.forward(x.detach().contiguous(), w.detach().contiguous(),
                                   labels.contiguous())
        if reduction == "none":
            raise NotImplementedError("use reduction sum or mean through autograd")
        ctx.save_for_backward(gi, gw)
        ctx.dtype = x.dtype
        return loss.reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        gi, gw = ctx.saved_tensors
        g = grad_out.detach().to(torch.float32).reshape(1).contiguous()
        _lib.fljsd_scale(_DT[ctx.dtype], gi, gi.numel(), g)
        _lib.fljsd_scale(_DT[ctx.dtype], gw, gw.numel(), g)
        return gi, gw, None, None, None, None, None, None, None


def fused_linear_cross_entropy(x, w, labels, *, reduction="mean", ignore_index=-100,
                               label_smoothing=0.0, lse_square_scale=0.0, softcap=0.0,
                               chunk_rows=0):
    """Cross-entropy of the logits x.w^T against int64 labels, differentiable in
    x and w (reduction sum or mean through autograd)."""
    return _FLCEFunction.apply(x, w, labels, reduction, int(ignore_index),
                               float(label_smoothing), float(lse_square_scale), float(softcap),
                               int(chunk_rows))


__all__ = ["FusedLinearJSD", "fused_linear_jsd", "jsd_logspace", "tvd",
           "FusedLinearCrossEntropy", "fused_linear_cross_entropy", "_lib"]
