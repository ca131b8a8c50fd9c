"""GB300 (sm_103a) per-row FP32 reductions: RMSNorm, LayerNorm, residual
LayerNorm, softmax, row sum and cross-entropy.

The computation is the CUDA library ``_lib/libmt_rowreduce.so`` (C ABI in
``include/mt_rowreduce.h``), built by :func:`row_reduction_gb300.build.build`.
``row_reduction_gb300.mt_*`` are its ctypes bindings under the C names; the
functions below allocate outputs with torch and call them.  PyTorch only
supplies device memory and streams.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    EXPORTS, LIB_PATH, MT_ERR_CUDA, MT_ERR_INVALID_ARGUMENT,
    MT_ERR_OUT_OF_RESOURCES, MT_ERR_UNSUPPORTED, MT_OK, MT_OP_CROSS_ENTROPY,
    MT_OP_LAYERNORM, MT_OP_RESIDUAL_LAYERNORM, MT_OP_RMSNORM, MT_OP_ROW_SUM,
    MT_OP_SOFTMAX, MT_PATH_LOOP, MT_PATH_REGISTERS, MT_PATH_STAGE, MT_PLAN_PDL,
    MT_PLAN_PREFETCH_NEXT, MT_PLAN_WHOLE_TILES, OP_IDS, DTYPE_IDS,
    MT_DTYPE_F32, MT_DTYPE_F16,
    MT_DTYPE_BF16, MTError, MtPlan, dtype_of, mt_row_reduce_with_plan,
    mt_plan_query_dtype, mt_plan_check_dtype, mt_rmsnorm_f16,
    mt_rmsnorm_bf16, mt_layernorm_f16, mt_layernorm_bf16,
    mt_residual_layernorm_f16, mt_residual_layernorm_bf16, mt_softmax_f16,
    mt_softmax_bf16, mt_row_sum_f16, mt_row_sum_bf16, mt_cross_entropy_f16,
    mt_cross_entropy_bf16, MT_OP_RESIDUAL_RMSNORM, MT_OP_LOG_SOFTMAX,
    MT_NO_IGNORE_INDEX, mt_residual_rmsnorm_f32,
    mt_residual_rmsnorm_f32_with_plan, mt_residual_rmsnorm_f16,
    mt_residual_rmsnorm_bf16, mt_log_softmax_f32,
    mt_log_softmax_f32_with_plan, mt_log_softmax_f16, mt_log_softmax_bf16,
    mt_cross_entropy_ignore_f32, mt_cross_entropy_ignore_f16,
    mt_cross_entropy_ignore_bf16,
    lib, make_plan, mt_cross_entropy_f32, mt_cross_entropy_f32_with_plan,
    mt_describe_plan, mt_last_cuda_error, mt_stage_wait_timeouts,
    mt_layernorm_f32,
    mt_layernorm_f32_with_plan, mt_plan_check, mt_plan_query,
    mt_private_slot_bound, mt_residual_layernorm_f32,
    mt_residual_layernorm_f32_with_plan, mt_rmsnorm_f32,
    mt_rmsnorm_f32_with_plan, mt_row_sum_f32, mt_row_sum_f32_with_plan,
    mt_softmax_f32, mt_softmax_f32_with_plan, mt_status_string,
    status_string)


def _shape(x):
    if x.dim() != 2:
        raise ValueError("x must be 2-D (rows, cols)")
    return x.shape[0], x.shape[1]


def rmsnorm(x, weight=None, eps=1e-6, out=None, plan=None, stream=None):
    """y = x / sqrt(mean(x^2) + eps) * weight, per row.  x may be FP32, FP16
    or BF16 (weight and y take x's type; arithmetic is FP32)."""
    import torch
    rows, cols = _shape(x)
    y = torch.empty_like(x) if out is None else out
    mt_row_reduce_with_plan("rmsnorm", dtype_of(x), x, weight=weight, y=y,
                            rows=rows, cols=cols, eps=eps, stream=stream,
                            plan=plan)
    return y


def layernorm(x, gamma=None, beta=None, eps=1e-5, out=None, plan=None,
              stream=None):
    """y = (x - mean) / sqrt(var + eps) * gamma + beta, per row."""
    import torch
    rows, cols = _shape(x)
    y = torch.empty_like(x) if out is None else out
    mt_row_reduce_with_plan("layernorm", dtype_of(x), x, weight=gamma,
                            beta=beta, y=y, rows=rows, cols=cols, eps=eps,
                            stream=stream, plan=plan)
    return y


def residual_layernorm(x, residual, gamma=None, beta=None, eps=1e-5,
                       out=None, h_out=None, return_h=False, plan=None,
                       stream=None):
    """y = layernorm(x + residual); with return_h also h = x + residual."""
    import torch
    rows, cols = _shape(x)
    y = torch.empty_like(x) if out is None else out
    if return_h and h_out is None:
        h_out = torch.empty_like(x)
    mt_row_reduce_with_plan("residual_layernorm", dtype_of(x), x,
                            residual=residual, weight=gamma, beta=beta, y=y,
                            h_out=h_out, rows=rows, cols=cols, eps=eps,
                            stream=stream, plan=plan)
    return (y, h_out) if return_h else y


def softmax(x, out=None, plan=None, stream=None):
    """Row-wise softmax."""
    import torch
    rows, cols = _shape(x)
    y = torch.empty_like(x) if out is None else out
    mt_row_reduce_with_plan("softmax", dtype_of(x), x, y=y, rows=rows,
                            cols=cols, stream=stream, plan=plan)
    return y


def row_sum(x, out=None, plan=None, stream=None):
    """out[r] = sum of row r (FP32 for every input type)."""
    import torch
    rows, cols = _shape(x)
    o = torch.empty(rows, dtype=torch.float32, device=x.device) \
        if out is None else out
    mt_row_reduce_with_plan("row_sum", dtype_of(x), x, out=o, rows=rows,
                            cols=cols, stream=stream, plan=plan)
    return o


def cross_entropy(logits, labels, mean=True, ignore_index=None, plan=None,
                  stream=None):
    """Per-row loss logsumexp(row) - row[label] and, with mean, its mean
    (both FP32).  Rows labelled `ignore_index` get loss 0 and leave the mean.
    Returns (loss, mean_loss) when mean is true (mean_loss a 1-element
    tensor), else loss."""
    import torch
    rows, cols = _shape(logits)
    loss = torch.empty(rows, dtype=torch.float32, device=logits.device)
    m = torch.empty(1, dtype=torch.float32, device=logits.device) if mean \
        else None
    mt_row_reduce_with_plan(
        "cross_entropy", dtype_of(logits), logits, labels=labels, out=loss,
        mean_loss=m, rows=rows, cols=cols, stream=stream, plan=plan,
        ignore_index=(MT_NO_IGNORE_INDEX if ignore_index is None
                      else ignore_index))
    return (loss, m) if mean else loss


def residual_rmsnorm(x, residual, weight=None, eps=1e-6, out=None,
                     h_out=None, return_h=False, plan=None, stream=None):
    """y = rmsnorm(x + residual) * weight; with return_h also h = x + r."""
    import torch
    rows, cols = _shape(x)
    y = torch.empty_like(x) if out is None else out
    if return_h and h_out is None:
        h_out = torch.empty_like(x)
    mt_row_reduce_with_plan("residual_rmsnorm", dtype_of(x), x,
                            residual=residual, weight=weight, y=y,
                            h_out=h_out, rows=rows, cols=cols, eps=eps,
                            stream=stream, plan=plan)
    return (y, h_out) if return_h else y


def log_softmax(x, out=None, plan=None, stream=None):
    """Row-wise log-softmax."""
    import torch
    rows, cols = _shape(x)
    y = torch.empty_like(x) if out is None else out
    mt_row_reduce_with_plan("log_softmax", dtype_of(x), x, y=y, rows=rows,
                            cols=cols, stream=stream, plan=plan)
    return y


def run(op: str, t: dict, plan=None, stream=None) -> dict:
    """Runs operator `op` on a dict of CUDA tensors named like the input
    generators' arrays (x, weight, gamma, beta, residual, labels, eps) and
    returns its outputs by name (y, h_out, out, loss, mean_loss)."""
    if op == "rmsnorm":
        return {"y": rmsnorm(t["x"], t.get("weight"), t["eps"], plan=plan,
                             stream=stream)}
    if op == "layernorm":
        return {"y": layernorm(t["x"], t.get("gamma"), t.get("beta"),
                               t["eps"], plan=plan, stream=stream)}
    if op == "residual_layernorm":
        y, h = residual_layernorm(t["x"], t["residual"], t.get("gamma"),
                                  t.get("beta"), t["eps"], return_h=True,
                                  plan=plan, stream=stream)
        return {"y": y, "h_out": h}
    if op == "softmax":
        return {"y": softmax(t["x"], plan=plan, stream=stream)}
    if op == "row_sum":
        return {"out": row_sum(t["x"], plan=plan, stream=stream)}
    if op == "cross_entropy":
        loss, m = cross_entropy(t["x"], t["labels"],
                                ignore_index=t.get("ignore_index"),
                                plan=plan, stream=stream)
        return {"loss": loss, "mean_loss": m}
    if op == "residual_rmsnorm":
        y, h = residual_rmsnorm(t["x"], t["residual"], t.get("weight"),
                                t["eps"], return_h=True, plan=plan,
                                stream=stream)
        return {"y": y, "h_out": h}
    if op == "log_softmax":
        return {"y": log_softmax(t["x"], plan=plan, stream=stream)}
    raise ValueError(f"unknown op {op!r}")
