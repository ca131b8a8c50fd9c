"""ctypes binding of ``libmt_rowreduce.so`` (argument marshalling only).

Every function named ``mt_*`` here calls the C function of the same name in
``include/mt_rowreduce.h``.  Pointer arguments accept a CUDA ``torch.Tensor``
(FP32 / int32, contiguous), a raw integer device address, or ``None`` for
NULL; ``stream`` accepts a ``torch.cuda.Stream``, a raw handle, or ``None``
for torch's current stream.  A status other than ``MT_OK`` raises
:class:`MTError`.  All computation happens in the library's CUDA kernels;
there is no fallback of any kind: if the library is not built, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmt_rowreduce.so")

MT_OK = 0
MT_ERR_INVALID_ARGUMENT = 1
MT_ERR_UNSUPPORTED = 2
MT_ERR_OUT_OF_RESOURCES = 3
MT_ERR_CUDA = 4

MT_OP_RMSNORM = 0
MT_OP_LAYERNORM = 1
MT_OP_RESIDUAL_LAYERNORM = 2
MT_OP_SOFTMAX = 3
MT_OP_ROW_SUM = 4
MT_OP_CROSS_ENTROPY = 5
MT_OP_RESIDUAL_RMSNORM = 6
MT_OP_LOG_SOFTMAX = 7
OP_IDS = {"rmsnorm": 0, "layernorm": 1, "residual_layernorm": 2,
          "softmax": 3, "row_sum": 4, "cross_entropy": 5,
          "residual_rmsnorm": 6, "log_softmax": 7}
MT_NO_IGNORE_INDEX = -(2 ** 31)

MT_DTYPE_F32 = 0
MT_DTYPE_F16 = 1
MT_DTYPE_BF16 = 2
DTYPE_IDS = {"f32": 0, "f16": 1, "bf16": 2}

MT_PATH_REGISTERS = 0
MT_PATH_LOOP = 1
MT_PATH_STAGE = 2

MT_PLAN_PDL = 1
MT_PLAN_PREFETCH_NEXT = 2
MT_PLAN_WHOLE_TILES = 4

# Symbols declared in include/mt_rowreduce.h.
EXPORTS = (
    "mt_rmsnorm_f32", "mt_rmsnorm_f32_with_plan",
    "mt_layernorm_f32", "mt_layernorm_f32_with_plan",
    "mt_residual_layernorm_f32", "mt_residual_layernorm_f32_with_plan",
    "mt_softmax_f32", "mt_softmax_f32_with_plan",
    "mt_row_sum_f32", "mt_row_sum_f32_with_plan",
    "mt_cross_entropy_f32", "mt_cross_entropy_f32_with_plan",
    "mt_plan_query", "mt_plan_check", "mt_private_slot_bound",
    "mt_describe_plan", "mt_status_string", "mt_last_cuda_error",
    "mt_stage_wait_timeouts",
    "mt_rmsnorm_f16", "mt_rmsnorm_bf16", "mt_layernorm_f16",
    "mt_layernorm_bf16", "mt_residual_layernorm_f16",
    "mt_residual_layernorm_bf16", "mt_softmax_f16", "mt_softmax_bf16",
    "mt_row_sum_f16", "mt_row_sum_bf16", "mt_cross_entropy_f16",
    "mt_cross_entropy_bf16", "mt_row_reduce_with_plan",
    "mt_plan_query_dtype", "mt_plan_check_dtype",
    "mt_residual_rmsnorm_f32", "mt_residual_rmsnorm_f32_with_plan",
    "mt_residual_rmsnorm_f16", "mt_residual_rmsnorm_bf16",
    "mt_log_softmax_f32", "mt_log_softmax_f32_with_plan",
    "mt_log_softmax_f16", "mt_log_softmax_bf16",
    "mt_cross_entropy_ignore_f32", "mt_cross_entropy_ignore_f16",
    "mt_cross_entropy_ignore_bf16",
    "mt_probe_copy", "mt_probe_read", "mt_probe_empty",
)


class MtPlan(ctypes.Structure):
    """``mt_plan_t``."""
    _fields_ = [("threads_per_row", ctypes.c_int32),
                ("values_per_thread", ctypes.c_int32),
                ("chunks", ctypes.c_int32),
                ("rows_per_block", ctypes.c_int32),
                ("path", ctypes.c_int32),
                ("grid", ctypes.c_int32),
                ("flags", ctypes.c_int32),
                ("cluster", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}

    def __repr__(self):
        return f"MtPlan({self.as_dict()})"


def make_plan(W, V, chunks=0, rows_per_block=1, path=MT_PATH_REGISTERS,
              grid=0, flags=0, cluster=0) -> MtPlan:
    return MtPlan(W, V, chunks, rows_per_block, path, grid, flags, cluster)


class MTError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {status_string(status)}"
        if status == MT_ERR_CUDA:
            msg += f" (cudaError {lib().mt_last_cuda_error()})"
        super().__init__(msg)


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library {LIB_PATH} is not built; run "
                    "row_reduction_gb300.build.build() (or "
                    "__graft_entry__.build()) first")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I32, F = (ctypes.c_void_p, ctypes.c_int64,
                              ctypes.c_int32, ctypes.c_float)
            PP = ctypes.POINTER(MtPlan)
            st = ctypes.c_int
            sig = {
                "mt_rmsnorm_f32": [P, P, P, I64, I64, F, P],
                "mt_rmsnorm_f32_with_plan": [P, P, P, I64, I64, F, P, PP],
                "mt_layernorm_f32": [P, P, P, P, I64, I64, F, P],
                "mt_layernorm_f32_with_plan": [P, P, P, P, I64, I64, F, P,
                                               PP],
                "mt_residual_layernorm_f32": [P, P, P, P, P, P, I64, I64, F,
                                              P],
                "mt_residual_layernorm_f32_with_plan": [P, P, P, P, P, P, I64,
                                                        I64, F, P, PP],
                "mt_softmax_f32": [P, P, I64, I64, P],
                "mt_softmax_f32_with_plan": [P, P, I64, I64, P, PP],
                "mt_row_sum_f32": [P, P, I64, I64, P],
                "mt_row_sum_f32_with_plan": [P, P, I64, I64, P, PP],
                "mt_cross_entropy_f32": [P, P, P, P, I64, I64, P],
                "mt_cross_entropy_f32_with_plan": [P, P, P, P, I64, I64, P,
                                                   PP],
                "mt_plan_query": [ctypes.c_int, I64, I64, PP],
                "mt_plan_check": [ctypes.c_int, I64, PP],
                "mt_row_reduce_with_plan": [ctypes.c_int, ctypes.c_int, P, P,
                                            P, P, P, I32, P, P, P, P, I64,
                                            I64, F, P, PP],
                "mt_residual_rmsnorm_f32": [P, P, P, P, P, I64, I64, F, P],
                "mt_residual_rmsnorm_f32_with_plan": [P, P, P, P, P, I64, I64,
                                                      F, P, PP],
                "mt_log_softmax_f32": [P, P, I64, I64, P],
                "mt_log_softmax_f32_with_plan": [P, P, I64, I64, P, PP],
                "mt_cross_entropy_ignore_f32": [P, P, I32, P, P, I64, I64, P],
                "mt_plan_query_dtype": [ctypes.c_int, ctypes.c_int, I64, I64,
                                        PP],
                "mt_plan_check_dtype": [ctypes.c_int, ctypes.c_int, I64, PP],
                "mt_probe_copy": [P, P, I64, I32, I32, I32, I32, P],
                "mt_probe_read": [P, I64, P, I64, I32, I32, I32, I32, P],
                "mt_probe_empty": [I32, I32, P],
                "mt_stage_wait_timeouts": [ctypes.POINTER(ctypes.c_uint64)],
            }
            for dt in ("f16", "bf16"):
                sig.update({
                    f"mt_rmsnorm_{dt}": [P, P, P, I64, I64, F, P],
                    f"mt_layernorm_{dt}": [P, P, P, P, I64, I64, F, P],
                    f"mt_residual_layernorm_{dt}": [P, P, P, P, P, P, I64,
                                                    I64, F, P],
                    f"mt_softmax_{dt}": [P, P, I64, I64, P],
                    f"mt_row_sum_{dt}": [P, P, I64, I64, P],
                    f"mt_cross_entropy_{dt}": [P, P, P, P, I64, I64, P],
                    f"mt_cross_entropy_ignore_{dt}": [P, P, I32, P, P, I64,
                                                      I64, P],
                    f"mt_residual_rmsnorm_{dt}": [P, P, P, P, P, I64, I64, F,
                                                  P],
                    f"mt_log_softmax_{dt}": [P, P, I64, I64, P],
                })
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = st
            L.mt_private_slot_bound.argtypes = [I64, I32, I32]
            L.mt_private_slot_bound.restype = I64
            L.mt_describe_plan.argtypes = [PP, ctypes.c_char_p,
                                           ctypes.c_size_t]
            L.mt_describe_plan.restype = ctypes.c_size_t
            L.mt_status_string.argtypes = [ctypes.c_int]
            L.mt_status_string.restype = ctypes.c_char_p
            L.mt_last_cuda_error.argtypes = []
            L.mt_last_cuda_error.restype = ctypes.c_int
            _lib = L
    return _lib


# ---- marshalling ------------------------------------------------------------
def _torch_dtype(name):
    import torch
    return {"float32": torch.float32, "f32": torch.float32,
            "f16": torch.float16, "bf16": torch.bfloat16,
            "int32": torch.int32}[name]


def dtype_of(t) -> str:
    """Storage type name ("f32", "f16", "bf16") of a torch tensor."""
    import torch
    return {torch.float32: "f32", torch.float16: "f16",
            torch.bfloat16: "bf16"}[t.dtype]


def _ptr(t, name, dtype="float32"):
    """Device address of a tensor (checked), a raw int, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a CUDA tensor, int or None")
    want = _torch_dtype(dtype)
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != want:
        raise TypeError(f"{name} must be {want}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _plan(p):
    if p is None:
        return None
    if isinstance(p, MtPlan):
        return ctypes.byref(p)
    if isinstance(p, dict):
        return ctypes.byref(MtPlan(**p))
    raise TypeError("plan must be an MtPlan, a dict or None")


def _check(st, where):
    if st != MT_OK:
        raise MTError(st, where)


# ---- the C ABI, one function per entry point ---------------------------------


def mt_rmsnorm_f32_with_plan(x, weight, y, rows, cols, eps, stream=None,
                             plan=None):
    _check(lib().mt_rmsnorm_f32_with_plan(
        _ptr(x, "x"), _ptr(weight, "weight"), _ptr(y, "y"), rows, cols, eps,
        _stream(stream), _plan(plan)), "mt_rmsnorm_f32_with_plan")




def mt_layernorm_f32_with_plan(x, gamma, beta, y, rows, cols, eps,
                               stream=None, plan=None):
    _check(lib().mt_layernorm_f32_with_plan(
        _ptr(x, "x"), _ptr(gamma, "gamma"), _ptr(beta, "beta"), _ptr(y, "y"),
        rows, cols, eps, _stream(stream), _plan(plan)),
        "mt_layernorm_f32_with_plan")




def mt_residual_layernorm_f32_with_plan(x, residual, gamma, beta, y, h_out,
                                        rows, cols, eps, stream=None,
                                        plan=None):
    _check(lib().mt_residual_layernorm_f32_with_plan(
        _ptr(x, "x"), _ptr(residual, "residual"), _ptr(gamma, "gamma"),
        _ptr(beta, "beta"), _ptr(y, "y"), _ptr(h_out, "h_out"), rows, cols,
        eps, _stream(stream), _plan(plan)),
        "mt_residual_layernorm_f32_with_plan")




def mt_softmax_f32_with_plan(x, y, rows, cols, stream=None, plan=None):
    _check(lib().mt_softmax_f32_with_plan(_ptr(x, "x"), _ptr(y, "y"), rows,
                                          cols, _stream(stream), _plan(plan)),
           "mt_softmax_f32_with_plan")




def mt_row_sum_f32_with_plan(x, out, rows, cols, stream=None, plan=None):
    _check(lib().mt_row_sum_f32_with_plan(_ptr(x, "x"), _ptr(out, "out"),
                                          rows, cols, _stream(stream),
                                          _plan(plan)),
           "mt_row_sum_f32_with_plan")




def mt_cross_entropy_f32_with_plan(logits, labels, loss, mean_loss, rows,
                                   cols, stream=None, plan=None):
    _check(lib().mt_cross_entropy_f32_with_plan(
        _ptr(logits, "logits"), _ptr(labels, "labels", "int32"),
        _ptr(loss, "loss"), _ptr(mean_loss, "mean_loss"), rows, cols,
        _stream(stream), _plan(plan)), "mt_cross_entropy_f32_with_plan")


def _half_entry_points(dt):
    def rmsnorm(x, weight, y, rows, cols, eps, stream=None):
        _check(getattr(lib(), f"mt_rmsnorm_{dt}")(
            _ptr(x, "x", dt), _ptr(weight, "weight", dt), _ptr(y, "y", dt),
            rows, cols, eps, _stream(stream)), f"mt_rmsnorm_{dt}")

    def layernorm(x, gamma, beta, y, rows, cols, eps, stream=None):
        _check(getattr(lib(), f"mt_layernorm_{dt}")(
            _ptr(x, "x", dt), _ptr(gamma, "gamma", dt),
            _ptr(beta, "beta", dt), _ptr(y, "y", dt), rows, cols, eps,
            _stream(stream)), f"mt_layernorm_{dt}")

    def residual_layernorm(x, residual, gamma, beta, y, h_out, rows, cols,
                           eps, stream=None):
        _check(getattr(lib(), f"mt_residual_layernorm_{dt}")(
            _ptr(x, "x", dt), _ptr(residual, "residual", dt),
            _ptr(gamma, "gamma", dt), _ptr(beta, "beta", dt),
            _ptr(y, "y", dt), _ptr(h_out, "h_out", dt), rows, cols, eps,
            _stream(stream)), f"mt_residual_layernorm_{dt}")

    def softmax(x, y, rows, cols, stream=None):
        _check(getattr(lib(), f"mt_softmax_{dt}")(
            _ptr(x, "x", dt), _ptr(y, "y", dt), rows, cols,
            _stream(stream)), f"mt_softmax_{dt}")

    def row_sum(x, out, rows, cols, stream=None):
        _check(getattr(lib(), f"mt_row_sum_{dt}")(
            _ptr(x, "x", dt), _ptr(out, "out"), rows, cols,
            _stream(stream)), f"mt_row_sum_{dt}")

    def cross_entropy(logits, labels, loss, mean_loss, rows, cols,
                      stream=None):
        _check(getattr(lib(), f"mt_cross_entropy_{dt}")(
            _ptr(logits, "logits", dt), _ptr(labels, "labels", "int32"),
            _ptr(loss, "loss"), _ptr(mean_loss, "mean_loss"), rows, cols,
            _stream(stream)), f"mt_cross_entropy_{dt}")
    def cross_entropy_ignore(logits, labels, ignore_index, loss, mean_loss,
                             rows, cols, stream=None):
        _check(getattr(lib(), f"mt_cross_entropy_ignore_{dt}")(
            _ptr(logits, "logits", dt), _ptr(labels, "labels", "int32"),
            ignore_index, _ptr(loss, "loss"), _ptr(mean_loss, "mean_loss"),
            rows, cols, _stream(stream)), f"mt_cross_entropy_ignore_{dt}")

    def residual_rmsnorm(x, residual, weight, y, h_out, rows, cols, eps,
                         stream=None):
        _check(getattr(lib(), f"mt_residual_rmsnorm_{dt}")(
            _ptr(x, "x", dt), _ptr(residual, "residual", dt),
            _ptr(weight, "weight", dt), _ptr(y, "y", dt),
            _ptr(h_out, "h_out", dt), rows, cols, eps, _stream(stream)),
            f"mt_residual_rmsnorm_{dt}")

    def log_softmax(x, y, rows, cols, stream=None):
        _check(getattr(lib(), f"mt_log_softmax_{dt}")(
            _ptr(x, "x", dt), _ptr(y, "y", dt), rows, cols,
            _stream(stream)), f"mt_log_softmax_{dt}")
    return (rmsnorm, layernorm, residual_layernorm, softmax, row_sum,
            cross_entropy, cross_entropy_ignore, residual_rmsnorm,
            log_softmax)


(mt_rmsnorm_f32, mt_layernorm_f32, mt_residual_layernorm_f32, mt_softmax_f32,
 mt_row_sum_f32, mt_cross_entropy_f32, mt_cross_entropy_ignore_f32,
 mt_residual_rmsnorm_f32, mt_log_softmax_f32) = _half_entry_points("f32")
(mt_rmsnorm_f16, mt_layernorm_f16, mt_residual_layernorm_f16, mt_softmax_f16,
 mt_row_sum_f16, mt_cross_entropy_f16, mt_cross_entropy_ignore_f16,
 mt_residual_rmsnorm_f16, mt_log_softmax_f16) = _half_entry_points("f16")
(mt_rmsnorm_bf16, mt_layernorm_bf16, mt_residual_layernorm_bf16,
 mt_softmax_bf16, mt_row_sum_bf16, mt_cross_entropy_bf16,
 mt_cross_entropy_ignore_bf16, mt_residual_rmsnorm_bf16,
 mt_log_softmax_bf16) = _half_entry_points("bf16")


def mt_residual_rmsnorm_f32_with_plan(x, residual, weight, y, h_out, rows,
                                      cols, eps, stream=None, plan=None):
    _check(lib().mt_residual_rmsnorm_f32_with_plan(
        _ptr(x, "x"), _ptr(residual, "residual"), _ptr(weight, "weight"),
        _ptr(y, "y"), _ptr(h_out, "h_out"), rows, cols, eps, _stream(stream),
        _plan(plan)), "mt_residual_rmsnorm_f32_with_plan")


def mt_log_softmax_f32_with_plan(x, y, rows, cols, stream=None, plan=None):
    _check(lib().mt_log_softmax_f32_with_plan(
        _ptr(x, "x"), _ptr(y, "y"), rows, cols, _stream(stream),
        _plan(plan)), "mt_log_softmax_f32_with_plan")


def mt_row_reduce_with_plan(op, dtype, x, residual=None, weight=None,
                            beta=None, labels=None, y=None, h_out=None,
                            out=None, mean_loss=None, rows=0, cols=0, eps=0.0,
                            stream=None, plan=None,
                            ignore_index=MT_NO_IGNORE_INDEX):
    """Any operator, any storage type, optional explicit plan."""
    op_id = OP_IDS.get(op, op)
    dt = dtype if isinstance(dtype, str) else \
        {v: k for k, v in DTYPE_IDS.items()}[dtype]
    _check(lib().mt_row_reduce_with_plan(
        op_id, DTYPE_IDS[dt], _ptr(x, "x", dt),
        _ptr(residual, "residual", dt), _ptr(weight, "weight", dt),
        _ptr(beta, "beta", dt), _ptr(labels, "labels", "int32"),
        ignore_index, _ptr(y, "y", dt), _ptr(h_out, "h_out", dt),
        _ptr(out, "out"),
        _ptr(mean_loss, "mean_loss"), rows, cols, eps, _stream(stream),
        _plan(plan)), "mt_row_reduce_with_plan")


def mt_plan_query_dtype(op, dtype, rows, cols) -> MtPlan:
    p = MtPlan()
    _check(lib().mt_plan_query_dtype(OP_IDS.get(op, op),
                                     DTYPE_IDS.get(dtype, dtype), rows, cols,
                                     ctypes.byref(p)), "mt_plan_query_dtype")
    return p


def mt_plan_check_dtype(op, dtype, cols, plan) -> int:
    return lib().mt_plan_check_dtype(OP_IDS.get(op, op),
                                     DTYPE_IDS.get(dtype, dtype), cols,
                                     _plan(plan))


def mt_plan_query(op, rows, cols) -> MtPlan:
    op = OP_IDS.get(op, op)
    p = MtPlan()
    _check(lib().mt_plan_query(op, rows, cols, ctypes.byref(p)),
           "mt_plan_query")
    return p


def mt_plan_check(op, cols, plan) -> int:
    """Status the *_with_plan call would return for this plan (no raise)."""
    op = OP_IDS.get(op, op)
    return lib().mt_plan_check(op, cols, _plan(plan))


def mt_private_slot_bound(n, W, V) -> int:
    return lib().mt_private_slot_bound(n, W, V)


def mt_describe_plan(plan) -> str:
    need = lib().mt_describe_plan(_plan(plan), None, 0)
    buf = ctypes.create_string_buffer(need + 1)
    lib().mt_describe_plan(_plan(plan), buf, need + 1)
    return buf.value.decode()


def status_string(st) -> str:
    return lib().mt_status_string(st).decode()


mt_status_string = status_string


def mt_last_cuda_error() -> int:
    return lib().mt_last_cuda_error()


def mt_stage_wait_timeouts() -> int:
    """Waits of the staged path that gave up on the current device (a
    diagnostic; synchronous)."""
    n = ctypes.c_uint64(0)
    _check(lib().mt_stage_wait_timeouts(ctypes.byref(n)),
           "mt_stage_wait_timeouts")
    return n.value


def mt_probe_copy(src, dst, nbytes, threads=512, unroll=4, grid=0,
                  flags=0, stream=None):
    """Measurement aid: a plain 16-byte-vector copy of `nbytes` bytes."""
    _check(lib().mt_probe_copy(_ptr(src, "src", _any_dtype(src)),
                               _ptr(dst, "dst", _any_dtype(dst)), nbytes,
                               threads, unroll, grid, flags,
                               _stream(stream)),
           "mt_probe_copy")


def mt_probe_empty(threads=32, grid=1, stream=None):
    """Measurement aid: a dependent launch that does no work."""
    _check(lib().mt_probe_empty(threads, grid, _stream(stream)),
           "mt_probe_empty")


def _any_dtype(t):
    """The storage name of a tensor argument (any of the library's types),
    so _ptr's checks apply without constraining the type."""
    if t is None or isinstance(t, int):
        return "float32"
    import torch
    return {torch.float32: "f32", torch.float16: "f16",
            torch.bfloat16: "bf16", torch.int32: "int32"}[t.dtype]
