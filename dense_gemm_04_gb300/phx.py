"""ctypes binding of libphx (include/phx.h): argument marshalling only.

Every function of the C ABI is available under its C name with raw integer pointers
(``phx_sgemm(M, N, K, alpha, A_ptr, B_ptr, beta, C_ptr, stream)`` etc.).  On top of
those, :func:`sgemm` and :func:`gemm_f16tc_f32acc` accept torch CUDA tensors and raise
:class:`PhxError` on a non-OK status.  All the arithmetic runs in libphx's CUDA kernels;
this module never computes a GEMM and has no fallback: if libphx.so was not built, importing
it raises.  PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
# PHX_LIBRARY=<path> loads another build of the same ABI (the bounds-checked one).
LIB_PATH = os.environ.get("PHX_LIBRARY") or os.path.join(_HERE, "_lib", "libphx.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "phx.h")

PHX_OK, PHX_ERR_INVALID, PHX_ERR_ARCH, PHX_ERR_LAUNCH = 0, 1, 2, 3
PHX_ERR_TIMEOUT, PHX_ERR_NOMEM, PHX_ERR_INTERNAL, PHX_ERR_CONFIG = 4, 5, 6, 7
VARIANT_SGEMM, VARIANT_F16TC = 0, 1

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python dense_gemm_04_gb300/build.py, or "
        "__graft_entry__.build()).  There is no fallback implementation.")

_lib = ctypes.CDLL(LIB_PATH)

_i64, _i32, _u64, _f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
_vp, _cp, _sz = ctypes.c_void_p, ctypes.c_char_p, ctypes.c_size_t

_SIGNATURES = {
    "phx_sgemm": (_i32, [_i64, _i64, _i64, _f32, _vp, _vp, _f32, _vp, _vp]),
    "phx_gemm_f16tc_f32acc": (_i32, [_i64, _i64, _i64, _f32, _vp, _vp, _f32, _vp, _vp]),
    "phx_gemm_f16tc_f32acc_noalloc": (_i32, [_i64, _i64, _i64, _f32, _vp, _vp, _f32, _vp, _vp]),
    "phx_sgemm_ex": (_i32, [_i32, _i32, _i64, _i64, _i64, _f32, _vp, _vp, _f32, _vp, _vp]),
    "phx_gemm_f16tc_f32acc_ex": (_i32, [_i32, _i32, _i64, _i64, _i64, _f32, _vp, _vp, _f32, _vp, _vp]),
    "phx_gemm_f16in_f32acc": (_i32, [_i32, _i32, _i64, _i64, _i64, _f32, _vp, _vp, _f32, _vp, _vp]),
    "phx_gemm_f16in_f16out": (_i32, [_i32, _i32, _i64, _i64, _i64, _f32, _vp, _vp, _f32, _vp, _vp]),
    "phx_f16tc_workspace_bytes": (_i32, [_i64, _i64, _i64, ctypes.POINTER(_sz)]),
    "phx_status_string": (_cp, [_i32]),
    "phx_check_device_status": (_i32, [_vp]),
    "phx_num_configs": (_i32, [_i32]),
    "phx_config_name": (_i32, [_i32, _i32, _cp, _sz]),
    "phx_set_config": (_i32, [_i32, _cp]),
    "phx_get_config": (_i32, [_i32, _i64, _i64, _i64, _cp, _sz]),
    "phx_last_config": (_i32, [_i32, _cp, _sz]),
    "phx_autotune": (_i32, [_i32, _i64, _i64, _i64, _i32, _i32, _i32, _vp]),
    "phx_tune_cache_save": (_i32, [_cp]),
    "phx_tune_cache_load": (_i32, [_cp]),
    "phx_device_tag": (_i32, [_cp, _sz]),
    "phx_autotune_report": (_i32, [_i32, _cp, _sz]),
    "phx_probe_ffma": (_i32, [_i32, _i64, _i32, _vp, _vp]),
    "phx_probe_stream_read": (_i32, [_vp, _i64, _vp, _i64, _vp]),
    "phx_probe_mma_f16": (_i32, [_i64, _i32, _i32, _vp, _vp]),
    "phx_selftest_bounded_wait": (_i32, [_u64, _vp]),
    "phx_selftest_bounded_wait_noalloc": (_i32, [_u64, _vp]),
    "phx_selftest_tuner": (_i32, [_i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_i32),
                                  ctypes.c_double, ctypes.c_double, _i32, _i32, _u64,
                                  ctypes.POINTER(_i32), ctypes.POINTER(_i64)]),
    "phx_selftest_sgemm_schedule": (_i32, [_i32, _i64, _i64, _i64, _i32, _i32, ctypes.POINTER(_i64)]),
    "phx_validate_args": (_i32, [_i64, _i64, _i64, _vp, _vp, _vp]),
    "phx_version": (_cp, []),
    "phx_profile_start": (_i32, []),
    "phx_debug_build": (_i32, []),
    "phx_debug_violations": (_i32, [ctypes.POINTER(_i64)]),
    "phx_profile_stop": (_i32, [ctypes.POINTER(_i64), ctypes.POINTER(ctypes.c_double)]),
}

for _name, (_res, _args) in _SIGNATURES.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args
    globals()[_name] = _fn


def declared_functions():
    """Names of the functions include/phx.h declares (for the export check)."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(phx_[a-z0-9_]+)\s*\(", text)))


class PhxError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        msg = phx_status_string(self.status).decode()
        super().__init__(f"{what}: {msg}" if what else msg)


def check(status: int, what: str = "") -> None:
    if status != PHX_OK:
        raise PhxError(status, what)


def version() -> str:
    return phx_version().decode()


def status_string(status: int) -> str:
    return phx_status_string(int(status)).decode()


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


OP_N, OP_T = 0, 1


def _operand_op(t, name):
    """PHX_OP_N for a contiguous matrix, PHX_OP_T for the transpose view of one."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D tensor")
    if t.is_contiguous():
        return OP_N
    if t.t().is_contiguous():
        return OP_T
    raise ValueError(f"{name} must be contiguous or the transpose of a contiguous matrix")


def _check_operands(A, B, C):
    """Shapes (M, N, K) and storage orders (op_a, op_b) of the GEMM's operands.  A or B may
    be the transpose view (t.t() or t.T) of a contiguous matrix; C must be contiguous."""
    import torch
    for name, t in (("A", A), ("B", B), ("C", C)):
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32, got {t.dtype}")
        if not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
    op_a, op_b = _operand_op(A, "A"), _operand_op(B, "B")
    if C.dim() != 2 or not C.is_contiguous():
        raise ValueError("C must be a contiguous 2-D tensor")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shapes do not match: A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    return M, N, K, op_a, op_b


def sgemm(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C <- alpha * A @ B + beta * C in f32 on the CUDA cores (in place; returns C).  A or B
    may be a transpose view of a contiguous matrix (stored transposed)."""
    M, N, K, op_a, op_b = _check_operands(A, B, C)
    if op_a == OP_N and op_b == OP_N:
        check(phx_sgemm(M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C.data_ptr(),
                        _stream_handle(stream)), "phx_sgemm")
    else:
        check(phx_sgemm_ex(op_a, op_b, M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C.data_ptr(),
                           _stream_handle(stream)), "phx_sgemm_ex")
    return C


def gemm_f16(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C <- alpha * A @ B + beta * C for half-precision A and B (torch.float16, contiguous or
    transpose views), summed in f32 on the tensor cores; C is float32 (phx_gemm_f16in_f32acc)
    or float16 (phx_gemm_f16in_f16out: rounded to f16 once).  In place; returns C."""
    import torch
    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float16:
            raise TypeError(f"{name} must be float16, got {t.dtype}")
        if not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
    if C.dtype not in (torch.float32, torch.float16) or not C.is_cuda:
        raise TypeError(f"C must be a float32 or float16 CUDA tensor, got {C.dtype}")
    op_a, op_b = _operand_op(A, "A"), _operand_op(B, "B")
    if C.dim() != 2 or not C.is_contiguous():
        raise ValueError("C must be a contiguous 2-D tensor")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shapes do not match: A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    fn, name = ((phx_gemm_f16in_f32acc, "phx_gemm_f16in_f32acc") if C.dtype == torch.float32
                else (phx_gemm_f16in_f16out, "phx_gemm_f16in_f16out"))
    check(fn(op_a, op_b, M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C.data_ptr(), _stream_handle(stream)),
          name)
    return C


def gemm_f16tc_f32acc(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C <- alpha * f16(A) @ f16(B) + beta * C with f32 accumulation on the tensor cores.  A or
    B may be a transpose view of a contiguous matrix (stored transposed)."""
    M, N, K, op_a, op_b = _check_operands(A, B, C)
    if op_a == OP_N and op_b == OP_N:
        check(phx_gemm_f16tc_f32acc(M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C.data_ptr(),
                                    _stream_handle(stream)), "phx_gemm_f16tc_f32acc")
    else:
        check(phx_gemm_f16tc_f32acc_ex(op_a, op_b, M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta,
                                       C.data_ptr(), _stream_handle(stream)), "phx_gemm_f16tc_f32acc_ex")
    return C


def f16tc_workspace_bytes(M: int, N: int, K: int) -> int:
    out = _sz()
    check(phx_f16tc_workspace_bytes(M, N, K, ctypes.byref(out)), "phx_f16tc_workspace_bytes")
    return int(out.value)


def check_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status as a phx_status."""
    return int(phx_check_device_status(_stream_handle(stream)))


def num_configs(variant: int) -> int:
    return int(phx_num_configs(variant))


def config_name(variant: int, index: int) -> str:
    buf = ctypes.create_string_buffer(160)
    check(phx_config_name(variant, index, buf, len(buf)), "phx_config_name")
    return buf.value.decode()


def config_names(variant: int):
    return [config_name(variant, i) for i in range(num_configs(variant))]


def set_config(variant: int, spec) -> None:
    check(phx_set_config(variant, None if spec is None else spec.encode()), "phx_set_config")


def get_config(variant: int, M: int, N: int, K: int) -> str:
    buf = ctypes.create_string_buffer(160)
    check(phx_get_config(variant, M, N, K, buf, len(buf)), "phx_get_config")
    return buf.value.decode()


def last_config(variant: int) -> str:
    """The configuration the last GEMM call of `variant` launched ("NONE" before the first)."""
    buf = ctypes.create_string_buffer(256)
    check(phx_last_config(variant, buf, 256), "phx_last_config")
    return buf.value.decode()


def autotune(variant: int, M: int, N: int, K: int, finalists: int = 4, rounds: int = 9,
             settle_ms: int = 250, stream=None) -> str:
    """Tune `variant` for (M, N, K); returns the name of the configuration chosen."""
    check(phx_autotune(variant, M, N, K, finalists, rounds, settle_ms, _stream_handle(stream)),
          "phx_autotune")
    return get_config(variant, M, N, K)


def debug_violations() -> int:
    """Failed index checks since the last call (bounds-checked build; 0 otherwise)."""
    n = _i64(0)
    check(phx_debug_violations(ctypes.byref(n)), "phx_debug_violations")
    return int(n.value)


def device_tag() -> str:
    """The current device's key in the tuning cache ("<name>:<SMs>", or "none")."""
    buf = ctypes.create_string_buffer(256)
    check(phx_device_tag(buf, len(buf)), "phx_device_tag")
    return buf.value.decode()


def autotune_report(variant: int) -> str:
    """The record of the last autotune of `variant` (finalists, median times and SM clocks)."""
    buf = ctypes.create_string_buffer(1 << 14)
    check(phx_autotune_report(variant, buf, len(buf)), "phx_autotune_report")
    return buf.value.decode()


def tune_cache_save(path: str) -> None:
    check(phx_tune_cache_save(path.encode()), "phx_tune_cache_save")


def tune_cache_load(path: str) -> None:
    check(phx_tune_cache_load(path.encode()), "phx_tune_cache_load")


def selftest_tuner(base_s, fail=None, noise=0.0, drift=0.0, finalists=4, rounds=9, seed=1):
    """Run the tuner's selection logic on simulated candidates; returns (picked, launches)."""
    n = len(base_s)
    b = (ctypes.c_double * n)(*base_s)
    f = (_i32 * n)(*(fail or [0] * n))
    picked, launches = _i32(), _i64()
    check(phx_selftest_tuner(n, b, f, noise, drift, finalists, rounds, seed,
                             ctypes.byref(picked), ctypes.byref(launches)), "phx_selftest_tuner")
    return picked.value, launches.value


KIND_SGEMM, KIND_F16_CAST, KIND_TC_GEMM, KIND_SCALE_C, KIND_TRANSPOSE, KIND_SKINNY = 0, 1, 2, 3, 4, 5
KIND_NAMES = ("sgemm", "f16_cast", "tc_gemm", "scale_c", "transpose", "skinny")


def profile_start() -> None:
    check(phx_profile_start(), "phx_profile_start")


def profile_stop():
    """Stop the profile; returns {kind name: (kernels launched, total device ms)}."""
    kinds = len(KIND_NAMES)
    n = (_i64 * kinds)()
    ms = (ctypes.c_double * kinds)()
    check(phx_profile_stop(n, ms), "phx_profile_stop")
    return {KIND_NAMES[k]: (int(n[k]), float(ms[k])) for k in range(kinds)}


def sgemm_schedule(config: str, M: int, N: int, K: int, ctas_per_sm: int = 2, num_sms: int = 152) -> dict:
    """The f32 GEMM's schedule for `config` on a GPU of `num_sms` SMs, worked out on the host
    (phx_selftest_sgemm_schedule)."""
    out = (_i64 * 6)()
    check(phx_selftest_sgemm_schedule(config_names(VARIANT_SGEMM).index(config), M, N, K, ctas_per_sm, num_sms, out),
          "phx_selftest_sgemm_schedule")
    keys = ("whole_tiles", "streamk_blocks", "streamk_k_tiles", "k_slices", "max_segments", "bookkeeping_ok")
    return dict(zip(keys, (int(v) for v in out)))


def validate_args(M, N, K, A, B, C) -> int:
    return int(phx_validate_args(M, N, K, A, B, C))
