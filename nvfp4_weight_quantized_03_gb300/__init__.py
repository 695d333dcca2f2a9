"""Python binding of libqerl (C ABI in include/qerl.h): NVFP4 weight-only
linear with a LoRA branch and Adaptive Quantization Noise on GB300.

Argument marshalling only: every function hands raw device pointers, sizes
and the current CUDA stream to the C library, whose CUDA kernels do all the
work.  There is no CPU path; if libqerl.so is missing every call raises.

The functions named like the C entry points take torch tensors:

    qerl_nvfp4_quantize(W, codes, scales, tensor_scale, workspace)
    qerl_nvfp4_quantize_with_scale(W, tensor_scale, codes, scales, workspace)
    qerl_nvfp4_amax(W, amax, workspace)
    qerl_aqn_sigma(stage, num_stages, sigma_start, sigma_end)       (host)
    qerl_aqn_stage(step, total_steps, num_stages)                   (host)
    qerl_aqn_sigma_schedule(schedule, stage, num_stages, ...)       (host)
    qerl_aqn_sample(z, sigma, seed, stream_id, counter)
    qerl_nvfp4_packed_size(n, k)                                    (host)
    qerl_nvfp4_pack(codes, scales, packed)
    qerl_lora_linear(x, wpacked, tensor_scale, z, A, B, alpha, y, workspace)
    qerl_lora_linear_noalloc(x, wpacked, tensor_scale, z, A, B, alpha, y)
    qerl_lora_linear_group(x, z, [(wpacked, tensor_scale, A, B, alpha, y), ...], workspace)
    qerl_read_status(workspace)

`linear_descs()` builds the descriptor array of a group once; passing it
instead of the list skips that marshalling on every call.

and return the qerl_status integer (QERL_OK == 0).  `check()` turns a
non-zero status into an exception.  `quantize()`, `pack()` and
`lora_linear()` are conveniences that allocate the outputs with torch (the
library itself never allocates).
"""
import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "QERL_OK", "QERL_F32", "QERL_BF16", "QerlError", "check", "lib", "lib_path", "status_string",
    "qerl_nvfp4_quantize", "qerl_nvfp4_quantize_with_scale", "qerl_nvfp4_amax",
    "qerl_nvfp4_quantize_workspace_size", "qerl_aqn_sigma", "qerl_aqn_stage", "qerl_aqn_sample",
    "qerl_aqn_sigma_schedule", "QERL_SCHEDULE_EXPONENTIAL", "QERL_SCHEDULE_LINEAR", "QERL_SCHEDULE_COSINE",
    "QERL_SCHEDULE_LOGARITHMIC",
    "qerl_nvfp4_packed_size", "qerl_nvfp4_pack", "pack",
    "qerl_lora_linear_workspace_size", "qerl_lora_linear", "qerl_lora_linear_noalloc", "qerl_read_status",
    "qerl_lora_linear_group", "qerl_lora_linear_group_workspace_size", "LinearDesc", "linear_descs",
    "quantize", "lora_linear", "workspace",
]

class LinearDesc(ctypes.Structure):
    """Mirror of qerl_linear_desc (include/qerl.h)."""
    _fields_ = [("wpacked", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p), ("n", ctypes.c_int64),
                ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("r", ctypes.c_int), ("alpha", ctypes.c_float),
                ("y", ctypes.c_void_p), ("y_dtype", ctypes.c_int), ("w_format", ctypes.c_int)]


QERL_OK = 0
QERL_F32, QERL_BF16 = 0, 1
QERL_W_NVFP4, QERL_W_NF4 = 0, 1
QERL_SCHEDULE_EXPONENTIAL, QERL_SCHEDULE_LINEAR, QERL_SCHEDULE_COSINE, QERL_SCHEDULE_LOGARITHMIC = 0, 1, 2, 3
STATUS_NAMES = {0: "QERL_OK", 1: "QERL_ERR_INVALID_ARGUMENT", 2: "QERL_ERR_UNSUPPORTED_SHAPE",
                3: "QERL_ERR_MISALIGNED", 4: "QERL_ERR_CUDA", 5: "QERL_ERR_TIMEOUT", 6: "QERL_ERR_NONFINITE",
                7: "QERL_ERR_WORKSPACE", 8: "QERL_ERR_RANGE"}

_lib = None
_lock = threading.Lock()
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


class QerlError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded libqerl.so.  Raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libqerl.so not built at {_build.LIB}; run "
                                   "nvfp4_weight_quantized_03_gb300.build.build() (nvcc, sm_103a)")
            L = ctypes.CDLL(_build.LIB)
            L.qerl_status_string.restype = ctypes.c_char_p
            L.qerl_status_string.argtypes = [ctypes.c_int]
            L.qerl_version.restype = ctypes.c_int
            L.qerl_version.argtypes = []
            L.qerl_nvfp4_quantize_workspace_size.restype = ctypes.c_size_t
            L.qerl_nvfp4_quantize_workspace_size.argtypes = []
            L.qerl_nvfp4_quantize.restype = ctypes.c_int
            L.qerl_nvfp4_quantize.argtypes = [_vp, ctypes.c_int, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                              ctypes.c_size_t, _vp]
            L.qerl_nvfp4_quantize_with_scale.restype = ctypes.c_int
            L.qerl_nvfp4_quantize_with_scale.argtypes = [_vp, ctypes.c_int, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                                         ctypes.c_size_t, _vp]
            L.qerl_nvfp4_pack_transposed.restype = ctypes.c_int
            L.qerl_nvfp4_pack_transposed.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp]
            L.qerl_lora_linear_backward_workspace_size.restype = ctypes.c_size_t
            L.qerl_lora_linear_backward_workspace_size.argtypes = [_i64, _i64, _i64, ctypes.c_int]
            L.qerl_lora_linear_backward.restype = ctypes.c_int
            L.qerl_lora_linear_backward.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _vp,
                                                    ctypes.c_int, ctypes.c_float, _vp, ctypes.c_int, _vp, _vp, _vp,
                                                    ctypes.c_size_t, _vp]
            L.qerl_nf4_quantize.restype = ctypes.c_int
            L.qerl_nf4_quantize.argtypes = [_vp, ctypes.c_int, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                            ctypes.c_size_t, _vp]
            L.qerl_mxfp4_quantize.restype = ctypes.c_int
            L.qerl_mxfp4_quantize.argtypes = [_vp, ctypes.c_int, _i64, _i64, _i64, _vp, _vp, _vp, ctypes.c_size_t,
                                              _vp]
            L.qerl_mxfp4_pack.restype = ctypes.c_int
            L.qerl_mxfp4_pack.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp, _vp, ctypes.c_size_t, _vp]
            L.qerl_nvfp4_amax.restype = ctypes.c_int
            L.qerl_nvfp4_amax.argtypes = [_vp, ctypes.c_int, _i64, _i64, _i64, _vp, _vp, ctypes.c_size_t, _vp]
            L.qerl_aqn_sigma.restype = ctypes.c_double
            L.qerl_aqn_sigma.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double]
            L.qerl_aqn_sigma_schedule.restype = ctypes.c_double
            L.qerl_aqn_sigma_schedule.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                  ctypes.c_double]
            L.qerl_aqn_stage.restype = ctypes.c_int
            L.qerl_aqn_stage.argtypes = [_i64, _i64, ctypes.c_int]
            L.qerl_aqn_sample.restype = ctypes.c_int
            L.qerl_aqn_sample.argtypes = [_vp, _i64, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32,
                                          ctypes.c_uint64, _vp]
            L.qerl_nvfp4_packed_size.restype = ctypes.c_size_t
            L.qerl_nvfp4_packed_size.argtypes = [_i64, _i64]
            L.qerl_nvfp4_pack.restype = ctypes.c_int
            L.qerl_nvfp4_pack.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp]
            L.qerl_lora_linear_workspace_size.restype = ctypes.c_size_t
            L.qerl_lora_linear_workspace_size.argtypes = [_i64, _i64, _i64, ctypes.c_int]
            L.qerl_lora_linear.restype = ctypes.c_int
            L.qerl_lora_linear.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _vp, _vp, _vp, ctypes.c_int,
                                           ctypes.c_float, _vp, ctypes.c_int, _vp, ctypes.c_size_t, _vp]
            L.qerl_lora_linear_group_workspace_size.restype = ctypes.c_size_t
            L.qerl_lora_linear_group_workspace_size.argtypes = [_i64, _i64, ctypes.POINTER(LinearDesc), ctypes.c_int]
            L.qerl_lora_linear_group.restype = ctypes.c_int
            L.qerl_lora_linear_group.argtypes = [_vp, _i64, _i64, _i64, _vp, ctypes.POINTER(LinearDesc), ctypes.c_int,
                                                 _vp, ctypes.c_size_t, _vp]
            L.qerl_nvfp4_tensor_scale.restype = ctypes.c_int
            L.qerl_nvfp4_tensor_scale.argtypes = [_vp, _vp, _vp]
            L.qerl_lora_linear_group_rowz.restype = ctypes.c_int
            L.qerl_lora_linear_group_rowz.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, ctypes.POINTER(LinearDesc),
                                                      ctypes.c_int, _vp, ctypes.c_size_t, _vp]
            L.qerl_rmsnorm_lora_linear_group_workspace_size.restype = ctypes.c_size_t
            L.qerl_rmsnorm_lora_linear_group_workspace_size.argtypes = [_i64, _i64, ctypes.POINTER(LinearDesc),
                                                                        ctypes.c_int]
            L.qerl_rmsnorm_lora_linear_group.restype = ctypes.c_int
            L.qerl_rmsnorm_lora_linear_group.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, ctypes.c_double,
                                                         ctypes.POINTER(LinearDesc), ctypes.c_int, _vp,
                                                         ctypes.c_size_t, _vp]
            L.qerl_rmsnorm_noise.restype = ctypes.c_int
            L.qerl_rmsnorm_noise.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, ctypes.c_double, _vp, _i64, _vp]
            L.qerl_lora_linear_noalloc.restype = ctypes.c_int
            L.qerl_lora_linear_noalloc.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _vp, _vp, _vp,
                                                   ctypes.c_int, ctypes.c_float, _vp, ctypes.c_int, _vp]
            L.qerl_read_status.restype = ctypes.c_int
            L.qerl_read_status.argtypes = [_vp, _vp]
            _lib = L
    return _lib


def status_string(st: int) -> str:
    return lib().qerl_status_string(int(st)).decode()


def check(st: int, where: str = "qerl") -> None:
    if st != QERL_OK:
        raise QerlError(st, where)


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _wdtype(W):
    if W.dtype == torch.float32:
        return QERL_F32
    if W.dtype == torch.bfloat16:
        return QERL_BF16
    raise TypeError("W must be float32 or bfloat16")


def _nbytes(t):
    return t.numel() * t.element_size()


# ---- C entry points ---------------------------------------------------------

def qerl_nvfp4_quantize_workspace_size() -> int:
    return lib().qerl_nvfp4_quantize_workspace_size()


def qerl_nvfp4_quantize(W, codes, scales, tensor_scale, workspace, stream=None) -> int:
    n, k = W.shape
    return lib().qerl_nvfp4_quantize(_p(W), _wdtype(W), n, k, W.stride(0), _p(codes), _p(scales),
                                     _p(tensor_scale), _p(workspace), _nbytes(workspace), _stream(stream))


def qerl_nvfp4_quantize_with_scale(W, tensor_scale, codes, scales, workspace, stream=None) -> int:
    n, k = W.shape
    return lib().qerl_nvfp4_quantize_with_scale(_p(W), _wdtype(W), n, k, W.stride(0), _p(tensor_scale),
                                                _p(codes), _p(scales), _p(workspace), _nbytes(workspace),
                                                _stream(stream))


def qerl_nvfp4_amax(W, amax, workspace, stream=None) -> int:
    n, k = W.shape
    return lib().qerl_nvfp4_amax(_p(W), _wdtype(W), n, k, W.stride(0), _p(amax), _p(workspace),
                                 _nbytes(workspace), _stream(stream))


def qerl_nvfp4_tensor_scale(amax, tensor_scale, stream=None) -> int:
    return lib().qerl_nvfp4_tensor_scale(_p(amax), _p(tensor_scale), _stream(stream))


def global_amax(amax, group=None):
    """All-reduce(max) of a shard's amax (a one-element float tensor, in place) over the
    process group: with it, qerl_nvfp4_tensor_scale and qerl_nvfp4_quantize_with_scale give
    every shard the codes and scales of the whole tensor.  Plain torch.distributed
    plumbing (any backend: gloo for CPU tensors, NCCL for device tensors)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    return amax


def qerl_aqn_sigma(stage: int, num_stages: int, sigma_start: float = 1e-2, sigma_end: float = 5e-4) -> float:
    return lib().qerl_aqn_sigma(int(stage), int(num_stages), float(sigma_start), float(sigma_end))


def qerl_aqn_sigma_schedule(schedule: int, stage: int, num_stages: int, sigma_start: float = 1e-2,
                            sigma_end: float = 5e-4) -> float:
    return lib().qerl_aqn_sigma_schedule(int(schedule), int(stage), int(num_stages), float(sigma_start),
                                         float(sigma_end))


def qerl_aqn_stage(step: int, total_steps: int, num_stages: int) -> int:
    return lib().qerl_aqn_stage(int(step), int(total_steps), int(num_stages))


def qerl_aqn_sample(z, sigma: float, seed: int, stream_id: int = 0, counter: int = 0, stream=None) -> int:
    return lib().qerl_aqn_sample(_p(z), z.numel(), float(sigma), int(seed) & (2**64 - 1),
                                 int(stream_id) & 0xFFFFFFFF, int(counter) & (2**64 - 1), _stream(stream))


def qerl_nvfp4_packed_size(n: int, k: int) -> int:
    return lib().qerl_nvfp4_packed_size(int(n), int(k))


def qerl_nvfp4_pack(codes, scales, packed, stream=None) -> int:
    """codes [n, k/2], scales [n, k/16] (uint8) -> packed (uint8, qerl_nvfp4_packed_size(n, k) bytes)."""
    n = codes.shape[0]
    k = codes.shape[1] * 2
    return lib().qerl_nvfp4_pack(_p(codes), _p(scales), n, k, _p(packed), _stream(stream))


def qerl_nvfp4_pack_transposed(codes, scales, packed_t, stream=None) -> int:
    """codes [n, k/2], scales [n, k/16] -> the transposed packed layout (qerl_nvfp4_packed_size(k, n) bytes)."""
    n = codes.shape[0]
    k = codes.shape[1] * 2
    return lib().qerl_nvfp4_pack_transposed(_p(codes), _p(scales), n, k, _p(packed_t), _stream(stream))


def qerl_lora_linear_backward_workspace_size(m: int, n: int, k: int, r: int) -> int:
    return lib().qerl_lora_linear_backward_workspace_size(int(m), int(n), int(k), int(r))


def qerl_lora_linear_backward(xt, dy, wpacked_t, tensor_scale, A, B, alpha, dxt, dA, dB, workspace,
                              stream=None) -> int:
    """xt [m, k] bf16 (the forward's x~), dy [m, n] bf16, wpacked_t from qerl_nvfp4_pack_transposed;
    dxt [m, k] bf16/fp32; dA [r, k], dB [n, r] fp32 or None."""
    m, n = dy.shape
    k = dxt.shape[1]
    r = 0 if A is None else A.shape[0]
    ddt = QERL_F32 if dxt.dtype == torch.float32 else QERL_BF16
    ldxt = xt.stride(0) if xt is not None else k
    return lib().qerl_lora_linear_backward(_p(xt), m, k, ldxt, _p(dy), n, dy.stride(0), _p(wpacked_t),
                                           _p(tensor_scale), _p(A), _p(B), r, float(alpha), _p(dxt), ddt, _p(dA),
                                           _p(dB), _p(workspace), _nbytes(workspace), _stream(stream))


def qerl_nf4_quantize(W, codes, scales, tensor_scale, workspace, stream=None) -> int:
    """W [n, k] f32/bf16 -> NF4 codes [n, k/2], E4M3 scales [n, k/16], tensor scale (the layout of
    qerl_nvfp4_quantize, so qerl_nvfp4_pack packs it; the linear takes w_format QERL_W_NF4)."""
    n, k = W.shape
    return lib().qerl_nf4_quantize(_p(W), _wdtype(W), n, k, W.stride(0), _p(codes), _p(scales), _p(tensor_scale),
                                   _p(workspace), _nbytes(workspace), _stream(stream))


def qerl_mxfp4_quantize(W, codes, scales, workspace, stream=None) -> int:
    """W [n, k] f32/bf16 -> codes [n, k/2], E8M0 scales [n, k/32] (uint8)."""
    n, k = W.shape
    return lib().qerl_mxfp4_quantize(_p(W), _wdtype(W), n, k, W.stride(0), _p(codes), _p(scales), _p(workspace),
                                     _nbytes(workspace), _stream(stream))


def qerl_mxfp4_pack(codes, scales, packed, tensor_scale, workspace, stream=None) -> int:
    """codes [n, k/2], E8M0 scales [n, k/32] -> packed (qerl_nvfp4_packed_size(n, k) bytes) and the
    power-of-two tensor scale the linear applies."""
    n = codes.shape[0]
    k = codes.shape[1] * 2
    return lib().qerl_mxfp4_pack(_p(codes), _p(scales), n, k, _p(packed), _p(tensor_scale), _p(workspace),
                                 _nbytes(workspace), _stream(stream))


def qerl_lora_linear_workspace_size(m: int, n: int, k: int, r: int) -> int:
    return lib().qerl_lora_linear_workspace_size(int(m), int(n), int(k), int(r))


def qerl_lora_linear(x, wpacked, tensor_scale, z, A, B, alpha, y, workspace, stream=None) -> int:
    """x [m, k] bf16; wpacked: the n x k weight packed by qerl_nvfp4_pack; y [m, n] (n taken from y);
    A: [r, k] bf16 (LoRA down-projection), B: [n, r] bf16 (LoRA up-projection)."""
    m, k = x.shape
    n = y.shape[1]
    r = 0 if A is None else A.shape[0]
    ydt = QERL_F32 if y.dtype == torch.float32 else QERL_BF16
    return lib().qerl_lora_linear(_p(x), m, k, x.stride(0), _p(wpacked), _p(tensor_scale), n, _p(z), _p(A), _p(B),
                                  r, float(alpha), _p(y), ydt, _p(workspace), _nbytes(workspace), _stream(stream))


def qerl_lora_linear_noalloc(x, wpacked, tensor_scale, z, A, B, alpha, y, stream=None) -> int:
    """qerl_lora_linear without a workspace, for callers that cannot allocate
    device memory at the call site; the library's own fixed scratch array is
    used (shared by all calls: keep them ordered)."""
    m, k = x.shape
    n = y.shape[1]
    r = 0 if A is None else A.shape[0]
    ydt = QERL_F32 if y.dtype == torch.float32 else QERL_BF16
    return lib().qerl_lora_linear_noalloc(_p(x), m, k, x.stride(0), _p(wpacked), _p(tensor_scale), n, _p(z),
                                          _p(A), _p(B), r, float(alpha), _p(y), ydt, _stream(stream))


def _descs(linears):
    """[(wpacked, tensor_scale, A, B, alpha, y[, w_format]), ...] -> ctypes array of LinearDesc
    (an array built before is passed through)."""
    if isinstance(linears, ctypes.Array):
        return linears
    arr = (LinearDesc * len(linears))()
    for d, item in zip(arr, linears):
        wp, ts, A, B, alpha, y = item[:6]
        d.w_format = int(item[6]) if len(item) > 6 else QERL_W_NVFP4
        d.wpacked, d.tensor_scale, d.n = _p(wp), _p(ts), y.shape[1]
        d.A, d.B, d.r = _p(A), _p(B), 0 if A is None else A.shape[0]
        d.alpha, d.y = float(alpha), _p(y)
        d.y_dtype = QERL_F32 if y.dtype == torch.float32 else QERL_BF16
    return arr


def linear_descs(linears):
    """The qerl_linear_desc array of a group, [(wpacked, tensor_scale, A, B, alpha, y), ...],
    built once: the array holds raw pointers, so the tensors must outlive it."""
    return _descs(linears)


def qerl_lora_linear_group_workspace_size(m: int, k: int, linears) -> int:
    arr = _descs(linears)
    return lib().qerl_lora_linear_group_workspace_size(int(m), int(k), arr, len(arr))


def qerl_lora_linear_group(x, z, linears, workspace, stream=None) -> int:
    """Up to four linears of one input x [m, k] (bf16) and noise z: linears is a list of
    (wpacked, tensor_scale, A, B, alpha, y) with y [m, n_i], or its linear_descs() array;
    one launch for all."""
    m, k = x.shape
    arr = _descs(linears)
    return lib().qerl_lora_linear_group(_p(x), m, k, x.stride(0), _p(z), arr, len(arr), _p(workspace),
                                        _nbytes(workspace), _stream(stream))


def qerl_lora_linear_group_rowz(x, z, linears, workspace, stream=None) -> int:
    """The grouped linear with per-row noise: z is None, a [k] vector (every row), or [m, k]
    float32 (row i of x uses z[i]; its row stride is passed)."""
    m, k = x.shape
    arr = _descs(linears)
    ldz = 0 if z is None or z.dim() == 1 else z.stride(0)
    return lib().qerl_lora_linear_group_rowz(_p(x), m, k, x.stride(0), _p(z), ldz, arr, len(arr), _p(workspace),
                                             _nbytes(workspace), _stream(stream))


def qerl_rmsnorm_lora_linear_group_workspace_size(m: int, k: int, linears) -> int:
    arr = _descs(linears)
    return lib().qerl_rmsnorm_lora_linear_group_workspace_size(int(m), int(k), arr, len(arr))


def qerl_rmsnorm_lora_linear_group(h, w_norm, Z, delta, linears, workspace, stream=None) -> int:
    """RMSNorm of h [m, k] (bf16) with the noise Z [k] (float32, or None) merged into its
    weight w_norm [k] (bf16), then the grouped linear of the result."""
    m, k = h.shape
    arr = _descs(linears)
    return lib().qerl_rmsnorm_lora_linear_group(_p(h), m, k, h.stride(0), _p(w_norm), _p(Z), float(delta), arr,
                                                len(arr), _p(workspace), _nbytes(workspace), _stream(stream))


def qerl_rmsnorm_noise(h, w_norm, Z, delta, out, stream=None) -> int:
    """The normalisation step alone: out [m, k] bf16 = bf16((w_norm + Z) * h / rms(h))."""
    m, k = h.shape
    return lib().qerl_rmsnorm_noise(_p(h), m, k, h.stride(0), _p(w_norm), _p(Z), float(delta), _p(out),
                                    out.stride(0), _stream(stream))


def qerl_read_status(workspace, stream=None) -> int:
    return lib().qerl_read_status(_p(workspace), _stream(stream))


# ---- conveniences (allocation by torch; compute by the library) -------------

def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled, 256-byte aligned device workspace of at least nbytes."""
    return torch.zeros(max(256, (nbytes + 255) // 256 * 256), dtype=torch.uint8, device=device or "cuda")


def quantize(W: torch.Tensor, ws: torch.Tensor = None):
    """NVFP4-quantize an n x k float32/bfloat16 CUDA tensor -> (codes, scales, tensor_scale)."""
    n, k = W.shape
    codes = torch.empty((n, k // 2), dtype=torch.uint8, device=W.device)
    scales = torch.empty((n, k // 16), dtype=torch.uint8, device=W.device)
    ts = torch.empty(1, dtype=torch.float32, device=W.device)
    ws = workspace(qerl_nvfp4_quantize_workspace_size(), W.device) if ws is None else ws
    check(qerl_nvfp4_quantize(W, codes, scales, ts, ws), "qerl_nvfp4_quantize")
    return codes, scales, ts


def pack(codes: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """Packed (kernel-native) form of quantized weights, for qerl_lora_linear."""
    n, k = codes.shape[0], codes.shape[1] * 2
    packed = torch.empty(qerl_nvfp4_packed_size(n, k), dtype=torch.uint8, device=codes.device)
    check(qerl_nvfp4_pack(codes, scales, packed), "qerl_nvfp4_pack")
    return packed


def pack_transposed(codes: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """The transposed packed layout of quantized weights, for qerl_lora_linear_backward."""
    n, k = codes.shape[0], codes.shape[1] * 2
    packed = torch.empty(qerl_nvfp4_packed_size(k, n), dtype=torch.uint8, device=codes.device)
    check(qerl_nvfp4_pack_transposed(codes, scales, packed), "qerl_nvfp4_pack_transposed")
    return packed


def nf4_quantize(W: torch.Tensor, ws: torch.Tensor = None):
    """NF4-quantize an n x k float32/bfloat16 CUDA tensor -> (codes, scales, tensor_scale)."""
    n, k = W.shape
    codes = torch.empty((n, k // 2), dtype=torch.uint8, device=W.device)
    scales = torch.empty((n, k // 16), dtype=torch.uint8, device=W.device)
    ts = torch.empty(1, dtype=torch.float32, device=W.device)
    ws = workspace(qerl_nvfp4_quantize_workspace_size(), W.device) if ws is None else ws
    check(qerl_nf4_quantize(W, codes, scales, ts, ws), "qerl_nf4_quantize")
    return codes, scales, ts


def mxfp4_quantize(W: torch.Tensor, ws: torch.Tensor = None):
    """MXFP4-quantize an n x k float32/bfloat16 CUDA tensor -> (codes, E8M0 scales)."""
    n, k = W.shape
    codes = torch.empty((n, k // 2), dtype=torch.uint8, device=W.device)
    scales = torch.empty((n, k // 32), dtype=torch.uint8, device=W.device)
    ws = workspace(qerl_nvfp4_quantize_workspace_size(), W.device) if ws is None else ws
    check(qerl_mxfp4_quantize(W, codes, scales, ws), "qerl_mxfp4_quantize")
    return codes, scales


def mxfp4_pack(codes: torch.Tensor, scales: torch.Tensor, ws: torch.Tensor = None):
    """Packed form of an MXFP4 weight for qerl_lora_linear -> (packed, tensor_scale)."""
    n, k = codes.shape[0], codes.shape[1] * 2
    packed = torch.empty(qerl_nvfp4_packed_size(n, k), dtype=torch.uint8, device=codes.device)
    ts = torch.empty(1, dtype=torch.float32, device=codes.device)
    ws = workspace(qerl_nvfp4_quantize_workspace_size(), codes.device) if ws is None else ws
    check(qerl_mxfp4_pack(codes, scales, packed, ts, ws), "qerl_mxfp4_pack")
    return packed, ts


def lora_linear(x, wpacked, tensor_scale, n, z=None, A=None, B=None, alpha=0.0, out_dtype=torch.bfloat16,
                ws=None):
    """y = x~ . dequant(W)^T + (alpha/r) (x~ A^T) B^T, x~ = bf16(x(1+z)), for bf16 x [m, k],
    W n x k packed by pack(), A [r, k], B [n, r]."""
    m, k = x.shape
    r = 0 if A is None else A.shape[0]
    y = torch.empty((m, n), dtype=out_dtype, device=x.device)
    ws = workspace(qerl_lora_linear_workspace_size(m, n, k, r), x.device) if ws is None else ws
    check(qerl_lora_linear(x, wpacked, tensor_scale, z, A, B, alpha, y, ws), "qerl_lora_linear")
    return y
