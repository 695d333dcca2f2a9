"""Plain CPU oracle for the NVFP4 weight-only linear with LoRA and AQN.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library (``nvfp4_weight_quantized_03_gb300``) never imports it and
shares no code with it.

The arithmetic lives in ``qerl_oracle.c`` (plain C, fp64 except where an fp32
decision fixes a discrete result); this module only marshals numpy arrays
through ctypes.  bf16 data is passed as uint16 bit patterns.

Sources: "QeRL: Beyond Efficiency -- Quantization-enhanced Reinforcement
Learning for LLMs" (paper-graph-ui digest), section 3.4: "NVFP4 Quantization"
(E2M1 levels, Eq. 6), "Low-Rank Adaptation" (Eq. 2), "Adaptive Quantization
Noise" (Eq. 7, Eq. 8), "Noise Merging" (Eq. 10-12), "Algorithm 1".
"""
import ctypes
import threading

import numpy as np

from . import build as _build

_lib = None
_lock = threading.Lock()

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64

OK, ERR_ARG, ERR_SHAPE, ERR_NONFINITE = 0, 1, 2, 6


class OracleError(RuntimeError):
    pass


def lib():
    """Load (building if needed) the oracle shared library."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            L.orc_e2m1_decode.restype = ctypes.c_double
            L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            L.orc_e2m1_encode.restype = ctypes.c_uint8
            L.orc_e2m1_encode.argtypes = [ctypes.c_float]
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_encode_pos.restype = ctypes.c_uint8
            L.orc_e4m3_encode_pos.argtypes = [ctypes.c_float]
            L.orc_f64_to_bf16.restype = ctypes.c_uint16
            L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
            L.orc_f64_to_bf16_array.restype = None
            L.orc_f64_to_bf16_array.argtypes = [_f64p, _i64, _u16p]
            L.orc_nvfp4_tensor_scale.restype = ctypes.c_int
            L.orc_nvfp4_tensor_scale.argtypes = [_f32p, _i64, _i64, _i64, _f32p]
            L.orc_nvfp4_quantize_with_scale.restype = ctypes.c_int
            L.orc_nvfp4_quantize_with_scale.argtypes = [_f32p, _i64, _i64, _i64, ctypes.c_float, _u8p, _u8p]
            L.orc_nvfp4_quantize.restype = ctypes.c_int
            L.orc_nvfp4_quantize.argtypes = [_f32p, _i64, _i64, _i64, _u8p, _u8p, _f32p]
            L.orc_nvfp4_dequant.restype = None
            L.orc_nvfp4_dequant.argtypes = [_u8p, _u8p, ctypes.c_float, _i64, _i64, _f64p]
            L.orc_aqn_sigma.restype = ctypes.c_double
            L.orc_aqn_sigma.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double]
            L.orc_aqn_sigma_schedule.restype = ctypes.c_double
            L.orc_aqn_sigma_schedule.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                 ctypes.c_double]
            L.orc_aqn_stage.restype = ctypes.c_int
            L.orc_aqn_stage.argtypes = [_i64, _i64, ctypes.c_int]
            L.orc_philox4x32_10.restype = None
            L.orc_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
            L.orc_aqn_sample.restype = None
            L.orc_aqn_sample.argtypes = [_f32p, _i64, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32,
                                         ctypes.c_uint64]
            L.orc_e8m0_decode.restype = ctypes.c_double
            L.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
            L.orc_mxfp4_quantize.restype = ctypes.c_int
            L.orc_mxfp4_quantize.argtypes = [_f32p, _i64, _i64, _i64, _u8p, _u8p]
            L.orc_mxfp4_dequant.restype = None
            L.orc_mxfp4_dequant.argtypes = [_u8p, _u8p, _i64, _i64, _f64p]
            L.orc_lora_linear_backward.restype = ctypes.c_int
            L.orc_lora_linear_backward.argtypes = [_u16p, _i64, _i64, _u8p, _u8p, ctypes.c_float, _i64, _u16p, _u16p,
                                                   ctypes.c_int, ctypes.c_float, _f64p, _f64p, _f64p, _f64p]
            L.orc_rmsnorm_noise.restype = None
            L.orc_rmsnorm_noise.argtypes = [_u16p, _i64, _i64, _i64, _u16p, _f32p, ctypes.c_double, _f64p, _u16p]
            L.orc_noise_apply.restype = None
            L.orc_noise_apply.argtypes = [_u16p, _i64, _i64, _i64, _f32p, _i64, _u16p]
            L.orc_lora_linear.restype = ctypes.c_int
            L.orc_lora_linear.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p, ctypes.c_float, _i64,
                                          _f32p, _i64, _u16p, _u16p, ctypes.c_int, ctypes.c_float,
                                          ctypes.c_int, _i64p, _i64, _f64p]
            L.orc_nf4_levels.restype = None
            L.orc_nf4_levels.argtypes = [_f64p]
            L.orc_nf4_encode.restype = ctypes.c_uint8
            L.orc_nf4_encode.argtypes = [ctypes.c_float]
            L.orc_nf4_quantize.restype = ctypes.c_int
            L.orc_nf4_quantize.argtypes = [_f32p, _i64, _i64, _i64, _u8p, _u8p, _f32p]
            L.orc_nf4_dequant.restype = None
            L.orc_nf4_dequant.argtypes = [_u8p, _u8p, ctypes.c_float, _i64, _i64, _f64p]
            L.orc_nf4_lora_linear.restype = ctypes.c_int
            L.orc_nf4_lora_linear.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p, ctypes.c_float, _i64,
                                              _f32p, _i64, _u16p, _u16p, ctypes.c_int, ctypes.c_float,
                                              ctypes.c_int, _i64p, _i64, _f64p]
            L.orc_mxfp4_lora_linear.restype = ctypes.c_int
            L.orc_mxfp4_lora_linear.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p, _i64,
                                                _f32p, _i64, _u16p, _u16p, ctypes.c_int, ctypes.c_float,
                                                ctypes.c_int, _i64p, _i64, _f64p]
            _lib = L
    return _lib


def _ptr(a, t):
    return None if a is None else a.ctypes.data_as(t)


def _check(st):
    if st != OK:
        raise OracleError(f"oracle status {st}")


# ---- element formats -------------------------------------------------------

def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code) & 0xF)


def e2m1_encode(v: float) -> int:
    return int(lib().orc_e2m1_encode(float(v)))


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(v: float) -> int:
    """Encode a non-negative value (nearest-even, saturating at 448)."""
    return int(lib().orc_e4m3_encode_pos(float(v)))


def f64_to_bf16(y: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (one rounding, nearest-even); returns uint16 bits."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    out = np.empty(y.shape, dtype=np.uint16)
    lib().orc_f64_to_bf16_array(_ptr(y, _f64p), y.size, _ptr(out, _u16p))
    return out


# ---- NVFP4 -----------------------------------------------------------------

def tensor_scale(W: np.ndarray) -> float:
    W = np.ascontiguousarray(W, dtype=np.float32)
    n, k = W.shape
    S = ctypes.c_float()
    _check(lib().orc_nvfp4_tensor_scale(_ptr(W, _f32p), n, k, k, ctypes.byref(S)))
    return S.value


def quantize(W: np.ndarray, S: float = None):
    """W: [n, k] fp32 (bf16 inputs converted exactly).  Returns (codes [n,k/2] u8,
    scales [n,k/16] u8, S float32)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    n, k = W.shape
    codes = np.zeros((n, k // 2), dtype=np.uint8)
    scales = np.zeros((n, k // 16), dtype=np.uint8)
    if S is None:
        Sc = ctypes.c_float()
        _check(lib().orc_nvfp4_quantize(_ptr(W, _f32p), n, k, k, _ptr(codes, _u8p), _ptr(scales, _u8p),
                                        ctypes.byref(Sc)))
        S = Sc.value
    else:
        S = float(np.float32(S))
        _check(lib().orc_nvfp4_quantize_with_scale(_ptr(W, _f32p), n, k, k, S, _ptr(codes, _u8p),
                                                   _ptr(scales, _u8p)))
    return codes, scales, np.float32(S)


def dequant(codes: np.ndarray, scales: np.ndarray, S: float) -> np.ndarray:
    """Eq. 6 in fp64.  Returns W_hat [n, k]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    n, k2 = codes.shape
    k = 2 * k2
    out = np.empty((n, k), dtype=np.float64)
    lib().orc_nvfp4_dequant(_ptr(codes, _u8p), _ptr(scales, _u8p), float(S), n, k, _ptr(out, _f64p))
    return out


def e8m0_decode(code: int) -> float:
    return lib().orc_e8m0_decode(int(code))


def mxfp4_quantize(W: np.ndarray):
    """MXFP4 (E2M1 elements, one E8M0 power-of-two scale per 32 along K): W [n, k] fp32 ->
    (codes [n, k/2] u8, scales [n, k/32] u8)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    n, k = W.shape
    codes = np.zeros((n, k // 2), dtype=np.uint8)
    scales = np.zeros((n, k // 32), dtype=np.uint8)
    _check(lib().orc_mxfp4_quantize(_ptr(W, _f32p), n, k, k, _ptr(codes, _u8p), _ptr(scales, _u8p)))
    return codes, scales


def mxfp4_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    n, k2 = codes.shape
    out = np.empty((n, 2 * k2), dtype=np.float64)
    lib().orc_mxfp4_dequant(_ptr(codes, _u8p), _ptr(scales, _u8p), n, 2 * k2, _ptr(out, _f64p))
    return out


# ---- AQN -------------------------------------------------------------------

def aqn_sigma(stage: int, num_stages: int, sigma_start: float = 1e-2, sigma_end: float = 5e-4) -> float:
    return lib().orc_aqn_sigma(int(stage), int(num_stages), float(sigma_start), float(sigma_end))


def aqn_sigma_schedule(schedule: int, stage: int, num_stages: int, sigma_start: float = 1e-2,
                       sigma_end: float = 5e-4) -> float:
    """Decay schedule 0 exponential (Eq. 8), 1 linear, 2 cosine, 3 logarithmic (digest, AQN section)."""
    return lib().orc_aqn_sigma_schedule(int(schedule), int(stage), int(num_stages), float(sigma_start),
                                        float(sigma_end))


def aqn_stage(step: int, total_steps: int, num_stages: int) -> int:
    return lib().orc_aqn_stage(int(step), int(total_steps), int(num_stages))


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    kk = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c, _u32p), _ptr(kk, _u32p), _ptr(out, _u32p))
    return out


def aqn_sample(k: int, sigma: float, seed: int, stream_id: int = 0, counter: int = 0) -> np.ndarray:
    z = np.empty(k, dtype=np.float32)
    lib().orc_aqn_sample(_ptr(z, _f32p), k, float(sigma), int(seed) & (2**64 - 1), int(stream_id) & 0xFFFFFFFF,
                         int(counter) & (2**64 - 1))
    return z


# ---- linear ----------------------------------------------------------------

def _noise_rows(z, m, k):
    """z: None, [k] (one vector for every row) or [m, k] (one per row) -> (array, row stride)."""
    if z is None:
        return None, 0
    zz = np.ascontiguousarray(z, dtype=np.float32)
    if zz.ndim == 1:
        assert zz.shape == (k,)
        return zz, 0
    assert zz.shape == (m, k)
    return zz, k


def noise_apply(x_bits: np.ndarray, z) -> np.ndarray:
    """x_bits [m, k] uint16 (bf16); z [k] or [m, k] float32; returns the bf16 bits of
    bf16(x * (1 + z))."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    m, k = x_bits.shape
    zz, ldz = _noise_rows(z, m, k)
    out = np.empty((m, k), dtype=np.uint16)
    lib().orc_noise_apply(_ptr(x_bits, _u16p), m, k, k, _ptr(zz, _f32p), ldz, _ptr(out, _u16p))
    return out


def lora_linear_backward(xt_bits, codes, scales, S, A_bits, B_bits, alpha, dy, want_dxt=True):
    """Gradients of the linear through the frozen NVFP4 weight, fp64: (d_xt [m, k], dA [r, k],
    dB [n, r]) for y = xt W_hat^T + (alpha/r)(xt A^T) B^T and the output gradient dy [m, n].
    xt_bits is the bf16 noisy activation; A_bits/B_bits None: no LoRA term (dA, dB None).
    want_dxt False: d_xt is not computed (None), only the adapters' gradients."""
    xt_bits = np.ascontiguousarray(xt_bits, dtype=np.uint16)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    dy = np.ascontiguousarray(dy, dtype=np.float64)
    m, k = xt_bits.shape
    n = codes.shape[0]
    assert dy.shape == (m, n)
    r = 0 if A_bits is None else A_bits.shape[0]
    A = None if A_bits is None else np.ascontiguousarray(A_bits, dtype=np.uint16)
    B = None if B_bits is None else np.ascontiguousarray(B_bits, dtype=np.uint16)
    dxt = np.empty((m, k), dtype=np.float64) if want_dxt else None
    dA = np.zeros((max(r, 1), k), dtype=np.float64)
    dB = np.zeros((n, max(r, 1)), dtype=np.float64)
    _check(lib().orc_lora_linear_backward(_ptr(xt_bits, _u16p), m, k, _ptr(codes, _u8p), _ptr(scales, _u8p),
                                          float(S), n, _ptr(A, _u16p), _ptr(B, _u16p), r, float(alpha),
                                          _ptr(dy, _f64p), _ptr(dxt, _f64p), _ptr(dA, _f64p), _ptr(dB, _f64p)))
    return dxt, (dA[:r] if r else None), (dB[:, :r] if r else None)


def rmsnorm_noise(h_bits, w_bits, Z=None, delta=1e-6):
    """Eq. 10 (digest, "Noise Merging"): (w + Z) * h / sqrt(mean(h^2) + delta) per row, fp64.
    h_bits [m, k] and w_bits [k] uint16 (bf16), Z [k] float32 or None.  Returns (fp64 values,
    their bf16 bits)."""
    h_bits = np.ascontiguousarray(h_bits, dtype=np.uint16)
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    m, k = h_bits.shape
    assert w_bits.shape == (k,)
    zz = None if Z is None else np.ascontiguousarray(Z, dtype=np.float32)
    out64 = np.empty((m, k), dtype=np.float64)
    bits = np.empty((m, k), dtype=np.uint16)
    lib().orc_rmsnorm_noise(_ptr(h_bits, _u16p), m, k, k, _ptr(w_bits, _u16p), _ptr(zz, _f32p), float(delta),
                            _ptr(out64, _f64p), _ptr(bits, _u16p))
    return out64, bits


def lora_linear(x_bits, codes, scales, S, z=None, A_bits=None, B_bits=None, alpha=0.0,
                round_xt=True, cols=None) -> np.ndarray:
    """fp64 y[m, len(cols)] of the NVFP4 + LoRA + AQN linear.

    x_bits: [m, k] uint16 bf16; codes [n, k/2]; scales [n, k/16]; S tensor scale;
    z: [k] float32 (one vector for every row), [m, k] (one per row) or None;
    A_bits [r, k] uint16 bf16; B_bits [n, r] uint16 bf16
    (the shapes of Eq. 2: A in R^{r x k}, B in R^{d x r}).
    """
    return _linear("nvfp4", x_bits, codes, scales, S, z, A_bits, B_bits, alpha, round_xt, cols)


def nf4_levels() -> np.ndarray:
    """The 16 NF4 levels, ascending (code c -> level c; code 7 is 0)."""
    out = np.empty(16, dtype=np.float64)
    lib().orc_nf4_levels(_ptr(out, _f64p))
    return out


def nf4_encode(q: float) -> int:
    return int(lib().orc_nf4_encode(float(q)))


def nf4_quantize(W: np.ndarray):
    """NF4 levels with NVFP4-style dual scaling: W [n, k] fp32 -> (codes [n, k/2], E4M3 scales
    [n, k/16], tensor scale S)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    n, k = W.shape
    codes = np.zeros((n, k // 2), dtype=np.uint8)
    scales = np.zeros((n, k // 16), dtype=np.uint8)
    S = np.zeros(1, dtype=np.float32)
    _check(lib().orc_nf4_quantize(_ptr(W, _f32p), n, k, k, _ptr(codes, _u8p), _ptr(scales, _u8p), _ptr(S, _f32p)))
    return codes, scales, float(S[0])


def nf4_dequant(codes: np.ndarray, scales: np.ndarray, S: float) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    n, k2 = codes.shape
    out = np.empty((n, 2 * k2), dtype=np.float64)
    lib().orc_nf4_dequant(_ptr(codes, _u8p), _ptr(scales, _u8p), float(S), n, 2 * k2, _ptr(out, _f64p))
    return out


def nf4_lora_linear(x_bits, codes, scales, S, z=None, A_bits=None, B_bits=None, alpha=0.0,
                    round_xt=True, cols=None) -> np.ndarray:
    """The same linear over an NF4 weight (codes [n, k/2], E4M3 scales [n, k/16], tensor scale S)."""
    return _linear("nf4", x_bits, codes, scales, S, z, A_bits, B_bits, alpha, round_xt, cols)


def mxfp4_lora_linear(x_bits, codes, scales, z=None, A_bits=None, B_bits=None, alpha=0.0,
                      round_xt=True, cols=None) -> np.ndarray:
    """The same linear over an MXFP4 weight: codes [n, k/2], E8M0 scales [n, k/32]."""
    return _linear("mxfp4", x_bits, codes, scales, 1.0, z, A_bits, B_bits, alpha, round_xt, cols)


def _linear(fmt, x_bits, codes, scales, S, z, A_bits, B_bits, alpha, round_xt, cols):
    mx = fmt == "mxfp4"
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    m, k = x_bits.shape
    n = codes.shape[0]
    assert codes.shape == (n, k // 2) and scales.shape == (n, k // (32 if mx else 16))
    r = 0
    if A_bits is not None and B_bits is not None:
        A_bits = np.ascontiguousarray(A_bits, dtype=np.uint16)
        B_bits = np.ascontiguousarray(B_bits, dtype=np.uint16)
        r = A_bits.shape[0]
        assert A_bits.shape == (r, k) and B_bits.shape == (n, r)
    else:
        A_bits = B_bits = None
    zz, ldz = _noise_rows(z, m, k)
    if cols is None:
        cols_arr, ncols = None, n
    else:
        cols_arr = np.ascontiguousarray(cols, dtype=np.int64)
        ncols = cols_arr.size
    y = np.empty((m, ncols), dtype=np.float64)
    rest = (_ptr(zz, _f32p), ldz, _ptr(A_bits, _u16p), _ptr(B_bits, _u16p), r, float(alpha),
            1 if round_xt else 0, _ptr(cols_arr, _i64p), ncols, _ptr(y, _f64p))
    if mx:
        _check(lib().orc_mxfp4_lora_linear(_ptr(x_bits, _u16p), m, k, k, _ptr(codes, _u8p), _ptr(scales, _u8p),
                                           n, *rest))
    elif fmt == "nf4":
        _check(lib().orc_nf4_lora_linear(_ptr(x_bits, _u16p), m, k, k, _ptr(codes, _u8p), _ptr(scales, _u8p),
                                         float(S), n, *rest))
    else:
        _check(lib().orc_lora_linear(_ptr(x_bits, _u16p), m, k, k, _ptr(codes, _u8p), _ptr(scales, _u8p),
                                     float(S), n, *rest))
    return y
