"""quantized_tensor_activation_gb300 -- Python binding of the GB300 codec library.

A thin ctypes layer over ``libqta.so`` (C ABI in ``include/qta.h``) with the
same call names: ``taco_compress``, ``taco_decompress``, ``qar_reduce``,
``qar_requant``, ``qar_reduce_requant``, ``taco_update_scale``, ``qta_copy``.  It only marshals
arguments (device pointers, sizes, the current CUDA stream); every step of
the codec runs in the library's CUDA kernels.  There is no CPU fallback: if
the library is missing or a call fails, an exception is raised.

Torch is used for device memory and streams only (``alloc_qtensor`` sizes
buffers from the library's own ``qta_*_bytes`` queries).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from . import _build

# ---------------------------------------------------------------- constants
QTA_OK, QTA_ERR_INVALID_ARG, QTA_ERR_ALIGNMENT, QTA_ERR_UNSUPPORTED, QTA_ERR_CUDA = range(5)
BF16, FP16, FP32 = 0, 1, 2
TACO_FP8, INT8_SYM_B64, INT4_ASYM_G128, INT8_ASYM_G128 = 0, 1, 2, 3
SCALE_DELAYED, SCALE_CURRENT = 0, 1
SCALE_ROUND_UP = 4    # OR into a TACO scale mode: block scales rounded up
MAX_RANKS = 16

SCHEMES = {"taco_fp8": TACO_FP8, "int8_sym": INT8_SYM_B64, "int4_asym": INT4_ASYM_G128,
           "int8_asym": INT8_ASYM_G128}


class QtaError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {_status_name(status)}")


class Desc(ctypes.Structure):
    _fields_ = [("scheme", ctypes.c_int32), ("block", ctypes.c_int32), ("batch", ctypes.c_int64),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("max_sms", ctypes.c_int32)]


class QTensorC(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zeros", ctypes.c_void_p),
                ("state", ctypes.c_void_p), ("chan", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return _build.LIB


def build(force: bool = False) -> str:
    """Compile libqta.so in-tree for sm_103a (nvcc)."""
    return _build.build(force=force)


def lib():
    """Load libqta.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libqta.so is not built ({path}); run quantized_tensor_activation_gb300.build()")
        L = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        PD, PQ = ctypes.POINTER(Desc), ctypes.POINTER(QTensorC)
        for name in ("qta_codes_bytes", "qta_scales_bytes", "qta_zeros_bytes", "qta_state_bytes"):
            getattr(L, name).argtypes = [PD]
            getattr(L, name).restype = sz
        L.taco_compress.argtypes = [PD, vp, i32, PQ, i32, vp]
        L.taco_decompress.argtypes = [PD, PQ, vp, i32, vp]
        L.qar_reduce.argtypes = [PD, PQ, i32, i64, i64, vp, vp]
        L.qar_requant.argtypes = [PD, vp, PQ, i32, vp]
        L.qar_reduce_requant.argtypes = [PD, PQ, i32, i64, i64, PD, PQ, i32, vp]
        L.qar_dequant_add.argtypes = [PD, PQ, vp, i32, vp, vp]
        L.qar_dequant_add_requant.argtypes = [PD, PQ, vp, i32, PQ, i32, vp]
        L.qta_sq_error.argtypes = [vp, i32, vp, i64, vp, vp]
        L.qta_wait_self_test.argtypes = [i32, vp]
        L.taco_update_scale.argtypes = [vp, i64, vp]
        L.qta_copy.argtypes = [vp, vp, sz, vp]
        L.qta_chan_bytes.argtypes = [i64]
        L.qta_chan_bytes.restype = sz
        L.taco_channel_amax.argtypes = [PD, vp, i32, vp, vp]
        L.taco_ash_update.argtypes = [vp, i64, vp]
        L.qta_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        for name in ("taco_compress", "taco_decompress", "qar_reduce", "qar_requant", "qar_reduce_requant",
                     "qar_dequant_add", "qar_dequant_add_requant", "qta_sq_error", "qta_wait_self_test",
                     "taco_update_scale", "qta_copy", "taco_channel_amax", "taco_ash_update",
                     "qta_device_error"):
            getattr(L, name).restype = ctypes.c_int
        L.qta_status_string.argtypes = [ctypes.c_int]
        L.qta_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _status_name(s: int) -> str:
    try:
        return lib().qta_status_string(s).decode()
    except Exception:  # library not loadable
        return f"status {s}"


def _check(call: str, status: int) -> None:
    if status != QTA_OK:
        raise QtaError(call, status)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def desc(scheme, block: int, rows: int, cols: int, batch: int = 1, max_sms: int = 0) -> Desc:
    """max_sms: SMs the calls may occupy (0: all)."""
    if isinstance(scheme, str):
        scheme = SCHEMES[scheme]
    return Desc(int(scheme), int(block), int(batch), int(rows), int(cols), int(max_sms))


@dataclass
class QTensor:
    """Device buffers of one quantized tensor (torch uint8/float32 tensors).
    chan: the adaptive rescaling state (float32 [3 * cols], see alloc_chan)
    or None."""
    desc: Desc
    codes: object
    scales: object
    zeros: object = None
    state: object = None
    chan: object = None

    def c(self) -> QTensorC:
        return QTensorC(_ptr(self.codes), _ptr(self.scales), _ptr(self.zeros), _ptr(self.state),
                        _ptr(self.chan))

    def shard(self, i: int) -> "QTensor":
        """View of tensor i of a batch as a batch-1 quantized tensor."""
        d = self.desc
        n = d.batch
        sub = Desc(d.scheme, d.block, 1, d.rows, d.cols, d.max_sms)
        cb, sb, zb = codes_bytes(sub), scales_bytes(sub), zeros_bytes(sub)
        return QTensor(sub, self.codes[i * cb:(i + 1) * cb], self.scales[i * sb:(i + 1) * sb],
                       None if self.zeros is None else self.zeros[i * zb:(i + 1) * zb],
                       None if self.state is None else self.state[2 * i:2 * i + 2], self.chan)


def codes_bytes(d: Desc) -> int:
    return lib().qta_codes_bytes(ctypes.byref(d))


def scales_bytes(d: Desc) -> int:
    return lib().qta_scales_bytes(ctypes.byref(d))


def zeros_bytes(d: Desc) -> int:
    return lib().qta_zeros_bytes(ctypes.byref(d))


def state_bytes(d: Desc) -> int:
    return lib().qta_state_bytes(ctypes.byref(d))


def alloc_qtensor(d: Desc, device="cuda", initial_scale: float | None = 1.0) -> QTensor:
    """Allocate the device buffers of a quantized tensor (byte buffers; the
    per-tensor state, when the scheme has one, as float32 [batch, 2] set to
    {initial_scale, 0})."""
    import torch
    cb, sb, zb, stb = codes_bytes(d), scales_bytes(d), zeros_bytes(d), state_bytes(d)
    codes = torch.empty(cb, dtype=torch.uint8, device=device)
    scales = torch.empty(sb, dtype=torch.uint8, device=device)
    zeros = torch.empty(zb, dtype=torch.uint8, device=device) if zb else None
    state = None
    if stb:
        state = torch.zeros(stb // 4, dtype=torch.float32, device=device)
        if initial_scale is not None:
            state[0::2] = initial_scale
    return QTensor(d, codes, scales, zeros, state)


# ---------------------------------------------------------------- the calls
def taco_compress(d: Desc, x, x_dtype: int, out: QTensor, mode: int = SCALE_DELAYED, stream=None) -> None:
    q = out.c()
    _check("taco_compress", lib().taco_compress(ctypes.byref(d), _ptr(x), x_dtype, ctypes.byref(q), mode,
                                                _stream(stream)))


def taco_decompress(d: Desc, q: QTensor, y, y_dtype: int, stream=None) -> None:
    qc = q.c()
    _check("taco_decompress", lib().taco_decompress(ctypes.byref(d), ctypes.byref(qc), _ptr(y), y_dtype,
                                                    _stream(stream)))


def qar_reduce(d: Desc, shards, row_begin: int, row_end: int, sum_out, stream=None) -> None:
    n = len(shards)
    arr = (QTensorC * max(n, 1))(*[s.c() for s in shards])
    _check("qar_reduce", lib().qar_reduce(ctypes.byref(d), arr, n, row_begin, row_end, _ptr(sum_out),
                                          _stream(stream)))


def qar_reduce_requant(d: Desc, shards, row_begin: int, row_end: int, out_desc: Desc, out: QTensor,
                       mode: int = SCALE_DELAYED, stream=None) -> None:
    n = len(shards)
    arr = (QTensorC * max(n, 1))(*[s.c() for s in shards])
    q = out.c()
    _check("qar_reduce_requant", lib().qar_reduce_requant(ctypes.byref(d), arr, n, row_begin, row_end,
                                                          ctypes.byref(out_desc), ctypes.byref(q), mode,
                                                          _stream(stream)))


def qar_requant(d: Desc, sum_in, out: QTensor, mode: int = SCALE_DELAYED, stream=None) -> None:
    q = out.c()
    _check("qar_requant", lib().qar_requant(ctypes.byref(d), _ptr(sum_in), ctypes.byref(q), mode,
                                            _stream(stream)))


def qar_dequant_add(d: Desc, q_in: QTensor, x, x_dtype: int, sum_out, stream=None) -> None:
    qi = q_in.c()
    _check("qar_dequant_add", lib().qar_dequant_add(ctypes.byref(d), ctypes.byref(qi), _ptr(x), x_dtype,
                                                    _ptr(sum_out), _stream(stream)))


def qar_dequant_add_requant(d: Desc, q_in: QTensor, x, x_dtype: int, out: QTensor, mode: int = SCALE_DELAYED,
                            stream=None) -> None:
    qi, qo = q_in.c(), out.c()
    _check("qar_dequant_add_requant", lib().qar_dequant_add_requant(ctypes.byref(d), ctypes.byref(qi), _ptr(x),
                                                                    x_dtype, ctypes.byref(qo), mode,
                                                                    _stream(stream)))


def qta_sq_error(a, a_dtype: int, b, n: int, out, stream=None) -> None:
    """out (device float64 [1]) = sum of (a - b)^2 over n elements."""
    _check("qta_sq_error", lib().qta_sq_error(_ptr(a), a_dtype, _ptr(b), n, _ptr(out), _stream(stream)))


def qta_wait_self_test(complete: bool, stream=None) -> None:
    _check("qta_wait_self_test", lib().qta_wait_self_test(1 if complete else 0, _stream(stream)))


def taco_update_scale(state, n_tensors: int, stream=None) -> None:
    _check("taco_update_scale", lib().taco_update_scale(_ptr(state), n_tensors, _stream(stream)))


def qta_copy(src, dst, nbytes: int, stream=None) -> None:
    _check("qta_copy", lib().qta_copy(_ptr(src), _ptr(dst), nbytes, _stream(stream)))


def qta_device_error(clear: bool = True) -> int:
    flags = ctypes.c_uint32(0)
    _check("qta_device_error", lib().qta_device_error(ctypes.byref(flags), 1 if clear else 0))
    return flags.value


# ---------------------------------------------------------------- adaptive rescaling
def alloc_chan(cols: int, device="cuda"):
    """Adaptive rescaling state of `cols` channels: float32 [3 * cols] =
    down (1), up (1), amax (0), i.e. no rescaling until taco_ash_update."""
    import torch
    n = lib().qta_chan_bytes(int(cols)) // 4
    c = torch.zeros(n, dtype=torch.float32, device=device)
    c[:2 * cols] = 1.0
    return c


def taco_channel_amax(d: Desc, x, x_dtype: int, chan, stream=None) -> None:
    _check("taco_channel_amax", lib().taco_channel_amax(ctypes.byref(d), _ptr(x), x_dtype, _ptr(chan),
                                                        _stream(stream)))


def taco_ash_update(chan, cols: int, stream=None) -> None:
    _check("taco_ash_update", lib().taco_ash_update(_ptr(chan), cols, _stream(stream)))
