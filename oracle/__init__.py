"""CPU oracle of the quantized tensor-activation codec -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports it, and the two share no code: the oracle is
plain single-threaded C (``qta_oracle.c``) wrapped here with ctypes and numpy.

Every function follows a passage of the pages (cited in ``qta_oracle.c``):
TACO (FP8 E4M3, block Hadamard, dual-scale), EQuARX (block-symmetric int8,
dequantize to FP32 before adding) and Flash Communication (asymmetric
group-128 INT4/INT8, two-step all-reduce).
"""
from __future__ import annotations

import ctypes
import functools
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qta_oracle.c")
_HDR = os.path.join(_HERE, "qta_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

# dtype / scheme / mode codes of the C oracle
BF16, FP16, FP32 = 0, 1, 2
TACO_FP8, INT8_SYM, INT4_ASYM, INT8_ASYM = 0, 1, 2, 3
DELAYED, CURRENT = 0, 1
ROUND_UP = 4          # OR into DELAYED / CURRENT: block scales rounded up (TACO)

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with strict IEEE binary32 semantics."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fexcess-precision=standard", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    """The loaded oracle library.  QTA_ORACLE_LIB names another build of it
    to load instead (the mutation tests load deliberately miswritten copies
    to show that the pins fail on them)."""
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(os.environ.get("QTA_ORACLE_LIB") or build())
            i64, i32, vp, fp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_decode.restype = ctypes.c_float
            L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            L.orc_f32_to_bf16.restype = ctypes.c_uint16
            L.orc_f32_to_f16.argtypes = [ctypes.c_float]
            L.orc_f32_to_f16.restype = ctypes.c_uint16
            L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_f32.restype = ctypes.c_float
            L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_f32.restype = ctypes.c_float
            for name in ("orc_e4m3_encode_array", "orc_f32_to_bf16_array", "orc_f32_to_f16_array"):
                getattr(L, name).argtypes = [vp, vp, i64]
                getattr(L, name).restype = None
            L.orc_fwht.argtypes = [fp, i32]
            L.orc_fwht_rows.argtypes = [fp, i64, i32]
            L.orc_scale_from_amax.argtypes = [ctypes.c_float]
            L.orc_scale_from_amax.restype = ctypes.c_float
            L.orc_taco_update_scale.argtypes = [fp, i64]
            L.orc_compress.argtypes = [i32, i32, vp, i32, i64, i64, i64, fp, i32, vp, vp, vp]
            L.orc_compress.restype = i32
            L.orc_decompress.argtypes = [i32, i32, vp, vp, vp, fp, i64, i64, i64, vp, i32]
            L.orc_decompress.restype = i32
            L.orc_reduce.argtypes = [i32, i32, i32, vp, vp, vp, vp, i64, i64, i64, i64, fp]
            L.orc_reduce.restype = i32
            L.orc_reduce_requant.argtypes = [i32, i32, i32, vp, vp, vp, vp, i64, i64, i64, i64,
                                             i32, i32, i64, fp, i32, vp, vp, vp]
            L.orc_reduce_requant.restype = i32
            L.orc_dequant_add.argtypes = [i32, i32, vp, vp, vp, fp, i64, i64, i64, vp, i32, fp]
            L.orc_dequant_add.restype = i32
            L.orc_compress_chan.argtypes = L.orc_compress.argtypes + [fp]
            L.orc_compress_chan.restype = i32
            L.orc_decompress_chan.argtypes = L.orc_decompress.argtypes + [fp]
            L.orc_decompress_chan.restype = i32
            L.orc_reduce_chan.argtypes = L.orc_reduce.argtypes + [fp]
            L.orc_reduce_chan.restype = i32
            L.orc_reduce_requant_chan.argtypes = L.orc_reduce_requant.argtypes + [fp]
            L.orc_reduce_requant_chan.restype = i32
            L.orc_channel_amax.argtypes = [vp, i32, i64, i64, i64, fp]
            L.orc_channel_amax.restype = i32
            L.orc_ash_update.argtypes = [fp, i64]
            L.orc_ash_update.restype = i32
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- formats
def e4m3_encode(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_ptr(v), _ptr(out), v.size)
    return out


@functools.lru_cache(maxsize=None)
def _e4m3_table() -> np.ndarray:
    return np.array([lib().orc_e4m3_decode(i) for i in range(256)], dtype=np.float32)


@functools.lru_cache(maxsize=None)
def _f16_table() -> np.ndarray:
    L = lib()
    return np.array([L.orc_f16_to_f32(i) for i in range(65536)], dtype=np.float32)


def e4m3_decode(c) -> np.ndarray:
    return _e4m3_table()[np.asarray(c, dtype=np.uint8)]


def f32_to_bf16(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(_ptr(v), _ptr(out), v.size)
    return out


def f32_to_f16(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_f32_to_f16_array(_ptr(v), _ptr(out), v.size)
    return out


def bf16_to_f32(h) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def f16_to_f32(h) -> np.ndarray:
    return _f16_table()[np.asarray(h, dtype=np.uint16)]


# ---------------------------------------------------------------- transform
def fwht(y, B: int) -> np.ndarray:
    """Unnormalised block Hadamard over consecutive blocks of B (in a copy)."""
    y = np.array(y, dtype=np.float32, copy=True).reshape(-1)
    assert y.size % B == 0
    lib().orc_fwht_rows(_ptr(y), y.size // B, B)
    return y


def scale_from_amax(amax: float) -> float:
    return lib().orc_scale_from_amax(float(amax))


def taco_update_scale(state: np.ndarray) -> None:
    assert state.dtype == np.float32 and state.flags.c_contiguous
    lib().orc_taco_update_scale(_ptr(state), state.size // 2)


# ---------------------------------------------------------------- codec
def codes_nbytes(scheme: int, n_elems: int) -> int:
    return n_elems // 2 if scheme == INT4_ASYM else n_elems


def _chan(chan, cols):
    if chan is None:
        return None
    assert chan.dtype == np.float32 and chan.flags.c_contiguous and chan.size == 3 * cols
    return chan


def compress(scheme: int, B: int, x: np.ndarray, in_dtype: int, batch: int, rows: int,
             cols: int, state: np.ndarray | None = None, mode: int = DELAYED, chan=None):
    """Returns (codes, scales, zeros); updates ``state`` in place for TACO.
    chan: the adaptive rescaling's per-channel state, float32 [3 * cols] =
    down, up, amax (TACO only; None: no rescaling)."""
    E = batch * rows * cols
    x = np.ascontiguousarray(x)
    assert x.size == E
    codes = np.zeros(codes_nbytes(scheme, E), dtype=np.int8 if scheme == INT8_SYM else np.uint8)
    zeros = None
    if scheme == TACO_FP8:
        scales = np.zeros(E // B, dtype=np.uint8)
        assert state is not None and state.dtype == np.float32 and state.size == 2 * batch
    elif scheme == INT8_SYM:
        scales = np.zeros(E // 64, dtype=np.float32)
    else:
        scales = np.zeros(E // 128, dtype=np.uint16)
        zeros = np.zeros(E // 128, dtype=np.uint16)
    rc = lib().orc_compress_chan(scheme, B, _ptr(x), in_dtype, batch, rows, cols,
                                 _ptr(state), mode, _ptr(codes), _ptr(scales), _ptr(zeros),
                                 _ptr(_chan(chan, cols)))
    if rc:
        raise ValueError(f"oracle compress rejected the arguments ({rc})")
    return codes, scales, zeros


def decompress(scheme: int, B: int, codes, scales, zeros, state, batch: int, rows: int,
               cols: int, out_dtype: int, chan=None) -> np.ndarray:
    E = batch * rows * cols
    out = np.zeros(E, dtype=np.float32 if out_dtype == FP32 else np.uint16)
    st = None if state is None else np.ascontiguousarray(state, dtype=np.float32)
    rc = lib().orc_decompress_chan(scheme, B, _ptr(np.ascontiguousarray(codes)),
                                   _ptr(np.ascontiguousarray(scales)),
                                   _ptr(None if zeros is None else np.ascontiguousarray(zeros)),
                                   _ptr(st), batch, rows, cols, _ptr(out), out_dtype, _ptr(_chan(chan, cols)))
    if rc:
        raise ValueError(f"oracle decompress rejected the arguments ({rc})")
    return out


def reduce(scheme: int, B: int, shards, rows: int, cols: int, row_begin: int = 0,
           row_end: int | None = None, chan=None) -> np.ndarray:
    """shards: list of (codes, scales, zeros, state) per rank, one tensor each."""
    if row_end is None:
        row_end = rows
    n = len(shards)
    keep = [tuple(None if a is None else np.ascontiguousarray(a) for a in s) for s in shards]
    VP = ctypes.c_void_p * n
    codes = VP(*[_ptr(s[0]) for s in keep])
    scales = VP(*[_ptr(s[1]) for s in keep])
    zeros = VP(*[_ptr(s[2]) for s in keep]) if keep[0][2] is not None else None
    st_keep = [None if s[3] is None else np.ascontiguousarray(s[3], dtype=np.float32) for s in keep]
    states = VP(*[_ptr(a) for a in st_keep]) if st_keep[0] is not None else None
    out = np.zeros((row_end - row_begin) * cols, dtype=np.float32)
    rc = lib().orc_reduce_chan(scheme, B, n, codes, scales, zeros, states, rows, cols,
                               row_begin, row_end, _ptr(out), _ptr(_chan(chan, cols)))
    if rc:
        raise ValueError(f"oracle reduce rejected the arguments ({rc})")
    return out


def _shard_arrays(shards):
    n = len(shards)
    keep = [tuple(None if a is None else np.ascontiguousarray(a) for a in s) for s in shards]
    VP = ctypes.c_void_p * n
    codes = VP(*[_ptr(s[0]) for s in keep])
    scales = VP(*[_ptr(s[1]) for s in keep])
    zeros = VP(*[_ptr(s[2]) for s in keep]) if keep[0][2] is not None else None
    st_keep = [None if s[3] is None else np.ascontiguousarray(s[3], dtype=np.float32) for s in keep]
    states = VP(*[_ptr(a) for a in st_keep]) if st_keep[0] is not None else None
    return keep, st_keep, codes, scales, zeros, states


def reduce_requant(scheme: int, B: int, shards, rows: int, cols: int, row_begin: int, row_end: int,
                   out_scheme: int, out_B: int, out_batch: int, out_state=None, mode: int = DELAYED,
                   chan=None):
    """Fused dequantize-reduce + requantize; returns (codes, scales, zeros) of
    the output tensors and updates ``out_state`` in place (TACO output)."""
    keep, st_keep, codes, scales, zeros, states = _shard_arrays(shards)
    E = (row_end - row_begin) * cols
    oc = np.zeros(codes_nbytes(out_scheme, E), dtype=np.int8 if out_scheme == INT8_SYM else np.uint8)
    oz = None
    if out_scheme == TACO_FP8:
        os_ = np.zeros(E // out_B, dtype=np.uint8)
        assert out_state is not None and out_state.dtype == np.float32 and out_state.size == 2 * out_batch
    elif out_scheme == INT8_SYM:
        os_ = np.zeros(E // 64, dtype=np.float32)
    else:
        os_ = np.zeros(E // 128, dtype=np.uint16)
        oz = np.zeros(E // 128, dtype=np.uint16)
    rc = lib().orc_reduce_requant_chan(scheme, B, len(shards), codes, scales, zeros, states, rows, cols,
                                       row_begin, row_end, out_scheme, out_B, out_batch, _ptr(out_state), mode,
                                       _ptr(oc), _ptr(os_), _ptr(oz), _ptr(_chan(chan, cols)))
    if rc:
        raise ValueError(f"oracle reduce_requant rejected the arguments ({rc})")
    return oc, os_, oz


# ---------------------------------------------------------------- ring
def dequant_add(scheme: int, B: int, codes, scales, zeros, state, batch: int, rows: int, cols: int,
                x: np.ndarray, x_dtype: int) -> np.ndarray:
    """One ring hop at the receiver: the incoming partial sum dequantized to
    FP32 as ``decompress`` does it, plus the local tensor x (one FP32 rounding
    per element).  x: 16-bit bits (uint16) or float32 values."""
    E = batch * rows * cols
    x = np.ascontiguousarray(x)
    assert x.size == E
    out = np.zeros(E, dtype=np.float32)
    st = None if state is None else np.ascontiguousarray(state, dtype=np.float32)
    rc = lib().orc_dequant_add(scheme, B, _ptr(np.ascontiguousarray(codes)),
                               _ptr(np.ascontiguousarray(scales)),
                               _ptr(None if zeros is None else np.ascontiguousarray(zeros)),
                               _ptr(st), batch, rows, cols, _ptr(x), x_dtype, _ptr(out))
    if rc:
        raise ValueError(f"oracle dequant_add rejected the arguments ({rc})")
    return out


def _compress_current(scheme: int, B: int, x, dtype: int, rows: int, cols: int):
    st = np.zeros(2, dtype=np.float32) if scheme == TACO_FP8 else None
    c, s, z = compress(scheme, B, x, dtype, 1, rows, cols, st, CURRENT)
    return c, s, z, st


def ring_chain(scheme: int, B: int, parts, dtype: int, rows: int, cols: int):
    """Adder chain [EQuARX Figs. 4-5]: the first rank quantizes its tensor;
    every following rank dequantizes the incoming partial sum, adds its own
    tensor in FP32 and requantizes the sum (CURRENT scale for TACO) before it
    travels on.  parts: the chain's tensors in visiting order.  Returns the
    quantized partial sum (codes, scales, zeros, state) leaving the last rank."""
    q = _compress_current(scheme, B, parts[0], dtype, rows, cols)
    for x in parts[1:]:
        s = dequant_add(scheme, B, *q, 1, rows, cols, x, dtype)
        q = _compress_current(scheme, B, s, FP32, rows, cols)
    return q


def ring_chunk_orders(n: int, j: int, semi: bool):
    """Visiting orders of the chains that end at the owner j of chunk j.
    Full loop: one chain j+1, j+2, ..., j+n-1.  Semi loop: two chains that
    meet at the owner, j+h, ..., j+1 and j-(n-1-h), ..., j-1 with h = n // 2."""
    if not semi:
        return [[(j + k) % n for k in range(1, n)]]
    h = n // 2
    chains = [[(j + k) % n for k in range(h, 0, -1)]]
    if n - 1 - h > 0:
        chains.append([(j - k) % n for k in range(n - 1 - h, 0, -1)])
    return chains


def ring_reduce_scatter(scheme: int, B: int, xs, dtype: int, rows: int, cols: int,
                        semi: bool = False) -> np.ndarray:
    """Quantized ring reduce-scatter of n = len(xs) tensors [rows, cols]:
    chunk j (rows j*rows/n .. (j+1)*rows/n) is reduced along the chain(s) of
    ring_chunk_orders and finished at its owner j, which adds its own chunk
    to the first chain's partial sum and then the second chain's (each
    dequantized to FP32 first).  Returns the FP32 sums [rows * cols]."""
    n = len(xs)
    assert n >= 2 and rows % n == 0
    rc = rows // n
    out = np.zeros(rows * cols, dtype=np.float32)
    for j in range(n):
        def chunk(r):
            return np.ascontiguousarray(np.asarray(xs[r]).reshape(rows, cols)[j * rc:(j + 1) * rc]).reshape(-1)
        qs = [ring_chain(scheme, B, [chunk(r) for r in order], dtype, rc, cols)
              for order in ring_chunk_orders(n, j, semi)]
        s = dequant_add(scheme, B, *qs[0], 1, rc, cols, chunk(j), dtype)
        for q in qs[1:]:
            s = dequant_add(scheme, B, *q, 1, rc, cols, s, FP32)
        out[j * rc * cols:(j + 1) * rc * cols] = s
    return out


def ring_allreduce(scheme: int, B: int, xs, dtype: int, rows: int, cols: int, semi: bool = False,
                   out_dtype: int = FP32):
    """Ring reduce-scatter, then the quantized all-gather: every reduced chunk
    is requantized (CURRENT scale for TACO) and every rank dequantizes the
    gathered chunks.  Returns (reduce-scatter FP32 sums, all-reduce output in
    out_dtype), both [rows * cols]."""
    s = ring_reduce_scatter(scheme, B, xs, dtype, rows, cols, semi)
    n = len(xs)
    rc = rows // n
    y = np.zeros(rows * cols, dtype=np.float32 if out_dtype == FP32 else np.uint16)
    for j in range(n):
        part = s[j * rc * cols:(j + 1) * rc * cols]
        q = _compress_current(scheme, B, part, FP32, rc, cols)
        y[j * rc * cols:(j + 1) * rc * cols] = decompress(scheme, B, *q, 1, rc, cols, out_dtype)
    return s, y


# ---------------------------------------------------------------- block choice
def block_errors(x, x_dtype: int, batch: int, rows: int, cols: int, candidates=(64, 128, 256),
                 mode: int = CURRENT) -> dict:
    """Squared reconstruction error of compress (TACO, CURRENT scale) ->
    decompress (FP32) for every candidate block size dividing cols, summed
    in float64 ([TACO] Core claim: the reshape is chosen from the data)."""
    xv = np.ascontiguousarray(x).reshape(-1)
    if x_dtype == BF16:
        xw = bf16_to_f32(xv).astype(np.float64)
    elif x_dtype == FP16:
        xw = f16_to_f32(xv).astype(np.float64)
    else:
        xw = xv.astype(np.float64)
    errs = {}
    for B in candidates:
        if cols % B:
            continue
        st = np.zeros(2 * batch, dtype=np.float32)
        c, s, z = compress(TACO_FP8, B, xv, x_dtype, batch, rows, cols, st, mode)
        y = decompress(TACO_FP8, B, c, s, z, st, batch, rows, cols, FP32).astype(np.float64)
        errs[B] = float(((xw - y) ** 2).sum())
    return errs


def choose_block(x, x_dtype: int, batch: int, rows: int, cols: int, candidates=(64, 128, 256)):
    errs = block_errors(x, x_dtype, batch, rows, cols, candidates)
    best = min(sorted(errs), key=lambda b: errs[b])
    return best, errs


# ---------------------------------------------------------------- adaptive rescaling
def new_chan_state(cols: int) -> np.ndarray:
    """Per-channel state of the adaptive rescaling: float32 [3 * cols] =
    down (all 1), up (all 1), amax (all 0)."""
    c = np.zeros(3 * cols, dtype=np.float32)
    c[:2 * cols] = 1.0
    return c


def channel_amax(x, dtype: int, batch: int, rows: int, cols: int, chan: np.ndarray) -> None:
    """Max-accumulate |x| per channel (column) into chan's amax part."""
    x = np.ascontiguousarray(x)
    assert x.size == batch * rows * cols
    rc = lib().orc_channel_amax(_ptr(x), dtype, batch, rows, cols, _ptr(_chan(chan, cols)))
    if rc:
        raise ValueError(f"oracle channel_amax rejected the arguments ({rc})")


def ash_update(chan: np.ndarray, cols: int) -> None:
    """Per-channel powers of two from the accumulated amax (median rule), amax reset."""
    rc = lib().orc_ash_update(_ptr(_chan(chan, cols)), cols)
    if rc:
        raise ValueError(f"oracle ash_update rejected the arguments ({rc})")
