"""The C ABI library builds, loads and exports every call the header
declares; host-side argument checks return their status codes without a GPU
(no compute call is made here)."""
import ctypes
import os
import re

import pytest

import quantized_tensor_activation_gb300 as qta

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    qta.build()
    return qta.lib()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z_0-9]*\s*\*?\s+\**([a-z_][a-z_0-9]*)\s*\(",
                             text, flags=re.M):
            names.append(m.group(1))
    return names


def test_exports_every_declared_call(L):
    names = _declared_functions()
    for must in ("taco_compress", "taco_decompress", "qar_reduce", "qar_requant", "taco_update_scale",
                 "qta_copy", "qta_device_error", "qta_status_string", "qta_codes_bytes"):
        assert must in names
    for n in names:
        assert hasattr(L, n), n


def test_sizes(L):
    d = qta.desc("taco_fp8", 128, 256, 1024, batch=4)
    assert (qta.codes_bytes(d), qta.scales_bytes(d), qta.zeros_bytes(d), qta.state_bytes(d)) == \
        (1048576, 8192, 0, 32)
    d = qta.desc("int8_sym", 64, 16, 512)
    assert (qta.codes_bytes(d), qta.scales_bytes(d), qta.zeros_bytes(d), qta.state_bytes(d)) == \
        (8192, 512, 0, 0)
    d = qta.desc("int4_asym", 128, 8, 256, batch=2)
    assert (qta.codes_bytes(d), qta.scales_bytes(d), qta.zeros_bytes(d)) == (2048, 64, 64)
    assert qta.codes_bytes(qta.desc("taco_fp8", 100, 1, 200)) == 0   # invalid block


def _c(L, name, *args):
    return getattr(L, name)(*args)


def test_argument_checks(L):
    D = lambda *a: ctypes.byref(qta.desc(*a))
    Q = lambda c=16, s=16, z=16, st=16: ctypes.byref(qta.QTensorC(c, s, z, st))
    OK, INV, ALN, UNS = qta.QTA_OK, qta.QTA_ERR_INVALID_ARG, qta.QTA_ERR_ALIGNMENT, qta.QTA_ERR_UNSUPPORTED
    # descriptor problems
    assert L.taco_compress(None, 16, 0, Q(), 0, None) == INV
    assert L.taco_compress(D(9, 128, 4, 128), 16, 0, Q(), 0, None) == UNS
    assert L.taco_compress(D(0, 96, 4, 192), 16, 0, Q(), 0, None) == UNS
    assert L.taco_compress(D(1, 128, 4, 128), 16, 0, Q(), 0, None) == UNS
    assert L.taco_compress(D(0, 128, 4, 192), 16, 0, Q(), 0, None) == INV      # cols % block
    assert L.taco_compress(D(0, 128, -1, 128), 16, 0, Q(), 0, None) == INV
    assert L.taco_compress(D(0, 128, 4, 128), 16, 7, Q(), 0, None) == UNS      # dtype
    for bad_mode in (2, 3, 6, 8, -1):                                        # mode (flag 4 allowed)
        assert L.taco_compress(D(0, 128, 4, 128), 16, 0, Q(), bad_mode, None) == INV
    # pointer problems
    assert L.taco_compress(D(0, 128, 4, 128), None, 0, Q(), 0, None) == INV
    assert L.taco_compress(D(0, 128, 4, 128), 24, 0, Q(), 0, None) == ALN
    assert L.taco_compress(D(0, 128, 4, 128), 16, 0, Q(c=40), 0, None) == ALN
    assert L.taco_compress(D(0, 128, 4, 128), 16, 0, Q(st=None), 0, None) == INV
    assert L.taco_compress(D(0, 128, 4, 128), 16, 0, Q(st=18), 0, None) == ALN
    assert L.taco_compress(D(2, 128, 4, 128), 16, 1, Q(z=None), 0, None) == INV
    assert L.taco_compress(D(2, 128, 4, 128), 16, 1, Q(s=17), 0, None) == ALN
    assert L.taco_compress(D(1, 64, 4, 128), 16, 1, Q(s=18), 0, None) == ALN
    # too many segments for 32-bit tile coordinates
    assert L.taco_compress(D(0, 128, 1 << 20, 1 << 17), 16, 0, Q(), 0, None) == UNS
    # empty tensors are a no-op
    assert L.taco_compress(D(0, 128, 0, 128), None, 0, None, 0, None) == OK
    assert L.taco_decompress(D(0, 128, 4, 0), None, None, 0, None) == OK
    # decompress / reduce / requant / update / copy checks
    assert L.taco_decompress(D(0, 128, 4, 128), Q(), 24, 0, None) == ALN
    assert L.taco_decompress(D(0, 128, 4, 128), Q(), 16, 3, None) == UNS
    arr = (qta.QTensorC * 2)(qta.QTensorC(16, 16, 16, 16), qta.QTensorC(16, 16, 16, 16))
    assert L.qar_reduce(D(0, 128, 4, 128, 2), arr, 2, 0, 4, 16, None) == INV   # batch must be 1
    assert L.qar_reduce(D(0, 128, 4, 128), arr, 0, 0, 4, 16, None) == INV
    assert L.qar_reduce(D(0, 128, 4, 128), arr, 17, 0, 4, 16, None) == UNS
    assert L.qar_reduce(D(0, 128, 4, 128), arr, 2, 3, 2, 16, None) == INV
    assert L.qar_reduce(D(0, 128, 4, 128), arr, 2, 0, 5, 16, None) == INV
    assert L.qar_reduce(D(0, 128, 4, 128), arr, 2, 2, 2, 16, None) == OK      # empty range
    assert L.qar_reduce(D(0, 128, 4, 128), arr, 2, 0, 4, 24, None) == ALN
    assert L.qar_reduce(D(0, 128, 4, 128), None, 2, 0, 4, 16, None) == INV
    bad = (qta.QTensorC * 2)(qta.QTensorC(16, 16, 16, 16), qta.QTensorC(8, 16, 16, 16))
    assert L.qar_reduce(D(0, 128, 4, 128), bad, 2, 0, 4, 16, None) == ALN
    assert L.qar_requant(D(0, 128, 4, 128), 20, Q(), 0, None) == ALN
    assert L.taco_update_scale(None, 3, None) == INV
    assert L.taco_update_scale(18, 3, None) == ALN
    assert L.taco_update_scale(None, 0, None) == OK
    assert L.taco_update_scale(16, -1, None) == INV
    assert L.qta_copy(16, 32, 24, None) == ALN
    assert L.qta_copy(None, 32, 32, None) == INV
    assert L.qta_copy(16, 32, 0, None) == OK
    assert L.qta_device_error(None, 0) == INV
    assert L.qta_status_string(qta.QTA_ERR_ALIGNMENT) == b"QTA_ERR_ALIGNMENT"


def test_reduce_requant_argument_checks(L):
    D = lambda *a: ctypes.byref(qta.desc(*a))
    OK, INV, ALN, UNS = qta.QTA_OK, qta.QTA_ERR_INVALID_ARG, qta.QTA_ERR_ALIGNMENT, qta.QTA_ERR_UNSUPPORTED
    arr = (qta.QTensorC * 2)(qta.QTensorC(16, 16, 16, 16), qta.QTensorC(16, 16, 16, 16))
    out = ctypes.byref(qta.QTensorC(16, 16, 16, 16))
    f = L.qar_reduce_requant
    assert f(D(0, 128, 8, 256), arr, 2, 0, 8, D(1, 64, 8, 256), out, 0, None) == UNS     # TACO -> INT8
    assert f(D(2, 128, 8, 256), arr, 2, 0, 8, D(0, 128, 8, 256), out, 0, None) == UNS
    assert f(D(0, 128, 8, 256), arr, 2, 0, 8, D(0, 128, 3, 256, 2), out, 0, None) == INV  # 2*3 != 8 rows
    assert f(D(0, 128, 8, 256), arr, 2, 0, 8, D(0, 128, 8, 512), out, 0, None) == INV    # cols differ
    assert f(D(0, 128, 8, 256), arr, 2, 0, 8, D(0, 128, 4, 256, 2), out, 7, None) == INV  # mode
    assert f(D(0, 128, 8, 256), arr, 2, 4, 4, D(0, 128, 0, 256, 1), out, 0, None) == OK   # empty range
    assert f(D(0, 128, 8, 256), arr, 2, 0, 8, D(0, 128, 4, 256, 2),
             ctypes.byref(qta.QTensorC(24, 16, 16, 16)), 0, None) == ALN
    assert f(D(0, 128, 8, 256), arr, 17, 0, 8, D(0, 128, 8, 256), out, 0, None) == UNS
    assert f(D(2, 128, 8, 256), arr, 2, 0, 8, D(3, 128, 8, 256),
             ctypes.byref(qta.QTensorC(16, 16, None, 16)), 0, None) == INV                # zeros needed


def test_ring_hop_argument_checks(L):
    D = lambda *a: ctypes.byref(qta.desc(*a))
    q = ctypes.byref(qta.QTensorC(16, 16, 16, 16))
    OK, INV, ALN, UNS = qta.QTA_OK, qta.QTA_ERR_INVALID_ARG, qta.QTA_ERR_ALIGNMENT, qta.QTA_ERR_UNSUPPORTED
    f, g = L.qar_dequant_add, L.qar_dequant_add_requant
    assert f(None, q, 16, 0, 16, None) == INV
    assert f(D(0, 96, 4, 192), q, 16, 0, 16, None) == UNS
    assert f(D(0, 128, 4, 128), q, 16, 5, 16, None) == UNS          # x dtype
    assert f(D(0, 128, 4, 128), q, None, 0, 16, None) == INV
    assert f(D(0, 128, 4, 128), q, 16, 0, None, None) == INV         # no sum buffer
    assert f(D(0, 128, 4, 128), q, 24, 0, 16, None) == ALN
    assert f(D(0, 128, 4, 128), q, 16, 0, 40, None) == ALN
    assert f(D(0, 128, 4, 128), None, 16, 0, 16, None) == INV
    assert f(D(0, 128, 4, 128), ctypes.byref(qta.QTensorC(16, 16, 16, None)), 16, 0, 16, None) == INV
    assert f(D(0, 128, 0, 128), None, None, 0, None, None) == OK     # empty
    assert g(D(0, 128, 4, 128), q, 16, 0, None, 0, None) == INV      # no output tensor
    assert g(D(0, 128, 4, 128), q, 16, 0, q, 9, None) == INV         # TACO scale mode
    assert g(D(2, 128, 4, 256), q, 16, 1, ctypes.byref(qta.QTensorC(16, 16, None, 16)), 0, None) == INV
    assert g(D(1, 64, 4, 128), q, 16, 2, ctypes.byref(qta.QTensorC(8, 16, 16, 16)), 0, None) == ALN


def test_descriptor_layout_and_sm_cap(L):
    # the C layout: two int32, three int64, one int32 (+ padding)
    assert ctypes.sizeof(qta.Desc) == 40
    assert qta.Desc.max_sms.offset == 32
    d = qta.desc("taco_fp8", 128, 4, 256, max_sms=48)
    assert d.max_sms == 48 and qta.desc("int8_sym", 64, 1, 64).max_sms == 0
    bad = qta.desc("taco_fp8", 128, 4, 256, max_sms=-1)
    assert L.taco_compress(ctypes.byref(bad), 16, 0, ctypes.byref(qta.QTensorC(16, 16, 16, 16)), 0,
                           None) == qta.QTA_ERR_INVALID_ARG


def test_sq_error_argument_checks(L):
    OK, INV, ALN, UNS = qta.QTA_OK, qta.QTA_ERR_INVALID_ARG, qta.QTA_ERR_ALIGNMENT, qta.QTA_ERR_UNSUPPORTED
    f = L.qta_sq_error
    assert f(16, 7, 16, 4, 16, None) == UNS
    assert f(16, 0, 16, -1, 16, None) == INV
    assert f(16, 0, 16, 4, None, None) == INV
    assert f(None, 0, 16, 4, 16, None) == INV
    assert f(16, 0, 18, 4, 16, None) == ALN
    assert f(16, 0, 16, 4, 20, None) == ALN


def test_ring_hop_rejects_overlapping_outputs(L):
    # an output that overlaps the local tensor x or a buffer of the incoming
    # tensor is refused on the host, before anything is enqueued (the
    # addresses below are never dereferenced)
    INV = qta.QTA_ERR_INVALID_ARG
    d = ctypes.byref(qta.desc(0, 128, 4, 128))                  # TACO, 512 elements
    qin = qta.QTensorC(0x100000, 0x200000, 0x300000, 0x400000)
    x = 0x500000                                                # bf16: 1024 bytes
    f, g = L.qar_dequant_add, L.qar_dequant_add_requant
    assert f(d, ctypes.byref(qin), x, 0, x + 512, None) == INV            # sum_out inside x
    assert f(d, ctypes.byref(qin), x, 0, x - 2032, None) == INV           # sum_out's end inside x
    assert f(d, ctypes.byref(qin), x, 0, 0x100000 - 16, None) == INV      # over the incoming codes
    assert f(d, ctypes.byref(qin), x, 0, 0x400000, None) == INV           # over the incoming state
    out = qta.QTensorC(0x600000, 0x700000, 0x800000, 0x200000)            # out state = in scales
    assert g(d, ctypes.byref(qin), x, 0, ctypes.byref(out), 0, None) == INV
    out = qta.QTensorC(x, 0x700000, 0x800000, 0x900000)                   # out codes = x
    assert g(d, ctypes.byref(qin), x, 0, ctypes.byref(out), 0, None) == INV


def test_ring_rejects_fewer_than_two_ranks():
    from quantized_tensor_activation_gb300 import ring
    with pytest.raises(ValueError):
        ring._chunk_desc(qta.desc("taco_fp8", 128, 4, 256), 1)
    assert ring._chunk_desc(qta.desc("taco_fp8", 128, 4, 256), 2).rows == 2


def test_rescaling_argument_checks(L):
    OK, INV, ALN, UNS = qta.QTA_OK, qta.QTA_ERR_INVALID_ARG, qta.QTA_ERR_ALIGNMENT, qta.QTA_ERR_UNSUPPORTED
    assert L.qta_chan_bytes(256) == 3 * 256 * 4 and L.qta_chan_bytes(0) == 0 and L.qta_chan_bytes(-5) == 0
    d = ctypes.byref(qta.desc(0, 128, 4, 256))
    f = L.taco_channel_amax
    assert f(d, 0x100000, 7, 0x200000, None) == UNS                    # dtype
    assert f(d, None, 0, 0x200000, None) == INV
    assert f(d, 0x100000, 0, None, None) == INV
    assert f(d, 0x100008, 0, 0x200000, None) == ALN
    assert f(d, 0x100000, 0, 0x200004, None) == ALN
    assert f(d, 0x100000, 0, 0x100000 + 1024, None) == INV             # chan inside x
    assert f(ctypes.byref(qta.desc(0, 128, 0, 256)), None, 0, None, None) == OK   # empty
    g = L.taco_ash_update
    assert g(None, 0, None) == OK and g(None, -1, None) == INV and g(None, 4, None) == INV
    assert g(0x200004, 4, None) == ALN
    # the factors go with TACO only, 16-byte aligned (checked before anything runs)
    q = ctypes.byref(qta.QTensorC(0x100000, 0x200000, 0x300000, 0x400000, 0x500000))
    assert L.taco_compress(ctypes.byref(qta.desc(1, 64, 4, 256)), 0x600000, 0, q, 0, None) == UNS
    qm = ctypes.byref(qta.QTensorC(0x100000, 0x200000, 0x300000, 0x400000, 0x500008))
    assert L.taco_compress(d, 0x600000, 0, qm, 0, None) == ALN
    # the ring hops take no rescaling
    out = ctypes.byref(qta.QTensorC(0x700000, 0x800000, 0x900000, 0xA00000, None))
    assert L.qar_dequant_add_requant(d, q, 0x600000, 0, out, 0, None) == UNS
    assert L.qar_dequant_add(d, q, 0x600000, 0, 0xB00000, None) == UNS
