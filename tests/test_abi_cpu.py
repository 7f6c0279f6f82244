"""Host-side checks of the C ABI that need no GPU: the library builds for sm_103a,
loads, exports every entry point include/lq.h declares, and its validation
rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

import bit_weight_quantized_dequant_gb300 as lq
from bit_weight_quantized_dequant_gb300 import _lq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = lq.build()
    return _lq.load_library(build_if_missing=False), path


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "lq.h")).read()
    return sorted(set(re.findall(r"LQ_API\s+[\w\s\*]+?\b(lq_\w+)\s*\(", src)))


def test_header_declares_the_binding_list():
    assert declared_symbols() == sorted(_lq.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    _, path = lib
    assert sorted(_lq.exported_symbols(path)) == declared_symbols()


def test_status_strings(lib):
    L, _ = lib
    for s in range(8):
        assert L.lq_status_string(s) != b"unknown status"
    assert L.lq_status_string(99) == b"unknown status"


def test_anchor_count_is_the_oracles(lib):
    """The library's default anchor count (floor of 3.5 % of K) equals the oracle's, which the
    oracle pins test ties to the listed workloads (8 at K = 256, 143 at 4096, ...)."""
    from oracle import oracle as O
    L, _ = lib
    for K in list(range(0, 2049)) + [4096, 5120, 8192, 11008, 13824, 28672, 1 << 20]:
        assert L.lq_anchor_count(K) == (O.anchor_count(K) if K > 0 else 0), K
    assert L.lq_anchor_count(-5) == 0


def _fake_handle():
    # Only used with arguments that fail validation, which happens before the handle is read.
    return ctypes.c_void_p(0x1000)


def test_validation_rejects_before_launch(lib):
    L, _ = lib
    h = _fake_handle()
    A16 = 0x10000          # 16-byte aligned fake device addresses (never dereferenced)
    # null handle
    assert L.lq_dequant(None, 1, A16, A16, A16, None, None, 0, 0, A16, 0, 4, 64, None) == _lq.LQ_ERR_INVALID_ARG
    # bad format
    assert L.lq_dequant(h, 7, A16, A16, A16, None, None, 0, 0, A16, 0, 4, 64, None) == _lq.LQ_ERR_INVALID_ARG
    # K not a multiple of the group
    assert L.lq_dequant(h, 1, A16, A16, A16, None, None, 0, 0, A16, 0, 4, 48, None) == _lq.LQ_ERR_INVALID_ARG
    # NF4 needs K % 64
    assert L.lq_dequant(h, 2, A16, A16, None, None, None, 0, 0, A16, 0, 4, 96, None) == _lq.LQ_ERR_INVALID_ARG
    # misaligned codes pointer
    assert L.lq_dequant(h, 1, A16 + 4, A16, A16, None, None, 0, 0, A16, 0, 4, 64, None) == _lq.LQ_ERR_ALIGNMENT
    # anchors given but no pointers
    assert L.lq_dequant(h, 1, A16, A16, A16, None, None, 3, 8, A16, 0, 4, 64, None) == _lq.LQ_ERR_INVALID_ARG
    # ld_anchor not a multiple of 8
    assert L.lq_dequant(h, 1, A16, A16, A16, A16, A16, 3, 4 + 1, A16, 0, 4, 64, None) == _lq.LQ_ERR_ALIGNMENT
    # ld_anchor < A
    assert L.lq_dequant(h, 1, A16, A16, A16, A16, A16, 9, 8, A16, 0, 4, 64, None) == _lq.LQ_ERR_INVALID_ARG
    # anchors with NF4
    assert L.lq_dequant(h, 2, A16, A16, None, A16, A16, 1, 8, A16, 0, 4, 64, None) == _lq.LQ_ERR_INVALID_ARG
    # bad output dtype
    assert L.lq_dequant(h, 1, A16, A16, A16, None, None, 0, 0, A16, 9, 4, 64, None) == _lq.LQ_ERR_INVALID_ARG
    # gemv: M out of range, bad x dtype, misaligned y
    assert L.lq_gemv(h, 1, A16, A16, A16, None, None, 0, 0, A16, 1, A16, 0, 33, 4, 64, None) == _lq.LQ_ERR_UNSUPPORTED
    assert L.lq_gemv(h, 1, A16, A16, A16, None, None, 0, 0, A16, 1, A16, 0, 0, 4, 64, None) == _lq.LQ_ERR_UNSUPPORTED
    assert L.lq_gemv(h, 1, A16, A16, A16, None, None, 0, 0, A16, 0, A16, 0, 1, 4, 64, None) == _lq.LQ_ERR_INVALID_ARG
    assert L.lq_gemv(h, 1, A16, A16, A16, None, None, 0, 0, A16, 1, A16 + 2, 0, 1, 4, 64, None) == _lq.LQ_ERR_ALIGNMENT
    # gemm: K % 64
    assert L.lq_gemm(h, 1, A16, A16, A16, None, None, 0, 0, A16, 2, A16, 0, 256, 4, 96, None) == _lq.LQ_ERR_UNSUPPORTED
    # NF4 with double quantization (format 4): needs the second-level constants, 16-byte
    # aligned, and no anchors
    assert L.lq_dequant(h, 4, A16, A16, None, None, None, 0, 0, A16, 0, 4, 64, None) == _lq.LQ_ERR_INVALID_ARG
    assert L.lq_dequant(h, 4, A16, A16, A16 + 4, None, None, 0, 0, A16, 0, 4, 64, None) == _lq.LQ_ERR_ALIGNMENT
    assert L.lq_dequant(h, 4, A16, A16, A16, A16, A16, 1, 8, A16, 0, 4, 64, None) == _lq.LQ_ERR_INVALID_ARG
    assert L.lq_dequant(h, 4, A16, A16, A16, None, None, 0, 0, A16, 0, 4, 96, None) == _lq.LQ_ERR_INVALID_ARG
    assert L.lq_gemm(h, 4, A16, A16, A16, None, None, 0, 0, A16, 2, A16, 0, 256, 4, 96, None) == _lq.LQ_ERR_INVALID_ARG


def test_grouped_validation(lib):
    L, _ = lib
    h = _fake_handle()
    A16 = 0x10000
    p = _lq.lq_problem()
    p.format, p.M, p.N, p.K = 1, 1, 64, 256
    p.codes = p.scales = p.offsets = p.x = p.y = A16
    p.x_dtype, p.y_dtype, p.batch = 1, 0, 1
    q = _lq.lq_problem.from_buffer_copy(p)
    q.M = 2                                         # mixed M in one launch
    arr = (_lq.lq_problem * 2)(p, q)
    assert L.lq_gemv_grouped(h, arr, 2, None) == _lq.LQ_ERR_UNSUPPORTED
    assert L.lq_gemv_grouped(h, arr, 0, None) == _lq.LQ_ERR_INVALID_ARG
    big = (_lq.lq_problem * 17)(*([p] * 17))
    assert L.lq_gemv_grouped(h, big, 17, None) == _lq.LQ_ERR_UNSUPPORTED
    r = _lq.lq_problem.from_buffer_copy(p)
    r.batch, r.stride_codes = 2, 8                  # stride not a multiple of 16 bytes
    assert L.lq_gemv_grouped(h, (_lq.lq_problem * 1)(r), 1, None) == _lq.LQ_ERR_ALIGNMENT


def test_layers_validation(lib):
    """lq_gemv_layers rejects bad layer lists on the host, before the handle or a device is touched."""
    L, _ = lib
    h = _fake_handle()
    A16 = 0x10000
    p = _lq.lq_problem()
    p.format, p.M, p.N, p.K = 1, 1, 64, 256
    p.codes = p.scales = p.offsets = p.x = p.y = A16
    p.x_dtype, p.y_dtype, p.batch = 1, 0, 1
    q = _lq.lq_problem.from_buffer_copy(p)
    q.M = 2
    arr = (_lq.lq_problem * 3)(p, p, q)
    counts = (ctypes.c_int * 2)(1, 2)                # the second layer mixes M
    assert L.lq_gemv_layers(h, arr, counts, 2, None) == _lq.LQ_ERR_UNSUPPORTED
    assert L.lq_gemv_layers(h, arr, counts, 0, None) == _lq.LQ_ERR_INVALID_ARG
    assert L.lq_gemv_layers(h, arr, None, 1, None) == _lq.LQ_ERR_INVALID_ARG
    zero = (ctypes.c_int * 2)(1, 0)
    assert L.lq_gemv_layers(h, arr, zero, 2, None) == _lq.LQ_ERR_INVALID_ARG
    big = (_lq.lq_problem * 17)(*([p] * 17))
    assert L.lq_gemv_layers(h, big, (ctypes.c_int * 1)(17), 1, None) == _lq.LQ_ERR_UNSUPPORTED
    r = _lq.lq_problem.from_buffer_copy(p)
    r.batch, r.stride_codes = 2, 8                  # stride not a multiple of 16 bytes
    assert L.lq_gemv_layers(h, (_lq.lq_problem * 2)(p, r), (ctypes.c_int * 2)(1, 1), 2, None) == _lq.LQ_ERR_ALIGNMENT


def test_create_without_device_reports_error(lib):
    """No GPU in this container: lq_create must fail cleanly, not crash."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L, _ = lib
    h = ctypes.c_void_p()
    st = L.lq_create(ctypes.byref(h), 0, 0)
    assert st in (_lq.LQ_ERR_CUDA, _lq.LQ_ERR_INVALID_ARG) and not h.value


def test_gemm_grouped_validation(lib):
    """lq_gemm_grouped rejects bad groups on the host, before the handle or a device is touched."""
    L, _ = lib
    h = _fake_handle()
    A16 = 0x10000

    def prob(fmt=1, K=256, batch=1, xdt=2):
        p = _lq.lq_problem()
        p.format, p.M, p.N, p.K = fmt, 256, 128, K
        p.codes = p.scales = p.x = p.y = A16
        p.offsets = A16 if fmt == 1 else None
        p.x_dtype, p.y_dtype, p.batch = xdt, 0, batch
        return p

    def call(ps):
        arr = (_lq.lq_problem * len(ps))(*ps)
        return L.lq_gemm_grouped(h, arr, len(ps), None)

    assert L.lq_gemm_grouped(h, None, 1, None) == _lq.LQ_ERR_INVALID_ARG
    assert call([prob() for _ in range(9)]) == _lq.LQ_ERR_UNSUPPORTED          # more than 8 problems
    assert call([prob(), prob(fmt=2)]) == _lq.LQ_ERR_UNSUPPORTED                # mixed formats
    assert call([prob(), prob(xdt=1)]) == _lq.LQ_ERR_UNSUPPORTED                # mixed x dtypes
    assert call([prob(batch=2)]) == _lq.LQ_ERR_UNSUPPORTED                      # batched members
    assert call([prob(K=96)]) == _lq.LQ_ERR_UNSUPPORTED                         # the tensor-core path needs K % 64


def test_quantizer_validation(lib):
    """The quantizer entry points reject bad shapes, pointers and alignment on the host."""
    L, _ = lib
    h = _fake_handle()
    A16 = 0x10000
    INV, ALN = _lq.LQ_ERR_INVALID_ARG, _lq.LQ_ERR_ALIGNMENT
    assert L.lq_select_anchors(None, A16, 4, 64, None, 2, A16, None) == INV
    assert L.lq_select_anchors(h, A16, 4, 64, None, 65, A16, None) == INV        # A > K
    assert L.lq_select_anchors(h, A16, 4, 64, None, 2, None, None) == INV        # no output
    assert L.lq_select_anchors(h, A16 + 4, 4, 64, None, 2, A16, None) == ALN
    assert L.lq_select_anchors(h, A16, 4, 64, A16 + 8, 2, A16, None) == ALN      # profile
    assert L.lq_quantize_2bit(h, A16, 4, 48, None, 0, A16, A16, A16, None, 0, None) == INV    # K % 32
    assert L.lq_quantize_2bit(h, A16, 4, 64, None, 2, A16, A16, A16, None, 8, None) == INV    # anchors, no pointers
    assert L.lq_quantize_2bit(h, A16, 4, 64, A16, 2, A16, A16, A16, A16, 1, None) == INV      # ld_anchor < A
    assert L.lq_quantize_2bit(h, A16, 4, 64, A16, 2, A16, A16, A16, A16, 12, None) == ALN     # ld_anchor % 8
    assert L.lq_quantize_2bit(h, A16, 4, 64, None, 0, A16 + 8, A16, A16, None, 0, None) == ALN
    assert L.lq_quantize_2bit(h, A16, 0, 64, None, 0, A16, A16, A16, None, 0, None) == INV
    assert L.lq_quantize_nf4(h, A16, 4, 96, A16, A16, None) == INV                # K % 64
    assert L.lq_quantize_nf4(h, A16, 4, 64, A16, A16 + 4, None) == ALN
    assert L.lq_quantize_nf4(None, A16, 4, 64, A16, A16, None) == INV


def test_stream_null_arguments(lib):
    """lq_stream_* reject a missing object or handle without touching a device."""
    L, _ = lib
    out = ctypes.c_void_p()
    assert L.lq_stream_create(ctypes.byref(out), None, 1 << 20) == _lq.LQ_ERR_INVALID_ARG
    assert L.lq_stream_create(None, _fake_handle(), 1 << 20) == _lq.LQ_ERR_INVALID_ARG
    assert L.lq_stream_run(None, 0x10000, 256, 256, 1, None, 1, 0, None) == _lq.LQ_ERR_INVALID_ARG
    assert L.lq_stream_destroy(None) == _lq.LQ_OK


def test_selftest_wait_validation(lib):
    L, _ = lib
    assert L.lq_selftest_wait(None, 1000, None) == _lq.LQ_ERR_INVALID_ARG
    assert L.lq_selftest_wait(_fake_handle(), 0, None) == _lq.LQ_ERR_INVALID_ARG
    assert L.lq_selftest_wait(_fake_handle(), 2000000, None) == _lq.LQ_ERR_INVALID_ARG
