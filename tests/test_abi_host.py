"""Host-side checks of the C ABI that need no GPU: the library builds, loads
and exports every entry point declared in include/qmm.h, and argument
validation rejects bad calls before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import mat_mul_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"QMM_API\s+[\w\s\*]*?\b(qmm\w*)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for want in ("qmm", "qmm_dequant", "qmm_quantize_act", "qmm_strerror", "qmm_last_error"):
        assert want in names


def test_library_exports_every_declared_symbol():
    path = q.build()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in _declared_symbols() if n not in exported]
    assert not missing, missing
    L = q.load()
    for n in _declared_symbols():
        assert hasattr(L, n)


def test_strerror_names():
    assert q._strerror(q.QMM_OK) == "QMM_OK"
    assert q._strerror(q.QMM_ETIMEOUT) == "QMM_ETIMEOUT"
    assert q._strerror(-99) == "QMM_UNKNOWN"


def test_validation_rejects_before_launch():
    L = q.load()
    null = ctypes.c_void_p(0)
    # unknown type
    assert L.qmm(7, null, 1, 256, null, 1, null, null) == q.QMM_EINVAL_TYPE
    assert b"unknown block type" in L.qmm_last_error()
    # K not a multiple of the block
    assert L.qmm(q.Q4_K, null, 4, 300, null, 1, null, null) == q.QMM_EINVAL_SHAPE
    assert L.qmm(q.Q8_0, null, 4, 48, null, 1, null, null) == q.QMM_EINVAL_SHAPE
    # negative sizes
    assert L.qmm(q.Q6_K, null, -1, 256, null, 1, null, null) == q.QMM_EINVAL_SHAPE
    assert L.qmm(q.Q6_K, null, 1, 256, null, -2, null, null) == q.QMM_EINVAL_SHAPE
    # null pointers on a non-empty problem
    assert L.qmm(q.Q6_K, null, 1, 256, null, 1, null, null) == q.QMM_EINVAL_PTR
    # misaligned W
    buf = ctypes.create_string_buffer(4096)
    base = (ctypes.addressof(buf) + 15) & ~15
    assert L.qmm(q.Q4_K, ctypes.c_void_p(base + 2), 1, 256, ctypes.c_void_p(base),
                 1, ctypes.c_void_p(base), null) == q.QMM_EINVAL_PTR
    # dequant
    assert L.qmm_dequant(6, null, 32, null) == q.QMM_EINVAL_TYPE
    assert L.qmm_dequant(q.Q4_K, null, 100, null) == q.QMM_EINVAL_SHAPE
    assert L.qmm_dequant(q.Q4_K, null, 256, null) == q.QMM_EINVAL_PTR
    assert L.qmm_quantize_act(null, 1, 33, null, null, null, null) == q.QMM_EINVAL_SHAPE


def test_group_validation_rejects_before_launch():
    L = q.load()
    null = ctypes.c_void_p(0)
    I64 = ctypes.c_int64

    def arrays(types, ns, ws=None, ys=None):
        n = len(types)
        return ((ctypes.c_int * n)(*types), (ctypes.c_void_p * n)(*(ws or [0] * n)),
                (I64 * n)(*ns), (ctypes.c_void_p * n)(*(ys or [0] * n)))
    t, w, n, y = arrays([q.Q4_K], [4])
    assert L.qmm_group(0, t, w, n, 256, null, 1, y, null) == q.QMM_EINVAL_SHAPE
    assert L.qmm_group(9, t, w, n, 256, null, 1, y, null) == q.QMM_EINVAL_SHAPE
    assert L.qmm_group(1, null, w, n, 256, null, 1, y, null) == q.QMM_EINVAL_PTR
    t, w, n, y = arrays([q.Q4_K, 7], [4, 4])
    assert L.qmm_group(2, t, w, n, 256, null, 1, y, null) == q.QMM_EINVAL_TYPE
    # K must suit every type of the group
    t, w, n, y = arrays([q.Q8_0, q.Q6_K], [4, 4])
    assert L.qmm_group(2, t, w, n, 96, null, 1, y, null) == q.QMM_EINVAL_SHAPE
    # a null W or y on a non-empty entry, found before anything runs
    buf = ctypes.create_string_buffer(4096)
    base = (ctypes.addressof(buf) + 15) & ~15
    t, w, n, y = arrays([q.Q4_K, q.Q6_K], [4, 4], ws=[base, 0], ys=[base, base])
    assert L.qmm_group(2, t, w, n, 256, ctypes.c_void_p(base), 1, y, null) == q.QMM_EINVAL_PTR
    assert b"entry 1" in L.qmm_last_error()
    # empty entries and M = 0 are no-ops without a launch
    before = L.qmm_launch_count()
    t, w, n, y = arrays([q.Q4_K, q.Q6_K], [0, 0])
    assert L.qmm_group(2, t, w, n, 256, null, 1, y, null) == q.QMM_OK
    t, w, n, y = arrays([q.Q4_K], [5])
    assert L.qmm_group(1, t, w, n, 256, null, 0, y, null) == q.QMM_OK
    assert L.qmm_launch_count() == before


def test_empty_problems_are_noops():
    L = q.load()
    null = ctypes.c_void_p(0)
    before = L.qmm_launch_count()
    assert L.qmm(q.Q4_K, null, 0, 256, null, 3, null, null) == q.QMM_OK
    assert L.qmm(q.Q4_K, null, 5, 256, null, 0, null, null) == q.QMM_OK
    assert L.qmm_dequant(q.Q6_K, null, 0, null) == q.QMM_OK
    assert L.qmm_quantize_act(null, 0, 64, null, null, null, null) == q.QMM_OK
    assert L.qmm_launch_count() == before


def test_binding_refuses_host_tensors():
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        q.qmm(q.Q4_K, torch.zeros(144, dtype=torch.uint8), 1, 256, torch.zeros(1, 256))


def test_decode_path_setter_validates_and_returns_the_previous_path():
    import mat_mul_gb300 as q
    L = q.load()
    assert L.qmm_set_decode_path(q.DECODE_BLOCK) == q.DECODE_AUTO
    assert L.qmm_set_decode_path(q.DECODE_TENSOR) == q.DECODE_BLOCK
    assert L.qmm_set_decode_path(7) == q.QMM_EINVAL_SHAPE
    assert b"decode path" in L.qmm_last_error()
    assert L.qmm_set_decode_path(q.DECODE_AUTO) == q.DECODE_TENSOR
    with pytest.raises(q.QmmError):
        q.set_decode_path(-1)


def test_qmm_t_validation_rejects_before_launch():
    L = q.load()
    null = ctypes.c_void_p(0)
    before = L.qmm_launch_count()
    # the KV cache format only
    assert L.qmm_t(q.Q4_K, null, 1, 4, 128, null, 1, null, null) == q.QMM_EINVAL_TYPE
    assert b"Q8_0" in L.qmm_last_error()
    assert L.qmm_t(9, null, 1, 4, 128, null, 1, null, null) == q.QMM_EINVAL_TYPE
    # K a multiple of 32, at most 256; sizes >= 0; H <= 65535
    assert L.qmm_t(q.Q8_0, null, 1, 4, 48, null, 1, null, null) == q.QMM_EINVAL_SHAPE
    assert L.qmm_t(q.Q8_0, null, 1, 4, 288, null, 1, null, null) == q.QMM_EINVAL_SHAPE
    assert L.qmm_t(q.Q8_0, null, -1, 4, 128, null, 1, null, null) == q.QMM_EINVAL_SHAPE
    assert L.qmm_t(q.Q8_0, null, 1, -4, 128, null, 1, null, null) == q.QMM_EINVAL_SHAPE
    assert L.qmm_t(q.Q8_0, null, 1, 4, 128, null, -1, null, null) == q.QMM_EINVAL_SHAPE
    assert L.qmm_t(q.Q8_0, null, 70000, 4, 128, null, 1, null, null) == q.QMM_EINVAL_SHAPE
    # empty problems
    assert L.qmm_t(q.Q8_0, null, 0, 4, 128, null, 1, null, null) == q.QMM_OK
    assert L.qmm_t(q.Q8_0, null, 2, 4, 128, null, 0, null, null) == q.QMM_OK
    assert L.qmm_t(q.Q8_0, null, 2, 4, 0, null, 3, null, null) == q.QMM_OK
    # null and misaligned pointers
    assert L.qmm_t(q.Q8_0, null, 1, 4, 128, null, 1, null, null) == q.QMM_EINVAL_PTR
    buf = ctypes.create_string_buffer(4096)
    base = (ctypes.addressof(buf) + 15) & ~15
    assert L.qmm_t(q.Q8_0, ctypes.c_void_p(base + 2), 1, 4, 128, ctypes.c_void_p(base), 1,
                   ctypes.c_void_p(base), null) == q.QMM_EINVAL_PTR
    assert L.qmm_t(q.Q8_0, ctypes.c_void_p(base), 1, 4, 128, ctypes.c_void_p(base + 2), 1,
                   ctypes.c_void_p(base), null) == q.QMM_EINVAL_PTR
    assert L.qmm_launch_count() == before


def test_other_k_quants_validation():
    """Q5_K, Q3_K and Q2_K: qmm_dequant and the products validate them like
    the others; qmm_t (the q8_0 KV cache) and qmm_noalloc reject them."""
    L = q.load()
    null = ctypes.c_void_p(0)
    for t in (q.Q5_K, q.Q3_K, q.Q2_K):
        assert L.qmm_dequant(t, null, 100, null) == q.QMM_EINVAL_SHAPE
        assert L.qmm_dequant(t, null, 256, null) == q.QMM_EINVAL_PTR
        assert L.qmm_dequant(t, null, 0, null) == q.QMM_OK
        assert L.qmm(t, null, 4, 128, null, 1, null, null) == q.QMM_EINVAL_SHAPE
        assert L.qmm(t, null, 4, 256, null, 1, null, null) == q.QMM_EINVAL_PTR
        assert L.qmm_t(t, null, 1, 4, 128, null, 1, null, null) == q.QMM_EINVAL_TYPE
        assert L.qmm_noalloc(t, null, 4, 256, null, 1, null, null) == q.QMM_EINVAL_TYPE
    assert L.qmm_dequant(6, null, 256, null) == q.QMM_EINVAL_TYPE
    assert L.qmm(6, null, 4, 256, null, 1, null, null) == q.QMM_EINVAL_TYPE



def test_prefill_path_setter_validates_and_returns_the_previous_path():
    L = q.load()
    assert L.qmm_set_prefill_path(q.PREFILL_INT8) == q.PREFILL_AUTO
    assert L.qmm_set_prefill_path(5) == q.QMM_EINVAL_SHAPE
    assert b"prefill path" in L.qmm_last_error()
    assert L.qmm_set_prefill_path(q.PREFILL_AUTO) == q.PREFILL_INT8
    with pytest.raises(q.QmmError):
        q.set_prefill_path(-1)


def test_noalloc_rejects_sizes_that_would_wrap_before_launch():
    """M*K products that wrap 64 bits (M*K = 2^67 here) or exceed the static
    scratch are rejected with QMM_EINVAL_SHAPE before anything is computed,
    and so is K > 2^24."""
    L = q.load()
    buf = ctypes.create_string_buffer(4096)
    base = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    before = L.qmm_launch_count()
    assert L.qmm_noalloc(q.Q4_K, base, 4, 1 << 24, base, 1 << 43, base, None) == q.QMM_EINVAL_SHAPE
    assert L.qmm_noalloc(q.Q8_0, base, 4, 1 << 14, base, (1 << 50) + 1, base, None) == q.QMM_EINVAL_SHAPE
    assert L.qmm_noalloc(q.Q4_K, base, 4, 1 << 25, base, 1, base, None) == q.QMM_EINVAL_SHAPE
    assert b"2^24" in L.qmm_last_error()
    assert L.qmm_noalloc(q.Q4_K, base, 4, 4096, base, 4097, base, None) == q.QMM_EINVAL_SHAPE
    assert b"scratch" in L.qmm_last_error()
    assert L.qmm_noalloc(q.Q5_K, base, 4, 256, base, 1, base, None) == q.QMM_EINVAL_TYPE
    assert b"Q8_0, Q4_K and Q6_K" in L.qmm_last_error()
    assert L.qmm_launch_count() == before


def test_noalloc_binding_checks_x_and_y():
    torch = pytest.importorskip("torch")
    W = torch.zeros(144, dtype=torch.uint8)
    x = torch.zeros(2, 256)
    y = torch.zeros(2, 1)
    # host tensors are refused before any size check reaches the library
    with pytest.raises(ValueError):
        q.qmm_noalloc(q.Q4_K, W, 1, 256, x, y)


def test_inject_stall_setter_validates_and_returns_the_previous_count():
    L = q.load()
    assert L.qmm_inject_stall(0) == 0
    assert L.qmm_inject_stall(2) == 0
    assert L.qmm_inject_stall(-1) == q.QMM_EINVAL_SHAPE
    assert L.qmm_inject_stall(0) == 2
    with pytest.raises(q.QmmError):
        q.inject_stall(-3)


def test_gate_up_validation_rejects_before_launch():
    L = q.load()
    null = ctypes.c_void_p(0)
    before = L.qmm_launch_count()
    assert L.qmm_gate_up(q.Q4_K, null, 9, null, 4, 256, null, 1, null, None) == q.QMM_EINVAL_TYPE
    assert L.qmm_gate_up(6, null, q.Q4_K, null, 4, 256, null, 1, null, None) == q.QMM_EINVAL_TYPE
    # K a multiple of both block sizes
    assert L.qmm_gate_up(q.Q8_0, null, q.Q4_K, null, 4, 96, null, 1, null, None) == q.QMM_EINVAL_SHAPE
    assert L.qmm_gate_up(q.Q4_K, null, q.Q4_K, null, -1, 256, null, 1, null, None) == q.QMM_EINVAL_SHAPE
    # empty problems launch nothing; null pointers on a real one are refused
    assert L.qmm_gate_up(q.Q4_K, null, q.Q4_K, null, 0, 256, null, 1, null, None) == q.QMM_OK
    assert L.qmm_gate_up(q.Q4_K, null, q.Q4_K, null, 4, 256, null, 0, null, None) == q.QMM_OK
    assert L.qmm_gate_up(q.Q4_K, null, q.Q4_K, null, 4, 256, null, 1, null, None) == q.QMM_EINVAL_PTR
    buf = ctypes.create_string_buffer(4096)
    base = (ctypes.addressof(buf) + 15) & ~15
    assert L.qmm_gate_up(q.Q4_K, ctypes.c_void_p(base), q.Q4_K, ctypes.c_void_p(base + 2), 4, 256,
                         ctypes.c_void_p(base), 1, ctypes.c_void_p(base), None) == q.QMM_EINVAL_PTR
    assert L.qmm_launch_count() == before
