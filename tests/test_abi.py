"""Host-side checks of the C ABI (no GPU needed).

The library builds, loads, and exports every function include/tj.h declares;
the ctypes binding knows each of them; argument and shape errors are reported
by status code before any launch (these calls return before touching a device).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "tj.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tj_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    path = __graft_entry__.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("tj_quantize_nvfp4", "tj_rht", "tj_linear_fwd", "tj_linear_bwd_dx", "tj_linear_bwd_dw",
              "tj_outlier_calibrate", "tj_osci_reset"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_covers_every_symbol():
    from nvfp4_bit_fully_gb300 import tj

    assert set(_declared()) <= set(tj.EXPORTED)


def test_status_strings_and_workspace(lib):
    from nvfp4_bit_fully_gb300 import tj

    l = tj.load()
    assert l.tj_status_str(0) == b"ok"
    assert l.tj_status_str(7) == b"workspace missing or too small"
    # dX workspace for 16384x4096x1024 with 103 outlier channels
    rp = lambda v: (v + 127) // 128 * 128
    def nv(r, c):
        return rp(r) * rp(c) // 2 + rp(r) * rp(c) // 16 + rp(r) * rp(c) // 128 * 4
    def mx(r, c):
        return rp(r) * rp(c) + rp(r) * rp(c) // 32
    assert tj.workspace_size(1, 16384, 4096, 1024, 103) == nv(16384, 4096) + nv(921, 4096) + mx(16384, 4096) + mx(103, 4096)
    assert tj.workspace_size(2, 256, 512, 512, 0) == nv(512, 256) + nv(512, 256)
    assert tj.workspace_size(1, 16, 16, 8, 9) == 0                       # k > K


def test_argument_errors_before_launch(lib):
    from nvfp4_bit_fully_gb300 import tj

    l = tj.load()
    q = tj.CNvfp4(0, 0, 0, 128, 128)
    # null input
    assert l.tj_quantize_nvfp4(None, 0, 128, 128, 128, 0, None, 0, 0, 0, 0, 0, 0, ctypes.byref(q), None) == 1
    # bad rounding mode
    assert l.tj_quantize_nvfp4(ctypes.c_void_p(256), 0, 128, 128, 128, 0, None, 0, 5, 0, 0, 0, 0,
                               ctypes.byref(q), None) == 1
    # misaligned input pointer (bf16 needs 2-byte alignment)
    assert l.tj_quantize_nvfp4(ctypes.c_void_p(257), 0, 128, 128, 128, 0, None, 0, 0, 0, 0, 0, 0,
                               ctypes.byref(q), None) == 3
    # output descriptor with null buffers
    assert l.tj_quantize_nvfp4(ctypes.c_void_p(256), 0, 128, 128, 128, 0, None, 0, 0, 0, 0, 0, 0,
                               ctypes.byref(q), None) == 1
    # RHT needs whole 128-blocks
    assert l.tj_rht(ctypes.c_void_p(256), ctypes.c_void_p(256), 4, 100, 0, 0, None) == 2
    # backward without workspace
    w = tj.CNvfp4(256, 256, 256, 128, 128)
    assert l.tj_linear_bwd_dx(ctypes.c_void_p(256), 128, 128, 128, ctypes.byref(w), None, None, None, 0, 1,
                              ctypes.c_void_p(256), 0, 128, None, 0, None) == 7
    # calibration: k larger than K
    assert l.tj_outlier_calibrate(None, 0, 0, 8, 8, ctypes.c_void_p(256), 1, 9, ctypes.c_void_p(256),
                                  ctypes.c_void_p(256), None) == 2


def test_block_count_limit(lib):
    """A descriptor whose padded size holds 2^31 or more 128-element blocks is a shape error,
    found before any launch."""
    from nvfp4_bit_fully_gb300 import tj

    l = tj.load()
    rows, cols = 1 << 24, 1 << 14                       # 2^24 rows x 128 blocks = 2^31 blocks
    q = tj.CNvfp4(256, 256, 256, rows, cols)
    assert l.tj_quantize_nvfp4(ctypes.c_void_p(256), 0, rows, cols, cols, 0, None, 0, 0, 0, 0, 0, 0,
                               ctypes.byref(q), None) == 2
    m = tj.CMxfp8(256, 256, rows, cols)
    assert l.tj_quantize_mxfp8(ctypes.c_void_p(256), 0, rows, cols, cols, 0, None, 0, ctypes.byref(m), None) == 2


def test_column_grid_limit(lib):
    """The transposed quantizers launch one grid row per 128 output columns (at most
    65535): a column quantization with more than 8,388,480 input rows, and the
    backward calls that would need one, are shape errors found before any launch."""
    from nvfp4_bit_fully_gb300 import tj

    l = tj.load()
    rows, cols = 65535 * 128 + 1, 128                   # one 128-block too many output columns
    q = tj.CNvfp4(256, 256, 256, cols, rows)            # transposed output [cols, rows]
    assert l.tj_quantize_nvfp4(ctypes.c_void_p(256), 0, rows, cols, cols, 1, None, 0, 0, 0, 0, 0, 0,
                               ctypes.byref(q), None) == 2
    m = tj.CMxfp8(256, 256, cols, rows)
    assert l.tj_quantize_mxfp8(ctypes.c_void_p(256), 0, rows, cols, cols, 1, None, 0, ctypes.byref(m), None) == 2
    src = tj.CNvfp4(256, 256, 256, rows, cols)
    assert l.tj_requantize_nvfp4(ctypes.byref(src), 1, 1, 0, 3, 0x100, ctypes.byref(q), None) == 2
    # dW over more tokens than the column grid holds
    xq = tj.CNvfp4(256, 256, 256, rows, 128)
    assert l.tj_linear_bwd_dw(ctypes.c_void_p(256), rows, 128, 128, ctypes.byref(xq), None, None, None, 0, 1,
                              ctypes.c_void_p(256), 128, ctypes.c_void_p(256), 1 << 40, None) == 2


def test_slice_format_checks(lib):
    """An MX slice descriptor with an unknown element format is an argument error, and packed
    FP6 / FP4 codes that do not start on 32 bytes an alignment error, before any launch."""
    from nvfp4_bit_fully_gb300 import tj

    l = tj.load()
    y = ctypes.c_void_p(256)
    assert ctypes.sizeof(tj.CMxfp8) == 40
    for fmt, want in ((1, 1), (2, 1), (6, 1), (-1, 1)):
        m = tj.CMxfp8(256, 256, 128, 128, fmt)
        assert l.tj_dequantize_mxfp8(ctypes.byref(m), y, 128, None) == want, fmt
    for fmt in (tj.TJ_MX_E2M3, tj.TJ_MX_E3M2, tj.TJ_MX_E2M1):
        m = tj.CMxfp8(256 + 16, 256, 128, 128, fmt)                 # 16- but not 32-byte aligned
        assert l.tj_dequantize_mxfp8(ctypes.byref(m), y, 128, None) == 3
        assert l.tj_quantize_mxfp8(ctypes.c_void_p(256), 0, 128, 128, 128, 0, None, 0, ctypes.byref(m), None) == 3
    m = tj.CMxfp8(256 + 16, 256, 128, 128, tj.TJ_MX_E4M3)           # E4M3 needs 16 bytes only
    assert l.tj_dequantize_mxfp8(ctypes.byref(m), y, 40, None) == 2   # (reaches the ldy check)


def test_binding_refuses_host_tensors(lib):
    """The binding marshals device tensors only: a host tensor, or a quantized tensor whose
    buffers live on the host, raises ValueError before any library call."""
    import torch

    from nvfp4_bit_fully_gb300 import tj

    x = torch.zeros(128, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        tj.quantize_nvfp4(x)
    with pytest.raises(ValueError, match="CUDA"):
        tj.dequantize_mxfp8(tj.MXFP8.empty(128, 256, device="cpu"))
    with pytest.raises(ValueError, match="CUDA"):
        tj.rht(torch.zeros(4, 128), 1, 2)


def test_binding_layout_dtype_and_length_rules(monkeypatch):
    """The binding's argument rules on host tensors, with its device check stubbed out: a
    matrix needs adjacent columns and a call's dtype; a single row is passed with its length
    as row stride; index lists are 1-D contiguous int32 with enough entries; state arrays
    are contiguous with the weight's size; a quantized tensor's buffers have their padded
    sizes."""
    import torch

    from nvfp4_bit_fully_gb300 import tj

    monkeypatch.setattr(tj, "_cuda", lambda t, name: None)
    x = torch.zeros(64, 256, dtype=torch.bfloat16)
    assert tj._mat(x, "x") is not None and tj._ld(x) == 256
    assert tj._ld(x[:, 8:72]) == 256                                     # a column slice keeps its row stride
    for bad, what in ((x.t(), "adjacent"), (x[:, ::2], "adjacent"), (x.float()[0], "2-D"),
                      (x.half(), "dtype")):
        with pytest.raises(ValueError, match=what):
            tj._mat(bad, "x")
    with pytest.raises(ValueError, match="dtype"):
        tj._mat(x, "x", tj._FP32)
    col = torch.zeros(256, 1, dtype=torch.bfloat16)
    assert tj._mat(col.t(), "x") is not None and tj._ld(col.t()) == 256   # one row: its own length
    idx = torch.arange(10, dtype=torch.int32)
    assert tj._idx(idx, "i", 10) is not None
    for bad, n, what in ((idx.long(), None, "dtype"), (idx[::2], None, "contiguous"), (idx.view(2, 5), None, "1-D"),
                         (idx, 11, "at least 11")):
        with pytest.raises(ValueError, match=what):
            tj._idx(bad, "i", n)
    st = torch.zeros(64, 256)
    assert tj._arr(st, "w", tj._FP32, st.numel()) is not None
    with pytest.raises(ValueError, match="elements"):
        tj._arr(st[:32], "w", tj._FP32, st.numel())
    with pytest.raises(ValueError, match="contiguous"):
        tj._arr(torch.zeros(64, 512)[:, :256], "w", tj._FP32, st.numel())
    q = tj.NVFP4.empty(100, 300, device="cpu")
    assert (q.codes.numel(), q.sf.numel(), q.outer.numel()) == (128 * 384 // 2, 128 * 384 // 16, 3 * 128)
    q.c()
    with pytest.raises(ValueError, match="codes"):
        tj.NVFP4(q.codes[:-1], q.sf, q.outer, 100, 300).c()
    with pytest.raises(ValueError, match="outer"):
        tj.NVFP4(q.codes, q.sf, q.outer.view(torch.int32), 100, 300).c()
    m = tj.MXFP8.empty(100, 300, device="cpu", fmt=tj.TJ_MX_E2M3)
    assert m.codes.numel() == 128 * 384 * 6 // 8
    m.c()
    m.fmt = 2
    with pytest.raises(ValueError, match="format"):
        m.c()
