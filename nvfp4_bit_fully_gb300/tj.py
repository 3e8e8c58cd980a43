"""ctypes binding of libtj (the C ABI in include/tj.h).

Argument marshalling only: every step of the NVFP4 linear path runs in the
CUDA kernels of libtj.  torch provides device memory and streams.  There is no
CPU fallback: if libtj.so is missing or no CUDA device is present, the calls
raise.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtj.so")

TJ_OK = 0
TJ_RTN, TJ_SR = 0, 1
TJ_BF16, TJ_FP32 = 0, 1
TJ_OP_BWD_DX, TJ_OP_BWD_DW, TJ_OP_FP8_BWD_DX, TJ_OP_FP8_BWD_DW = 1, 2, 3, 4
# element formats of an MX slice (E4M3 = the FP8 slice; E2M3 / E3M2 / E2M1 for FP6 x FP4)
TJ_MX_E4M3, TJ_MX_E2M3, TJ_MX_E3M2, TJ_MX_E2M1 = 0, 3, 4, 5
MX_BITS = {TJ_MX_E4M3: 8, TJ_MX_E2M3: 6, TJ_MX_E3M2: 6, TJ_MX_E2M1: 4}
TAG_DY_ROW, TAG_DY_COL, TAG_WT, TAG_XT = 1, 2, 3, 4
TAG_RHT_DX, TAG_RHT_DW = 0x100, 0x101
STATUS = {0: "ok", 1: "invalid argument", 2: "shape", 3: "alignment", 4: "unsupported", 5: "CUDA error",
          6: "device wait timed out", 7: "workspace"}


class TjError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s failed: %s (%d)" % (fn, STATUS.get(code, "?"), code))
        self.code = code


class CNvfp4(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("outer", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class CMxfp8(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("sf", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("fmt", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_U32 = ctypes.c_uint32
_U64 = ctypes.c_uint64
_F = ctypes.c_float
_SIGS = {
    "tj_quantize_nvfp4": [_P, _I, _I64, _I64, _I64, _I, _P, _I64, _I, _I, _U64, _U32, _U32, ctypes.POINTER(CNvfp4), _P],
    "tj_quantize_mxfp8": [_P, _I, _I64, _I64, _I64, _I, _P, _I64, ctypes.POINTER(CMxfp8), _P],
    "tj_quantize_split": [_P, _I, _I64, _I64, _I64, _P, _I64, _P, _I64, ctypes.POINTER(CNvfp4),
                          ctypes.POINTER(CMxfp8), _P],
    "tj_quantize_nvfp4_mxfp8": [_P, _I, _I64, _I64, _I64, _I, _P, _I64, _I, _I, _U64, _U32, _U32,
                                ctypes.POINTER(CNvfp4), ctypes.POINTER(CMxfp8), _P],
    "tj_requantize_nvfp4": [ctypes.POINTER(CNvfp4), _I, _I, _U64, _U32, _U32, ctypes.POINTER(CNvfp4), _P],
    "tj_requantize_mxfp8": [ctypes.POINTER(CMxfp8), ctypes.POINTER(CMxfp8), _P],
    "tj_requantize_nvfp4_mxfp8": [ctypes.POINTER(CNvfp4), _I, _I, _U64, _U32, _U32, ctypes.POINTER(CNvfp4),
                                  ctypes.POINTER(CMxfp8), ctypes.POINTER(CMxfp8), _P],
    "tj_rht": [_P, _P, _I64, _I64, _U64, _U32, _P],
    "tj_dequantize_nvfp4": [ctypes.POINTER(CNvfp4), _P, _I64, _P],
    "tj_dequantize_mxfp8": [ctypes.POINTER(CMxfp8), _P, _I64, _P],
    "tj_gemm_nvfp4": [ctypes.POINTER(CNvfp4), ctypes.POINTER(CNvfp4), ctypes.POINTER(CMxfp8),
                      ctypes.POINTER(CMxfp8), _F, _P, _I, _I64, _P, _P],
    "tj_gemm_mxfp8": [ctypes.POINTER(CMxfp8), ctypes.POINTER(CMxfp8), _P, _I, _I64, _P, _P],
    "tj_gemm_pair": [ctypes.POINTER(CNvfp4), ctypes.POINTER(CNvfp4), _F, _P, _I, _I64, _P, ctypes.POINTER(CMxfp8),
                     ctypes.POINTER(CMxfp8), _P, _I, _I64, _P, _P],
    "tj_gemm_pair_f32": [ctypes.POINTER(CNvfp4), ctypes.POINTER(CNvfp4), _F, _P, ctypes.POINTER(CMxfp8),
                         ctypes.POINTER(CMxfp8), _P, _P, _I64, _I64, _P],
    "tj_linear_fwd": [_P, _I64, _I64, _I64, ctypes.POINTER(CNvfp4), ctypes.POINTER(CMxfp8), _P, _P, _I64,
                      ctypes.POINTER(CNvfp4), ctypes.POINTER(CMxfp8), _P, _I, _I64, _P],
    "tj_linear_bwd_dx": [_P, _I64, _I64, _I64, ctypes.POINTER(CNvfp4), ctypes.POINTER(CMxfp8), _P, _P, _I64, _U64,
                         _P, _I, _I64, _P, ctypes.c_size_t, _P],
    "tj_linear_bwd_dw": [_P, _I64, _I64, _I64, ctypes.POINTER(CNvfp4), ctypes.POINTER(CMxfp8), _P, _P, _I64, _U64,
                         _P, _I64, _P, ctypes.c_size_t, _P],
    "tj_fp8_linear_fwd": [_P, _I64, _I64, _I64, ctypes.POINTER(CMxfp8), ctypes.POINTER(CMxfp8), ctypes.POINTER(CMxfp8),
                          _P, _I, _I64, _P],
    "tj_fp8_linear_bwd_dx": [_P, _I64, _I64, _I64, ctypes.POINTER(CMxfp8), _P, _I, _I64, _P, ctypes.c_size_t, _P],
    "tj_fp8_linear_bwd_dw": [_P, _I64, _I64, _I64, ctypes.POINTER(CMxfp8), _P, _I64, _P, ctypes.c_size_t, _P],
    "tj_workspace_size": [_I, _I64, _I64, _I64, _I64],
    "tj_outlier_calibrate": [_P, _I, _I64, _I64, _I64, _P, _I, _I64, _P, _P, _P],
    "tj_osci_reset": [_P, _P, _P, _P, ctypes.POINTER(CNvfp4), ctypes.POINTER(CNvfp4), _P, _I64, _I64, _F, _F, _F,
                      _I, _P],
    "tj_adamw_osci_reset": [_P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(CNvfp4), ctypes.POINTER(CNvfp4), _P, _I64,
                            _I64, _F, _F, _F, _F, _F, _I64, _F, _F, _I, _P],
    "tj_linear_bwd_dx_noalloc": [_P, _I64, _I64, _I64, ctypes.POINTER(CNvfp4), ctypes.POINTER(CMxfp8), _P, _P, _I64,
                                 _U64, _P, _I, _I64, _P],
    "tj_noalloc_scratch_bytes": [],
    "tj_get_device_status": [],
    "tj_debug_gemm_fault": [_I, _I64],
    "tj_status_str": [_I],
}
EXPORTED = sorted(_SIGS)


def load(path=LIB_PATH):
    """Load libtj.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError("libtj.so not built (run __graft_entry__.build()); no CPU fallback exists")
        lib = ctypes.CDLL(path)
        for name, args in _SIGS.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_size_t if name in ("tj_workspace_size", "tj_noalloc_scratch_bytes") else (
                ctypes.c_char_p if name == "tj_status_str" else ctypes.c_int)
        _lib = lib
    return _lib


def _call(name, *args):
    code = getattr(load(), name)(*args)
    if code != TJ_OK:
        raise TjError(name, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_DENSE = (torch.bfloat16, torch.float32)
_BF16 = (torch.bfloat16,)
_FP32 = (torch.float32,)
_MASK = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())


def _cuda(t, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s: a CUDA tensor is expected, got %s" % (name, type(t).__name__ if not
                                                                     isinstance(t, torch.Tensor) else t.device))


def _mat(t, name, dtypes=_DENSE):
    """Pointer to a 2-D CUDA matrix in one of `dtypes`.  The library addresses element (r, c)
    at r * ld + c, so the columns must be adjacent (stride(1) == 1); the row stride is free."""
    if t is None:
        return None
    _cuda(t, name)
    if t.dim() != 2:
        raise ValueError("%s: a 2-D tensor is expected, got shape %s" % (name, tuple(t.shape)))
    if t.dtype not in dtypes:
        raise ValueError("%s: dtype %s, expected %s" % (name, t.dtype, " or ".join(map(str, dtypes))))
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("%s: the columns must be adjacent in memory (stride %s); pass .contiguous()"
                         % (name, tuple(t.stride())))
    return ctypes.c_void_p(t.data_ptr())


def _ld(t):
    """Row stride of a matrix checked by _mat; a single row has no row stride of its own."""
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


def _arr(t, name, dtypes, numel=None, at_least=False):
    """Pointer to a contiguous CUDA array in one of `dtypes` with `numel` elements (or at
    least that many): index lists, column maps, optimizer state, masks."""
    if t is None:
        return None
    _cuda(t, name)
    if t.dtype not in dtypes:
        raise ValueError("%s: dtype %s, expected %s" % (name, t.dtype, " or ".join(map(str, dtypes))))
    if not t.is_contiguous():
        raise ValueError("%s: a contiguous tensor is expected (stride %s)" % (name, tuple(t.stride())))
    if numel is not None and (t.numel() < numel if at_least else t.numel() != numel):
        raise ValueError("%s: %d elements, expected %s%d" % (name, t.numel(), "at least " if at_least else "",
                                                              numel))
    return ctypes.c_void_p(t.data_ptr())


def _idx(t, name, numel=None):
    """An int32 index list (channel selection, column map)."""
    if t is not None and t.dim() != 1:
        raise ValueError("%s: a 1-D index tensor is expected, got shape %s" % (name, tuple(t.shape)))
    return _arr(t, name, (torch.int32,), numel, at_least=True)


def _workspace(t, name="workspace"):
    """(pointer, size in bytes) of a contiguous CUDA scratch buffer of any dtype."""
    _arr(t, name, (t.dtype,))
    return ctypes.c_void_p(t.data_ptr()), t.numel() * t.element_size()


_NO_COLUMN = ctypes.c_int32(0)


def _sel_ptr(sel):
    """A channel selection: None -> NULL (all columns); an empty index tensor, whose data
    pointer is NULL, -> a non-NULL address that the library does not read (no column)."""
    if sel is None:
        return None
    p = _idx(sel, "sel")
    return p if sel.numel() else ctypes.cast(ctypes.byref(_NO_COLUMN), ctypes.c_void_p)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _round_up(v, m):
    return (v + m - 1) // m * m


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return TJ_BF16
    if t.dtype == torch.float32:
        return TJ_FP32
    raise TypeError("bf16 or fp32 tensor expected, got %s" % t.dtype)


def _buf(t, name, dtype, numel):
    """Address of a packed buffer of a quantized tensor: contiguous, CUDA, at least the
    padded size of its layout."""
    if t.dtype != dtype:
        raise ValueError("%s: dtype %s, expected %s" % (name, t.dtype, dtype))
    return _arr(t, name, (dtype,), numel, at_least=True).value


class NVFP4:
    """Device buffers of a double-block NVFP4 tensor (layout documented in tj.h)."""

    def __init__(self, codes, sf, outer, rows, cols):
        self.codes, self.sf, self.outer, self.rows, self.cols = codes, sf, outer, rows, cols

    @staticmethod
    def empty(rows, cols, device="cuda"):
        rp, cp = _round_up(rows, 128), _round_up(cols, 128)
        return NVFP4(torch.empty(rp * cp // 2, dtype=torch.uint8, device=device),
                     torch.empty(rp * cp // 16, dtype=torch.uint8, device=device),
                     torch.empty((cp // 128) * rp, dtype=torch.float32, device=device), rows, cols)

    def c(self):
        rp, cp = _round_up(self.rows, 128), _round_up(self.cols, 128)
        return CNvfp4(_buf(self.codes, "NVFP4 codes", torch.uint8, rp * cp // 2),
                      _buf(self.sf, "NVFP4 inner scales", torch.uint8, rp * cp // 16),
                      _buf(self.outer, "NVFP4 outer scales", torch.float32, (cp // 128) * rp), self.rows, self.cols)


class MXFP8:
    """Device buffers of an MX outlier slice in element format fmt (TJ_MX_*; E4M3 = the FP8
    slice; layout documented in tj.h)."""

    def __init__(self, codes, sf, rows, cols, fmt=TJ_MX_E4M3):
        self.codes, self.sf, self.rows, self.cols, self.fmt = codes, sf, rows, cols, fmt

    @staticmethod
    def empty(rows, cols, device="cuda", fmt=TJ_MX_E4M3):
        rp, cp = _round_up(rows, 128), _round_up(cols, 128)
        return MXFP8(torch.empty(rp * cp * MX_BITS[fmt] // 8, dtype=torch.uint8, device=device),
                     torch.empty(rp * cp // 32, dtype=torch.uint8, device=device), rows, cols, fmt)

    def c(self):
        if self.fmt not in MX_BITS:
            raise ValueError("MX slice: unknown element format %r" % (self.fmt,))
        rp, cp = _round_up(self.rows, 128), _round_up(self.cols, 128)
        return CMxfp8(_buf(self.codes, "MX slice codes", torch.uint8, rp * cp * MX_BITS[self.fmt] // 8),
                      _buf(self.sf, "MX slice scales", torch.uint8, rp * cp // 32), self.rows, self.cols, self.fmt)


def _ref(obj):
    return None if obj is None else ctypes.byref(obj)


def quantize_nvfp4(x, along_cols=False, sel=None, mode=TJ_RTN, rht=False, seed=0, tag=0, rht_tag=0, out=None,
                   stream=None):
    """Double-block NVFP4 quantization of a 2-D bf16/fp32 CUDA tensor (tj_quantize_nvfp4)."""
    rows_x, cols_x = x.shape
    ncols = cols_x if sel is None else sel.numel()
    orows, ocols = (ncols, rows_x) if along_cols else (rows_x, ncols)
    out = out if out is not None else NVFP4.empty(orows, ocols, x.device)
    c = out.c()
    _call("tj_quantize_nvfp4", _mat(x, "x"), _dtype_code(x), rows_x, cols_x, _ld(x), int(along_cols), _sel_ptr(sel),
          0 if sel is None else sel.numel(), mode, int(rht), seed, tag, rht_tag, ctypes.byref(c), _stream(stream))
    return out


def quantize_mxfp8(x, along_cols=False, sel=None, out=None, stream=None, fmt=TJ_MX_E4M3):
    """MX slice quantization (tj_quantize_mxfp8), in `out`'s format or, when out is None, in fmt."""
    rows_x, cols_x = x.shape
    ncols = cols_x if sel is None else sel.numel()
    orows, ocols = (ncols, rows_x) if along_cols else (rows_x, ncols)
    out = out if out is not None else MXFP8.empty(orows, ocols, x.device, fmt)
    c = out.c()
    _call("tj_quantize_mxfp8", _mat(x, "x"), _dtype_code(x), rows_x, cols_x, _ld(x), int(along_cols), _sel_ptr(sel),
          0 if sel is None else sel.numel(), ctypes.byref(c), _stream(stream))
    return out


def quantize_nvfp4_mxfp8(x, along_cols=False, sel=None, mode=TJ_RTN, rht=False, seed=0, tag=0, rht_tag=0,
                         out=None, out8=None, stream=None, fmt8=TJ_MX_E4M3):
    """NVFP4 and an MX slice (format fmt8 unless out8 is given) of the same input from one
    read (tj_quantize_nvfp4_mxfp8)."""
    rows_x, cols_x = x.shape
    ncols = cols_x if sel is None else sel.numel()
    orows, ocols = (ncols, rows_x) if along_cols else (rows_x, ncols)
    out = out if out is not None else NVFP4.empty(orows, ocols, x.device)
    out8 = out8 if out8 is not None else MXFP8.empty(orows, ocols, x.device, fmt8)
    c, c8 = out.c(), out8.c()
    _call("tj_quantize_nvfp4_mxfp8", _mat(x, "x"), _dtype_code(x), rows_x, cols_x, _ld(x), int(along_cols),
          _sel_ptr(sel), 0 if sel is None else sel.numel(), mode, int(rht), seed, tag, rht_tag, ctypes.byref(c),
          ctypes.byref(c8), _stream(stream))
    return out, out8


def quantize_split(x, normal_idx, outlier_idx, out=None, out8=None, stream=None, fmt8=TJ_MX_E4M3):
    """OutControl split, row-wise, one read: NVFP4 RTN of the normal channels and the MX slice
    (format fmt8 unless out8 is given) of the outlier channels (tj_quantize_split)."""
    rows, cols = x.shape
    kn, k = normal_idx.numel(), (0 if outlier_idx is None else outlier_idx.numel())
    out = out if out is not None else NVFP4.empty(rows, kn, x.device)
    if k > 0 and out8 is None:
        out8 = MXFP8.empty(rows, k, x.device, fmt8)
    c = out.c()
    c8 = out8.c() if k > 0 else None
    _call("tj_quantize_split", _mat(x, "x"), _dtype_code(x), rows, cols, _ld(x), _idx(normal_idx, "normal_idx"), kn,
          _idx(outlier_idx, "outlier_idx") if k > 0 else None, k, ctypes.byref(c), ctypes.byref(c8) if c8 is not None else None,
          _stream(stream))
    return out, out8


def requantize_nvfp4(q, mode=TJ_SR, rht=True, seed=0, tag=0, rht_tag=0, out=None, stream=None):
    """Transposed re-alignment of a forward NVFP4 operand [rows, cols] -> [cols, rows]."""
    out = out if out is not None else NVFP4.empty(q.cols, q.rows, q.codes.device)
    ci, co = q.c(), out.c()
    _call("tj_requantize_nvfp4", ctypes.byref(ci), mode, int(rht), seed, tag, rht_tag, ctypes.byref(co),
          _stream(stream))
    return out


def requantize_mxfp8(q, out=None, stream=None, fmt=None):
    """Transposed re-alignment of a slice [rows, cols] -> [cols, rows] (RTN), in `out`'s
    format or fmt (default: the input's)."""
    out = out if out is not None else MXFP8.empty(q.cols, q.rows, q.codes.device, q.fmt if fmt is None else fmt)
    ci, co = q.c(), out.c()
    _call("tj_requantize_mxfp8", ctypes.byref(ci), ctypes.byref(co), _stream(stream))
    return out


def requantize_nvfp4_mxfp8(q, q8, mode=TJ_SR, rht=True, seed=0, tag=0, rht_tag=0, out=None, out8=None, stream=None):
    """Both backward re-alignments of a forward operand (NVFP4 q [rows, cols] and its slice q8) in
    one launch (tj_requantize_nvfp4_mxfp8); returns (out, out8)."""
    out = out if out is not None else NVFP4.empty(q.cols, q.rows, q.codes.device)
    out8 = out8 if out8 is not None else MXFP8.empty(q8.cols, q8.rows, q8.codes.device, q8.fmt)
    ci, co, ci8, co8 = q.c(), out.c(), q8.c(), out8.c()
    _call("tj_requantize_nvfp4_mxfp8", ctypes.byref(ci), mode, int(rht), seed, tag, rht_tag, ctypes.byref(co),
          ctypes.byref(ci8), ctypes.byref(co8), _stream(stream))
    return out, out8


def rht(x, seed, tag, out=None, stream=None):
    """128-point random Hadamard transform of each 128-block of the rows of x (fp32)."""
    _arr(x, "x", _FP32)
    if x.dim() != 2:
        raise ValueError("x: a 2-D tensor is expected, got shape %s" % (tuple(x.shape),))
    out = out if out is not None else torch.empty_like(x)
    _call("tj_rht", _ptr(x), _arr(out, "out", _FP32, x.numel()), x.shape[0], x.shape[1], seed, tag, _stream(stream))
    return out


def dequantize_nvfp4(q, stream=None):
    y = torch.empty(q.rows, q.cols, dtype=torch.float32, device=q.codes.device)
    c = q.c()
    _call("tj_dequantize_nvfp4", ctypes.byref(c), _ptr(y), q.cols, _stream(stream))
    return y


def dequantize_mxfp8(q, stream=None):
    y = torch.empty(q.rows, q.cols, dtype=torch.float32, device=q.codes.device)
    c = q.c()
    _call("tj_dequantize_mxfp8", ctypes.byref(c), _ptr(y), q.cols, _stream(stream))
    return y


def gemm_nvfp4(a, b, a8=None, b8=None, alpha=1.0, out=None, out_dtype=torch.float32, col_map=None, stream=None):
    """D = alpha * A B^T (+ A8 B8^T), block-scaled FP4 on the tensor cores."""
    if out is None:
        out = torch.empty(a.rows, b.rows, dtype=out_dtype, device=a.codes.device)
    ca, cb = a.c(), b.c()
    c8a = a8.c() if a8 is not None else None
    c8b = b8.c() if b8 is not None else None
    _call("tj_gemm_nvfp4", ctypes.byref(ca), ctypes.byref(cb), _ref(c8a), _ref(c8b), alpha, _mat(out, "out"),
          _dtype_code(out), _ld(out), _idx(col_map, "col_map", b.rows), _stream(stream))
    return out


def gemm_mxfp8(a8, b8, out=None, out_dtype=torch.float32, col_map=None, stream=None):
    if out is None:
        out = torch.empty(a8.rows, b8.rows, dtype=out_dtype, device=a8.codes.device)
    ca, cb = a8.c(), b8.c()
    _call("tj_gemm_mxfp8", ctypes.byref(ca), ctypes.byref(cb), _mat(out, "out"), _dtype_code(out), _ld(out),
          _idx(col_map, "col_map", b8.rows), _stream(stream))
    return out


def gemm_pair(a, b, a8, b8, alpha=1.0, out=None, out8=None, col_map=None, col_map8=None, stream=None):
    """An FP4 product and an FP8-only product in one launch (tj_gemm_pair); out / out8 may be
    the same tensor when the column maps are disjoint."""
    ca, cb, ca8, cb8 = a.c(), b.c(), a8.c(), b8.c()
    _call("tj_gemm_pair", ctypes.byref(ca), ctypes.byref(cb), float(alpha), _mat(out, "out"), _dtype_code(out),
          _ld(out), _idx(col_map, "col_map", b.rows), ctypes.byref(ca8), ctypes.byref(cb8), _mat(out8, "out8"),
          _dtype_code(out8), _ld(out8), _idx(col_map8, "col_map8", b8.rows), _stream(stream))
    return out, out8


def gemm_pair_f32(a, b, a8, b8, out, col_map, col_map8, alpha=1.0, stream=None):
    """A pair launch whose fp32 products fill `out` through their column maps
    (tj_gemm_pair_f32): the call may zero `out` and split a long K in two."""
    ca, cb, ca8, cb8 = a.c(), b.c(), a8.c(), b8.c()
    _call("tj_gemm_pair_f32", ctypes.byref(ca), ctypes.byref(cb), float(alpha), _idx(col_map, "col_map", b.rows),
          ctypes.byref(ca8), ctypes.byref(cb8), _idx(col_map8, "col_map8", b8.rows), _mat(out, "out", _FP32),
          out.shape[1], _ld(out), _stream(stream))
    return out


def workspace_size(op, M, N, K, k):
    return int(load().tj_workspace_size(op, M, N, K, k))


def linear_fwd(x, wq, w8=None, normal_idx=None, outlier_idx=None, out_dtype=torch.bfloat16, xq=None, x8=None,
               out=None, stream=None, fmt_x8=TJ_MX_E4M3):
    """Forward Y = X W^T of the NVFP4 linear layer; returns (Y, X-hat NVFP4, X-hat slice).
    X's slice is quantized in x8's format, or fmt_x8 when x8 is None."""
    M, K = x.shape
    k = 0 if outlier_idx is None else outlier_idx.numel()
    xq = xq if xq is not None else NVFP4.empty(M, K - k, x.device)
    if k and x8 is None:
        x8 = MXFP8.empty(M, k, x.device, fmt_x8)
    out = out if out is not None else torch.empty(M, wq.rows, dtype=out_dtype, device=x.device)
    cw, cx = wq.c(), xq.c()
    cw8 = w8.c() if k else None
    cx8 = x8.c() if k else None
    _call("tj_linear_fwd", _mat(x, "x", _BF16), M, K, _ld(x), ctypes.byref(cw), _ref(cw8),
          _idx(normal_idx, "normal_idx", K - k), _idx(outlier_idx, "outlier_idx", k), k, ctypes.byref(cx), _ref(cx8),
          _mat(out, "out"), _dtype_code(out), _ld(out), _stream(stream))
    return out, xq, (x8 if k else None)


def linear_bwd_dx(dy, wq, w8=None, normal_idx=None, outlier_idx=None, seed=0, out_dtype=torch.bfloat16,
                  workspace=None, out=None, stream=None):
    M, N = dy.shape
    k = 0 if outlier_idx is None else outlier_idx.numel()
    K = wq.cols + k
    ws_bytes = workspace_size(TJ_OP_BWD_DX, M, N, K, k)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dy.device)
    out = out if out is not None else torch.empty(M, K, dtype=out_dtype, device=dy.device)
    cw = wq.c()
    cw8 = w8.c() if k else None
    _call("tj_linear_bwd_dx", _mat(dy, "dy", _BF16), M, N, _ld(dy), ctypes.byref(cw), _ref(cw8),
          _idx(normal_idx, "normal_idx", K - k), _idx(outlier_idx, "outlier_idx", k), k, seed, _mat(out, "out"),
          _dtype_code(out), _ld(out), *_workspace(workspace), _stream(stream))
    return out


def linear_bwd_dw(dy, xq, x8=None, normal_idx=None, outlier_idx=None, seed=0, workspace=None, out=None,
                  stream=None):
    M, N = dy.shape
    k = 0 if outlier_idx is None else outlier_idx.numel()
    K = xq.cols + k
    ws_bytes = workspace_size(TJ_OP_BWD_DW, M, N, K, k)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dy.device)
    out = out if out is not None else torch.empty(N, K, dtype=torch.float32, device=dy.device)
    cx = xq.c()
    cx8 = x8.c() if k else None
    _call("tj_linear_bwd_dw", _mat(dy, "dy", _BF16), M, N, _ld(dy), ctypes.byref(cx), _ref(cx8),
          _idx(normal_idx, "normal_idx", K - k), _idx(outlier_idx, "outlier_idx", k), k, seed,
          _mat(out, "out", _FP32), _ld(out), *_workspace(workspace), _stream(stream))
    return out


def linear_bwd_dx_noalloc(dy, wq, w8=None, normal_idx=None, outlier_idx=None, seed=0, out_dtype=torch.bfloat16,
                          out=None, stream=None):
    """dX like linear_bwd_dx, with the library's fixed internal scratch instead of a workspace
    (for callers that cannot allocate device memory when the backward runs)."""
    M, N = dy.shape
    k = 0 if outlier_idx is None else outlier_idx.numel()
    out = out if out is not None else torch.empty(M, wq.cols + k, dtype=out_dtype, device=dy.device)
    cw = wq.c()
    cw8 = w8.c() if k else None
    K = wq.cols + k
    _call("tj_linear_bwd_dx_noalloc", _mat(dy, "dy", _BF16), M, N, _ld(dy), ctypes.byref(cw), _ref(cw8),
          _idx(normal_idx, "normal_idx", K - k), _idx(outlier_idx, "outlier_idx", k), k, seed, _mat(out, "out"),
          _dtype_code(out), _ld(out), _stream(stream))
    return out


def fp8_linear_fwd(x, w8, out_dtype=torch.bfloat16, x8=None, xt8=None, save_xt=True, out=None, stream=None):
    """FP8 baseline forward (tj_fp8_linear_fwd); returns (Y, X along K, X^T along M or None)."""
    M, K = x.shape
    x8 = x8 if x8 is not None else MXFP8.empty(M, K, x.device)
    if save_xt and xt8 is None:
        xt8 = MXFP8.empty(K, M, x.device)
    out = out if out is not None else torch.empty(M, w8.rows, dtype=out_dtype, device=x.device)
    cw, cx = w8.c(), x8.c()
    cxt = xt8.c() if save_xt else None
    _call("tj_fp8_linear_fwd", _mat(x, "x", _BF16), M, K, _ld(x), ctypes.byref(cw), ctypes.byref(cx), _ref(cxt),
          _mat(out, "out"), _dtype_code(out), _ld(out), _stream(stream))
    return out, x8, (xt8 if save_xt else None)


def fp8_linear_bwd_dx(dy, wt8, out_dtype=torch.bfloat16, workspace=None, out=None, stream=None):
    """FP8 baseline input gradient (tj_fp8_linear_bwd_dx); wt8 = MXFP8 of W^T along N."""
    M, N = dy.shape
    K = wt8.rows
    ws_bytes = workspace_size(TJ_OP_FP8_BWD_DX, M, N, K, 0)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dy.device)
    out = out if out is not None else torch.empty(M, K, dtype=out_dtype, device=dy.device)
    cw = wt8.c()
    _call("tj_fp8_linear_bwd_dx", _mat(dy, "dy", _BF16), M, N, _ld(dy), ctypes.byref(cw), _mat(out, "out"),
          _dtype_code(out), _ld(out), *_workspace(workspace), _stream(stream))
    return out


def fp8_linear_bwd_dw(dy, xt8, workspace=None, out=None, stream=None):
    """FP8 baseline weight gradient (tj_fp8_linear_bwd_dw); xt8 from fp8_linear_fwd."""
    M, N = dy.shape
    K = xt8.rows
    ws_bytes = workspace_size(TJ_OP_FP8_BWD_DW, M, N, K, 0)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dy.device)
    out = out if out is not None else torch.empty(N, K, dtype=torch.float32, device=dy.device)
    cx = xt8.c()
    _call("tj_fp8_linear_bwd_dw", _mat(dy, "dy", _BF16), M, N, _ld(dy), ctypes.byref(cx), _mat(out, "out", _FP32),
          _ld(out), *_workspace(workspace), _stream(stream))
    return out


def outlier_calibrate(x, sumsq, finalize=False, k=0, stream=None):
    """Accumulate per-channel sums of squares (x may be None); on finalize return
    (outlier_idx [k], normal_idx [K-k]) as int32 CUDA tensors."""
    K = sumsq.numel()
    outl = torch.empty(max(k, 1), dtype=torch.int32, device=sumsq.device)
    norm = torch.empty(max(K - k, 1), dtype=torch.int32, device=sumsq.device)
    if x is not None:
        _call("tj_outlier_calibrate", _mat(x, "x"), _dtype_code(x), x.shape[0], x.shape[1], _ld(x),
              _arr(sumsq, "sumsq", (torch.float64,)), 0, 0, None, None, _stream(stream))
    if finalize:
        _call("tj_outlier_calibrate", None, TJ_BF16, 0, K, K, _arr(sumsq, "sumsq", (torch.float64,)), 1, k,
              _ptr(outl), _ptr(norm), _stream(stream))
        return outl[:k], norm[:K - k]
    return None


def osci_reset(w, w_prev, dist_q, dist_m, q_prev, q_out, mask, lr, lr_thr, risk_thr, track=True, stream=None):
    """One OsciReset pass (tj_osci_reset); w, w_prev, dist_q, dist_m updated in place."""
    rows, cols = w.shape
    n = w.numel()
    cp, co = q_prev.c(), q_out.c()
    _call("tj_osci_reset", _arr(w, "w", _FP32, n), _arr(w_prev, "w_prev", _FP32, n), _arr(dist_q, "dist_q", _FP32, n),
          _arr(dist_m, "dist_m", _FP32, n), ctypes.byref(cp), ctypes.byref(co),
          _arr(mask, "mask", _MASK, rows * ((cols + 31) // 32), at_least=True), rows, cols, lr, lr_thr, risk_thr,
          int(track), _stream(stream))


def adamw_osci_reset(w, g, m, v, w_prev, dist_q, dist_m, q_prev, q_out, mask, lr, beta1, beta2, eps, weight_decay,
                     step, lr_thr, risk_thr, track=True, stream=None):
    """AdamW then OsciReset in one pass (tj_adamw_osci_reset); w, m, v, w_prev and the
    distances are updated in place."""
    rows, cols = w.shape
    n = w.numel()
    cp, co = q_prev.c(), q_out.c()
    _call("tj_adamw_osci_reset", _arr(w, "w", _FP32, n), _arr(g, "g", _FP32, n), _arr(m, "m", _FP32, n),
          _arr(v, "v", _FP32, n), _arr(w_prev, "w_prev", _FP32, n), _arr(dist_q, "dist_q", _FP32, n),
          _arr(dist_m, "dist_m", _FP32, n), ctypes.byref(cp), ctypes.byref(co),
          _arr(mask, "mask", _MASK, rows * ((cols + 31) // 32), at_least=True), rows, cols, lr, beta1, beta2, eps, weight_decay, int(step),
          lr_thr, risk_thr, int(track), _stream(stream))


def device_status():
    """Reads and clears the sticky device flag; raises TjError on a timed-out device wait."""
    code = load().tj_get_device_status()
    if code != TJ_OK:
        raise TjError("tj_get_device_status", code)
