"""Test harness: read the library's HBM layouts back into the oracle's logical
arrays, and the GEMM tolerance check.

The layouts are re-derived here from their documentation in include/tj.h (not
from the CUDA sources), so a layout bug in a kernel shows up as a mismatch.
"""
import numpy as np
import torch


def _round_up(v, m):
    return (v + m - 1) // m * m


def _sf_untile(sf_bytes, rows_p, n_groups, group_tiles_per_row):
    """Scale tile layout -> logical [rows_p, n_groups]: the scale of row r, group g
    sits at byte (rt * group_tiles_per_row + g//4) * 512 + 16*(r%32) + 4*((r%128)//32) + g%4."""
    r = np.arange(rows_p)[:, None]
    g = np.arange(n_groups)[None, :]
    rt, rr = r // 128, r % 128
    off = (rt * group_tiles_per_row + g // 4) * 512 + 16 * (rr % 32) + 4 * (rr // 32) + g % 4
    return np.asarray(sf_bytes)[off]


def nvfp4_to_logical(q):
    """tj.NVFP4 -> (codes [rows, cols_p] uint8, sf [rows, cols_p/16] uint8, outer [rows, cols_p/128] f32)."""
    rows_p, cols_p = _round_up(q.rows, 128), _round_up(q.cols, 128)
    raw = q.codes.cpu().numpy().reshape(rows_p, cols_p // 2)
    codes = np.empty((rows_p, cols_p), dtype=np.uint8)
    codes[:, 0::2] = raw & 15
    codes[:, 1::2] = raw >> 4
    sf = _sf_untile(q.sf.cpu().numpy(), rows_p, cols_p // 16, cols_p // 64)
    outer = q.outer.cpu().numpy().reshape(cols_p // 128, rows_p).T
    return codes[: q.rows], sf[: q.rows], np.ascontiguousarray(outer[: q.rows])


def nvfp4_padding_is_zero(q):
    rows_p, cols_p = _round_up(q.rows, 128), _round_up(q.cols, 128)
    c, s, o = nvfp4_to_logical_full(q)
    return (not c[q.rows:].any()) and (not s[q.rows:].any()) and (not o[q.rows:].any())


def nvfp4_to_logical_full(q):
    rows_p, cols_p = _round_up(q.rows, 128), _round_up(q.cols, 128)
    raw = q.codes.cpu().numpy().reshape(rows_p, cols_p // 2)
    codes = np.empty((rows_p, cols_p), dtype=np.uint8)
    codes[:, 0::2] = raw & 15
    codes[:, 1::2] = raw >> 4
    sf = _sf_untile(q.sf.cpu().numpy(), rows_p, cols_p // 16, cols_p // 64)
    outer = q.outer.cpu().numpy().reshape(cols_p // 128, rows_p).T
    return codes, sf, outer


MX_BITS = {0: 8, 3: 6, 4: 6, 5: 4}


def unpack_mx_codes(raw, rows_p, cols_p, fmt):
    """Packed slice rows -> one code per element [rows_p, cols_p] (tj.h: E4M3 bytes; 6-bit
    codes as a little-endian bit stream per row, element c at bits 6c..6c+5; 4-bit codes
    two per byte, element 2j in the low nibble)."""
    raw = np.asarray(raw, dtype=np.uint8).reshape(rows_p, cols_p * MX_BITS[fmt] // 8)
    if fmt == 0:
        return raw.copy()
    if fmt == 5:
        codes = np.empty((rows_p, cols_p), dtype=np.uint8)
        codes[:, 0::2] = raw & 15
        codes[:, 1::2] = raw >> 4
        return codes
    bits = np.unpackbits(raw, axis=1, bitorder="little").reshape(rows_p, cols_p, 6)
    return (bits.astype(np.uint8) << np.arange(6, dtype=np.uint8)).sum(axis=2).astype(np.uint8)


def pack_mx_codes(codes, fmt):
    """Inverse of unpack_mx_codes: [rows, cols_p] codes -> packed bytes [rows, cols_p*bits/8]."""
    codes = np.asarray(codes, dtype=np.uint8)
    if fmt == 0:
        return codes.copy()
    if fmt == 5:
        return (codes[:, 0::2] & 15) | ((codes[:, 1::2] & 15) << 4)
    r, c = codes.shape
    bits = ((codes[:, :, None] >> np.arange(6, dtype=np.uint8)) & 1).reshape(r, c * 6)
    return np.packbits(bits, axis=1, bitorder="little")


def mxfp8_to_logical(q):
    """tj.MXFP8 (any slice format) -> (codes [rows, cols_p] uint8, one per element;
    scale bytes [rows, cols_p/32] uint8)."""
    rows_p, cols_p = _round_up(q.rows, 128), _round_up(q.cols, 128)
    fmt = getattr(q, "fmt", 0)
    nbytes = rows_p * cols_p * MX_BITS[fmt] // 8
    codes = unpack_mx_codes(q.codes[:nbytes].cpu().numpy(), rows_p, cols_p, fmt)
    sb = _sf_untile(q.sf.cpu().numpy(), rows_p, cols_p // 32, cols_p // 128)
    return codes[: q.rows], sb[: q.rows]


def assert_nvfp4_equal(q, ref, what=""):
    got = nvfp4_to_logical(q)
    for name, g, r in zip(("codes", "inner scales", "outer scales"), got, ref):
        r = np.asarray(r)
        assert g.shape == r.shape, (what, name, g.shape, r.shape)
        if not np.array_equal(g, r):
            bad = np.argwhere(g != r)
            i = tuple(bad[0])
            raise AssertionError("%s %s differ at %d positions; first %s: gpu %r oracle %r"
                                 % (what, name, len(bad), i, g[i], r[i]))


def assert_mxfp8_equal(q, ref, what=""):
    got = mxfp8_to_logical(q)
    for name, g, r in zip(("codes", "scales"), got, ref):
        assert g.shape == r.shape, (what, name, g.shape, r.shape)
        if not np.array_equal(g, r):
            bad = np.argwhere(g != r)
            i = tuple(bad[0])
            raise AssertionError("%s %s differ at %d positions; first %s: gpu %r oracle %r"
                                 % (what, name, len(bad), i, g[i], r[i]))


def abs_product(qa, qb, alpha=1.0):
    """sum_k |a_mk| |b_nk| of two oracle double-block operands (fp64)."""
    from oracle import quant as Q

    a = np.abs(Q.dequantize_nvfp4_f64(*qa))
    b = np.abs(Q.dequantize_nvfp4_f64(*qb))
    return alpha * (a @ b.T)


def abs_product_fp8(qa, qb):
    from oracle import quant as Q

    return np.abs(Q.dequantize_mxfp8_f64(*qa)) @ np.abs(Q.dequantize_mxfp8_f64(*qb)).T


GEMM_TOL = 2e-3


def assert_gemm_close(got, ref, absprod, tol=GEMM_TOL, bf16=False, what=""):
    """|got - ref| <= tol * sum|a||b| per output (+ half a bf16 ulp of ref for bf16 outputs)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    absprod = np.asarray(absprod, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    bound = tol * absprod + 1e-30
    if bf16:
        bound = bound + np.abs(ref) * 2.0 ** -8
    err = np.abs(got - ref)
    if not np.all(err <= bound):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError("%s: %d outputs outside tolerance; worst %s: gpu %r oracle %r bound %r"
                             % (what, int((err > bound).sum()), i, got[i], ref[i], bound[i]))
    assert np.all(np.isfinite(got))


def to_numpy_f32(t):
    return t.detach().float().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float32)


def carve_workspace(ws, parts):
    """Views of a backward workspace, carved in the documented order.

    parts: list of ("nv" | "mx", rows, cols[, slice format]); every buffer (codes, sf,
    outer) starts on a 256-byte boundary, and a slice reserves its FP8 size whatever its
    format.  Returns tj.NVFP4 / tj.MXFP8 objects."""
    from nvfp4_bit_fully_gb300 import tj

    out, off = [], 0

    def take(nbytes, dtype=torch.uint8):
        nonlocal off
        view = ws[off: off + nbytes]
        off += _round_up(nbytes, 256)
        return view.view(dtype) if dtype != torch.uint8 else view

    for part in parts:
        kind, rows, cols = part[:3]
        rp, cp = _round_up(rows, 128), _round_up(cols, 128)
        if kind == "nv":
            codes = take(rp * cp // 2)
            sf = take(rp * cp // 16)
            outer = take(rp * (cp // 128) * 4, torch.float32)
            out.append(tj.NVFP4(codes, sf, outer, rows, cols))
        else:
            codes = take(rp * cp)
            sf = take(rp * cp // 32)
            out.append(tj.MXFP8(codes, sf, rows, cols, part[3] if len(part) > 3 else 0))
    return out
