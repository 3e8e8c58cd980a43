"""GPU parity: quantize kernels vs the CPU oracle, bit for bit.

Codes, E4M3 inner scales, FP32 outer scales, SR decisions, MXFP8 codes and
scales must equal the oracle's exactly, on seeded inputs that span several
128-blocks, ragged tails (rows and columns not multiples of 128), fp32 and
bf16 inputs, channel selection (OutControl's normal / outlier channels), both
orientations, RTN and SR, with and without the RHT.
"""
import numpy as np
import pytest
import torch

from layouts import assert_mxfp8_equal, assert_nvfp4_equal, nvfp4_to_logical_full
from oracle import linear as OL
from oracle import quant as Q
from oracle.philox import rht_signs
from oracle.rht import rht_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


def _input(rows, cols, dtype, seed, heavy=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g)
    if heavy:
        x[:, torch.randperm(cols, generator=g)[: max(1, cols // 50)]] *= 30
    x[min(3, rows - 1), : min(128, cols)] = 0.0          # an all-zero block
    return x.to(dtype)


def _oracle_rows(xf, mode, seed, tag, rht, rht_tag):
    if rht:
        d = rht_signs(seed, rht_tag)
        return Q.quantize_nvfp4(rht_f32(Q.pad_cols(xf, 128), d), mode, seed=seed, tag=tag)
    return Q.quantize_nvfp4(xf, mode, seed=seed, tag=tag)


CASES = [  # rows, cols, dtype
    (256, 512, torch.bfloat16),
    (200, 300, torch.float32),
    (130, 1024, torch.bfloat16),
    (64, 136, torch.bfloat16),
]


@pytest.mark.parametrize("rows,cols,dtype", CASES)
@pytest.mark.parametrize("mode,rht", [(0, False), (1, False), (1, True), (0, True)])
def test_quantize_rows_bit_exact(tj, rows, cols, dtype, mode, rht):
    x = _input(rows, cols, dtype, rows + cols)
    q = tj.quantize_nvfp4(x.cuda(), mode=mode, rht=rht, seed=77, tag=5, rht_tag=0x100)
    torch.cuda.synchronize()
    ref = _oracle_rows(x.float().numpy(), mode, 77, 5, rht, 0x100)
    assert_nvfp4_equal(q, ref, "rows")
    c, s, o = nvfp4_to_logical_full(q)                       # padded rows written as zero
    assert not c[rows:].any() and not s[rows:].any() and not o[rows:].any()


@pytest.mark.parametrize("rows,cols,dtype", CASES)
@pytest.mark.parametrize("mode,rht", [(0, False), (1, False), (1, True)])
def test_quantize_cols_bit_exact(tj, rows, cols, dtype, mode, rht):
    x = _input(rows, cols, dtype, 3 * rows + cols)
    q = tj.quantize_nvfp4(x.cuda(), along_cols=True, mode=mode, rht=rht, seed=91, tag=2, rht_tag=0x101)
    torch.cuda.synchronize()
    xt = np.ascontiguousarray(x.float().numpy().T)
    ref = _oracle_rows(xt, mode, 91, 2, rht, 0x101)
    assert_nvfp4_equal(q, ref, "cols")


@pytest.mark.parametrize("along", [False, True])
def test_quantize_channel_selection(tj, along):
    rows, cols = 256, 520
    x = _input(rows, cols, torch.bfloat16, 5)
    rng = np.random.default_rng(1)
    outl = np.sort(rng.choice(cols, 52, replace=False))
    normal = OL.normal_channels(cols, outl)
    sel = torch.from_numpy(normal.astype(np.int32)).cuda()
    q = tj.quantize_nvfp4(x.cuda(), along_cols=along, sel=sel, mode=1, seed=3, tag=4)
    torch.cuda.synchronize()
    xs = x.float().numpy()[:, normal]
    ref = Q.quantize_nvfp4(np.ascontiguousarray(xs.T) if along else xs, 1, seed=3, tag=4)
    assert_nvfp4_equal(q, ref, "selected")
    # the FP8 slice of the outlier channels
    q8 = tj.quantize_mxfp8(x.cuda(), along_cols=along, sel=torch.from_numpy(outl.astype(np.int32)).cuda())
    torch.cuda.synchronize()
    xo = x.float().numpy()[:, outl]
    assert_mxfp8_equal(q8, Q.quantize_mxfp8(np.ascontiguousarray(xo.T) if along else xo), "fp8 slice")


@pytest.mark.parametrize("rows,cols,dtype", CASES)
@pytest.mark.parametrize("along", [False, True])
def test_quantize_mxfp8_bit_exact(tj, rows, cols, dtype, along):
    x = _input(rows, cols, dtype, rows * 7 + cols)
    x[1, 5] = 1e-30 if dtype == torch.float32 else 0.0      # tiny values -> the smallest normal inner scale / zero
    q8 = tj.quantize_mxfp8(x.cuda(), along_cols=along)
    torch.cuda.synchronize()
    xf = x.float().numpy()
    assert_mxfp8_equal(q8, Q.quantize_mxfp8(np.ascontiguousarray(xf.T) if along else xf), "mxfp8")


@pytest.mark.parametrize("rows,cols,dtype", CASES)
@pytest.mark.parametrize("along", [False, True])
@pytest.mark.parametrize("mode,rht", [(1, True), (0, False)])
def test_quantize_dual_bit_exact(tj, rows, cols, dtype, along, mode, rht):
    """NVFP4 + MXFP8 of one input from one read: both outputs equal the oracle's."""
    x = _input(rows, cols, dtype, 11 * rows + cols)
    q, q8 = tj.quantize_nvfp4_mxfp8(x.cuda(), along_cols=along, mode=mode, rht=rht, seed=19, tag=1, rht_tag=0x100)
    torch.cuda.synchronize()
    xf = x.float().numpy()
    xo = np.ascontiguousarray(xf.T) if along else xf
    assert_nvfp4_equal(q, _oracle_rows(xo, mode, 19, 1, rht, 0x100), "dual nvfp4")
    assert_mxfp8_equal(q8, Q.quantize_mxfp8(xo), "dual mxfp8")


@pytest.mark.parametrize("rows,cols,dtype,n_out", [(256, 520, torch.bfloat16, 52), (200, 300, torch.float32, 30),
                                                    (130, 1024, torch.bfloat16, 103), (64, 136, torch.bfloat16, 1),
                                                    (96, 517, torch.bfloat16, 40), (40, 4100, torch.bfloat16, 410)])
def test_quantize_split_bit_exact(tj, rows, cols, dtype, n_out):
    """The OutControl split from one read equals the oracle's NVFP4 / MXFP8 of the two channel sets."""
    x = _input(rows, cols, dtype, 13 * rows + cols)
    outl = np.sort(np.random.default_rng(rows).choice(cols, n_out, replace=False))
    normal = OL.normal_channels(cols, outl)
    ni = torch.from_numpy(normal.astype(np.int32)).cuda()
    oi = torch.from_numpy(outl.astype(np.int32)).cuda()
    q, q8 = tj.quantize_split(x.cuda(), ni, oi)
    torch.cuda.synchronize()
    xf = x.float().numpy()
    assert_nvfp4_equal(q, Q.quantize_nvfp4(np.ascontiguousarray(xf[:, normal]), 0), "split nvfp4")
    assert_mxfp8_equal(q8, Q.quantize_mxfp8(np.ascontiguousarray(xf[:, outl])), "split mxfp8")
    c, s, o = nvfp4_to_logical_full(q)                       # padded rows written as zero
    assert not c[rows:].any() and not s[rows:].any() and not o[rows:].any()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_split_unaligned_rows(tj, dtype):
    """Rows that start off a 16-byte boundary (a column slice of a wider tensor) take the
    element-wise staging path; same results."""
    rows, cols, n_out = 70, 333, 33
    big = _input(rows, cols + 3, dtype, 5)
    x = big.cuda()[:, 1:cols + 1]
    outl = np.sort(np.random.default_rng(7).choice(cols, n_out, replace=False))
    normal = OL.normal_channels(cols, outl)
    q, q8 = tj.quantize_split(x, torch.from_numpy(normal.astype(np.int32)).cuda(),
                              torch.from_numpy(outl.astype(np.int32)).cuda())
    torch.cuda.synchronize()
    xf = big[:, 1:cols + 1].float().numpy()
    assert_nvfp4_equal(q, Q.quantize_nvfp4(np.ascontiguousarray(xf[:, normal]), 0), "split nvfp4")
    assert_mxfp8_equal(q8, Q.quantize_mxfp8(np.ascontiguousarray(xf[:, outl])), "split mxfp8")


def test_rht_standalone_bit_exact(tj):
    x = torch.randn(96, 512, generator=torch.Generator().manual_seed(4))
    y = tj.rht(x.cuda(), seed=12345, tag=0x100)
    torch.cuda.synchronize()
    ref = rht_f32(x.numpy(), rht_signs(12345, 0x100))
    assert np.array_equal(y.cpu().numpy(), ref)


def test_dequantize_matches_oracle(tj):
    x = _input(200, 300, torch.bfloat16, 8)
    q = tj.quantize_nvfp4(x.cuda(), mode=1, seed=1, tag=1)
    y = tj.dequantize_nvfp4(q)
    torch.cuda.synchronize()
    c, s, o = Q.quantize_nvfp4(x.float().numpy(), 1, seed=1, tag=1)
    assert np.array_equal(y.cpu().numpy(), Q.dequantize_nvfp4_f32(c, s, o)[:, :300])


def test_edge_cases(tj):
    # all zeros, a single nonzero, huge and tiny magnitudes, exact grid values
    x = torch.zeros(128, 256)
    x[1, 7] = 1.0
    x[2, :] = 3.0e38 / 3
    x[3, :16] = 1e-38
    x[4, :] = torch.tensor([0.0, 0.5, 1, 1.5, 2, 3, 4, 6] * 32) * 2.0 ** -3
    x[5, ::2] = -0.25
    # signed zeros and products that underflow next to a huge group maximum: a negative
    # element whose scaled value rounds to -0 keeps its sign bit, a -0 input gets code 0
    x[6, :8] = torch.tensor([3.0e38, -1.4e-45, -0.0, 0.0, 1.0e-45, -3.0e-39, -1.0, 2.0e-38])
    x[7, 16:32] = -0.0
    for mode in (0, 1):
        q = tj.quantize_nvfp4(x.cuda(), mode=mode, seed=5, tag=9)
        torch.cuda.synchronize()
        assert_nvfp4_equal(q, Q.quantize_nvfp4(x.numpy(), mode, seed=5, tag=9), "edge")


def test_argument_errors(tj):
    x = torch.randn(128, 128).cuda()
    with pytest.raises(tj.TjError):
        tj.quantize_nvfp4(x, mode=7)
    bad = tj.NVFP4.empty(64, 128)                          # wrong output shape
    with pytest.raises(tj.TjError):
        tj.quantize_nvfp4(x, out=bad)


@pytest.mark.parametrize("rows,cols", [(256, 512), (200, 328), (4096, 921)])
def test_requantize_bit_exact(tj, rows, cols):
    """Transposed re-alignment (X-hat^T, W-hat^T) of forward operands, NVFP4 and FP8."""
    x = _input(rows, cols, torch.bfloat16, rows + 3 * cols)
    q = tj.quantize_nvfp4(x.cuda())
    r = tj.requantize_nvfp4(q, mode=1, rht=True, seed=21, tag=3, rht_tag=0x100)
    q8 = tj.quantize_mxfp8(x.cuda())
    r8 = tj.requantize_mxfp8(q8)
    torch.cuda.synchronize()
    c, s, o = Q.quantize_nvfp4(x.float().numpy(), 0)
    xh = Q.dequantize_nvfp4_f32(c, s, o)[:, :cols]
    ref = _oracle_rows(np.ascontiguousarray(xh.T), 1, 21, 3, True, 0x100)
    assert_nvfp4_equal(r, ref, "requantize nvfp4")
    c8, s8 = Q.quantize_mxfp8(x.float().numpy())
    xh8 = Q.dequantize_mxfp8_f32(c8, s8)[:, :cols]
    assert_mxfp8_equal(r8, Q.quantize_mxfp8(np.ascontiguousarray(xh8.T)), "requantize mxfp8")


def test_dequantize_mxfp8_exact(tj):
    """tj_dequantize_mxfp8 returns E4M3 value x 2^(e - 127) of every element, exactly."""
    x = _input(200, 300, torch.bfloat16, 77)
    q8 = tj.quantize_mxfp8(x.cuda())
    y = tj.dequantize_mxfp8(q8)
    torch.cuda.synchronize()
    codes, sb = Q.quantize_mxfp8(x.float().numpy())
    ref = Q.dequantize_mxfp8_f32(codes, sb)[:, :300]
    assert np.array_equal(y.cpu().numpy(), ref)
