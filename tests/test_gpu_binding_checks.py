"""GPU: the Python binding refuses tensors that the C ABI would misread.

The C ABI takes a matrix as (pointer, row stride) with adjacent columns, index lists as
contiguous int32 arrays, optimizer state as contiguous fp32 arrays and the quantized
tensors as packed buffers of a fixed padded size.  A transposed or column-strided view,
an int64 index list, a short column map or a short buffer would be read as something
else; the binding raises ValueError before any launch instead.  A matrix with a single
row has no row stride of its own: any view of one row is accepted.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


def _x(rows, cols, seed=0, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(rows, cols, generator=g).to(dtype).cuda()


def test_column_strided_and_transposed_views_are_refused(tj):
    x = _x(256, 256)
    for bad in (x.t(), x[:, ::2]):
        with pytest.raises(ValueError, match="adjacent"):
            tj.quantize_nvfp4(bad)
        with pytest.raises(ValueError, match="adjacent"):
            tj.quantize_mxfp8(bad)
        with pytest.raises(ValueError, match="adjacent"):
            tj.outlier_calibrate(bad, torch.zeros(bad.shape[1], dtype=torch.float64, device="cuda"))
    a, b = tj.quantize_nvfp4(_x(128, 256)), tj.quantize_nvfp4(_x(128, 256, 1))
    with pytest.raises(ValueError, match="adjacent"):
        tj.gemm_nvfp4(a, b, out=torch.empty(128, 128, device="cuda").t())


def test_wrong_dtypes_are_refused(tj):
    with pytest.raises(ValueError, match="dtype"):
        tj.quantize_nvfp4(_x(128, 128, dtype=torch.float16))
    K, N = 256, 128
    w = _x(N, K, 2)
    wq = tj.quantize_nvfp4(w)
    with pytest.raises(ValueError, match="dtype"):            # the linear layer reads X as bf16 only
        tj.linear_fwd(_x(64, K, dtype=torch.float32), wq)
    with pytest.raises(ValueError, match="dtype"):
        tj.linear_bwd_dx(_x(64, N, dtype=torch.float32), wq)
    with pytest.raises(ValueError, match="dtype"):            # dW is fp32
        xq = tj.quantize_nvfp4(_x(64, K))
        tj.linear_bwd_dw(_x(64, N), xq, out=torch.empty(N, K, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError, match="dtype"):
        tj.rht(_x(4, 128), 1, 2)                              # the transform is fp32 in, fp32 out


def test_index_lists_must_be_int32_and_long_enough(tj):
    x = _x(64, 256)
    ni = torch.arange(0, 200, device="cuda")                  # int64
    oi = torch.arange(200, 256, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError, match="dtype"):
        tj.quantize_split(x, ni, oi)
    with pytest.raises(ValueError, match="dtype"):
        tj.quantize_nvfp4(x, sel=ni)
    with pytest.raises(ValueError, match="1-D"):
        tj.quantize_nvfp4(x, sel=oi.view(8, 7))
    with pytest.raises(ValueError, match="contiguous"):
        tj.quantize_nvfp4(x, sel=torch.arange(0, 256, dtype=torch.int32, device="cuda")[::2])
    a, b = tj.quantize_nvfp4(_x(128, 256)), tj.quantize_nvfp4(_x(136, 256, 1))
    short = torch.arange(0, 100, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError, match="at least 136"):     # one target column per output column
        tj.gemm_nvfp4(a, b, out=torch.empty(128, 300, device="cuda"), col_map=short)


def test_optimizer_state_must_be_contiguous_and_whole(tj):
    rows, cols = 128, 256
    w = _x(rows, cols, dtype=torch.float32)
    q = [tj.quantize_nvfp4(w), tj.NVFP4.empty(rows, cols)]
    mask = torch.empty(rows * cols // 32, dtype=torch.int32, device="cuda")
    z = torch.zeros_like(w)
    wide = torch.zeros(rows, 2 * cols, device="cuda")
    with pytest.raises(ValueError, match="contiguous"):
        tj.osci_reset(w, w.clone(), wide[:, :cols], z.clone(), q[0], q[1], mask, 1e-5, 1e-4, 4.0)
    with pytest.raises(ValueError, match="at least"):
        tj.osci_reset(w, w.clone(), z.clone(), z.clone(), q[0], q[1], mask[:-1], 1e-5, 1e-4, 4.0)
    with pytest.raises(ValueError, match="elements"):
        tj.adamw_osci_reset(w, z[:64], z.clone(), z.clone(), w.clone(), z.clone(), z.clone(), q[0], q[1], mask,
                            1e-4, 0.9, 0.95, 1e-8, 0.1, 1, 1e-4, 4.0)


def test_short_or_foreign_buffers_of_a_quantized_tensor_are_refused(tj):
    q = tj.NVFP4.empty(128, 256)
    short = tj.NVFP4(q.codes[:-1], q.sf, q.outer, 128, 256)
    with pytest.raises(ValueError, match="codes"):
        tj.dequantize_nvfp4(short)
    wrong = tj.NVFP4(q.codes, q.sf, q.outer.view(torch.int32), 128, 256)
    with pytest.raises(ValueError, match="outer"):
        tj.dequantize_nvfp4(wrong)
    m = tj.MXFP8.empty(128, 256, fmt=tj.TJ_MX_E2M3)
    m.fmt = 7
    with pytest.raises(ValueError, match="format"):
        tj.dequantize_mxfp8(m)
    with pytest.raises(ValueError, match="CUDA"):
        tj.quantize_nvfp4(torch.zeros(128, 128, dtype=torch.bfloat16))


def test_any_view_of_a_single_row_is_read_as_that_row(tj):
    """One row: the binding passes its length as the row stride, whatever stride torch gives
    the size-1 dimension, and the result equals that of the contiguous row."""
    K = 512
    col = _x(K, 1, 5)                                          # [K, 1]: .t() has strides (1, 1)
    row_t = col.t()
    assert row_t.stride() == (1, 1)
    big = _x(8, 2 * K, 5)
    row_v = big[3:4, K:]                                       # row stride 2K
    for row in (row_t, row_v):
        ref = tj.quantize_nvfp4(row.contiguous(), mode=tj.TJ_SR, rht=True, seed=3, tag=1, rht_tag=2)
        got = tj.quantize_nvfp4(row, mode=tj.TJ_SR, rht=True, seed=3, tag=1, rht_tag=2)
        torch.cuda.synchronize()
        assert torch.equal(got.codes, ref.codes) and torch.equal(got.sf, ref.sf)
        assert np.array_equal(got.outer.cpu().numpy().view(np.uint32), ref.outer.cpu().numpy().view(np.uint32))
