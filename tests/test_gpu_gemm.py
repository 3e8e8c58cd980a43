"""GPU parity: the tcgen05 block-scaled GEMM vs the oracle's fp64 product.

The operands are quantized on the GPU (bit-exact against the oracle, checked
here again), then |D_gpu - D_oracle| <= 2e-3 * sum_k |a_mk||b_nk| per output.
Shapes cover one tile, several tiles, an odd number of 128-K blocks (a half
pipeline stage), ragged M / N, the FP8 slice alone and combined, column
scatter and bf16 output.
"""
import numpy as np
import pytest
import torch

from layouts import abs_product, abs_product_fp8, assert_gemm_close, assert_mxfp8_equal, assert_nvfp4_equal
from oracle import linear as OL
from oracle import quant as Q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


def _rand(rows, cols, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * scale
    x[:, torch.randperm(cols, generator=g)[: max(1, cols // 64)]] *= 20
    return x.to(torch.bfloat16)


def _operands(tj, M, N, K, mode=0, seed=0):
    A = _rand(M, K, seed + 1)
    B = _rand(N, K, seed + 2, 0.05)
    qa = tj.quantize_nvfp4(A.cuda(), mode=mode, seed=seed, tag=1)
    qb = tj.quantize_nvfp4(B.cuda(), mode=mode, seed=seed, tag=2)
    ra = Q.quantize_nvfp4(A.float().numpy(), mode, seed=seed, tag=1)
    rb = Q.quantize_nvfp4(B.float().numpy(), mode, seed=seed, tag=2)
    torch.cuda.synchronize()
    assert_nvfp4_equal(qa, ra, "A")
    assert_nvfp4_equal(qb, rb, "B")
    return qa, qb, ra, rb


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 512), (128, 128, 384), (200, 300, 640),
                                   (512, 256, 1024)])
def test_gemm_fp4(tj, M, N, K):
    qa, qb, ra, rb = _operands(tj, M, N, K, mode=1, seed=M + N + K)
    d = tj.gemm_nvfp4(qa, qb)
    torch.cuda.synchronize()
    tj.device_status()
    ref = OL.gemm_fp4(ra, rb)
    assert_gemm_close(d.cpu().numpy(), ref, abs_product(ra, rb), what="fp4 %dx%dx%d" % (M, N, K))


def test_gemm_fp4_alpha_bf16_and_scatter(tj):
    M, N, K = 256, 200, 256
    qa, qb, ra, rb = _operands(tj, M, N, K, seed=9)
    cmap = torch.randperm(300, generator=torch.Generator().manual_seed(2))[:N].to(torch.int32)
    out = torch.full((M, 300), -7.0, dtype=torch.bfloat16, device="cuda")
    tj.gemm_nvfp4(qa, qb, alpha=2.0 ** -7, out=out, col_map=cmap.cuda())
    torch.cuda.synchronize()
    ref = OL.gemm_fp4(ra, rb, 2.0 ** -7)
    got = out.float().cpu().numpy()
    assert_gemm_close(got[:, cmap.numpy()], ref, abs_product(ra, rb, 2.0 ** -7), bf16=True, what="scatter")
    untouched = np.setdiff1d(np.arange(300), cmap.numpy())
    assert np.all(got[:, untouched] == -7.0)


def _fp8_operands(tj, M, N, k, seed):
    A = _rand(M, k, seed + 5, 30.0)
    B = _rand(N, k, seed + 6, 0.05)
    a8 = tj.quantize_mxfp8(A.cuda())
    b8 = tj.quantize_mxfp8(B.cuda())
    ra = Q.quantize_mxfp8(A.float().numpy())
    rb = Q.quantize_mxfp8(B.float().numpy())
    torch.cuda.synchronize()
    assert_mxfp8_equal(a8, ra, "A8")
    assert_mxfp8_equal(b8, rb, "B8")
    return a8, b8, ra, rb


@pytest.mark.parametrize("M,N,k", [(128, 128, 128), (256, 103, 103), (300, 410, 410)])
def test_gemm_fp8_slice(tj, M, N, k):
    a8, b8, ra, rb = _fp8_operands(tj, M, N, k, seed=k)
    d = tj.gemm_mxfp8(a8, b8)
    torch.cuda.synchronize()
    ref = OL.gemm_fp8(ra, rb)
    assert_gemm_close(d.cpu().numpy(), ref, abs_product_fp8(ra, rb), what="fp8")


def test_gemm_fp4_plus_fp8_same_tile(tj):
    M, N, K, k = 256, 256, 384, 40
    qa, qb, ra, rb = _operands(tj, M, N, K, seed=3)
    a8, b8, ra8, rb8 = _fp8_operands(tj, M, N, k, seed=4)
    d = tj.gemm_nvfp4(qa, qb, a8, b8)
    torch.cuda.synchronize()
    ref = OL.gemm_fp4(ra, rb) + OL.gemm_fp8(ra8, rb8)
    bound = abs_product(ra, rb) + abs_product_fp8(ra8, rb8)
    assert_gemm_close(d.cpu().numpy(), ref, bound, what="fp4+fp8")


def test_gemm_pipeline_over_many_tiles(tj):
    """More tiles than SMs (each CTA walks several), an odd number of FP4 blocks (a half
    last stage) and an FP8 slice of six 128-K stages in the same tiles, so that partial
    slots, scale-factor slots and the outer-scale ring all wrap across tile boundaries."""
    M, N, K, k = 2048, 1536, 640, 700
    qa, qb, ra, rb = _operands(tj, M, N, K, seed=21)
    a8, b8, ra8, rb8 = _fp8_operands(tj, M, N, k, seed=22)
    d = tj.gemm_nvfp4(qa, qb, a8, b8, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    tj.device_status()
    rows = np.random.default_rng(5).choice(M, 96, replace=False)
    sub = lambda q: tuple(x[rows] for x in q)
    ref = OL.gemm_fp4(sub(ra), rb) + OL.gemm_fp8(sub(ra8), rb8)
    bound = abs_product(sub(ra), rb) + abs_product_fp8(sub(ra8), rb8)
    assert_gemm_close(d.float().cpu().numpy()[rows], ref, bound, bf16=True, what="many tiles fp4+fp8")


def test_gemm_fp8_slice_long(tj):
    """An FP8-only product whose K spans more stages than the FP8 scale-factor slots."""
    M, N, k = 384, 256, 1500
    a8, b8, ra, rb = _fp8_operands(tj, M, N, k, seed=31)
    d = tj.gemm_mxfp8(a8, b8)
    torch.cuda.synchronize()
    tj.device_status()
    ref = OL.gemm_fp8(ra, rb)
    assert_gemm_close(d.cpu().numpy(), ref, abs_product_fp8(ra, rb), what="fp8 long")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_pair_equals_the_two_products(tj, out_dtype):
    """An FP4 product and an FP8-only product in one launch, written through disjoint column
    maps into one output: each matches the oracle, and both equal the separate calls."""
    M, N, K, k = 384, 300, 640, 700
    qa, qb, ra, rb = _operands(tj, M, N, K, seed=41)
    a8, b8, ra8, rb8 = _fp8_operands(tj, M, 96, k, seed=42)
    perm = torch.randperm(N + 96, generator=torch.Generator().manual_seed(7)).to(torch.int32)
    cm, cm8 = perm[:N].sort().values, perm[N:].sort().values
    out = torch.full((M, N + 96), -3.0, dtype=out_dtype, device="cuda")
    tj.gemm_pair(qa, qb, a8, b8, alpha=2.0 ** -7, out=out, out8=out, col_map=cm.cuda(), col_map8=cm8.cuda())
    ref_sep = torch.full_like(out, -3.0)
    tj.gemm_nvfp4(qa, qb, alpha=2.0 ** -7, out=ref_sep, col_map=cm.cuda())
    tj.gemm_mxfp8(a8, b8, out=ref_sep, col_map=cm8.cuda())
    torch.cuda.synchronize()
    tj.device_status()
    assert torch.equal(out, ref_sep)
    got = out.float().cpu().numpy()
    bf = out_dtype == torch.bfloat16
    assert_gemm_close(got[:, cm.numpy()], OL.gemm_fp4(ra, rb, 2.0 ** -7), abs_product(ra, rb, 2.0 ** -7), bf16=bf,
                      what="pair fp4")
    assert_gemm_close(got[:, cm8.numpy()], OL.gemm_fp8(ra8, rb8), abs_product_fp8(ra8, rb8), bf16=bf, what="pair fp8")


@pytest.mark.parametrize("K,k", [(2048, 1024), (640, 256)])
def test_gemm_pair_f32_whole_output(tj, K, k):
    """tj_gemm_pair_f32: both fp32 products fill one matrix through their column maps.  With 8
    or more stages of K in both products and few tiles the call zeroes the matrix and splits K
    in two (first case); the result matches the oracle, agrees with tj_gemm_pair to fp32
    rounding, and repeats bit for bit.  Without a split (second case) it is tj_gemm_pair's."""
    M, N, N8 = 384, 300, 96
    qa, qb, ra, rb = _operands(tj, M, N, K, seed=51)
    a8, b8, ra8, rb8 = _fp8_operands(tj, M, N8, k, seed=52)
    perm = torch.randperm(N + N8, generator=torch.Generator().manual_seed(8)).to(torch.int32)
    cm, cm8 = perm[:N].sort().values.cuda(), perm[N:].sort().values.cuda()
    out = torch.full((M, N + N8), 5.0, dtype=torch.float32, device="cuda")
    tj.gemm_pair_f32(qa, qb, a8, b8, out, cm, cm8, alpha=2.0 ** -7)
    again = torch.full_like(out, -1.0)
    tj.gemm_pair_f32(qa, qb, a8, b8, again, cm, cm8, alpha=2.0 ** -7)
    ref = torch.full_like(out, 5.0)
    tj.gemm_pair(qa, qb, a8, b8, alpha=2.0 ** -7, out=ref, out8=ref, col_map=cm, col_map8=cm8)
    torch.cuda.synchronize()
    tj.device_status()
    assert torch.equal(out, again)
    if K < 2048:
        assert torch.equal(out, ref)
    else:
        assert float((out - ref).abs().max()) <= 1e-5 * float(ref.abs().max())
    got = out.cpu().numpy()
    assert_gemm_close(got[:, cm.cpu().numpy()], OL.gemm_fp4(ra, rb, 2.0 ** -7), abs_product(ra, rb, 2.0 ** -7),
                      what="pair_f32 fp4")
    assert_gemm_close(got[:, cm8.cpu().numpy()], OL.gemm_fp8(ra8, rb8), abs_product_fp8(ra8, rb8), what="pair_f32 fp8")


@pytest.mark.parametrize("mode,rht,fmt", [(1, True, 0), (0, False, 5), (1, True, 3)])
def test_realignment_pair_equals_the_two_calls(tj, mode, rht, fmt):
    """tj_requantize_nvfp4_mxfp8: the NVFP4 operand and its slice re-aligned in one launch are
    byte for byte the two separate calls."""
    g = torch.Generator().manual_seed(17 + fmt)
    X = torch.randn(300, 700, generator=g).to(torch.bfloat16)
    q = tj.quantize_nvfp4(X[:, :597].contiguous().cuda())
    q8 = tj.quantize_mxfp8(X[:, 597:].contiguous().cuda(), fmt=fmt)
    a, a8 = tj.requantize_nvfp4_mxfp8(q, q8, mode, rht, 99, 4, 0x101)
    b = tj.requantize_nvfp4(q, mode, rht, 99, 4, 0x101)
    b8 = tj.requantize_mxfp8(q8)
    torch.cuda.synchronize()
    for x, y in ((a.codes, b.codes), (a.sf, b.sf), (a.outer, b.outer), (a8.codes, b8.codes), (a8.sf, b8.sf)):
        assert torch.equal(x, y)
