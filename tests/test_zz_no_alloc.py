"""GPU test of tj_linear_bwd_dx_noalloc, the input-gradient entry point for callers
that cannot allocate device memory when the backward runs (code below the
framework's allocator, or deployments that only use buffers registered up front).
It uses a fixed scratch array inside the library instead of a caller workspace.

Through the C ABI: a call of another shape, with another seed and the other
outlier setting, first leaves the shared scratch holding unrelated bytes.  Then
two calls in a row must each give the oracle's dX (oracle.linear.bwd_dx) within
the GEMM tolerance the other tests use, 2e-3 * sum|a||b| over the oracle's
quantized operands, and the same bits as tj_linear_bwd_dx with a caller
workspace; so no byte the previous call left in the scratch reaches the result.
A problem larger than the fixed scratch is rejected before any launch.  The call
also works inside a captured CUDA graph, whose replays give the same bits.  This file
is named to be collected last, and passes alone or after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from layouts import abs_product, assert_gemm_close
from oracle import linear as OL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


def _call_noalloc(tj, dy, wq, w8, ni, oi, seed, out):
    """Call the entry point directly through ctypes (no Python-side buffers besides dX)."""
    lib = tj.load()
    k = 0 if oi is None else oi.numel()
    cw = wq.c()
    cw8 = w8.c() if k else None
    code = lib.tj_linear_bwd_dx_noalloc(
        ctypes.c_void_p(dy.data_ptr()), dy.shape[0], dy.shape[1], dy.stride(0), ctypes.byref(cw),
        ctypes.byref(cw8) if cw8 is not None else None,
        ctypes.c_void_p(ni.data_ptr()) if ni is not None else None,
        ctypes.c_void_p(oi.data_ptr()) if oi is not None else None, k, seed,
        ctypes.c_void_p(out.data_ptr()), tj.TJ_FP32, out.stride(0),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, tj.STATUS.get(code, code)


def _problem(tj, M, N, K, with_outliers, seed):
    """Inputs of one backward: dY, the forward-quantized weight, and the channel lists."""
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    dY = (torch.randn(M, N, generator=g) * 1e-3).to(torch.bfloat16)
    if with_outliers:
        outl = np.arange(3, K, 10)[: max(1, K // 10)]
        normal = OL.normal_channels(K, outl)
        ni = torch.from_numpy(normal.astype(np.int32)).cuda()
        oi = torch.from_numpy(outl.astype(np.int32)).cuda()
        wq = tj.quantize_nvfp4(W.cuda(), sel=ni)
        w8 = tj.quantize_mxfp8(W.cuda(), sel=oi)
    else:
        outl = np.array([], dtype=np.int64)
        ni = oi = w8 = None
        wq = tj.quantize_nvfp4(W.cuda())
    return W, dY, outl, wq, w8, ni, oi


@pytest.mark.parametrize("with_outliers", [False, True])
def test_noalloc_matches_oracle_and_workspace_version_twice(tj, with_outliers):
    M, N, K, seed = 256, 512, 512, 77
    W, dY, outl, wq, w8, ni, oi = _problem(tj, M, N, K, with_outliers, seed=0)
    dyd = dY.cuda()
    ref = tj.linear_bwd_dx(dyd, wq, w8, ni, oi, seed=seed, out_dtype=torch.float32)
    # a call of another shape, seed and outlier setting fills the scratch with other bytes
    W2, dY2, _, wq2, w82, ni2, oi2 = _problem(tj, 384, 640, 768, not with_outliers, seed=5)
    junk = torch.empty(384, 768, device="cuda")
    _call_noalloc(tj, dY2.cuda(), wq2, w82, ni2, oi2, 991, junk)
    torch.cuda.synchronize()
    ref_np = ref.cpu().numpy()
    # the oracle's dX and the tolerance of the other GEMM tests: 2e-3 * sum|a||b| over the
    # quantized operands (FP4 product on the normal channels, FP8 slice on the outliers)
    _, _, fw = OL.forward(np.zeros((1, K), np.float32), W.float().numpy(), outl)
    dx_oracle = OL.bwd_dx(dY.float().numpy(), fw, outl, seed)
    s_dy, s_w, q8_dy, q8_w = OL.bwd_dx_operands(dY.float().numpy(), fw, seed)
    bound = np.zeros(ref_np.shape)
    bound[:, OL.normal_channels(K, outl)] = abs_product(s_dy, s_w, OL.ALPHA_RHT)[:, : K - len(outl)]
    if len(outl):
        from layouts import abs_product_fp8
        bound[:, outl] = abs_product_fp8(q8_dy, q8_w)[:, : len(outl)]
    for call in range(2):                                      # two calls in a row share the scratch
        out = torch.full_like(ref, float("nan"))
        _call_noalloc(tj, dyd, wq, w8, ni, oi, seed, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert_gemm_close(got, dx_oracle, bound, what="noalloc call %d" % call)
        assert np.array_equal(got, ref_np)
    tj.device_status()


def test_noalloc_rejects_problems_beyond_the_scratch(tj):
    lib = tj.load()
    limit = int(lib.tj_noalloc_scratch_bytes())
    assert limit == 16 << 20
    M, N, K = 16384, 4096, 1024                               # needs ~45 MB of scratch
    assert tj.workspace_size(tj.TJ_OP_BWD_DX, M, N, K, 0) > limit
    wq = tj.CNvfp4(256, 256, 256, N, K)
    code = lib.tj_linear_bwd_dx_noalloc(ctypes.c_void_p(256), M, N, N, ctypes.byref(wq), None, None, None, 0, 1,
                                        ctypes.c_void_p(256), tj.TJ_FP32, K, None)
    assert code == 7                                           # TJ_ERR_WORKSPACE, before any launch


def test_noalloc_in_a_cuda_graph(tj):
    """Captured into a CUDA graph (the scratch address is looked up while capturing) and
    replayed, the call writes the workspace version's dX byte for byte; after the scratch
    has been overwritten by an eager call of another shape, a replay still does."""
    M, N, K, seed = 256, 512, 512, 31
    W, dY, outl, wq, w8, ni, oi = _problem(tj, M, N, K, True, seed=2)
    dyd = dY.cuda()
    ref = tj.linear_bwd_dx(dyd, wq, w8, ni, oi, seed=seed, out_dtype=torch.float32)
    out = torch.empty_like(ref)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            tj.linear_bwd_dx_noalloc(dyd, wq, w8, ni, oi, seed=seed, out_dtype=torch.float32, out=out)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        W2, dY2, _, wq2, w82, ni2, oi2 = _problem(tj, 384, 640, 768, False, seed=5)
        tj.linear_bwd_dx_noalloc(dY2.cuda(), wq2, w82, ni2, oi2, seed=991, out_dtype=torch.float32)
        torch.cuda.synchronize()
    tj.device_status()
