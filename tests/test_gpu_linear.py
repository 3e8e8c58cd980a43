"""GPU parity: the NVFP4 linear layer (forward, dX, dW) through the C ABI.

Every quantized operand the calls produce (saved X-hat, the SR + RHT operands
of the backward, the re-aligned W-hat^T / X-hat^T, the FP8 slices) is compared
bit for bit with the oracle; the products are compared within
2e-3 * sum|a||b| of the oracle's fp64 GEMM on those same operands.
"""
import numpy as np
import pytest
import torch

from layouts import (abs_product, abs_product_fp8, assert_gemm_close, assert_mxfp8_equal, assert_nvfp4_equal,
                     carve_workspace)
from nvfp4_bit_fully_gb300 import workloads
from oracle import linear as OL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


def _setup(tj, X, W, outl):
    K = X.shape[1]
    if len(outl):
        normal = OL.normal_channels(K, outl)
        ni = torch.from_numpy(normal.astype(np.int32)).cuda()
        oi = torch.from_numpy(np.asarray(outl, np.int32)).cuda()
        wq = tj.quantize_nvfp4(W.cuda(), sel=ni)
        w8 = tj.quantize_mxfp8(W.cuda(), sel=oi)
    else:
        ni = oi = None
        wq = tj.quantize_nvfp4(W.cuda())
        w8 = None
    return ni, oi, wq, w8


def _run_and_check(tj, X, W, dY, outl, seed):
    M, K = X.shape
    N = W.shape[0]
    k = len(outl)
    ni, oi, wq, w8 = _setup(tj, X, W, outl)
    y, xq, x8 = tj.linear_fwd(X.cuda(), wq, w8, ni, oi, out_dtype=torch.float32)
    ws_dx = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DX, M, N, K, k), dtype=torch.uint8, device="cuda")
    ws_dw = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DW, M, N, K, k), dtype=torch.uint8, device="cuda")
    dx = tj.linear_bwd_dx(dY.cuda(), wq, w8, ni, oi, seed=seed, out_dtype=torch.float32, workspace=ws_dx)
    dw = tj.linear_bwd_dw(dY.cuda(), xq, x8, ni, oi, seed=seed, workspace=ws_dw)
    torch.cuda.synchronize()
    tj.device_status()

    Xf, Wf, dYf = X.float().numpy(), W.float().numpy(), dY.float().numpy()
    Y_ref, fx, fw = OL.forward(Xf, Wf, outl)
    # forward: saved context bit-exact, product within tolerance
    assert_nvfp4_equal(xq, fx["q"], "X-hat")
    bound = abs_product(fx["q"], fw["q"])
    if k:
        assert_mxfp8_equal(x8, fx["q8"], "X-hat FP8 slice")
        bound = bound + abs_product_fp8(fx["q8"], fw["q8"])
    assert_gemm_close(y.cpu().numpy(), Y_ref, bound, what="Y")

    # dX: operands in the workspace bit-exact, product within tolerance
    K_N = K - k
    s_dy, s_w, q8_dy, q8_w = OL.bwd_dx_operands(dYf, fw, seed)
    parts = [("nv", M, N), ("nv", K_N, N)] + ([("mx", M, N), ("mx", k, N)] if k else [])
    views = carve_workspace(ws_dx, parts)
    assert_nvfp4_equal(views[0], s_dy, "S_dY")
    assert_nvfp4_equal(views[1], s_w, "S_W (re-aligned W-hat^T)")
    if k:
        assert_mxfp8_equal(views[2], q8_dy, "Q8(dY)")
        assert_mxfp8_equal(views[3], q8_w, "Q8(W-hat_O^T)")
    dx_ref = OL.bwd_dx(dYf, fw, outl, seed)
    nc = OL.normal_channels(K, outl)
    bx = np.zeros((M, K))
    bx[:, nc] = abs_product(s_dy, s_w, OL.ALPHA_RHT)[:, :K_N]
    if k:
        bx[:, outl] = abs_product_fp8(q8_dy, q8_w)[:, :k]
    assert_gemm_close(dx.cpu().numpy(), dx_ref, bx, what="dX")

    # dW
    s_dyt, s_x, q8_dyt, q8_x = OL.bwd_dw_operands(dYf, fx, seed)
    parts = [("nv", N, M), ("nv", K_N, M)] + ([("mx", N, M), ("mx", k, M)] if k else [])
    views = carve_workspace(ws_dw, parts)
    assert_nvfp4_equal(views[0], s_dyt, "S_dY^T")
    assert_nvfp4_equal(views[1], s_x, "S_X (re-aligned X-hat^T)")
    if k:
        assert_mxfp8_equal(views[2], q8_dyt, "Q8(dY^T)")
        assert_mxfp8_equal(views[3], q8_x, "Q8(X-hat_O^T)")
    dw_ref = OL.bwd_dw(dYf, fx, outl, seed)
    bw = np.zeros((N, K))
    bw[:, nc] = abs_product(s_dyt, s_x, OL.ALPHA_RHT)[:, :K_N]
    if k:
        bw[:, outl] = abs_product_fp8(q8_dyt, q8_x)[:, :k]
    assert_gemm_close(dw.cpu().numpy(), dw_ref, bw, what="dW")


def test_tiny_linear_no_outliers(tj):
    X, W, dY = workloads.tiny(seed=0)
    _run_and_check(tj, X, W, dY, np.array([], dtype=np.int64), seed=0)


def test_tiny_linear_with_outcontrol(tj):
    X, W, dY = workloads.tiny(seed=0)
    heavy = workloads.heavy_columns(512, 8, 0, 1 + 7919).numpy()
    s = (X.float() ** 2).sum(dim=0).numpy()
    outl = np.sort(np.argsort(-s, kind="stable")[:52])          # top 10% channels
    assert set(heavy) <= set(outl)
    _run_and_check(tj, X, W, dY, outl, seed=5)


def test_every_channel_an_outlier(tj):
    """The degenerate OutControl split with p = 100%: no NVFP4 channels, the whole layer in
    the FP8 slice (the empty NVFP4 parts are skipped, the products are the slice's alone)."""
    g = torch.Generator().manual_seed(29)
    M, N, K = 200, 136, 256
    X = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    dY = (torch.randn(M, N, generator=g) * 1e-3).to(torch.bfloat16)
    _run_and_check(tj, X, W, dY, np.arange(K), seed=9)


def _random_case(case):
    """A seeded random layer: M, N, K anywhere from one element to a few tiles (so every
    dimension is ragged in its own way), and 0 to 80 outlier channels at random positions
    (every channel, when K is that small)."""
    rng = np.random.default_rng(4000 + case)
    M, N, K = int(rng.integers(1, 520)), int(rng.integers(1, 400)), int(rng.integers(1, 600))
    k = int(rng.integers(0, min(K, 80) + 1))
    outl = np.sort(rng.choice(K, k, replace=False)).astype(np.int64)
    g = torch.Generator().manual_seed(4000 + case)
    X = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    dY = (torch.randn(M, N, generator=g) * 1e-3).to(torch.bfloat16)
    return X, W, dY, outl


@pytest.mark.parametrize("case", range(12))
def test_random_ragged_shapes(tj, case):
    """Twelve seeded random shapes and outlier sets through forward, dX and dW, checked like
    the fixed cases: every quantized operand bit for bit, the products within tolerance."""
    X, W, dY, outl = _random_case(case)
    _run_and_check(tj, X, W, dY, outl, seed=17 + case)


def test_ragged_linear(tj):
    g = torch.Generator().manual_seed(11)
    M, N, K = 200, 136, 328
    X = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    dY = (torch.randn(M, N, generator=g) * 1e-3).to(torch.bfloat16)
    outl = np.array([3, 40, 41, 200, 327])
    _run_and_check(tj, X, W, dY, outl, seed=17)


@pytest.mark.parametrize("k_out", [0, 26])
def test_long_token_dw_splits_k(tj, k_out):
    """2048 tokens and a few output tiles: the dW launch halves its K over two works per tile
    that add into the zeroed fp32 output (two additions onto zero, so the bits do not depend
    on their order).  Same checks as above, and a second call gives the same bits."""
    g = torch.Generator().manual_seed(23)
    M, N, K = 2048, 200, 264
    X = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    dY = (torch.randn(M, N, generator=g) * 1e-3).to(torch.bfloat16)
    outl = np.sort(np.random.default_rng(3).choice(K, k_out, replace=False))
    _run_and_check(tj, X, W, dY, outl, seed=29)
    ni, oi, wq, w8 = _setup(tj, X, W, outl)
    _, xq, x8 = tj.linear_fwd(X.cuda(), wq, w8, ni, oi)
    dw1 = tj.linear_bwd_dw(dY.cuda(), xq, x8, ni, oi, seed=29)
    dw2 = tj.linear_bwd_dw(dY.cuda(), xq, x8, ni, oi, seed=29)
    torch.cuda.synchronize()
    assert torch.equal(dw1, dw2)
    if k_out:
        # the same dW from the public steps, the GEMM as tj_gemm_pair_f32: bit-identical
        dYc = dY.cuda()
        s_dyt = tj.quantize_nvfp4(dYc, along_cols=True, mode=tj.TJ_SR, rht=True, seed=29, tag=tj.TAG_DY_COL,
                                  rht_tag=tj.TAG_RHT_DW)
        s_x = tj.requantize_nvfp4(xq, tj.TJ_SR, True, 29, tj.TAG_XT, tj.TAG_RHT_DW)
        dw3 = torch.full((N, K), 7.0, device="cuda")
        tj.gemm_pair_f32(s_dyt, s_x, tj.quantize_mxfp8(dYc, along_cols=True), tj.requantize_mxfp8(x8), dw3, ni, oi,
                         alpha=2.0 ** -7)
        torch.cuda.synchronize()
        assert torch.equal(dw1, dw3)


def test_linear_calls_equal_their_steps(tj):
    """tj_linear_fwd / bwd_dx / bwd_dw give bit-identical results to the sequence of
    public step calls (quantize, requantize, GEMM) that the benchmark times one by one."""
    g = torch.Generator().manual_seed(12)
    M, N, K = 256, 384, 520
    X = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16).cuda()
    dY = (torch.randn(M, N, generator=g) * 1e-3).to(torch.bfloat16).cuda()
    outl = np.sort(np.random.default_rng(3).choice(K, 52, replace=False))
    ni, oi, wq, w8 = _setup(tj, X.cpu(), W.cpu(), outl)
    seed = 99
    y, xq, x8 = tj.linear_fwd(X, wq, w8, ni, oi, out_dtype=torch.float32)
    dx = tj.linear_bwd_dx(dY, wq, w8, ni, oi, seed=seed, out_dtype=torch.float32)
    dw = tj.linear_bwd_dw(dY, xq, x8, ni, oi, seed=seed)
    # the same step, call by call
    xq2 = tj.quantize_nvfp4(X, sel=ni)
    x82 = tj.quantize_mxfp8(X, sel=oi)
    y2 = tj.gemm_nvfp4(xq2, wq, x82, w8)
    s_dy = tj.quantize_nvfp4(dY, mode=tj.TJ_SR, rht=True, seed=seed, tag=tj.TAG_DY_ROW, rht_tag=tj.TAG_RHT_DX)
    s_w = tj.requantize_nvfp4(wq, tj.TJ_SR, True, seed, tj.TAG_WT, tj.TAG_RHT_DX)
    dx2 = torch.zeros(M, K, device="cuda")
    tj.gemm_nvfp4(s_dy, s_w, alpha=2.0 ** -7, out=dx2, col_map=ni)
    tj.gemm_mxfp8(tj.quantize_mxfp8(dY), tj.requantize_mxfp8(w8), out=dx2, col_map=oi)
    s_dyt = tj.quantize_nvfp4(dY, along_cols=True, mode=tj.TJ_SR, rht=True, seed=seed, tag=tj.TAG_DY_COL,
                              rht_tag=tj.TAG_RHT_DW)
    s_x = tj.requantize_nvfp4(xq2, tj.TJ_SR, True, seed, tj.TAG_XT, tj.TAG_RHT_DW)
    dw2 = torch.zeros(N, K, device="cuda")
    tj.gemm_nvfp4(s_dyt, s_x, alpha=2.0 ** -7, out=dw2, col_map=ni)
    tj.gemm_mxfp8(tj.quantize_mxfp8(dY, along_cols=True), tj.requantize_mxfp8(x82), out=dw2, col_map=oi)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(dx, dx2) and torch.equal(dw, dw2)


def test_linear_is_deterministic(tj):
    """Every output of the layer is a fixed function of its inputs: two runs over 4096 tokens
    (many tiles per CTA, split-K dW, the FP8 slice) give the same bytes."""
    g = torch.Generator().manual_seed(31)
    M, N, K = 4096, 1536, 1024
    X = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    dY = (torch.randn(M, N, generator=g) * 1e-3).to(torch.bfloat16).cuda()
    outl = np.sort(np.random.default_rng(5).choice(K, 103, replace=False))
    ni, oi, wq, w8 = _setup(tj, X.cpu(), W, outl)
    runs = []
    for _ in range(2):
        y, xq, x8 = tj.linear_fwd(X, wq, w8, ni, oi)
        dx = tj.linear_bwd_dx(dY, wq, w8, ni, oi, seed=17)
        dw = tj.linear_bwd_dw(dY, xq, x8, ni, oi, seed=17)
        runs.append([y, xq.codes, xq.sf, xq.outer, x8.codes, x8.sf, dx, dw])
    torch.cuda.synchronize()
    tj.device_status()
    for a, b in zip(*runs):
        assert torch.equal(a, b)


def test_strided_inputs_and_outputs(tj):
    """X, dY and the outputs as column slices of wider buffers (row strides K + 40, N + 24,
    N + 16, K + 8): every result equals the contiguous call byte for byte, and the columns
    beyond each view are left untouched."""
    g = torch.Generator().manual_seed(37)
    M, N, K = 300, 200, 328
    outl = np.sort(np.random.default_rng(7).choice(K, 33, replace=False))
    Xw = torch.randn(M, K + 40, generator=g).to(torch.bfloat16).cuda()
    dYw = (torch.randn(M, N + 24, generator=g) * 1e-3).to(torch.bfloat16).cuda()
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    ni, oi, wq, w8 = _setup(tj, Xw[:, :K].cpu(), W, outl)
    X, dY = Xw[:, :K], dYw[:, :N]
    y_ref, xq_ref, x8_ref = tj.linear_fwd(X.contiguous(), wq, w8, ni, oi)
    dx_ref = tj.linear_bwd_dx(dY.contiguous(), wq, w8, ni, oi, seed=3)
    dw_ref = tj.linear_bwd_dw(dY.contiguous(), xq_ref, x8_ref, ni, oi, seed=3)
    yw = torch.full((M, N + 16), 5.0, dtype=torch.bfloat16, device="cuda")
    dxw = torch.full((M, K + 8), 5.0, dtype=torch.bfloat16, device="cuda")
    dww = torch.full((N, K + 8), 5.0, device="cuda")
    y, xq, x8 = tj.linear_fwd(X, wq, w8, ni, oi, out=yw[:, :N])
    dx = tj.linear_bwd_dx(dY, wq, w8, ni, oi, seed=3, out=dxw[:, :K])
    dw = tj.linear_bwd_dw(dY, xq, x8, ni, oi, seed=3, out=dww[:, :K])
    torch.cuda.synchronize()
    tj.device_status()
    for a, b in ((y, y_ref), (dx, dx_ref), (dw, dw_ref), (xq.codes, xq_ref.codes), (xq.sf, xq_ref.sf),
                 (xq.outer, xq_ref.outer), (x8.codes, x8_ref.codes), (x8.sf, x8_ref.sf)):
        assert torch.equal(a, b)
    assert bool((yw[:, N:] == 5.0).all()) and bool((dxw[:, K:] == 5.0).all()) and bool((dww[:, K:] == 5.0).all())


def test_concurrent_streams(tj):
    """Two layers forward and backward on two streams at once equal the same calls run one
    after the other: the launches share no hidden state and honour their stream."""
    g = torch.Generator().manual_seed(41)
    M, N, K = 2048, 640, 512
    outl = np.sort(np.random.default_rng(9).choice(K, 52, replace=False))
    layers = []
    for _ in range(2):
        X = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
        W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
        dY = (torch.randn(M, N, generator=g) * 1e-3).to(torch.bfloat16).cuda()
        ni, oi, wq, w8 = _setup(tj, X.cpu(), W, outl)
        layers.append((X, dY, ni, oi, wq, w8))

    def run(L, stream=None):
        X, dY, ni, oi, wq, w8 = L
        y, xq, x8 = tj.linear_fwd(X, wq, w8, ni, oi, stream=stream)
        dx = tj.linear_bwd_dx(dY, wq, w8, ni, oi, seed=5, stream=stream)
        dw = tj.linear_bwd_dw(dY, xq, x8, ni, oi, seed=5, stream=stream)
        return [y, dx, dw, xq.codes, xq.sf, xq.outer, x8.codes, x8.sf]

    ref = [run(L) for L in layers]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    got = []
    for L, s in zip(layers, streams):
        with torch.cuda.stream(s):
            got.append(run(L, stream=s))
    torch.cuda.synchronize()
    tj.device_status()
    for r, o in zip(ref, got):
        for a, b in zip(r, o):
            assert torch.equal(a, b)


def test_cuda_graph_capture(tj):
    """The layer's launches (forward, dX, dW) captured into one CUDA graph and replayed give
    the eager calls' bytes; a replay after the inputs change gives the new results."""
    g = torch.Generator().manual_seed(43)
    M, N, K = 1024, 512, 512
    k = 52
    outl = np.sort(np.random.default_rng(11).choice(K, k, replace=False))
    X = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    dY = (torch.randn(M, N, generator=g) * 1e-3).to(torch.bfloat16).cuda()
    ni, oi, wq, w8 = _setup(tj, X.cpu(), W, outl)
    # buffers the graph writes, allocated up front
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    xq, x8 = tj.NVFP4.empty(M, K - k), tj.MXFP8.empty(M, k)
    dx = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    dw = torch.empty(N, K, dtype=torch.float32, device="cuda")
    ws_dx = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DX, M, N, K, k), dtype=torch.uint8, device="cuda")
    ws_dw = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DW, M, N, K, k), dtype=torch.uint8, device="cuda")

    def layer():
        tj.linear_fwd(X, wq, w8, ni, oi, xq=xq, x8=x8, out=y)
        tj.linear_bwd_dx(dY, wq, w8, ni, oi, seed=13, workspace=ws_dx, out=dx)
        tj.linear_bwd_dw(dY, xq, x8, ni, oi, seed=13, workspace=ws_dw, out=dw)

    def snapshot():
        return [t.clone() for t in (y, dx, dw, xq.codes, xq.sf, xq.outer, x8.codes, x8.sf)]

    layer()                                  # eager (also sets the kernels' launch attributes)
    torch.cuda.synchronize()
    eager = snapshot()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            layer()
    torch.cuda.current_stream().wait_stream(s)
    for t in (y, dx, dw):
        t.fill_(7.0)
    graph.replay()
    torch.cuda.synchronize()
    tj.device_status()
    for a, b in zip(eager, snapshot()):
        assert torch.equal(a, b)
    # new inputs in the same buffers: the replay computes them
    X.copy_(torch.randn(M, K, generator=g).to(torch.bfloat16))
    dY.mul_(-2.0)
    layer()
    torch.cuda.synchronize()
    eager2 = snapshot()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager2, snapshot()):
        assert torch.equal(a, b)
    assert not torch.equal(eager[0], eager2[0])
