"""GPU test of the GEMM's time-out path, made on the host with the test hook
tj_debug_gemm_fault: the producers of one launch never load one stage, and the
launch's waits are bounded by a short limit.  That launch must give up, report
TJ_ERR_TIMEOUT through tj_get_device_status, and return; the GPU must go on answering,
and the next normal launch must match the oracle.

Nothing faults, traps or hangs the GPU: the wait that runs out is an mbarrier wait with
a time bound, and the CPU model in test_gemm_abort_model.py shows that the hardware
named barriers of the abort path always complete.
"""
import numpy as np
import pytest
import torch

from layouts import abs_product, abs_product_fp8, assert_gemm_close
from oracle import linear as OL
from test_gpu_gemm import _fp8_operands, _operands

pytestmark = pytest.mark.gpu

TJ_ERR_TIMEOUT = 6
WAIT_CLK = 200000                # about 0.1 ms at the maximum SM clock


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


def _status(tj):
    return tj.load().tj_get_device_status()


@pytest.mark.parametrize("M,N,K,skip", [(256, 512, 512, 1),       # 8 tiles of 4 blocks: 2 stages per CTA
                                         (2048, 1536, 512, 3)])     # 192 tiles: two per CTA on 40 CTAs
def test_skipped_stage_times_out_and_the_next_launch_is_correct(tj, M, N, K, skip):
    qa, qb, ra, rb = _operands(tj, M, N, K, seed=61)
    out = torch.empty(M, N, device="cuda")
    torch.cuda.synchronize()
    assert _status(tj) == 0
    assert tj.load().tj_debug_gemm_fault(skip, WAIT_CLK) == 0
    tj.gemm_nvfp4(qa, qb, out=out)
    torch.cuda.synchronize()
    assert _status(tj) == TJ_ERR_TIMEOUT
    assert _status(tj) == 0                       # read and cleared
    # the GPU answers, and a normal launch is correct
    assert torch.cuda.is_available() and torch.ones(4, device="cuda").sum().item() == 4.0
    tj.gemm_nvfp4(qa, qb, out=out)
    torch.cuda.synchronize()
    assert _status(tj) == 0
    assert_gemm_close(out.cpu().numpy(), OL.gemm_fp4(ra, rb), abs_product(ra, rb), what="after time-out")


def test_skipped_fp8_stage_of_a_pair_launch(tj):
    """The FP8 slice's stages follow the FP4 stages of a tile; skipping one of them aborts
    a launch whose partial slots and barriers hold both kinds of block."""
    M, N, K, k = 384, 300, 640, 700
    qa, qb, ra, rb = _operands(tj, M, N, K, seed=62)
    a8, b8, ra8, rb8 = _fp8_operands(tj, M, 96, k, seed=63)
    out = torch.zeros(M, N + 96, device="cuda")
    cm = torch.arange(N, dtype=torch.int32, device="cuda")
    cm8 = torch.arange(N, N + 96, dtype=torch.int32, device="cuda")
    assert tj.load().tj_debug_gemm_fault(4, WAIT_CLK) == 0
    tj.gemm_pair(qa, qb, a8, b8, out=out, out8=out, col_map=cm, col_map8=cm8)
    torch.cuda.synchronize()
    assert _status(tj) == TJ_ERR_TIMEOUT
    tj.gemm_pair(qa, qb, a8, b8, out=out, out8=out, col_map=cm, col_map8=cm8)
    torch.cuda.synchronize()
    assert _status(tj) == 0
    got = out.cpu().numpy()
    assert_gemm_close(got[:, :N], OL.gemm_fp4(ra, rb), abs_product(ra, rb), what="pair fp4 after time-out")
    assert_gemm_close(got[:, N:], OL.gemm_fp8(ra8, rb8), abs_product_fp8(ra8, rb8), what="pair fp8 after time-out")


def test_armed_hook_without_a_reachable_stage_changes_nothing(tj):
    """A skipped stage beyond every CTA's stages and a short bound: the launch completes."""
    M, N, K = 256, 256, 1024
    qa, qb, ra, rb = _operands(tj, M, N, K, seed=64)
    assert tj.load().tj_debug_gemm_fault(10 ** 6, 50_000_000) == 0
    out = tj.gemm_nvfp4(qa, qb)
    torch.cuda.synchronize()
    assert _status(tj) == 0
    assert_gemm_close(out.cpu().numpy(), OL.gemm_fp4(ra, rb), abs_product(ra, rb), what="armed, no fault")


def test_hook_argument_errors(tj):
    assert tj.load().tj_debug_gemm_fault(-2, 0) == 1
    assert tj.load().tj_debug_gemm_fault(0, -1) == 1
    assert tj.load().tj_debug_gemm_fault(-1, 0) == 0               # disarmed
