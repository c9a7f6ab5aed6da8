"""The tcgen05/TMA GEMM pipeline in isolation: every operand majorness and tile
width against torch's matmul of the same bf16 inputs (fp32 accumulation)."""
import pytest
import torch

from lm_head_kl_fkl_b300 import api

pytestmark = pytest.mark.gpu


def _case(M, N, K, a_mn, b_mn, bn, seed=0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    A_in = A.t().contiguous() if a_mn else A
    B_in = B.t().contiguous() if b_mn else B
    C = api.selftest_gemm(A_in, B_in, M, N, K, a_mn, b_mn, bn)
    ref = A.float() @ B.float().t()
    err = (C - ref).norm() / ref.norm()
    assert err < 1e-5, (M, N, K, a_mn, b_mn, bn, float(err))
    # elementwise: fp32 sums of the same products differ only in order
    tol = 1e-4 * (A.float().abs() @ B.float().abs().t())
    assert torch.all((C - ref).abs() <= tol + 1e-5), float((C - ref).abs().max())


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("bn", [512, 256, 192, 128])
def test_single_tile_exact_k(a_mn, b_mn, bn):
    _case(128, bn, 64, a_mn, b_mn, bn)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("bn", [512, 256, 192, 128])
def test_ragged_multi_tile(a_mn, b_mn, bn):
    # tails in M, N and K; several k-blocks and tiles per CTA
    _case(392, 584, 456, a_mn, b_mn, bn, seed=1)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1)])
def test_many_tiles_persistent(a_mn, b_mn):
    # more tiles than SMs: exercises the double-buffered accumulator and ring wrap-around
    _case(2048, 2304, 2880, a_mn, b_mn, 192 if b_mn else 256, seed=2)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 1), (1, 1), (0, 0)])
@pytest.mark.parametrize("N", [2880, 2816, 2624, 2936, 2968, 2504, 2560])
def test_wide_tiles_ragged_last_sub_tile(a_mn, b_mn, N):
    # 512-wide tiles.  Columns left for the last tile's second sub-tile, and the
    # sub-tile width that follows: 2880: 64 -> 64; 2816: 0 -> skipped; 2624: the
    # first sub-tile is itself ragged; 2936: 120 -> 128; 2968: 152 -> 192;
    # 2504: 200 -> 256; 2560: no ragged tile.
    _case(1000, N, 1216, a_mn, b_mn, 512, seed=3)
