"""ssm_proj (the x_proj / dt_proj products on the tensor cores) against the
oracle's fp64 product of the same bf16 inputs, bf16 outputs checked
element-wise against 2e-3 max|ref| + 2^-8 |ref|: ragged m, n and k (partial
tiles, K not a multiple of the 64-wide stage), batches, strided views (dt_proj
reads the first R rows of x_proj's output), the bias + softplus epilogue, and
the x_proj -> dt_proj chain at the Mamba-1.4B layer's shape on sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import assert_close, to_np

pytestmark = pytest.mark.gpu


def _lib():
    import selective_state_space_147_b300 as L
    return L


@pytest.mark.parametrize("batch,m,n,k", [(1, 128, 128, 64), (2, 288, 256, 4096), (1, 100, 200, 200),
                                         (3, 300, 1000, 520), (2, 4096, 384, 256), (1, 8, 8, 8),
                                         # more tiles than SMs at K <= 256: contiguous tile ranges that
                                         # cross row tiles, W reloaded inside a CTA
                                         (2, 4096, 2560, 256), (3, 1000, 3000, 200)])
def test_products(batch, m, n, k):
    L = _lib()
    W = S.normal(40, 1, (m, k), torch.bfloat16, std=k ** -0.5)
    X = S.normal(40, 2, (batch, k, n), torch.bfloat16)
    out = L.ssm_proj(W.cuda(), X.cuda())
    assert L.device_status() == 0
    assert_close(out, oracle.proj(W, X), torch.bfloat16, torch.bfloat16, what=f"{batch}x{m}x{n}x{k}")


def test_bias_softplus_epilogue():
    L = _lib()
    m, n, k = 200, 256, 192
    W = S.normal(41, 1, (m, k), torch.bfloat16, std=k ** -0.5)
    X = S.normal(41, 2, (2, k, n), torch.bfloat16)
    b = S.normal(41, 3, (m,), torch.float32)
    out = L.ssm_proj(W.cuda(), X.cuda(), bias=b.cuda(), softplus=True)
    assert_close(out, oracle.proj(W, X, bias=b, softplus=True), torch.bfloat16, torch.bfloat16)


def test_strided_views():
    """X a row slice of a wider tensor, out a slice of a wider buffer."""
    L = _lib()
    R, N, L_ = 64, 16, 320
    big = S.normal(42, 1, (2, R + 2 * N, L_), torch.bfloat16).cuda()
    W = S.normal(42, 2, (96, R), torch.bfloat16, std=R ** -0.5).cuda()
    buf = torch.zeros(2, 100, L_ + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[:, 2:98, 8:]
    L.ssm_proj(W, big[:, :R], out=out)
    ref = oracle.proj(W.cpu(), big[:, :R].cpu())
    assert_close(out, ref, torch.bfloat16, torch.bfloat16)
    assert torch.count_nonzero(buf[:, :2]) == 0 and torch.count_nonzero(buf[:, 98:]) == 0
    assert torch.count_nonzero(buf[..., :8]) == 0


def test_x_dt_proj_mamba1p4b_sampled_tokens():
    """d_inner 4096, dt_rank 256, d_state 16, batch 8, L 16384: delta, B, C on
    sampled token columns (the oracle rounds dt_raw to bf16 as the library stores it)."""
    L = _lib()
    seed = S.config_seed(2)
    b, D, T, N, R = 8, 4096, 16384, 16, 256
    xc = S.normal(seed, S.STREAM["u"], (b, D, T), torch.bfloat16, "cuda")
    W_x, W_dt = S.proj_weights(seed, D, R, N, "cuda")
    delta, Bm, Cm, x_dbl = L.x_dt_proj(xc, W_x, W_dt, N)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    rng = np.random.default_rng(5)
    cols = np.sort(rng.choice(T, size=16, replace=False))
    for bb in (0, 5):
        X = xc[bb][:, cols].cpu()[None]
        ref_dbl = oracle.proj(W_x.cpu(), X)
        assert_close(x_dbl[bb][:, cols][None], ref_dbl, torch.bfloat16, torch.bfloat16, what=f"x_dbl b{bb}")
        assert_close(Bm[bb][:, cols][None], ref_dbl[:, R:R + N], torch.bfloat16, torch.bfloat16, what="B")
        assert_close(Cm[bb][:, cols][None], ref_dbl[:, R + N:], torch.bfloat16, torch.bfloat16, what="C")
        dt_raw = x_dbl[bb][:R, cols].cpu()[None]          # the bf16 values the library stored
        ref_delta = oracle.proj(W_dt.cpu(), dt_raw)
        assert_close(delta[bb][:, cols][None], ref_delta, torch.bfloat16, torch.bfloat16, what=f"delta b{bb}")
