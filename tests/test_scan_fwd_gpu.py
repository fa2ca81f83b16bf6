"""ssm_scan_fwd on the GPU against the fp64 oracle, element by element."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import assert_close, to_np

pytestmark = pytest.mark.gpu

THREADS = oracle.default_threads()


def _lib():
    import selective_state_space_147_b300 as L
    return L


def make(seed, batch, dim, L, N, dtype, device="cuda", delta_range=(1e-3, 1e-1), with_z=True,
         with_h0=False):
    g = S.scan_inputs(seed, batch, dim, L, N, dtype=dtype, device="cpu", delta_range=delta_range,
                      with_z=with_z, with_h0=with_h0)
    return {k: (v.to(device) if v is not None else None) for k, v in g.items()}


def run_gpu(g, zoh=True, out_dtype=torch.float32, softplus=True, use_D=True, use_bias=True,
            final=False, **kw):
    L = _lib()
    return L.ssm_scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], D=g["D"] if use_D else None,
                          delta_bias=g["bias"] if use_bias else None, z=g["z"], h0=g["h0"],
                          bbar_mode=L.SSM_BBAR_ZOH if zoh else L.SSM_BBAR_SIMPLE,
                          delta_softplus=softplus, out_dtype=out_dtype, return_final_state=final, **kw)


def run_oracle(g, zoh=True, softplus=True, use_D=True, use_bias=True):
    return oracle.scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["D"] if use_D else None,
                           g["bias"] if use_bias else None, g["z"], g["h0"], zoh=zoh,
                           delta_softplus=softplus, threads=THREADS)


@pytest.fixture
def schedule():
    """Force a (G, nseg) schedule: the forward then goes through ssm_scan_fwd_scheduled."""
    state = {}

    def set_(G=None, nseg=None):
        state.clear()
        state.update(lanes_per_channel=G or 0, segments=nseg or 0)
    set_.kw = lambda: {"schedule": dict(state)} if state else {}
    return set_


def test_tiny_fp32_config():
    """B1 D16 N16 L256, fp32, ZOH: the small exact-parity workload (1e-5)."""
    g = make(S.config_seed(0), 1, 16, 256, 16, torch.float32)
    out, hN = run_gpu(g, final=True)
    ref, href = run_oracle(g)
    assert_close(out, ref, torch.float32, what="out")
    assert_close(hN, href, torch.float32, what="final_state")


@pytest.mark.parametrize("zoh", [True, False])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("G,nseg", [(1, 1), (2, 1), (4, 1), (1, 3), (4, 5)])
def test_schedules_and_modes(schedule, zoh, dtype, G, nseg):
    schedule(G, nseg)
    # dim 100 is not a multiple of any channel group; L 1000 leaves a ragged tile and sub-block
    g = make(7, 2, 100, 1000, 16, dtype, with_h0=True)
    out, hN = run_gpu(g, zoh=zoh, final=True, **schedule.kw())
    ref, href = run_oracle(g, zoh=zoh)
    assert_close(out, ref, dtype, what="out")
    assert_close(hN, href, dtype, what="final_state")


@pytest.mark.parametrize("N", [1, 3, 4, 8, 13, 16, 17, 24, 32, 33, 48, 64])
def test_state_sizes(N):
    g = make(8, 1, 40, 300, N, torch.bfloat16)
    out, hN = run_gpu(g, final=True)
    ref, href = run_oracle(g)
    assert_close(out, ref, torch.bfloat16, what="out")
    assert_close(hN, href, torch.bfloat16, what="final_state")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("zoh", [True, False])
def test_large_state_with_checkpoints_and_segments(dtype, zoh, schedule):
    """d_state 40 (three state groups): outputs, final state and every checkpoint,
    also under the segmented schedule."""
    schedule(None, 3)
    N, L, K = 40, 600, 8
    g = make(16, 2, 36, L, N, dtype, with_h0=True)
    lib = _lib()
    ck = lib.checkpoint_buffer(2, 36, L, N, every=K).fill_(float("nan"))
    out, hN = run_gpu(g, final=True, checkpoints=ck, checkpoint_every=K, zoh=zoh, **schedule.kw())
    ref, href = run_oracle(g, zoh=zoh)
    assert_close(out, ref, dtype, what="out")
    assert_close(hN, href, dtype, what="final_state")
    cs = lib.checkpoint_states(ck, N)
    for k in (1, 37, (L - 1) // K):
        _, hk = oracle.scan_fwd(g["u"][..., :k * K], g["dt"][..., :k * K], g["A"], g["B"][..., :k * K],
                                g["C"][..., :k * K], g["D"], g["bias"], g["z"][..., :k * K], g["h0"], zoh=zoh,
                                threads=THREADS)
        assert_close(cs[:, k], hk, dtype, what=f"checkpoint {k}")


@pytest.mark.parametrize("L", [1, 3, 7, 8, 9, 63, 64, 65, 129])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_short_and_ragged_lengths(L, dtype):
    g = make(9, 2, 33, L, 16, dtype, with_h0=True)
    out, hN = run_gpu(g, final=True)
    ref, href = run_oracle(g)
    assert_close(out, ref, dtype, what="out")
    assert_close(hN, href, dtype, what="final_state")


def test_seqlen_zero_copies_h0():
    g = make(10, 2, 5, 0, 16, torch.bfloat16, with_h0=True)
    out, hN = run_gpu(g, final=True)
    assert out.shape == (2, 5, 0)
    assert torch.equal(hN, g["h0"])


@pytest.mark.parametrize("softplus,use_D,use_bias,with_z", [
    (False, True, True, True), (True, False, True, True), (True, True, False, False),
    (False, False, False, False)])
def test_optional_inputs(softplus, use_D, use_bias, with_z):
    g = make(11, 2, 64, 200, 16, torch.float32, with_z=with_z)
    if not softplus:
        # without softplus delta = dt + bias must stay positive by construction
        g["dt"] = g["dt"].abs() * 0.05 + 1e-3
        g["bias"] = torch.full_like(g["bias"], 0.01)
    out = run_gpu(g, softplus=softplus, use_D=use_D, use_bias=use_bias)
    ref, _ = run_oracle(g, softplus=softplus, use_D=use_D, use_bias=use_bias)
    assert_close(out, ref, torch.float32)


@pytest.mark.parametrize("zoh", [True, False])
def test_bf16_output_bound(zoh):
    g = make(12, 2, 96, 777, 16, torch.bfloat16)
    out = run_gpu(g, zoh=zoh, out_dtype=torch.bfloat16)
    ref, _ = run_oracle(g, zoh=zoh)
    assert out.dtype == torch.bfloat16
    assert_close(out, ref, torch.bfloat16, torch.bfloat16)


def test_unaligned_and_strided_rows():
    # L = 37 leaves bf16 rows 2-byte aligned only; the inputs are also views into a
    # wider buffer (row stride 40), which the 16-byte path must not assume away
    g = make(13, 2, 24, 37, 16, torch.bfloat16)
    wide = {}
    for k in ("u", "dt", "z"):
        buf = torch.zeros(2, 24, 40, dtype=torch.bfloat16, device="cuda")
        buf[..., 1:38] = g[k]
        wide[k] = buf[..., 1:38]
    g2 = dict(g, **wide)
    out = run_gpu(g2)
    ref, _ = run_oracle(g)
    assert_close(out, ref, torch.bfloat16)


def test_zero_A_takes_the_limit():
    g = make(14, 1, 64, 150, 16, torch.bfloat16)
    A = g["A"].clone()
    A[5, 3] = 0.0
    A[40, 0] = 0.0
    g["A"] = A
    out = run_gpu(g)
    ref, _ = run_oracle(g)
    assert_close(out, ref, torch.bfloat16)


@pytest.mark.parametrize("K", [4, 8, 12, 64, 136])
def test_checkpoints(schedule, K):
    schedule(None, 3)
    g = make(15, 2, 40, 700, 16, torch.bfloat16, with_h0=True)
    L = 700
    nck = (L + K - 1) // K
    lib = _lib()
    ck = lib.checkpoint_buffer(2, 40, L, 16, every=K).fill_(float("nan"))
    run_gpu(g, checkpoints=ck, checkpoint_every=K, **schedule.kw())
    ck = lib.checkpoint_states(ck, 16)
    for k in range(nck):
        t = k * K
        if t == 0:
            ref = to_np(g["h0"])
        else:
            _, ref = oracle.scan_fwd(g["u"][..., :t], g["dt"][..., :t], g["A"], g["B"][..., :t],
                                     g["C"][..., :t], g["D"], g["bias"], g["z"][..., :t], g["h0"],
                                     threads=THREADS)
        assert_close(ck[:, k], ref, torch.bfloat16, what=f"checkpoint {k}")


@pytest.mark.parametrize("zoh", [True, False])
def test_mamba130m_layer_full_size(zoh):
    """B8 D1536 N16 L2048 bf16 inputs: every output element against the oracle."""
    g = make(S.config_seed(1), 8, 1536, 2048, 16, torch.bfloat16)
    out = run_gpu(g, zoh=zoh)
    ref, _ = run_oracle(g, zoh=zoh)
    assert_close(out, ref, torch.bfloat16, what="out")


def test_deterministic():
    g = make(16, 4, 512, 1024, 16, torch.bfloat16)
    a = run_gpu(g)
    b = run_gpu(g)
    assert torch.equal(a, b)


@pytest.mark.parametrize("zoh", [True, False])
@pytest.mark.parametrize("L,N,out_dtype", [(1000, 16, torch.float32), (256, 16, torch.bfloat16), (5000, 12, torch.float32),
                                           (1, 16, torch.float32), (777, 3, torch.bfloat16)])
def test_warp_scan_schedule(zoh, L, N, out_dtype):
    """The warp-shuffle chunked schedule: ragged chunks (L not a multiple of 256),
    d_state below 16, h0 and the final state, both output dtypes."""
    g = make(17, 2, 40, L, N, torch.bfloat16, with_h0=True)
    out, hN = run_gpu(g, zoh=zoh, final=True, out_dtype=out_dtype, schedule={"warp_scan": 1})
    ref, href = run_oracle(g, zoh=zoh)
    assert_close(out, ref, torch.bfloat16, out_dtype, what="out")
    assert_close(hN, href, torch.bfloat16, what="final_state")


def test_warp_scan_long_sequence_and_groups():
    """L 2^17 at batch 1 (many chunks: the carry across chunks), and B/C groups."""
    g = make(18, 1, 8, 1 << 17, 16, torch.bfloat16, delta_range=(1e-4, 1e-2), with_h0=True)
    out, hN = run_gpu(g, final=True, schedule={"warp_scan": 1})
    ref, href = run_oracle(g)
    assert_close(out, ref, torch.bfloat16, what="out")
    assert_close(hN, href, torch.bfloat16, what="final_state")
    L = _lib()
    gg = S.scan_inputs(19, 2, 256, 600, 16, dtype=torch.bfloat16)
    Bg = S.normal(19, 40, (2, 2, 16, 600), torch.bfloat16)
    Cg = S.normal(19, 41, (2, 2, 16, 600), torch.bfloat16)
    dev = {k: (v.cuda() if v is not None else None) for k, v in gg.items()}
    out = L.ssm_scan_fwd(dev["u"], dev["dt"], dev["A"], Bg.cuda(), Cg.cuda(), D=dev["D"], delta_bias=dev["bias"],
                         z=dev["z"], out_dtype=torch.float32, schedule={"warp_scan": 1})
    for grp in range(2):
        sl = slice(128 * grp, 128 * grp + 128)
        ref, _ = oracle.scan_fwd(gg["u"][:, sl], gg["dt"][:, sl], gg["A"][sl], Bg[:, grp], Cg[:, grp], gg["D"][sl],
                                 gg["bias"][sl], gg["z"][:, sl], threads=THREADS)
        assert_close(out[:, sl], ref, torch.bfloat16, what=f"group {grp}")
