"""GPU parity of the FP8 (E4M3) forward (fa_fwd_fp8) against the fp64 oracle
on the same E4M3 inputs and descale factors.

The scores are exact products accumulated in fp32, so LSE meets the plain
forward's 1e-3.  O is different: P is rounded to E4M3 (3 mantissa bits,
relative error at most 2^-4) before the P V product, so
|O_i - O_ref,i| <= 2^-4 * sum_j p_ij |v_j| / sum_j p_ij <= 2^-4 max |v| for
every element (plus the bf16 output rounding, 2^-8 relative); with the
roundings of different keys independent, the root-mean-square error stays
below 2^-4 / sqrt(3) times the rms of v.  Both bounds are checked, the
second being the sharper test.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from attention_forward_10_gb300 import build
    build.build()
    import attention_forward_10_gb300 as fa_mod
    fa_mod.fa_set_max_ctas(0)
    fa_mod.fa_set_wait_timeout_us(2_000_000)
    return fa_mod


def _inputs(B, H, H_kv, N, seed, mult=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, N, 128, generator=g) * mult).to(torch.float8_e4m3fn)
    k = (torch.randn(B, H_kv, N, 128, generator=g) * mult).to(torch.float8_e4m3fn)
    v = torch.randn(B, H_kv, N, 128, generator=g).to(torch.float8_e4m3fn)
    return q, k, v


def _run(fa, q, k, v, scale, dq, dk, dv, causal, window=(-1, -1)):
    o, lse = fa.fwd_fp8(q.cuda(), k.cuda(), v.cuda(), scale=scale, descale_q=dq, descale_k=dk,
                        descale_v=dv, causal=causal, window=window)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    return o, lse


def _check(o, lse, o_ref, l_ref, v, dv, what):
    o_np = o.float().cpu().numpy()
    l_np = lse.cpu().numpy()
    assert np.isfinite(o_np).all() and np.isfinite(l_np).all(), what
    err_l = float(np.abs(l_np - l_ref).max())
    assert err_l <= 1e-3, f"{what}: max|dLSE| = {err_l:.3e}"
    vv = v.float().numpy() * dv
    diff = np.abs(o_np - o_ref)
    bound = 2.0 ** -4 * float(np.abs(vv).max()) + 2.0 ** -8 * float(np.abs(o_ref).max())
    assert float(diff.max()) <= bound, f"{what}: max|dO| = {diff.max():.3e} > {bound:.3e}"
    rms = float(np.sqrt((diff ** 2).mean()))
    rms_bound = 2.0 ** -4 / math.sqrt(3) * float(np.sqrt((vv ** 2).mean()))
    assert rms <= rms_bound, f"{what}: rms dO = {rms:.3e} > {rms_bound:.3e}"
    return float(diff.max()), rms


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("N", [1, 127, 128, 300, 1000])
def test_shapes(fa, causal, N):
    q, k, v = _inputs(2, 2, 2, N, seed=1000 + N)
    o, lse = _run(fa, q, k, v, 1 / math.sqrt(128), 1.0, 1.0, 1.0, causal)
    o_ref, l_ref = oracle.attention_fp8(q, k, v, 1 / math.sqrt(128), 1.0, 1.0, 1.0, causal)
    _check(o, lse, o_ref, l_ref, v, 1.0, f"N={N} causal={causal}")


@pytest.mark.parametrize("descales", [(0.5, 2.0, 0.25), (0.125, 0.5, 3.0)])
@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 1)])
@pytest.mark.parametrize("window", [(-1, -1), (100, 0), (64, 64)])
def test_descales_groups_windows(fa, descales, H, H_kv, window):
    q, k, v = _inputs(1, H, H_kv, 700, seed=1100 + H_kv, mult=2.0)
    o, lse = _run(fa, q, k, v, 0.09, *descales, False, window)
    o_ref, l_ref = oracle.attention_fp8(q, k, v, 0.09, *descales, False, *window)
    _check(o, lse, o_ref, l_ref, v, descales[2], f"{descales} H={H}/{H_kv} window={window}")


@pytest.mark.parametrize("ctas", [1, 3])
def test_persistent_loop(fa, ctas):
    q, k, v = _inputs(1, 3, 3, 1500, seed=1200 + ctas)
    fa.fa_set_max_ctas(ctas)
    try:
        o, lse = _run(fa, q, k, v, 0.088, 1.0, 1.0, 1.0, True)
    finally:
        fa.fa_set_max_ctas(0)
    o_ref, l_ref = oracle.attention_fp8(q, k, v, 0.088, 1.0, 1.0, 1.0, True)
    _check(o, lse, o_ref, l_ref, v, 1.0, f"ctas={ctas}")


def test_print_error_levels(fa, capsys):
    """Reports the measured error levels of a mid-size case (kept in the log)."""
    q, k, v = _inputs(2, 4, 4, 2048, seed=1300)
    o, lse = _run(fa, q, k, v, 1 / math.sqrt(128), 1.0, 1.0, 1.0, False)
    o_ref, l_ref = oracle.attention_fp8(q, k, v, 1 / math.sqrt(128), 1.0, 1.0, 1.0, False)
    mx, rms = _check(o, lse, o_ref, l_ref, v, 1.0, "N=2048")
    with capsys.disabled():
        print(f"\nFP8 N=2048: max|dO| {mx:.3e}, rms dO {rms:.3e}, "
              f"max|dLSE| {np.abs(lse.cpu().numpy() - l_ref).max():.3e}")
