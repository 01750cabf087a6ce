"""GPU parity of the FP8 (E4M3) forward (fa_fwd_fp8) against the fp64 oracle
on the same E4M3 inputs and descale factors.

The scores are exact products accumulated in fp32, so LSE meets the plain
forward's 1e-3.  O differs from the oracle's by the E4M3 rounding of P
before the P V product (the page's FP8 path rounds P to the input type).
With the kernel's exponent offset, every p_j sent to E4M3 lies in
(0, 2^8]; the row sum l that O is divided by uses the unrounded p and is at
least 2^6 (the largest p of the row).  A normal E4M3 value has 3 fraction
bits, so its rounding error e_j is at most 2^-4 p_j; below 2^-6 (the
subnormal range) it is at most 2^-10 absolute, i.e. 2^-16 of l.  Taking
each e_j uniform over its interval and independent of the others (the
usual model of round-to-nearest), the error of O_ic = sum_j p~_j v_jc / l
has variance at most

    sigma_ic^2 = (2^-4)^2 / 3 * sum_j P_ij^2 v_jc^2
               + (2^-16)^2 / 3 * sum_{j in J(i)} v_jc^2

with P_ij the exact softmax weights.  The first sum comes from the oracle
itself: run on v^2 with the scale doubled it returns
O2_ic = sum_j exp(2 s_ij - LSE2_i) v_jc^2, and
sum_j P_ij^2 v_jc^2 = O2_ic * exp(LSE2_i - 2 LSE_i).  The second is the
oracle with Q = 0 (the mean of v^2 over the admissible keys) times |J(i)|.

Checks, each with the bf16 output rounding (2^-8 relative) on top:
  * every element within 6 sigma_ic (a single dominant key gives at most
    sqrt(3) sigma; many keys give an error close to normal with standard
    deviation at most sigma);
  * the RMS error of every row within 2.5 times that row's RMS sigma;
  * the RMS error of the whole output within 1.2 times the RMS sigma (the
    expected ratio is about 0.73: the bound takes every p at the bottom of
    its binade).
A host-side negative control adds 5e-3 to one row of a GPU result and
requires the check to fail.
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


def _real_bf16(x, descale):
    """The real values descale * x of an E4M3 tensor as bfloat16 (exact: an
    E4M3 value has 4 significant bits and the descales here are powers of
    two)."""
    real = x.float() * descale
    out = real.to(torch.bfloat16)
    assert torch.equal(out.float(), real), "descaled E4M3 values must be exact in bf16"
    return out


def _sigma(q, k, v, scale, dq, dk, dv, causal, window, l_ref):
    """Per-element standard deviation bound sigma_ic of the E4M3 rounding of P
    (module docstring), from two more oracle calls."""
    qr, kr = _real_bf16(q, dq), _real_bf16(k, dk)
    v2 = ((v.float() * dv) ** 2).to(torch.bfloat16)   # rounding: 2^-9 of a variance
    o2, lse2 = oracle.attention_ex(qr, kr, v2, 2.0 * scale, causal, *window)
    sum_p2v2 = o2 * np.exp(lse2 - 2.0 * l_ref)[..., None]
    o0, lse0 = oracle.attention_ex(torch.zeros_like(qr), kr, v2, scale, causal, *window)
    sum_v2 = o0 * np.exp(lse0)[..., None]
    var = (2.0 ** -4) ** 2 / 3.0 * sum_p2v2 + (2.0 ** -16) ** 2 / 3.0 * sum_v2
    return np.sqrt(var)


def _check_o(o_np, o_ref, sigma, what):
    """The three O checks of the module docstring; returns (max err, rms err,
    rms sigma)."""
    diff = np.abs(o_np - o_ref)
    out_round = 2.0 ** -8 * np.abs(o_ref)
    elem_bound = 6.0 * sigma + out_round + 1e-5
    worst = np.unravel_index(np.argmax(diff - elem_bound), diff.shape)
    assert (diff <= elem_bound).all(), (
        f"{what}: |dO| {diff[worst]:.3e} > 6 sigma + rounding {elem_bound[worst]:.3e} at {worst}")
    row_rms = np.sqrt((diff ** 2).mean(axis=-1))
    row_sigma = np.sqrt((sigma ** 2).mean(axis=-1))
    row_bound = 2.5 * row_sigma + 2.0 ** -8 * np.sqrt((o_ref ** 2).mean(axis=-1)) + 1e-5
    worst = np.unravel_index(np.argmax(row_rms - row_bound), row_rms.shape)
    assert (row_rms <= row_bound).all(), (
        f"{what}: row rms dO {row_rms[worst]:.3e} > {row_bound[worst]:.3e} at row {worst}")
    rms = float(np.sqrt((diff ** 2).mean()))
    rms_sigma = float(np.sqrt((sigma ** 2).mean()))
    rms_bound = 1.2 * rms_sigma + 2.0 ** -8 * float(np.sqrt((o_ref ** 2).mean())) + 1e-6
    assert rms <= rms_bound, f"{what}: rms dO {rms:.3e} > {rms_bound:.3e}"
    return float(diff.max()), rms, rms_sigma


def _check(o, lse, o_ref, l_ref, sigma, what):
    o_np = o.float().cpu().numpy()
    l_np = lse.cpu().numpy()
    assert np.isfinite(o_np).all() and np.isfinite(l_np).all(), what
    err_l = float(np.abs(l_np - l_ref).max())
    assert err_l <= 1e-3, f"{what}: max|dLSE| = {err_l:.3e}"
    return _check_o(o_np, o_ref, sigma, what)


def _case(fa, B, H, H_kv, N, seed, scale, descales, causal, window=(-1, -1), mult=1.0):
    q, k, v = _inputs(B, H, H_kv, N, seed, mult)
    o, lse = _run(fa, q, k, v, scale, *descales, causal, window)
    o_ref, l_ref = oracle.attention_fp8(q, k, v, scale, *descales, causal, *window)
    sigma = _sigma(q, k, v, scale, *descales, causal, window, l_ref)
    return o, lse, o_ref, l_ref, sigma


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("N", [1, 127, 128, 300, 1000])
def test_shapes(fa, causal, N):
    o, lse, o_ref, l_ref, sigma = _case(fa, 2, 2, 2, N, 1000 + N, 1 / math.sqrt(128),
                                        (1.0, 1.0, 1.0), causal)
    _check(o, lse, o_ref, l_ref, sigma, f"N={N} causal={causal}")


@pytest.mark.parametrize("descales", [(0.5, 2.0, 0.25), (0.125, 0.5, 3.0)])
@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 1)])
@pytest.mark.parametrize("window", [(-1, -1), (100, 0), (64, 64)])
def test_descales_groups_windows(fa, descales, H, H_kv, window):
    o, lse, o_ref, l_ref, sigma = _case(fa, 1, H, H_kv, 700, 1100 + H_kv, 0.09, descales, False,
                                        window, mult=2.0)
    _check(o, lse, o_ref, l_ref, sigma, f"{descales} H={H}/{H_kv} window={window}")


@pytest.mark.parametrize("ctas", [1, 3])
def test_persistent_loop(fa, ctas):
    fa.fa_set_max_ctas(ctas)
    try:
        o, lse, o_ref, l_ref, sigma = _case(fa, 1, 3, 3, 1500, 1200 + ctas, 0.088,
                                            (1.0, 1.0, 1.0), True)
    finally:
        fa.fa_set_max_ctas(0)
    _check(o, lse, o_ref, l_ref, sigma, f"ctas={ctas}")


def test_error_levels_and_negative_control(fa, capsys):
    """A mid-size case: reports the measured error against the bound, then
    shifts one row of the GPU result by 5e-3 on the host and requires the
    same check to reject it."""
    o, lse, o_ref, l_ref, sigma = _case(fa, 2, 4, 4, 2048, 1300, 1 / math.sqrt(128),
                                        (1.0, 1.0, 1.0), False)
    mx, rms, rms_sigma = _check(o, lse, o_ref, l_ref, sigma, "N=2048")
    with capsys.disabled():
        print(f"\nFP8 N=2048: max|dO| {mx:.3e}, rms dO {rms:.3e}, rms sigma bound "
              f"{rms_sigma:.3e} (rms test limit {1.2 * rms_sigma:.3e}), "
              f"max|dLSE| {np.abs(lse.cpu().numpy() - l_ref).max():.3e}")
    shifted = o.float().cpu().numpy().copy()
    shifted[1, 2, 777, :] += 5e-3
    with pytest.raises(AssertionError):
        _check_o(shifted, o_ref, sigma, "shifted row")
