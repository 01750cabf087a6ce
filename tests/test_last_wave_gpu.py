"""GPU parity of the last-wave split of the forward kernel (d = 64 and 128)
against the fp64 oracle.

When the 256-row query-pair units do not fill the last wave of CTAs, each
pair of that wave runs as two single-tile units, one per CTA; with fewer
pairs than CTAs, as many pairs as there are idle CTAs are split.  The grid is
capped with fa_set_max_ctas so that small problems take this path; every case
asserts that its shape does.  The cases add to the split tests of the main
parity file: d = 64, both parities of the key-tile count, heads with a
single key tile, grouped heads and windows, one dominant key, repeat-run
bit identity and the FP8 forward.

Tolerances are the forward's: max |O - O_ref| <= 2e-2, max |LSE - LSE_ref|
<= 1e-3 (the FP8 case uses the FP8 bounds of its own test file).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import make_random_qkv

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module")
def fa():
    from attention_forward_10_gb300 import build
    build.build()
    import attention_forward_10_gb300 as fa_mod
    fa_mod.fa_set_max_ctas(0)
    fa_mod.fa_set_wait_timeout_us(2_000_000)
    return fa_mod


def _splits_last_wave(B, H, N, ctas):
    """The launcher's rule: the partial last wave of L pair units is split
    when 2 L units fit in one wave."""
    pairs = B * H * ((N + 255) // 256)
    part = pairs % ctas
    return pairs > ctas and part > 0 and 2 * part <= ctas


def _run(fa, q, k, v, scale, causal, window, ctas):
    fa.fa_set_max_ctas(ctas)
    try:
        o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal,
                        window=window)
        torch.cuda.synchronize()
    finally:
        fa.fa_set_max_ctas(0)
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    return o, lse


def _check(o, lse, o_ref, lse_ref, what):
    o_np = o.float().cpu().numpy()
    l_np = lse.cpu().numpy()
    assert np.isfinite(o_np).all() and np.isfinite(l_np).all(), what
    err_o = float(np.abs(o_np - o_ref).max())
    err_l = float(np.abs(l_np - lse_ref).max())
    assert err_l <= LSE_TOL, f"{what}: max|dLSE| = {err_l:.3e} (O err {err_o:.3e})"
    assert err_o <= O_TOL, f"{what}: max|dO| = {err_o:.3e} (LSE err {err_l:.3e})"


# N, ctas: 9 key tiles (odd), 8 (even), 5 (odd), a ragged 900, and 200 rows
# (tile 0 of a causal head sees one key tile)
CASES = [(1100, 6), (1024, 5), (640, 4), (640, 6), (900, 5), (200, 5)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("N,ctas", CASES)
def test_split_units(fa, N, ctas, causal, d):
    B, H = (1, 7) if N == 200 else (1, 3)
    assert _splits_last_wave(B, H, N, ctas)
    q, k, v = make_random_qkv(B, H, N, d, torch.bfloat16, seed=1500 + N + ctas + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, scale, causal, (-1, -1), ctas)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    _check(o, lse, o_ref, lse_ref, f"N={N} ctas={ctas} causal={causal} d={d}")


def test_one_key_tile_per_head(fa):
    """128-row heads: each split tile has a single key tile."""
    q, k, v = make_random_qkv(1, 7, 128, 128, torch.float16, seed=1530)
    assert _splits_last_wave(1, 7, 128, 5)
    for causal in (False, True):
        o, lse = _run(fa, q, k, v, 0.1, causal, (-1, -1), 5)
        o_ref, lse_ref = oracle.attention(q, k, v, 0.1, causal)
        _check(o, lse, o_ref, lse_ref, f"causal={causal}")


@pytest.mark.parametrize("window", [(200, 0), (64, 64), (-1, 130)])
@pytest.mark.parametrize("H,H_kv", [(4, 2), (4, 1)])
def test_split_groups_and_windows(fa, H, H_kv, window):
    N, ctas = 1100, 6
    assert _splits_last_wave(1, H, N, ctas)
    q, _, _ = make_random_qkv(1, H, N, 128, torch.bfloat16, seed=1540 + H_kv)
    _, k, v = make_random_qkv(1, H_kv, N, 128, torch.bfloat16, seed=1541 + H_kv)
    o, lse = _run(fa, q, k, v, 0.09, False, window, ctas)
    o_ref, lse_ref = oracle.attention_ex(q, k, v, 0.09, False, *window)
    _check(o, lse, o_ref, lse_ref, f"H={H}/{H_kv} window={window}")


# the split units are rows 512-1023 of head 2 (full) and rows 0-255 of
# heads 1 and 2 (causal: heaviest pairs first); the key sits in an odd or an
# even key tile
@pytest.mark.parametrize("causal,j0", [(False, 3 * 128 + 17), (False, 4 * 128 + 5),
                                       (True, 128 + 2), (True, 5)],
                         ids=["full_odd_tile", "full_even_tile", "causal_odd_tile",
                              "causal_even_tile"])
def test_dominant_key_in_split_units(fa, j0, causal):
    """One key scores ~30 nats above the rest for every query that sees it:
    the running maximum jumps by ~43 (log2 units) inside a split unit."""
    N, ctas, d = 1024, 5, 128
    assert _splits_last_wave(1, 3, N, ctas)
    g = torch.Generator().manual_seed(1550 + j0)
    u = torch.randn(d, generator=g)
    u /= u.norm()
    c = 18.0
    q = torch.randn(1, 3, N, d, generator=g) + c * u
    k = torch.randn(1, 3, N, d, generator=g)
    k[:, :, j0, :] = c * u
    v = torch.randn(1, 3, N, d, generator=g)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, scale, causal, (-1, -1), ctas)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    _check(o, lse, o_ref, lse_ref, f"j0={j0} causal={causal}")
    # rows that see the key take (almost exactly) its value row
    rows = np.arange(j0 if causal else 0, N)
    np.testing.assert_allclose(o[0, 2, rows].float().cpu().numpy(),
                               np.broadcast_to(v[0, 2, j0].float().numpy(), (len(rows), d)),
                               atol=2e-2)


def test_split_runs_are_bit_identical(fa):
    q, k, v = make_random_qkv(1, 3, 1100, 128, torch.bfloat16, seed=1560)
    outs = [_run(fa, q, k, v, 0.09, True, (-1, -1), 6) for _ in range(3)]
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_split_fp8(fa, causal):
    """The FP8 forward shares the kernel; bounds as in its own parity file."""
    N, ctas = 1100, 6
    assert _splits_last_wave(1, 3, N, ctas)
    g = torch.Generator().manual_seed(1570)
    q = torch.randn(1, 3, N, 128, generator=g).to(torch.float8_e4m3fn)
    k = torch.randn(1, 3, N, 128, generator=g).to(torch.float8_e4m3fn)
    v = torch.randn(1, 3, N, 128, generator=g).to(torch.float8_e4m3fn)
    fa.fa_set_max_ctas(ctas)
    try:
        o, lse = fa.fwd_fp8(q.cuda(), k.cuda(), v.cuda(), scale=0.088, descale_q=1.0,
                            descale_k=1.0, descale_v=1.0, causal=causal)
        torch.cuda.synchronize()
    finally:
        fa.fa_set_max_ctas(0)
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    o_ref, l_ref = oracle.attention_fp8(q, k, v, 0.088, 1.0, 1.0, 1.0, causal)
    o_np, l_np = o.float().cpu().numpy(), lse.cpu().numpy()
    assert float(np.abs(l_np - l_ref).max()) <= 1e-3
    vv = v.float().numpy()
    bound = 2.0 ** -4 * float(np.abs(vv).max()) + 2.0 ** -8 * float(np.abs(o_ref).max())
    assert float(np.abs(o_np - o_ref).max()) <= bound


# ----------------------------------------------- fewer pairs than CTAs
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,ctas", [
    (1, 3, 256, 5),    # 3 pairs, 2 idle CTAs: 2 pairs split, 1 kept
    (1, 2, 1000, 0),   # 8 pairs on every SM: all split
    (1, 1, 300, 3),    # 2 pairs, the second holding a ragged 44-row tile
])
def test_first_wave_split(fa, B, H, N, ctas, causal, d):
    """With fewer 256-row pair units than CTAs, as many pairs as there are
    idle CTAs run as two single-tile units each."""
    q, k, v = make_random_qkv(B, H, N, d, torch.bfloat16, seed=90 + N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, scale, causal, (-1, -1), ctas)
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal)
    err_o = float(np.abs(o.float().cpu().numpy() - o_ref).max())
    err_l = float(np.abs(lse.cpu().numpy() - l_ref).max())
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)
