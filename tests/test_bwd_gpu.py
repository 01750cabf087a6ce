"""GPU parity of the backward pass (fa_bwd) against the fp64 oracle.

The forward kernel provides O and LSE; fa_bwd then gives dQ, dK, dV for a
seeded dO.  The oracle recomputes everything in double from the same 16-bit
Q, K, V, dO.  Tolerance: the kernels round P and dS to the input type (2^-9
relative for bf16) before the P^T dO, dS^T Q and dS K products and round the
gradients on output, so each gradient must satisfy
max |dX - dX_ref| <= 2e-2 * max |dX_ref| + 1e-4, element by element (the
floor covers gradients that vanish exactly, such as dQ for N = 1, where the
kernels' D = rowsum(dO * O) uses the 16-bit O).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import make_random_qkv

pytestmark = pytest.mark.gpu

REL_TOL = 2e-2
ABS_FLOOR = 1e-4


@pytest.fixture(scope="module")
def fa():
    from attention_forward_10_gb300 import build
    build.build()
    import attention_forward_10_gb300 as fa_mod
    fa_mod.fa_set_max_ctas(0)
    fa_mod.fa_set_wait_timeout_us(2_000_000)
    return fa_mod


def _case(fa, B, H, H_kv, N, d, dtype, causal, window=(-1, -1), seed=0):
    q, _, _ = make_random_qkv(B, H, N, d, dtype, seed=800 + seed)
    _, k, v = make_random_qkv(B, H_kv, N, d, dtype, seed=801 + seed)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(802 + seed)).to(dtype)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, scale=scale, causal=causal, window=window)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal, window=window)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    ref = oracle.attention_bwd(q, k, v, do, scale, causal, *window)
    return (dq, dk, dv), ref


def _check(got, ref, what):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        gn = g.float().cpu().numpy()
        assert np.isfinite(gn).all(), f"{what}: non-finite {name}"
        err = float(np.abs(gn - r).max())
        bound = REL_TOL * float(np.abs(r).max()) + ABS_FLOOR
        assert err <= bound, f"{what}: {name} max err {err:.3e} > {bound:.3e}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("N", [1, 127, 128, 300, 513])
def test_shapes(fa, d, causal, dtype, N):
    got, ref = _case(fa, 2, 2, 2, N, d, dtype, causal, seed=N + d)
    _check(got, ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(4, 2), (4, 1)])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("window", [(-1, -1), (40, 40), (200, 0), (0, 0)])
def test_grouped_heads_and_windows(fa, d, H, H_kv, causal, window):
    got, ref = _case(fa, 1, H, H_kv, 400, d, torch.bfloat16, causal, window, seed=H_kv + d)
    _check(got, ref, f"d={d} H={H}/{H_kv} causal={causal} window={window}")


@pytest.mark.parametrize("ctas", [1, 3, 4, 5])
def test_persistent_loop(fa, ctas):
    """18 units of each kernel on 1-5 CTAs: with 4 the last wave (even) is
    partial, with 5 the last wave is partial and odd, so it runs reversed
    within itself."""
    fa.fa_set_max_ctas(ctas)
    try:
        got, ref = _case(fa, 1, 3, 3, 700, 128, torch.bfloat16, True, seed=50 + ctas)
    finally:
        fa.fa_set_max_ctas(0)
    _check(got, ref, f"ctas={ctas}")


@pytest.mark.parametrize("ctas", [1, 2, 5])
@pytest.mark.parametrize("d,H,H_kv,N,causal,window", [
    (128, 4, 2, 700, False, (-1, -1)),   # units spanning two query heads
    (64, 4, 1, 513, True, (-1, -1)),     # d = 64, four query heads per unit
    (128, 2, 2, 600, True, (0, 0)),      # one-step units (diagonal only)
    (128, 2, 1, 900, False, (100, 50)),  # banded: units of two or three steps
])
def test_many_units_per_cta(fa, ctas, d, H, H_kv, N, causal, window):
    """Every CTA walks many units: the per-step barriers, the unit tiles and
    the rings carry their phases across unit boundaries, and the pipelines run
    ahead into the next unit."""
    fa.fa_set_max_ctas(ctas)
    try:
        got, ref = _case(fa, 1, H, H_kv, N, d, torch.bfloat16, causal, window,
                         seed=70 + ctas + d + H_kv)
    finally:
        fa.fa_set_max_ctas(0)
    _check(got, ref, f"ctas={ctas} d={d} H={H}/{H_kv} N={N} causal={causal} window={window}")


def test_deterministic(fa):
    """No atomics: repeated launches give identical bits."""
    q, k, v = (t.cuda() for t in make_random_qkv(2, 4, 1000, 128, torch.bfloat16, seed=60))
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(61)).to(torch.bfloat16)
    do = do.cuda()
    o, lse = fa.fwd(q, k, v, causal=True)
    first = fa.bwd(q, k, v, o, lse, do, causal=True)
    for _ in range(3):
        again = fa.bwd(q, k, v, o, lse, do, causal=True)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    torch.cuda.synchronize()
    st, _ = fa.fa_get_device_status(None)
    assert st == fa.FA_OK


@pytest.mark.parametrize("index", [2, 3])
def test_workload_size_heads(fa, index):
    """The backward on a whole workload (B*H heads launched together); the
    gradients of the first and the last head checked against the oracle run
    on those heads alone."""
    from workloads import make_qkv, workload
    wl = workload(index)
    q, k, v = make_qkv(wl)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(4000 + wl.index))
    do = do.to(q.dtype)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, scale=wl.scale, causal=wl.causal)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, scale=wl.scale, causal=wl.causal)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    for (b, h) in ((0, 0), (wl.B - 1, wl.H - 1)):
        sl = lambda t: t[b:b + 1, h:h + 1].contiguous()
        ref = oracle.attention_bwd(sl(q), sl(k), sl(v), sl(do), wl.scale, wl.causal)
        got = tuple(g[b:b + 1, h:h + 1] for g in (dq, dk, dv))
        _check(got, ref, f"{wl.name} head ({b},{h})")
