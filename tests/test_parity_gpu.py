"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (stated for bf16/fp16 inputs with fp32 accumulation): max |O - O_ref|
<= 2e-2 and max |LSE - LSE_ref| <= 1e-3, element by element.  Small shapes
are compared in full (several tiles plus ragged tails); the large workloads in
full (tiny and N=2048) or on seeded row samples.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, make_qkv, make_random_qkv, sample_rows, workload

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


def _run(fa, q, k, v, scale, causal, dev="cuda:0", stream=None):
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o, lse = fa.fwd(qd, kd, vd, scale=scale, causal=causal, stream=stream)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    return o, lse


def _check(o, lse, o_ref, lse_ref, what):
    o_np = o.float().cpu().numpy() if torch.is_tensor(o) else o
    l_np = lse.cpu().numpy() if torch.is_tensor(lse) else lse
    assert np.isfinite(o_np).all(), f"{what}: non-finite O"
    assert np.isfinite(l_np).all(), f"{what}: non-finite LSE"
    err_o = float(np.abs(o_np - o_ref).max()) if o_np.size else 0.0
    err_l = float(np.abs(l_np - lse_ref).max()) if l_np.size else 0.0
    assert err_l <= LSE_TOL, f"{what}: max|dLSE| = {err_l:.3e} (O err {err_o:.3e})"
    assert err_o <= O_TOL, f"{what}: max|dO| = {err_o:.3e} (LSE err {err_l:.3e})"
    return err_o, err_l


# ------------------------------------------------------------ small, full
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", [1, 5, 63, 64, 65, 127, 128, 129, 255, 256, 257, 384, 640])
def test_small_shapes_full_compare(fa, N, d, causal, dtype):
    q, k, v = make_random_qkv(1, 2, N, d, dtype, seed=100 + N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    _check(o, lse, o_ref, lse_ref, f"N={N} d={d} causal={causal} {dtype}")


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_peaky_scores_trigger_rescale(fa, causal, d):
    """Large scores make the running maximum jump across tiles (O rescales)."""
    q, k, v = make_random_qkv(2, 2, 700, d, torch.bfloat16, seed=31, qk_mult=4.0)
    # a growing ramp of key norms so later tiles keep raising the maximum
    ramp = torch.linspace(0.2, 3.0, 700).to(torch.bfloat16)[None, None, :, None]
    k = (k * ramp).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    _check(o, lse, o_ref, lse_ref, "peaky")


# ------------------------------------------------------ structured inputs
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_constant_values_give_constant_output(fa, causal, d):
    q, k, _ = make_random_qkv(1, 3, 300, d, torch.bfloat16, seed=41)
    v = torch.full_like(q, 0.625)
    o, _ = _run(fa, q, k, v, 0.088, causal)
    assert torch.all(o.float().cpu() == 0.625)


def test_one_hot_values_expose_probabilities(fa):
    """V = identity (N = d = 128): O_i is the probability row P_i."""
    q, k, _ = make_random_qkv(1, 1, 128, 128, torch.bfloat16, seed=42)
    v = torch.eye(128, dtype=torch.bfloat16)[None, None].contiguous()
    o, lse = _run(fa, q, k, v, 0.1, False)
    p_ref, lse_ref = oracle.attention(q, k, v, 0.1, False)
    _check(o, lse, p_ref, lse_ref, "one-hot")
    assert np.abs(o.float().cpu().numpy().sum(-1) - 1.0).max() < 2e-2


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_zero_queries_uniform_weights(fa, causal):
    _, k, v = make_random_qkv(1, 2, 333, 64, torch.float16, seed=43)
    q = torch.zeros_like(k)
    o, lse = _run(fa, q, k, v, 0.125, causal)
    n = np.arange(1, 334) if causal else np.full(333, 333)
    np.testing.assert_allclose(lse.cpu().numpy(), np.broadcast_to(np.log(n), (1, 2, 333)),
                               rtol=0, atol=LSE_TOL)
    o_ref, _ = oracle.attention(q, k, v, 0.125, causal)
    _check(o, lse, o_ref, np.log(np.broadcast_to(n, (1, 2, 333)).astype(float)), "Q=0")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_causal_first_row_is_first_value_row(fa, d):
    q, k, v = make_random_qkv(2, 2, 200, d, torch.bfloat16, seed=44)
    o, _ = _run(fa, q, k, v, 0.088, True)
    _assert_first_row_is_v0(o, v)


# ------------------------------------------- persistent scheduler, streams
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("ctas", [1, 2, 3, 5, 7])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_persistent_loop_many_units_per_cta(fa, ctas, causal, d):
    """Many units per CTA; causal launches reverse every other wave (with 7
    CTAs the 27 units of d <= 128 end in a partial odd wave, with 5 the 48
    units of d = 256 do)."""
    q, k, v = make_random_qkv(2, 3, 1000, d, torch.bfloat16, seed=50 + ctas)
    scale = 1.0 / math.sqrt(d)
    fa.fa_set_max_ctas(ctas)
    try:
        o, lse = _run(fa, q, k, v, scale, causal)
    finally:
        fa.fa_set_max_ctas(0)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    _check(o, lse, o_ref, lse_ref, f"ctas={ctas}")


@pytest.mark.parametrize("ctas,N", [(5, 1024), (5, 900), (5, 800), (7, 2000), (30, 4096)])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_last_wave_split_into_single_tiles(fa, ctas, N, causal):
    """Pair units of a partial last wave run as single-tile units."""
    q, k, v = make_random_qkv(1, 3, N, 128, torch.bfloat16, seed=70 + ctas + N)
    scale = 1.0 / math.sqrt(128)
    fa.fa_set_max_ctas(ctas)
    try:
        o, lse = _run(fa, q, k, v, scale, causal)
    finally:
        fa.fa_set_max_ctas(0)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    _check(o, lse, o_ref, lse_ref, f"ctas={ctas} N={N}")


def test_side_stream_and_no_lse(fa):
    q, k, v = make_random_qkv(1, 2, 260, 64, torch.bfloat16, seed=60)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.fwd(qd, kd, vd, scale=0.125, causal=True, return_lse=False)
    s.synchronize()
    assert lse is None
    o_ref, _ = oracle.attention(q, k, v, 0.125, True)
    assert float(np.abs(o.float().cpu().numpy() - o_ref).max()) <= O_TOL


def test_deterministic_and_guard_bands(fa):
    q, k, v = make_random_qkv(2, 2, 513, 128, torch.bfloat16, seed=61)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    G = 64
    numel = q.numel()
    pattern = torch.tensor([0x7FC1], dtype=torch.int16).view(torch.bfloat16)
    obuf = pattern.repeat(numel + 2 * G).cuda()
    lbuf = torch.full((2 * 2 * 513 + 2 * G,), -7.25, dtype=torch.float32, device="cuda")
    o = obuf[G:G + numel].view(q.shape)
    lse = lbuf[G:G + 2 * 2 * 513].view(2, 2, 513)
    outs = []
    for _ in range(2):
        fa.fwd(qd, kd, vd, scale=0.09, causal=False, out=o, lse=lse)
        torch.cuda.synchronize()
        outs.append((o.clone(), lse.clone()))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])
    guard = torch.cat([obuf[:G], obuf[G + numel:]]).view(torch.int16).cpu()
    assert torch.all(guard == 0x7FC1)
    lg = torch.cat([lbuf[:G], lbuf[G + 2 * 2 * 513:]]).cpu()
    assert torch.all(lg == -7.25)


# ------------------------------------------- grouped heads, local window
def _run_ext(fa, q, k, v, scale, causal, window):
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal, window=window)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    return o, lse


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 2), (4, 1)])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("window", [(-1, -1), (40, 40), (200, 0), (0, 0), (300, -1),
                                    (-1, 130)])
def test_grouped_heads_and_window(fa, d, H, H_kv, causal, window):
    q, _, _ = make_random_qkv(2, H, 700, d, torch.bfloat16, seed=90 + d + H_kv)
    _, k, v = make_random_qkv(2, H_kv, 700, d, torch.bfloat16, seed=91 + d + H_kv)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run_ext(fa, q, k, v, scale, causal, window)
    o_ref, lse_ref = oracle.attention_ex(q, k, v, scale, causal, *window)
    _check(o, lse, o_ref, lse_ref, f"d={d} H={H}/{H_kv} causal={causal} window={window}")


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("ctas", [1, 3])
@pytest.mark.parametrize("window", [(64, 64), (500, 0)])
def test_window_persistent_loop(fa, ctas, window, d):
    """Windowed units see different numbers of key tiles, so the K/V ring's
    slots and phases (and, at d = 256, the separate K and V producers and
    the S and P V issuers) run on across units of uneven length."""
    q, k, v = make_random_qkv(1, 3, 1500, d, torch.float16, seed=95 + ctas)
    fa.fa_set_max_ctas(ctas)
    try:
        o, lse = _run_ext(fa, q, k, v, 0.09, False, window)
    finally:
        fa.fa_set_max_ctas(0)
    o_ref, lse_ref = oracle.attention_ex(q, k, v, 0.09, False, *window)
    _check(o, lse, o_ref, lse_ref, f"d={d} ctas={ctas} window={window}")


# ------------------------------------------------------------- watchdog
def test_watchdog_times_out_cleanly(fa):
    st = fa.fa_selftest_watchdog(20_000, None)
    assert st == fa.FA_OK
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_ERR_DEVICE_TIMEOUT and site == 15
    st, _ = fa.fa_get_device_status(None)       # the word was cleared
    assert st == fa.FA_OK
    # the context is still usable
    q, k, v = make_random_qkv(1, 1, 130, 64, torch.bfloat16, seed=62)
    o, lse = _run(fa, q, k, v, 0.125, False)
    o_ref, lse_ref = oracle.attention(q, k, v, 0.125, False)
    _check(o, lse, o_ref, lse_ref, "after watchdog")


# ------------------------------------------------------- the workloads
def _varlen_workload_case(fa, wl):
    """Packed sequences: every row of the sample is checked against the oracle
    evaluated on its own sequence."""
    q, k, v = make_qkv(wl)
    cu = wl.cu_seqlens()
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o, lse = fa.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_t, max(wl.seqlens()),
                           scale=wl.scale, causal=wl.causal)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    rows = sample_rows(wl)
    o_s, l_s, o_r, l_r = [], [], [], []
    for b in sorted(set(r[0] for r in rows)):
        s0, s1 = cu[b], cu[b + 1]
        trip = [(0, h, i) for (bb, h, i) in rows if bb == b]
        to_bhnd = lambda t: t[s0:s1].permute(1, 0, 2).unsqueeze(0).contiguous()
        ref_o, ref_l = oracle.attention_rows(to_bhnd(q), to_bhnd(k), to_bhnd(v), wl.scale,
                                             wl.causal, trip)
        for t, (_, h, i) in enumerate(trip):
            o_s.append(o[s0 + i, h].float().cpu().numpy())
            l_s.append(lse[h, s0 + i].item())
            o_r.append(ref_o[t])
            l_r.append(ref_l[t])
    err = _check(np.array(o_s), np.array(l_s), np.array(o_r), np.array(l_r),
                 wl.name + " (sampled)")
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    return err


def _fp8_workload_case(fa, wl):
    """E4M3 inputs (descales 1): LSE to 1e-3 and O within the E4M3 bound on P
    (|dO| <= 2^-4 max|v| + 2^-8 max|O|, rms <= 2^-4/sqrt(3) rms(v)), in full."""
    q, k, v = make_qkv(wl)
    o, lse = fa.fwd_fp8(q.cuda(), k.cuda(), v.cuda(), scale=wl.scale, causal=wl.causal)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    o_ref, l_ref = oracle.attention_fp8(q, k, v, wl.scale, 1.0, 1.0, 1.0, wl.causal)
    o_np, l_np = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.abs(l_np - l_ref).max() <= LSE_TOL
    vv = v.float().numpy()
    diff = np.abs(o_np - o_ref)
    assert diff.max() <= 2.0 ** -4 * np.abs(vv).max() + 2.0 ** -8 * np.abs(o_ref).max()
    assert np.sqrt((diff ** 2).mean()) <= 2.0 ** -4 / math.sqrt(3) * np.sqrt((vv ** 2).mean())
    return float(diff.max()), float(np.abs(l_np - l_ref).max())


def _decode_workload_case(fa, wl):
    """The decode workload at full size through fa_fwd_varlen_qk (grouped
    heads packed into shared tiles), against the oracle on a seeded sample
    of 6 whole sequences (every head and query row) and the first and last
    sequence."""
    q, k, v = make_qkv(wl)
    nq, N, B = wl.n_q, wl.N, wl.B
    cu_q = torch.arange(0, B + 1, dtype=torch.int32, device="cuda") * nq
    cu_k = torch.arange(0, B + 1, dtype=torch.int32, device="cuda") * N
    o, lse = fa.fwd_varlen_qk(q.cuda(), k.cuda(), v.cuda(), cu_q, cu_k, nq, N,
                              scale=wl.scale, causal=wl.causal)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    g = torch.Generator().manual_seed(2000 + wl.index)
    seqs = sorted({0, B - 1} | set(torch.randint(0, B, (6,), generator=g).tolist()))
    worst = (0.0, 0.0)
    for b in seqs:
        o_ref, l_ref = oracle.attention_varlen_qk(q[b * nq:(b + 1) * nq], k[b * N:(b + 1) * N],
                                                  v[b * N:(b + 1) * N], [0, nq], [0, N],
                                                  wl.scale, wl.causal)
        err = _check(o[b * nq:(b + 1) * nq], lse[:, b * nq:(b + 1) * nq], o_ref, l_ref,
                     f"{wl.name} sequence {b}")
        worst = (max(worst[0], err[0]), max(worst[1], err[1]))
    return worst


def _workload_case(fa, wl, full):
    if wl.decode:
        return _decode_workload_case(fa, wl)
    if wl.varlen:
        return _varlen_workload_case(fa, wl)
    if wl.dtype == "fp8":
        return _fp8_workload_case(fa, wl)
    q, k, v = make_qkv(wl)
    if wl.splitkv:
        o, lse = fa.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), scale=wl.scale,
                                causal=wl.causal, num_splits=0)
        torch.cuda.synchronize()
        st, site = fa.fa_get_device_status(None)
        assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    else:
        o, lse = _run(fa, q, k, v, wl.scale, wl.causal)
    if full:
        o_ref, lse_ref = oracle.attention(q, k, v, wl.scale, wl.causal)
        return _check(o, lse, o_ref, lse_ref, wl.name)
    rows = sample_rows(wl)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, wl.scale, wl.causal, rows)
    idx = torch.tensor(rows, dtype=torch.long)
    o_s = o[idx[:, 0], idx[:, 1], idx[:, 2]].float().cpu().numpy()
    l_s = lse[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy()
    err = _check(o_s, l_s, o_ref, lse_ref, wl.name + " (sampled)")
    # properties that hold at any size, over every row
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    if wl.causal:
        _assert_first_row_is_v0(o, v)
    return err


def _assert_first_row_is_v0(o, v):
    """Causal row 0 attends to key 0 alone: O_0 = V_0 up to the output rounding."""
    got = o[:, :, 0, :].float().cpu()
    want = v[:, :, 0, :].float()
    diff = (got - want).abs()
    bad = (diff > 0).nonzero()
    assert bad.numel() == 0, (f"{bad.shape[0]} elements of O[:,:,0,:] differ from V[:,:,0,:]; "
                              f"max |diff| {diff.max().item():.3e}; first {bad[:4].tolist()}")


@pytest.mark.parametrize("index", [w.index for w in WORKLOADS])
def test_workload(fa, index):
    wl = workload(index)
    full = wl.B * wl.H * wl.N * wl.N * wl.d <= 4 * 16 * 2048 * 2048 * 128
    _workload_case(fa, wl, full)


@pytest.mark.parametrize("index", [2, 3])
def test_repeat_runs_bit_identical_full_size(fa, index):
    """Full-size launches repeated back to back give the same bits: the order
    of every MMA, every reduction and every rescale decision is fixed, so
    nothing varies from run to run."""
    wl = workload(index)
    q, k, v = (t.cuda() for t in make_qkv(wl))
    o0, l0 = fa.fwd(q, k, v, scale=wl.scale, causal=wl.causal)
    for _ in range(8):
        o, lse = fa.fwd(q, k, v, scale=wl.scale, causal=wl.causal)
        assert torch.equal(o, o0) and torch.equal(lse, l0)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
