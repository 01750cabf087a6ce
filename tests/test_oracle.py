"""Pins for the fp64 oracle: each check ties it to something other than itself.

Every test here runs on the CPU.  The checks are chosen so that a plausible
mistake in the oracle (a dropped scale, a wrong sign, swapped Q/K roles, the
causal mask pointing the wrong way, a missing max subtraction, the LSE in the
wrong base, a wrong 16-bit decoder) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import make_random_qkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _num(x):
    """Parse the fixture's closed forms: numbers, 'lnK' and 'a/b'."""
    if isinstance(x, (int, float)):
        return float(x)
    if x.startswith("ln"):
        return math.log(float(x[2:]))
    if "/" in x:
        a, b = x.split("/")
        return float(a) / float(b)
    return float(x)


def _as4d(rows):
    return np.asarray(rows, dtype=np.float64)[None, None]


# --------------------------------------------------------------------------
# Closed forms worked by hand (tests/golden/hand_worked.json).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("path", ["f64", "bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_golden_hand_worked(path, causal):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        scale = _num(case["scale"])
        q, k, v = (_as4d(case[n]) for n in ("q", "k", "v"))
        want = case["causal" if causal else "full"]
        want_o = np.array([[_num(x) for x in r] for r in want["o"]])
        want_lse = np.array([_num(x) for x in want["lse"]])
        if path == "f64":
            o, lse = oracle.attention_f64(q, k, v, scale, causal)
        else:
            dt = torch.bfloat16 if path == "bf16" else torch.float16
            tq, tk, tv = (torch.from_numpy(a).to(dt) for a in (q, k, v))
            o, lse = oracle.attention(tq, tk, tv, scale, causal)
        np.testing.assert_allclose(o[0, 0], want_o, rtol=0, atol=1e-12,
                                   err_msg=case["name"])
        np.testing.assert_allclose(lse[0, 0], want_lse, rtol=0, atol=1e-12,
                                   err_msg=case["name"])


# --------------------------------------------------------------------------
# The 16-bit decoders, exhaustively, against PyTorch's own conversions.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_decoder_exhaustive(dtype):
    words = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    ref = words.view(dtype).to(torch.float64).numpy()
    is_bf16 = dtype == torch.bfloat16
    got = np.array([oracle.widen(w, is_bf16) for w in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# --------------------------------------------------------------------------
# Library routines: PyTorch CPU float64 attention, logsumexp, softmax.
# --------------------------------------------------------------------------
def _torch_ref(q, k, v, scale, causal):
    qt, kt, vt = (torch.from_numpy(np.asarray(a, dtype=np.float64)) for a in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, is_causal=causal, scale=scale)
    s = scale * torch.matmul(qt, kt.transpose(-1, -2))
    if causal:
        n = s.shape[-1]
        mask = torch.ones(n, n, dtype=torch.bool).triu(1)
        s = s.masked_fill(mask, float("-inf"))
    return o.numpy(), torch.logsumexp(s, dim=-1).numpy()


@pytest.mark.parametrize("shape", [(1, 1, 1, 4), (1, 2, 7, 8), (2, 3, 33, 16),
                                   (1, 1, 130, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_f64(shape, causal):
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal(shape) for _ in range(3))
    scale = 0.37
    o, lse = oracle.attention_f64(q, k, v, scale, causal)
    o_ref, lse_ref = _torch_ref(q, k, v, scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_16bit(dtype, causal):
    q, k, v = make_random_qkv(2, 2, 45, 32, dtype, seed=11)
    scale = 1 / math.sqrt(32)
    o, lse = oracle.attention(q, k, v, scale, causal)
    o_ref, lse_ref = _torch_ref(q.double().numpy(), k.double().numpy(),
                                v.double().numpy(), scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_large_scores_no_overflow():
    """Scores near 1e3 overflow exp() unless the row maximum is subtracted."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 20, 8)) * 30
    k = rng.standard_normal((1, 1, 20, 8)) * 30
    v = rng.standard_normal((1, 1, 20, 8))
    o, lse = oracle.attention_f64(q, k, v, 1.0, False)
    o_ref, lse_ref = _torch_ref(q, k, v, 1.0, False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-14, atol=0)


# --------------------------------------------------------------------------
# Invariants of the definition.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_probabilities_sum_to_one(causal):
    """V = identity makes O_i the probability row P_i itself."""
    n = 24
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 1, n, n))
    k = rng.standard_normal((1, 1, n, n))
    v = np.eye(n)[None, None]
    scale = 0.5
    p, lse = oracle.attention_f64(q, k, v, scale, causal)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert (p >= 0).all()
    s = scale * torch.from_numpy(q[0, 0]) @ torch.from_numpy(k[0, 0]).T
    if causal:
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(p[0, 0], torch.softmax(s, -1).numpy(), rtol=0,
                               atol=1e-12)
    if causal:
        assert np.all(np.triu(p[0, 0], 1) == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values(causal):
    q, k, _ = make_random_qkv(1, 2, 40, 16, torch.bfloat16, seed=21)
    v = torch.full_like(q, 1.75)
    o, _ = oracle.attention(q, k, v, 0.25, causal)
    np.testing.assert_allclose(o, 1.75, rtol=0, atol=1e-12)


def test_causal_row_zero():
    q, k, v = make_random_qkv(2, 2, 19, 16, torch.float16, seed=22)
    scale = 0.3
    o, lse = oracle.attention(q, k, v, scale, True)
    np.testing.assert_array_equal(o[:, :, 0, :], v[:, :, 0, :].double().numpy())
    want = scale * (q[:, :, 0, :].double() * k[:, :, 0, :].double()).sum(-1)
    np.testing.assert_allclose(lse[:, :, 0], want.numpy(), rtol=0, atol=1e-13)


def test_causal_row_independent_of_later_keys():
    q, k, v = make_random_qkv(1, 1, 32, 16, torch.bfloat16, seed=23)
    o1, l1 = oracle.attention(q, k, v, 0.25, True)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 20:] = -k2[:, :, 20:] * 3
    v2[:, :, 20:] = 5.0
    o2, l2 = oracle.attention(q, k2, v2, 0.25, True)
    np.testing.assert_array_equal(o1[:, :, :20], o2[:, :, :20])
    np.testing.assert_array_equal(l1[:, :, :20], l2[:, :, :20])
    assert not np.allclose(o1[:, :, 20:], o2[:, :, 20:])


def test_key_value_permutation_invariance():
    q, k, v = make_random_qkv(1, 2, 50, 32, torch.bfloat16, seed=24)
    perm = torch.randperm(50, generator=torch.Generator().manual_seed(1))
    o1, l1 = oracle.attention(q, k, v, 0.2, False)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.2, False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_score_shift():
    """Adding u to every key adds scale*q_i.u to row i: O fixed, LSE shifted."""
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 1, 30, 8))
    k = rng.standard_normal((1, 1, 30, 8))
    v = rng.standard_normal((1, 1, 30, 8))
    u = rng.standard_normal(8)
    scale = 0.7
    for causal in (False, True):
        o1, l1 = oracle.attention_f64(q, k, v, scale, causal)
        o2, l2 = oracle.attention_f64(q, k + u, v, scale, causal)
        np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
        np.testing.assert_allclose((l2 - l1)[0, 0], scale * q[0, 0] @ u, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_closed_form(causal):
    """Q = 0: uniform weights, O_i = mean of admissible v_j, LSE_i = ln |J(i)|."""
    n, d = 37, 8
    rng = np.random.default_rng(4)
    q = np.zeros((1, 1, n, d))
    k = rng.standard_normal((1, 1, n, d))
    v = rng.standard_normal((1, 1, n, d))
    o, lse = oracle.attention_f64(q, k, v, 1.3, causal)
    for i in range(n):
        cnt = i + 1 if causal else n
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :cnt].mean(0), rtol=0, atol=1e-13)
        assert abs(lse[0, 0, i] - math.log(cnt)) < 1e-13


def test_single_key_closed_form():
    """N = 1: O = V and LSE = scale * q.k, whatever the mask."""
    q, k, v = make_random_qkv(3, 2, 1, 64, torch.float16, seed=25)
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, 0.125, causal)
        np.testing.assert_array_equal(o, v.double().numpy())
        want = 0.125 * (q.double() * k.double()).sum(-1)
        np.testing.assert_allclose(lse, want.numpy(), rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# Brute force by a different route: blockwise online softmax (test-only).
# --------------------------------------------------------------------------
def _online_softmax_attention(q, k, v, scale, causal, block=7):
    """Separately written tiled evaluation with a running max and sum."""
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                run_max, run_sum = -np.inf, 0.0
                acc = np.zeros(d)
                last = i if causal else N - 1
                for j0 in range(0, last + 1, block):
                    j1 = min(j0 + block, last + 1)
                    sc = scale * (k[b, h, j0:j1] @ q[b, h, i])
                    new_max = max(run_max, sc.max())
                    corr = math.exp(run_max - new_max) if run_max > -np.inf else 0.0
                    w = np.exp(sc - new_max)
                    acc = acc * corr + w @ v[b, h, j0:j1]
                    run_sum = run_sum * corr + w.sum()
                    run_max = new_max
                o[b, h, i] = acc / run_sum
                lse[b, h, i] = run_max + math.log(run_sum)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_matches_online_softmax(causal):
    q, k, v = make_random_qkv(1, 2, 29, 16, torch.bfloat16, seed=26, qk_mult=2.0)
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    o, lse = oracle.attention(q, k, v, 0.25, causal)
    o2, l2 = _online_softmax_attention(qd, kd, vd, 0.25, causal)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, l2, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# The row-sampling entry agrees with the full evaluation.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_rows_match_full(causal):
    q, k, v = make_random_qkv(2, 3, 70, 32, torch.bfloat16, seed=27)
    o, lse = oracle.attention(q, k, v, 0.17, causal)
    rows = [(0, 0, 0), (1, 2, 69), (0, 1, 33), (1, 0, 5), (0, 0, 64)]
    o_r, l_r = oracle.attention_rows(q, k, v, 0.17, causal, rows)
    for t, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(o_r[t], o[b, h, i])
        assert l_r[t] == lse[b, h, i]


def test_bad_arguments_rejected():
    q, k, v = make_random_qkv(1, 1, 8, 16, torch.bfloat16, seed=28)
    with pytest.raises(RuntimeError):
        oracle.attention_rows(q, k, v, 0.1, False, [(0, 0, 8)])
    with pytest.raises(TypeError):
        oracle.attention(q.float(), k, v, 0.1, False)


# --------------------------------------------------------------------------
# Grouped K/V heads and the local window.
# --------------------------------------------------------------------------
def _window_mask(n, causal, wl, wr):
    i = torch.arange(n)[:, None]
    j = torch.arange(n)[None, :]
    ok = torch.ones(n, n, dtype=torch.bool)
    if causal:
        ok &= j <= i
    if wl >= 0:
        ok &= j >= i - wl
    if wr >= 0:
        ok &= j <= i + wr
    return ok


@pytest.mark.parametrize("causal", [False, True])
def test_window_matches_sdpa_mask(causal):
    """Library routine with an explicit boolean mask."""
    q, k, v = make_random_qkv(1, 2, 70, 16, torch.bfloat16, seed=81)
    for wl, wr in ((5, 3), (0, 9), (17, -1), (-1, 4), (0, 0), (100, 100)):
        o, lse = oracle.attention_ex(q, k, v, 0.3, causal, wl, wr)
        mask = _window_mask(70, causal, wl, wr)
        qd, kd, vd = (t.double() for t in (q, k, v))
        o_ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask,
                                                                 scale=0.3)
        s = (0.3 * qd @ kd.transpose(-1, -2)).masked_fill(~mask, float("-inf"))
        np.testing.assert_allclose(o, o_ref.numpy(), rtol=0, atol=1e-12, err_msg=str((wl, wr)))
        np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def test_window_closed_forms():
    q, k, v = make_random_qkv(1, 2, 40, 16, torch.float16, seed=82)
    # a window of zero width leaves each row with its own key only
    o, lse = oracle.attention_ex(q, k, v, 0.25, False, 0, 0)
    np.testing.assert_array_equal(o, v.double().numpy())
    np.testing.assert_allclose(lse, (0.25 * (q.double() * k.double()).sum(-1)).numpy(),
                               rtol=0, atol=1e-13)
    # windows wider than the sequence are full attention; right bound 0 is causal
    o_full, l_full = oracle.attention(q, k, v, 0.25, False)
    o_w, l_w = oracle.attention_ex(q, k, v, 0.25, False, 40, 40)
    np.testing.assert_array_equal(o_w, o_full)
    np.testing.assert_array_equal(l_w, l_full)
    o_c, l_c = oracle.attention(q, k, v, 0.25, True)
    o_r, l_r = oracle.attention_ex(q, k, v, 0.25, False, -1, 0)
    np.testing.assert_array_equal(o_r, o_c)
    np.testing.assert_array_equal(l_r, l_c)
    # Q = 0: uniform weights over the window
    z = torch.zeros_like(q)
    o_z, l_z = oracle.attention_ex(z, k, v, 0.25, False, 3, 2)
    vd = v.double().numpy()
    for i in range(40):
        lo, hi = max(0, i - 3), min(40, i + 3)
        np.testing.assert_allclose(o_z[:, :, i], vd[:, :, lo:hi].mean(2), rtol=0, atol=1e-13)
        np.testing.assert_allclose(l_z[:, :, i], math.log(hi - lo), rtol=0, atol=1e-13)


def test_grouped_heads_equal_repeated_heads():
    """H_kv < H equals repeating each K/V head H / H_kv times."""
    q, _, _ = make_random_qkv(2, 6, 33, 16, torch.bfloat16, seed=83)
    _, k, v = make_random_qkv(2, 2, 33, 16, torch.bfloat16, seed=84)
    for causal in (False, True):
        o, lse = oracle.attention_ex(q, k, v, 0.2, causal)
        kr = k.repeat_interleave(3, dim=1)
        vr = v.repeat_interleave(3, dim=1)
        o_ref, l_ref = oracle.attention(q, kr, vr, 0.2, causal)
        np.testing.assert_array_equal(o, o_ref)
        np.testing.assert_array_equal(lse, l_ref)
        rows = [(0, 0, 0), (1, 5, 32), (1, 2, 10), (0, 4, 7)]
        o_r, l_r = oracle.attention_rows_ex(q, k, v, 0.2, causal, rows)
        for t, (b, h, i) in enumerate(rows):
            np.testing.assert_array_equal(o_r[t], o[b, h, i])
            assert l_r[t] == lse[b, h, i]


# ------------------------------------------------- variable-length batches
def _pack(t):
    """[B, H, N, d] -> [B*N, H, d] (sequences of equal length, packed)."""
    B, H, N, d = t.shape
    return t.permute(0, 2, 1, 3).reshape(B * N, H, d).contiguous()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [(-1, -1), (5, 3), (0, -1)])
def test_varlen_equal_lengths_is_the_batched_definition(causal, window):
    """Equal-length sequences packed along the rows give the [B,H,N,d] result."""
    q, _, _ = make_random_qkv(3, 4, 29, 16, torch.bfloat16, seed=400)
    _, k, v = make_random_qkv(3, 2, 29, 16, torch.bfloat16, seed=401)
    o, lse = oracle.attention_ex(q, k, v, 0.3, causal, *window)
    cu = [0, 29, 58, 87]
    o_v, l_v = oracle.attention_varlen(_pack(q), _pack(k), _pack(v), cu, 0.3, causal, *window)
    np.testing.assert_array_equal(o_v, o.transpose(0, 2, 1, 3).reshape(87, 4, 16))
    np.testing.assert_array_equal(l_v, lse.transpose(1, 0, 2).reshape(4, 87))


def _sdpa_rows(qs, ks, vs, scale, causal, window):
    """torch float64 attention of one sequence ([n, H, d] slices) with an
    explicit boolean mask built from the window's definition."""
    n, H, _ = qs.shape
    group = H // ks.shape[1]
    i = torch.arange(n)[:, None]
    j = torch.arange(n)[None, :]
    allowed = torch.ones(n, n, dtype=torch.bool)
    if causal:
        allowed &= j <= i
    if window[0] >= 0:
        allowed &= j >= i - window[0]
    if window[1] >= 0:
        allowed &= j <= i + window[1]
    qd = qs.double().permute(1, 0, 2)
    kd = ks.double().repeat_interleave(group, 1).permute(1, 0, 2)
    vd = vs.double().repeat_interleave(group, 1).permute(1, 0, 2)
    o = torch.nn.functional.scaled_dot_product_attention(
        qd[None], kd[None], vd[None], attn_mask=allowed, scale=scale)[0]
    s = scale * qd @ kd.transpose(-1, -2)
    lse = torch.logsumexp(s.masked_fill(~allowed, float("-inf")), -1)
    return o.permute(1, 0, 2).numpy(), lse.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [(-1, -1), (4, 2)])
def test_varlen_matches_torch_per_sequence(causal, window):
    """Ragged lengths (with an empty and a one-row sequence) against torch's
    float64 attention of each sequence on its own; rows after the last
    sequence stay unwritten."""
    lens = [5, 0, 17, 1, 33]
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    total = cu[-1] + 3
    q = torch.randn(total, 6, 16, generator=torch.Generator().manual_seed(410)).to(torch.bfloat16)
    k = torch.randn(total, 3, 16, generator=torch.Generator().manual_seed(411)).to(torch.bfloat16)
    v = torch.randn(total, 3, 16, generator=torch.Generator().manual_seed(412)).to(torch.bfloat16)
    o, lse = oracle.attention_varlen(q, k, v, cu, 0.27, causal, *window)
    for b, n in enumerate(lens):
        if n == 0:
            continue
        s0 = cu[b]
        o_ref, l_ref = _sdpa_rows(q[s0:s0 + n], k[s0:s0 + n], v[s0:s0 + n], 0.27, causal,
                                  window)
        np.testing.assert_allclose(o[s0:s0 + n], o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, s0:s0 + n], l_ref, rtol=0, atol=1e-12)
    assert np.isnan(o[cu[-1]:]).all() and np.isnan(lse[:, cu[-1]:]).all()


def test_varlen_sequences_are_isolated():
    """Changing one sequence's tokens leaves every other sequence's rows bit
    for bit unchanged."""
    lens = [9, 14, 6]
    cu = [0, 9, 23, 29]
    q, k, v = (torch.randn(29, 2, 16, generator=torch.Generator().manual_seed(420 + t))
               .to(torch.float16) for t in range(3))
    o, lse = oracle.attention_varlen(q, k, v, cu, 0.25, False)
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    for t in (q2, k2, v2):
        t[9:23] = -t[9:23] * 2
    o2, l2 = oracle.attention_varlen(q2, k2, v2, cu, 0.25, False)
    keep = np.r_[0:9, 23:29]
    np.testing.assert_array_equal(o2[keep], o[keep])
    np.testing.assert_array_equal(l2[:, keep], lse[:, keep])
    assert not np.array_equal(o2[9:23], o[9:23])
    assert sum(lens) == 29


def test_varlen_zero_queries_closed_form():
    """Q = 0: every admissible key of the row's own sequence weighs the same."""
    cu = [0, 7, 20]
    k = torch.randn(20, 1, 16, generator=torch.Generator().manual_seed(430)).to(torch.bfloat16)
    v = torch.randn(20, 1, 16, generator=torch.Generator().manual_seed(431)).to(torch.bfloat16)
    q = torch.zeros(20, 2, 16, dtype=torch.bfloat16)
    o, lse = oracle.attention_varlen(q, k, v, cu, 0.5, True, 3, -1)
    vd = v.double().numpy()[:, 0]
    for b in range(2):
        s0, n = cu[b], cu[b + 1] - cu[b]
        for i in range(n):
            lo = max(0, i - 3)
            for h in range(2):
                np.testing.assert_allclose(o[s0 + i, h], vd[s0 + lo:s0 + i + 1].mean(0),
                                           rtol=0, atol=1e-13)
                np.testing.assert_allclose(lse[h, s0 + i], math.log(i + 1 - lo), rtol=0,
                                           atol=1e-13)


def test_varlen_rejects_malformed_offsets():
    q = torch.zeros(10, 1, 16, dtype=torch.bfloat16)
    for cu in ([0, 6, 4], [0, 11], [-1, 5]):
        with pytest.raises(RuntimeError):
            oracle.attention_varlen(q, q, q, cu, 0.5, False)


# ------------------- separate query / key sequences, used lengths (KV cache)
def _sdpa_qk(qs, ks, vs, scale, causal, window):
    """torch float64 attention of one sequence with n_q queries ([n_q, H, d])
    and n_k keys ([n_k, H_kv, d]); the mask is built from its bottom-right
    definition (query i at key position i + n_k - n_q).  Rows with no
    admissible key are returned as O = 0, LSE = -inf."""
    nq, H, _ = qs.shape
    nk = ks.shape[0]
    group = H // ks.shape[1]
    pos = torch.arange(nq)[:, None] + (nk - nq)
    j = torch.arange(nk)[None, :]
    allowed = torch.ones(nq, nk, dtype=torch.bool)
    if causal:
        allowed &= j <= pos
    if window[0] >= 0:
        allowed &= j >= pos - window[0]
    if window[1] >= 0:
        allowed &= j <= pos + window[1]
    qd = qs.double().permute(1, 0, 2)
    kd = ks.double().repeat_interleave(group, 1).permute(1, 0, 2)
    vd = vs.double().repeat_interleave(group, 1).permute(1, 0, 2)
    s = scale * qd @ kd.transpose(-1, -2)
    lse = torch.logsumexp(s.masked_fill(~allowed, float("-inf")), -1)
    p = torch.softmax(s.masked_fill(~allowed, float("-inf")), -1)
    p = torch.nan_to_num(p, nan=0.0)   # rows without keys: all weights 0
    o = p @ vd
    return o.permute(1, 0, 2).numpy(), lse.numpy(), allowed.any(1).numpy()


QK_CASES = [
    # (n_q per sequence, n_k per sequence): cross-attention, decode, prefill
    # continuation, fewer keys than queries, an empty query sequence
    ([5, 1, 17, 0, 9], [12, 40, 17, 6, 3]),
    ([1, 1, 1], [64, 1, 33]),
    ([33, 8], [20, 8]),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [(-1, -1), (4, 2), (0, -1)])
@pytest.mark.parametrize("case", range(len(QK_CASES)))
def test_varlen_qk_matches_torch_per_sequence(causal, window, case):
    """Separate query and key offsets against torch's float64 attention of
    each sequence with the bottom-right mask; rows past the last sequence
    stay unwritten."""
    lq, lk = QK_CASES[case]
    cu_q = np.concatenate([[0], np.cumsum(lq)]).tolist()
    cu_k = np.concatenate([[0], np.cumsum(lk)]).tolist()
    total_q, total_k = cu_q[-1] + 2, cu_k[-1] + 5
    g = torch.Generator().manual_seed(440 + case)
    q = torch.randn(total_q, 4, 16, generator=g).to(torch.bfloat16)
    k = torch.randn(total_k, 2, 16, generator=g).to(torch.bfloat16)
    v = torch.randn(total_k, 2, 16, generator=g).to(torch.bfloat16)
    o, lse = oracle.attention_varlen_qk(q, k, v, cu_q, cu_k, 0.31, causal, *window)
    for b in range(len(lq)):
        if lq[b] == 0:
            continue
        q0, k0 = cu_q[b], cu_k[b]
        o_ref, l_ref, _ = _sdpa_qk(q[q0:q0 + lq[b]], k[k0:k0 + lk[b]], v[k0:k0 + lk[b]], 0.31,
                                   causal, window)
        np.testing.assert_allclose(o[q0:q0 + lq[b]], o_ref, rtol=0, atol=1e-12)
        np.testing.assert_array_equal(np.isinf(lse[:, q0:q0 + lq[b]]), np.isinf(l_ref))
        fin = np.isfinite(l_ref)
        np.testing.assert_allclose(lse[:, q0:q0 + lq[b]][fin], l_ref[fin], rtol=0, atol=1e-12)
    assert np.isnan(o[cu_q[-1]:]).all() and np.isnan(lse[:, cu_q[-1]:]).all()


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_qk_used_lengths_are_a_prefix(causal):
    """seqused_q / seqused_k: only the first used rows of each sequence's
    buffer rows take part (a KV cache with spare capacity); the result equals
    the same call on buffers packed with the used rows alone, and query rows
    past the used count stay unwritten."""
    cap_q, cap_k = [6, 4, 9], [30, 16, 25]
    used_q, used_k = [3, 4, 1], [21, 9, 25]
    cu_q = np.concatenate([[0], np.cumsum(cap_q)]).tolist()
    cu_k = np.concatenate([[0], np.cumsum(cap_k)]).tolist()
    g = torch.Generator().manual_seed(450)
    q = torch.randn(cu_q[-1], 2, 16, generator=g).to(torch.float16)
    k = torch.randn(cu_k[-1], 1, 16, generator=g).to(torch.float16)
    v = torch.randn(cu_k[-1], 1, 16, generator=g).to(torch.float16)
    o, lse = oracle.attention_varlen_qk(q, k, v, cu_q, cu_k, 0.4, causal, seqused_q=used_q,
                                        seqused_k=used_k)
    take_q = np.concatenate([np.arange(cu_q[b], cu_q[b] + used_q[b]) for b in range(3)])
    take_k = np.concatenate([np.arange(cu_k[b], cu_k[b] + used_k[b]) for b in range(3)])
    pq = np.concatenate([[0], np.cumsum(used_q)]).tolist()
    pk = np.concatenate([[0], np.cumsum(used_k)]).tolist()
    o2, l2 = oracle.attention_varlen_qk(q[take_q], k[take_k], v[take_k], pq, pk, 0.4, causal)
    np.testing.assert_array_equal(o[take_q], o2)
    np.testing.assert_array_equal(lse[:, take_q], l2)
    rest = np.setdiff1d(np.arange(cu_q[-1]), take_q)
    assert np.isnan(o[rest]).all() and np.isnan(lse[:, rest]).all()
    # and the torch reference on the used rows of sequence 0
    o_ref, l_ref, _ = _sdpa_qk(q[0:3], k[0:21], v[0:21], 0.4, causal, (-1, -1))
    np.testing.assert_allclose(o[0:3], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[:, 0:3], l_ref, rtol=0, atol=1e-12)


def test_varlen_qk_decode_and_zero_query_closed_forms():
    """One query per sequence (decode) under the causal mask sees every key
    of its sequence: with Q = 0 its O is the mean of the sequence's V rows
    and LSE = ln n_k; a window of w keeps the last w + 1 keys; with fewer
    keys than queries the first n_q - n_k causal rows have no key (O = 0,
    LSE = -inf) and row n_q - n_k + t sees keys 0..t."""
    lk = [7, 30, 1]
    cu_k = np.concatenate([[0], np.cumsum(lk)]).tolist()
    g = torch.Generator().manual_seed(460)
    k = torch.randn(cu_k[-1], 1, 16, generator=g).to(torch.bfloat16)
    v = torch.randn(cu_k[-1], 1, 16, generator=g).to(torch.bfloat16)
    q = torch.zeros(3, 3, 16, dtype=torch.bfloat16)
    vd = v.double().numpy()[:, 0]
    for window in ((-1, -1), (5, -1)):
        o, lse = oracle.attention_varlen_qk(q, k, v, [0, 1, 2, 3], cu_k, 0.7, True, *window)
        for b in range(3):
            n = lk[b]
            lo = 0 if window[0] < 0 else max(0, n - 1 - window[0])
            for h in range(3):
                np.testing.assert_allclose(o[b, h], vd[cu_k[b] + lo:cu_k[b] + n].mean(0),
                                           rtol=0, atol=1e-13)
                np.testing.assert_allclose(lse[h, b], math.log(n - lo), rtol=0, atol=1e-13)
    # more queries than keys, causal
    qz = torch.zeros(10, 1, 16, dtype=torch.bfloat16)
    o, lse = oracle.attention_varlen_qk(qz, k, v, [0, 10], [0, 7], 0.7, True)
    assert (o[:3] == 0).all() and np.isneginf(lse[0, :3]).all()
    for t in range(7):
        np.testing.assert_allclose(o[3 + t, 0], vd[0:t + 1].mean(0), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 3 + t], math.log(t + 1), rtol=0, atol=1e-13)


def test_varlen_qk_equal_offsets_is_the_self_attention_mode():
    """cu_seqlens_k = cu_seqlens_q and no used lengths: the self-attention
    packed mode, checked against the [B,H,N,d] definition."""
    q, _, _ = make_random_qkv(2, 2, 23, 16, torch.bfloat16, seed=470)
    _, k, v = make_random_qkv(2, 1, 23, 16, torch.bfloat16, seed=471)
    o, lse = oracle.attention_ex(q, k, v, 0.3, True, 6, -1)
    o_v, l_v = oracle.attention_varlen_qk(_pack(q), _pack(k), _pack(v), [0, 23, 46], [0, 23, 46],
                                          0.3, True, 6, -1)
    np.testing.assert_array_equal(o_v, o.transpose(0, 2, 1, 3).reshape(46, 2, 16))
    np.testing.assert_array_equal(l_v, lse.transpose(1, 0, 2).reshape(2, 46))


def test_varlen_qk_rejects_malformed_lengths():
    q = torch.zeros(10, 1, 16, dtype=torch.bfloat16)
    k = torch.zeros(12, 1, 16, dtype=torch.bfloat16)
    bad = [dict(cu_seqlens_q=[0, 6, 4], cu_seqlens_k=[0, 6, 12]),
           dict(cu_seqlens_q=[0, 5, 10], cu_seqlens_k=[0, 6, 13]),
           dict(cu_seqlens_q=[0, 5, 10], cu_seqlens_k=[0, 6, 12], seqused_k=[7, 1]),
           dict(cu_seqlens_q=[0, 5, 10], cu_seqlens_k=[0, 6, 12], seqused_q=[1, -1])]
    for kw in bad:
        with pytest.raises(RuntimeError):
            oracle.attention_varlen_qk(q, k, k, scale=0.5, causal=False, **kw)


# --------------------------------------------------------------- backward
def _torch_attention_f64(q, k, v, scale, causal, window):
    """Reference forward in torch float64 with an explicit mask (autograd)."""
    N = q.shape[-2]
    group = q.shape[1] // k.shape[1]
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    allowed = torch.ones(N, N, dtype=torch.bool)
    if causal:
        allowed &= j <= i
    if window[0] >= 0:
        allowed &= j >= i - window[0]
    if window[1] >= 0:
        allowed &= j <= i + window[1]
    kr = k.repeat_interleave(group, 1)
    vr = v.repeat_interleave(group, 1)
    s = scale * q @ kr.transpose(-1, -2)
    p = torch.softmax(s.masked_fill(~allowed, float("-inf")), -1)
    return p @ vr


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [(-1, -1), (6, 3)])
@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 2)])
def test_bwd_matches_torch_autograd(causal, window, H, H_kv):
    """dQ, dK, dV equal torch float64 autograd through softmax attention."""
    q, _, _ = make_random_qkv(2, H, 37, 16, torch.bfloat16, seed=700 + H_kv)
    _, k, v = make_random_qkv(2, H_kv, 37, 16, torch.bfloat16, seed=701 + H_kv)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(702)).to(torch.bfloat16)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.3, causal, *window)
    qd, kd, vd = (t.double().requires_grad_() for t in (q, k, v))
    o = _torch_attention_f64(qd, kd, vd, 0.3, causal, window)
    o.backward(do.double())
    np.testing.assert_allclose(dq, qd.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, kd.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, vd.grad.numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_directional_finite_difference(causal):
    """<dQ,Eq> + <dK,Ek> + <dV,Ev> equals the central difference of
    L = sum(O * dO) along (Eq, Ek, Ev), with O from the double forward."""
    q, k, v = make_random_qkv(1, 2, 23, 8, torch.bfloat16, seed=710)
    g = torch.Generator().manual_seed(711)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    eq, ek, ev = (torch.randn(q.shape, generator=g, dtype=torch.float64) for _ in range(3))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.35, causal)
    qd, kd, vd, dod = (t.double().numpy() for t in (q, k, v, do))
    eps = 1e-4

    def loss(sign):
        o, _ = oracle.attention_f64(qd + sign * eps * eq.numpy(), kd + sign * eps * ek.numpy(),
                                    vd + sign * eps * ev.numpy(), 0.35, causal)
        return float((o * dod).sum())

    fd = (loss(+1) - loss(-1)) / (2 * eps)
    an = float((dq * eq.numpy()).sum() + (dk * ek.numpy()).sum() + (dv * ev.numpy()).sum())
    assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (fd, an)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [(-1, -1), (5, 2)])
def test_bwd_sum_identities(causal, window):
    """Every row of P sums to one and every row of dS to zero, so
    sum_j dV_j = sum_i dO_i (over the heads sharing a K/V head) and
    sum_j dK_j = 0."""
    q, _, _ = make_random_qkv(1, 4, 41, 16, torch.float16, seed=720)
    _, k, v = make_random_qkv(1, 2, 41, 16, torch.float16, seed=721)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(722)).to(torch.float16)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.25, causal, *window)
    dod = do.double().numpy().reshape(1, 2, 2, 41, 16)
    np.testing.assert_allclose(dv.sum(2), dod.sum((2, 3)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk.sum(2), 0.0, rtol=0, atol=1e-12)
    assert np.abs(dq).max() > 1e-3


def _torch_attention_qk_f64(q, k, v, scale, causal, window):
    """Reference forward in torch float64 for Nq query and Nk key rows, masks
    aligned bottom-right (query i at key position i + Nk - Nq); a row without
    keys outputs 0 (its softmax runs unmasked and is multiplied by 0, so
    autograd sees no NaN)."""
    Nq, Nk = q.shape[-2], k.shape[-2]
    group = q.shape[1] // k.shape[1]
    pos = torch.arange(Nq)[:, None] + (Nk - Nq)
    j = torch.arange(Nk)[None, :]
    allowed = torch.ones(Nq, Nk, dtype=torch.bool)
    if causal:
        allowed &= j <= pos
    if window[0] >= 0:
        allowed &= j >= pos - window[0]
    if window[1] >= 0:
        allowed &= j <= pos + window[1]
    has_key = allowed.any(-1, keepdim=True)
    allowed = allowed | ~has_key
    kr = k.repeat_interleave(group, 1)
    vr = v.repeat_interleave(group, 1)
    s = scale * q @ kr.transpose(-1, -2)
    p = torch.softmax(s.masked_fill(~allowed, float("-inf")), -1) * has_key
    return p @ vr


@pytest.mark.parametrize("Nq,Nk", [(9, 23), (23, 9), (1, 30), (17, 17)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [(-1, -1), (4, 2)])
def test_bwd_qk_matches_torch_autograd(Nq, Nk, causal, window):
    """Separate query and key lengths: dQ, dK, dV equal torch float64
    autograd through the bottom-right masked softmax attention."""
    q, _, _ = make_random_qkv(1, 4, Nq, 16, torch.bfloat16, seed=730 + Nq)
    _, k, v = make_random_qkv(1, 2, Nk, 16, torch.bfloat16, seed=731 + Nk)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(732)).to(torch.bfloat16)
    dq, dk, dv = oracle.attention_bwd_qk(q, k, v, do, 0.3, causal, *window)
    qd, kd, vd = (t.double().requires_grad_() for t in (q, k, v))
    o = _torch_attention_qk_f64(qd, kd, vd, 0.3, causal, window)
    o.backward(do.double())
    np.testing.assert_allclose(dq, qd.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, kd.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, vd.grad.numpy(), rtol=0, atol=1e-11)


def test_bwd_qk_keyless_rows_drop_out():
    """Causal with more queries than keys: the first Nq - Nk rows see no key,
    so their dQ is exactly 0 and dK, dV are those of the last Nk rows alone
    (which then align on the plain diagonal)."""
    Nq, Nk = 29, 12
    q, _, _ = make_random_qkv(1, 2, Nq, 16, torch.float16, seed=740)
    _, k, v = make_random_qkv(1, 2, Nk, 16, torch.float16, seed=741)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(742)).to(torch.float16)
    dq, dk, dv = oracle.attention_bwd_qk(q, k, v, do, 0.4, True)
    assert (dq[:, :, :Nq - Nk] == 0).all()
    tail = lambda t: t[:, :, Nq - Nk:].contiguous()
    dq2, dk2, dv2 = oracle.attention_bwd(tail(q), k, v, tail(do), 0.4, True)
    np.testing.assert_allclose(dq[:, :, Nq - Nk:], dq2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, dk2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dv2, rtol=0, atol=1e-13)


def test_bwd_qk_equal_lengths_is_the_backward():
    q, k, v = make_random_qkv(2, 2, 19, 8, torch.bfloat16, seed=750)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(751)).to(torch.bfloat16)
    for causal, window in ((False, (-1, -1)), (True, (-1, -1)), (False, (3, 5))):
        a = oracle.attention_bwd_qk(q, k, v, do, 0.5, causal, *window)
        b = oracle.attention_bwd(q, k, v, do, 0.5, causal, *window)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


# ------------------------------------------------------------ FP8 inputs
def test_e4m3_decoder_exhaustive():
    """All 256 E4M3 codes decode as PyTorch's float8_e4m3fn does (NaN codes
    included)."""
    codes = torch.arange(256, dtype=torch.uint8)
    want = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3(c) for c in range(256)])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])
    assert oracle.e4m3(0x7E) == 448.0 and oracle.e4m3(0x01) == 2.0 ** -9


def _fp8_inputs(B, H, H_kv, N, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, N, d, generator=g).to(torch.float8_e4m3fn)
    k = torch.randn(B, H_kv, N, d, generator=g).to(torch.float8_e4m3fn)
    v = torch.randn(B, H_kv, N, d, generator=g).to(torch.float8_e4m3fn)
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_matches_torch_on_decoded_inputs(causal):
    """The FP8 definition equals torch float64 attention of the decoded,
    descaled inputs (library routine on PyTorch's own FP8 decoding)."""
    q, k, v = _fp8_inputs(2, 4, 2, 33, 16, seed=900)
    o, lse = oracle.attention_fp8(q, k, v, 0.2, 0.5, 2.0, 0.25, causal, 5, -1)
    qd, kd, vd = q.double() * 0.5, k.double() * 2.0, v.double() * 0.25
    o_ref = _torch_attention_f64(qd, kd, vd, 0.2, causal, (5, -1))
    np.testing.assert_allclose(o, o_ref.numpy(), rtol=0, atol=1e-12)
    kr = kd.repeat_interleave(2, 1)
    s = 0.2 * qd @ kr.transpose(-1, -2)
    N = 33
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    allowed = j >= i - 5
    if causal:
        allowed &= j <= i
    l_ref = torch.logsumexp(s.masked_fill(~allowed, float("-inf")), -1)
    np.testing.assert_allclose(lse, l_ref.numpy(), rtol=0, atol=1e-12)


def test_fp8_descale_folds_into_scale():
    """Scaling Q's descale by c equals scaling the softmax scale by c, and V's
    descale scales O linearly (the descales are plain multipliers)."""
    q, k, v = _fp8_inputs(1, 2, 2, 40, 32, seed=910)
    o1, l1 = oracle.attention_fp8(q, k, v, 0.3, 2.0, 1.0, 1.0, False)
    o2, l2 = oracle.attention_fp8(q, k, v, 0.6, 1.0, 1.0, 1.0, False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
    o3, l3 = oracle.attention_fp8(q, k, v, 0.6, 1.0, 1.0, 4.0, False)
    np.testing.assert_allclose(o3, 4.0 * o2, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(l3, l2)
