"""GPU parity of the split-KV forward (fa_fwd_splitkv) against the fp64 oracle.

The keys of every row are cut into splits that run as separate work units;
a merge kernel combines the partial outputs by their log-sum-exps.  The
result must meet the tolerances of the plain forward (max |O - O_ref| <=
2e-2, max |LSE - LSE_ref| <= 1e-3) for every split count, mask, window and
head grouping, including rows that have no admissible key in some splits.
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


def _status_ok(fa):
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"


def _split(fa, q, k, v, scale, causal, window=(-1, -1), num_splits=0, **kw):
    o, lse = fa.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal,
                            window=window, num_splits=num_splits, **kw)
    _status_ok(fa)
    return o, lse


def _check(o, lse, o_ref, lse_ref, what):
    o_np = o.float().cpu().numpy() if torch.is_tensor(o) else o
    l_np = lse.cpu().numpy() if torch.is_tensor(lse) else lse
    assert np.isfinite(o_np).all(), f"{what}: non-finite O"
    assert np.isfinite(l_np).all(), f"{what}: non-finite LSE"
    err_o = float(np.abs(o_np - o_ref).max())
    err_l = float(np.abs(l_np - lse_ref).max())
    assert err_l <= LSE_TOL, f"{what}: max|dLSE| = {err_l:.3e} (O err {err_o:.3e})"
    assert err_o <= O_TOL, f"{what}: max|dO| = {err_o:.3e} (LSE err {err_l:.3e})"


def _splits_used(fa, q, causal, window, num_splits):
    B, H, N, d = q.shape
    st, nbytes = fa.fa_splitkv_workspace_bytes(B, H, N, d, int(causal), window[0], window[1],
                                               num_splits)
    assert st == fa.FA_OK
    if nbytes == 0:
        return 1
    per_split = B * H * N * (d * 2 + 4)
    return round(nbytes / per_split)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("num_splits", [2, 3, 5, 64])
def test_split_counts(fa, d, causal, num_splits):
    q, k, v = make_random_qkv(2, 2, 1000, d, torch.bfloat16, seed=300 + d + num_splits)
    scale = 1.0 / math.sqrt(d)
    assert _splits_used(fa, q, causal, (-1, -1), num_splits) > 1
    o, lse = _split(fa, q, k, v, scale, causal, num_splits=num_splits)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    _check(o, lse, o_ref, lse_ref, f"d={d} causal={causal} splits={num_splits}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 1)])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("window", [(40, 40), (200, 0), (0, 0), (300, -1), (-1, 130)])
def test_windows_and_grouped_heads(fa, d, H, H_kv, causal, window):
    """Narrow windows leave most splits without admissible keys for a row."""
    q, _, _ = make_random_qkv(1, H, 900, d, torch.bfloat16, seed=310 + d + H_kv)
    _, k, v = make_random_qkv(1, H_kv, 900, d, torch.bfloat16, seed=311 + d + H_kv)
    scale = 1.0 / math.sqrt(d)
    o, lse = _split(fa, q, k, v, scale, causal, window=window, num_splits=4)
    o_ref, lse_ref = oracle.attention_ex(q, k, v, scale, causal, *window)
    _check(o, lse, o_ref, lse_ref, f"d={d} H={H}/{H_kv} causal={causal} window={window}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("N", [129, 257, 640, 1537])
def test_ragged_lengths(fa, dtype, N):
    q, k, v = make_random_qkv(1, 3, N, 128, dtype, seed=320 + N)
    o, lse = _split(fa, q, k, v, 0.09, True, num_splits=3)
    o_ref, lse_ref = oracle.attention(q, k, v, 0.09, True)
    _check(o, lse, o_ref, lse_ref, f"N={N} {dtype}")


@pytest.mark.parametrize("ctas", [1, 3])
@pytest.mark.parametrize("d", [128, 256])
def test_persistent_loop(fa, ctas, d):
    q, k, v = make_random_qkv(1, 2, 1300, d, torch.bfloat16, seed=330 + ctas)
    fa.fa_set_max_ctas(ctas)
    try:
        o, lse = _split(fa, q, k, v, 0.07, True, num_splits=4)
    finally:
        fa.fa_set_max_ctas(0)
    o_ref, lse_ref = oracle.attention(q, k, v, 0.07, True)
    _check(o, lse, o_ref, lse_ref, f"ctas={ctas} d={d}")


def test_one_split_is_the_plain_forward(fa):
    """With one split the call is fa_fwd_ext: bit-identical outputs."""
    q, k, v = make_random_qkv(2, 2, 700, 128, torch.bfloat16, seed=340)
    o1, l1 = _split(fa, q, k, v, 0.1, True, num_splits=1)
    o2, l2 = fa.fwd(q.cuda(), k.cuda(), v.cuda(), scale=0.1, causal=True)
    _status_ok(fa)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_auto_split_small_batch_long_sequence(fa):
    """One head of 8192 causal rows: 32 query units cannot fill the SMs, so the
    automatic count splits the keys; sampled rows against the oracle."""
    q, k, v = make_random_qkv(1, 1, 8192, 128, torch.bfloat16, seed=350)
    assert _splits_used(fa, q, True, (-1, -1), 0) > 1
    o, lse = _split(fa, q, k, v, 1.0 / math.sqrt(128), True, num_splits=0)
    g = torch.Generator().manual_seed(351)
    rows = sorted(set(torch.randint(0, 8192, (200,), generator=g).tolist())
                  | {0, 1, 127, 128, 255, 256, 4095, 4096, 8191})
    trip = [(0, 0, r) for r in rows]
    o_ref, lse_ref = oracle.attention_rows(q, k, v, 1.0 / math.sqrt(128), True, trip)
    idx = torch.tensor(rows)
    _check(o[0, 0, idx], lse[0, 0, idx], o_ref, lse_ref, "auto split, N=8192 causal")
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_workspace_and_outputs_stay_in_bounds(fa):
    """Guard bands around the workspace and the outputs are left untouched,
    and two calls on the same workspace give identical results."""
    q, k, v = make_random_qkv(1, 2, 600, 64, torch.float16, seed=360)
    B, H, N, d = q.shape
    st, need = fa.fa_splitkv_workspace_bytes(B, H, N, d, 0, -1, -1, 3)
    assert st == fa.FA_OK and need > 0
    G = 4096
    ws_all = torch.full((need + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = ws_all[G:G + need]
    numel = q.numel()
    pattern = torch.tensor([0x7E01], dtype=torch.int16).view(torch.float16)
    obuf = pattern.repeat(numel + 2 * 64).cuda()
    lbuf = torch.full((B * H * N + 2 * 64,), -3.5, dtype=torch.float32, device="cuda")
    o = obuf[64:64 + numel].view(q.shape)
    lse = lbuf[64:64 + B * H * N].view(B, H, N)
    outs = []
    for _ in range(2):
        _split(fa, q, k, v, 0.125, False, num_splits=3, out=o, lse=lse, workspace=ws)
        outs.append((o.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert (ws_all[:G] == 0xA5).all() and (ws_all[G + need:] == 0xA5).all()
    og = torch.cat([obuf[:64], obuf[64 + numel:]]).view(torch.int16).cpu()
    assert (og == 0x7E01).all()
    lg = torch.cat([lbuf[:64], lbuf[64 + B * H * N:]]).cpu()
    assert (lg == -3.5).all()
    o_ref, lse_ref = oracle.attention(q, k, v, 0.125, False)
    _check(o, lse, o_ref, lse_ref, "guarded")


def test_side_stream_without_lse(fa):
    q, k, v = make_random_qkv(1, 2, 1024, 128, torch.bfloat16, seed=370)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, _ = fa.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), scale=0.1, causal=False,
                              num_splits=4, return_lse=False, stream=s)
    s.synchronize()
    _status_ok(fa)
    o_ref, lse_ref = oracle.attention(q, k, v, 0.1, False)
    err = float(np.abs(o.float().cpu().numpy() - o_ref).max())
    assert err <= O_TOL
