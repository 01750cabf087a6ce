"""GPU checks of fa_fwd_host, the forward on host buffers.

The chunked copy-in / compute / copy-out pipeline must give exactly the
device forward's result (same kernel, same per-tile arithmetic), so most
cases compare bit for bit with fa_fwd_ext on the same inputs; the fp64 oracle
pins the host path itself at the forward's tolerances (max |O - O_ref| <=
2e-2, max |LSE - LSE_ref| <= 1e-3).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import make_random_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from attention_forward_10_gb300 import build
    build.build()
    import attention_forward_10_gb300 as fa_mod
    fa_mod.fa_set_max_ctas(0)
    fa_mod.fa_set_wait_timeout_us(2_000_000)
    return fa_mod


def _status_ok(fa):
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"


def _device(fa, q, k, v, scale, causal, window=(-1, -1)):
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal, window=window)
    torch.cuda.synchronize()
    _status_ok(fa)
    return o.cpu(), lse.cpu()


def _slot_bytes(B, H, H_kv, N, d, groups_per_chunk, with_lse=True):
    a256 = lambda x: (x + 255) // 256 * 256
    grp = H // H_kv
    g = groups_per_chunk
    return 2 * a256(g * grp * N * d * 2) + 2 * a256(g * N * d * 2) + \
        (a256(g * grp * N * 4) if with_lse else 0)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_host_forward_matches_oracle(fa, d, causal):
    q, k, v = make_random_qkv(2, 3, 700, d, torch.bfloat16, seed=1600 + d)
    q, k, v = (t.pin_memory() for t in (q, k, v))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd_host(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    _status_ok(fa)
    assert not o.is_cuda and not lse.is_cuda
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    assert float(np.abs(lse.numpy() - lse_ref).max()) <= 1e-3
    assert float(np.abs(o.float().numpy() - o_ref).max()) <= 2e-2


@pytest.mark.parametrize("shape", [(4, 16, 16, 1024, 128), (2, 8, 2, 777, 64),
                                   (1, 6, 1, 1500, 128), (3, 2, 2, 300, 256)])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_host_forward_bit_identical_to_device(fa, shape, causal):
    B, H, H_kv, N, d = shape
    q, _, _ = make_random_qkv(B, H, N, d, torch.float16, seed=1610 + N)
    _, k, v = make_random_qkv(B, H_kv, N, d, torch.float16, seed=1611 + N)
    q, k, v = (t.pin_memory() for t in (q, k, v))
    o_d, lse_d = _device(fa, q, k, v, 0.07, causal)
    o, lse = fa.fwd_host(q, k, v, scale=0.07, causal=causal)
    torch.cuda.synchronize()
    _status_ok(fa)
    assert torch.equal(o, o_d) and torch.equal(lse, lse_d)


@pytest.mark.parametrize("slots,groups_per_chunk", [(1, 1), (2, 1), (3, 1), (2, 3)])
def test_small_workspace_shrinks_the_chunks(fa, slots, groups_per_chunk):
    """A workspace of `slots` slots of `groups_per_chunk` groups: the plan
    shrinks to fit it, and the result does not change."""
    B, H, H_kv, N, d = 2, 8, 4, 640, 128
    q, _, _ = make_random_qkv(B, H, N, d, torch.bfloat16, seed=1620)
    _, k, v = make_random_qkv(B, H_kv, N, d, torch.bfloat16, seed=1621)
    q, k, v = (t.pin_memory() for t in (q, k, v))
    o_d, lse_d = _device(fa, q, k, v, 0.09, True)
    nbytes = slots * _slot_bytes(B, H, H_kv, N, d, groups_per_chunk)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    o, lse = fa.fwd_host(q, k, v, scale=0.09, causal=True, workspace=ws)
    torch.cuda.synchronize()
    _status_ok(fa)
    assert torch.equal(o, o_d) and torch.equal(lse, lse_d)


def test_workspace_below_one_group_is_rejected(fa):
    B, H, H_kv, N, d = 1, 4, 2, 512, 128
    q, _, _ = make_random_qkv(B, H, N, d, torch.bfloat16, seed=1625)
    _, k, v = make_random_qkv(B, H_kv, N, d, torch.bfloat16, seed=1626)
    need = _slot_bytes(B, H, H_kv, N, d, 1)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H_kv,
            N, d, 0.09, 0, -1, -1, fa.FA_DTYPE_BF16, ws.data_ptr())
    assert fa.fa_fwd_host(*args, need - 1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_host(*args, need, None) == fa.FA_OK
    torch.cuda.synchronize()
    _status_ok(fa)


def test_pageable_memory_and_no_lse(fa):
    q, k, v = make_random_qkv(2, 4, 900, 128, torch.bfloat16, seed=1630)
    assert not q.is_pinned()
    o_d, _ = _device(fa, q, k, v, 0.09, False)
    o, lse = fa.fwd_host(q, k, v, scale=0.09, return_lse=False)
    torch.cuda.synchronize()
    _status_ok(fa)
    assert lse is None and torch.equal(o, o_d)


@pytest.mark.parametrize("window", [(200, 0), (64, 64)])
def test_groups_and_windows(fa, window):
    q, _, _ = make_random_qkv(2, 8, 1100, 128, torch.bfloat16, seed=1640)
    _, k, v = make_random_qkv(2, 2, 1100, 128, torch.bfloat16, seed=1641)
    q, k, v = (t.pin_memory() for t in (q, k, v))
    o_d, lse_d = _device(fa, q, k, v, 0.09, False, window)
    o, lse = fa.fwd_host(q, k, v, scale=0.09, window=window)
    torch.cuda.synchronize()
    _status_ok(fa)
    assert torch.equal(o, o_d) and torch.equal(lse, lse_d)


def test_side_stream(fa):
    q, k, v = make_random_qkv(4, 8, 1024, 128, torch.bfloat16, seed=1650)
    q, k, v = (t.pin_memory() for t in (q, k, v))
    o_d, lse_d = _device(fa, q, k, v, 0.09, True)
    side = torch.cuda.Stream()
    o, lse = fa.fwd_host(q, k, v, scale=0.09, causal=True, stream=side)
    side.synchronize()
    _status_ok(fa)
    assert torch.equal(o, o_d) and torch.equal(lse, lse_d)


def test_graph_capture_and_replay(fa):
    """Pinned buffers: the call is captured once and replayed on new inputs
    written into the same host buffers."""
    B, H, N, d = 4, 8, 1024, 128
    q, k, v = (t.pin_memory() for t in make_random_qkv(B, H, N, d, torch.bfloat16, seed=1660))
    o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    st, need = fa.fa_fwd_host_workspace_bytes(B, H, H, N, d, 1)
    assert st == fa.FA_OK
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    # the first call outside capture makes the library's helper streams
    fa.fwd_host(q, k, v, scale=0.09, out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            fa.fwd_host(q, k, v, scale=0.09, out=o, lse=lse, workspace=ws, stream=cap)
    for seed in (1661, 1662):
        q2, k2, v2 = make_random_qkv(B, H, N, d, torch.bfloat16, seed=seed)
        q.copy_(q2), k.copy_(k2), v.copy_(v2)
        graph.replay()
        torch.cuda.synchronize()
        _status_ok(fa)
        o_d, lse_d = _device(fa, q2, k2, v2, 0.09, False)
        assert torch.equal(o, o_d) and torch.equal(lse, lse_d)
