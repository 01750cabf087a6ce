"""GPU check of fa_fwd_splitkv_noalloc, the split-KV forward that keeps its
partials in the library's fixed per-device scratch instead of a caller
workspace.

Each case calls it through the C ABI twice in a row on the same inputs and
compares both results with the fp64 oracle and with the existing entry
points: within the parity tolerances (max |dO| <= 2e-2, max |dLSE| <= 1e-3)
of the oracle (every row, or 512 seeded rows plus the edge rows of the
long case) and of the unsplit fa_fwd_ext, and bit for bit with
fa_fwd_splitkv run with the same split count on a torch-allocated
workspace.  For the automatic count the case is one where the planned
count does not fit the scratch, and the comparison is with fa_fwd_splitkv
at the count the library must lower it to.  The file sorts last so that it
also runs after every other test in one session; it depends on no state
they leave.
"""
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


def _dcode(fa, t):
    return fa.FA_DTYPE_BF16 if t.dtype == torch.bfloat16 else fa.FA_DTYPE_F16


def _sync_ok(fa):
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"


def _noalloc(fa, q, k, v, scale, causal, window, S):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, k.shape[1], N, d, scale, int(causal),
                                   window[0], window[1], _dcode(fa, q), S,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o, lse


def _with_workspace(fa, q, k, v, scale, causal, window, S):
    B, H, N, d = q.shape
    st, need = fa.fa_splitkv_workspace_bytes(B, H, N, d, int(causal), window[0], window[1], S)
    assert st == fa.FA_OK
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = fa.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), B, H, k.shape[1], N, d, scale, int(causal),
                           window[0], window[1], _dcode(fa, q), S, ws.data_ptr(), need,
                           torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o, lse, need


def _unsplit(fa, q, k, v, scale, causal, window):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = fa.fa_fwd_ext(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       B, H, k.shape[1], N, d, scale, int(causal), window[0], window[1],
                       _dcode(fa, q), torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o, lse


CASES = [
    # B, H, H_kv, N, d, dtype, causal, window, num_splits
    (1, 2, 2, 1000, 128, torch.bfloat16, True, (-1, -1), 4),
    (2, 2, 1, 777, 64, torch.float16, False, (-1, -1), 3),
    (1, 4, 2, 1200, 256, torch.bfloat16, True, (300, -1), 5),
    (1, 2, 2, 900, 128, torch.bfloat16, False, (100, 100), 4),
    # automatic count: on 152 SMs the planner picks 7 splits (60 MB of
    # partials) for these 128 units, which the scratch limit lowers to 3
    (1, 1, 1, 32768, 128, torch.bfloat16, False, (-1, -1), 0),
]


def _oracle_check(q, k, v, scale, causal, window, results):
    """Both results against the fp64 oracle: every row of the small cases,
    512 seeded rows plus the edge rows of the long one."""
    B, H, N, _ = q.shape
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    if N <= 4096:
        o_ref, l_ref = oracle.attention_ex(qc, kc, vc, scale, causal, *window)
        pick = lambda o, lse: (o.float().cpu().numpy(), lse.cpu().numpy())
    else:
        g = torch.Generator().manual_seed(520)
        rows = {(b, h, i) for b in range(B) for h in range(H)
                for i in (0, 1, 127, 128, N // 2, N - 2, N - 1)}
        rows |= {(int(torch.randint(B, (1,), generator=g)), int(torch.randint(H, (1,), generator=g)),
                  int(torch.randint(N, (1,), generator=g))) for _ in range(512)}
        rows = sorted(rows)
        o_ref, l_ref = oracle.attention_rows_ex(qc, kc, vc, scale, causal, rows, *window)
        idx = tuple(np.array(rows).T)
        pick = lambda o, lse: (o.float().cpu().numpy()[idx], lse.cpu().numpy()[idx])
    for o, lse in results:
        o_np, l_np = pick(o, lse)
        err_o = float(np.abs(o_np - o_ref).max())
        err_l = float(np.abs(l_np - l_ref).max())
        assert err_o <= O_TOL and err_l <= LSE_TOL, ("oracle", err_o, err_l)


def _lowered_count(fa, B, H, N, d, causal, window):
    """The automatic split count and the count fa_fwd_splitkv_noalloc must
    lower it to: the largest count (as resolved by the planner) whose
    partials fit the scratch."""
    st, auto_bytes = fa.fa_splitkv_workspace_bytes(B, H, N, d, int(causal), *window, 0)
    assert st == fa.FA_OK
    per_split = B * H * N * (2 * d + 4)
    auto = auto_bytes // per_split
    for want in range(auto, 0, -1):
        st, need = fa.fa_splitkv_workspace_bytes(B, H, N, d, int(causal), *window, want)
        assert st == fa.FA_OK
        if need <= fa.FA_NOALLOC_SCRATCH_BYTES:
            return auto_bytes, want
    return auto_bytes, 1


@pytest.mark.parametrize("case", CASES, ids=[f"N{c[3]}_d{c[4]}_S{c[8]}" for c in CASES])
def test_noalloc_twice_matches_existing_entry_points(fa, case):
    B, H, H_kv, N, d, dtype, causal, window, S = case
    q, _, _ = make_random_qkv(B, H, N, d, dtype, seed=500 + N)
    _, k, v = make_random_qkv(B, H_kv, N, d, dtype, seed=501 + N)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    scale = d ** -0.5
    first = _noalloc(fa, q, k, v, scale, causal, window, S)
    second = _noalloc(fa, q, k, v, scale, causal, window, S)
    _sync_ok(fa)
    o_ref, l_ref = _unsplit(fa, q, k, v, scale, causal, window)
    _sync_ok(fa)
    for o, lse in (first, second):
        assert torch.isfinite(o).all() and torch.isfinite(lse).all()
        err_o = (o.float() - o_ref.float()).abs().max().item()
        err_l = (lse - l_ref).abs().max().item()
        assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)
    assert torch.equal(first[0], second[0]) and torch.equal(first[1], second[1])
    _oracle_check(q, k, v, scale, causal, window, (first, second))
    explicit = S
    if S == 0:
        # the planned count must not fit, so that the lowering really ran
        auto_bytes, explicit = _lowered_count(fa, B, H, N, d, causal, window)
        assert auto_bytes > fa.FA_NOALLOC_SCRATCH_BYTES, auto_bytes
        assert explicit > 1
    o_w, l_w, need = _with_workspace(fa, q, k, v, scale, causal, window, explicit)
    _sync_ok(fa)
    assert 0 < need <= fa.FA_NOALLOC_SCRATCH_BYTES
    assert torch.equal(first[0], o_w) and torch.equal(first[1], l_w)


def test_noalloc_beyond_the_scratch_is_rejected_untouched(fa):
    q, k, v = make_random_qkv(1, 8, 8192, 128, torch.bfloat16, seed=510)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(q, 3.0)
    lse = torch.full((1, 8, 8192), 5.0, dtype=torch.float32, device="cuda")
    st = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), 1, 8, 8, 8192, 128, 0.088, 0, -1, -1,
                                   fa.FA_DTYPE_BF16, 8, None)
    assert st == fa.FA_ERR_SCRATCH_LIMIT
    _sync_ok(fa)
    assert (o == 3.0).all() and (lse == 5.0).all()
