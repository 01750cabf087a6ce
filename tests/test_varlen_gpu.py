"""GPU parity of the variable-length forward (fa_fwd_varlen) against the fp64
oracle's packed-sequence evaluation.

Sequences of different lengths are packed along the rows of [total, H, d]
tensors; each is attended on its own.  Tolerances as for the plain forward
(max |dO| <= 2e-2, max |dLSE| <= 1e-3), compared element by element over
every row that belongs to a sequence; rows outside every sequence must stay
untouched.
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


def _packed(lens, H, H_kv, d, dtype, seed, extra_rows=0):
    total = sum(lens) + extra_rows
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(total, H, d, generator=g).to(dtype)
    k = torch.randn(total, H_kv, d, generator=g).to(dtype)
    v = torch.randn(total, H_kv, d, generator=g).to(dtype)
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    return q, k, v, cu


def _run(fa, q, k, v, cu, scale, causal, window=(-1, -1), out=None, lse=None, max_seqlen=None):
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    lens = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    ms = max(lens) if max_seqlen is None else max_seqlen
    o, l = fa.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_t, ms, scale=scale, causal=causal,
                         window=window, out=out, lse=lse)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    return o, l


def _check(o, lse, o_ref, l_ref, cu, what):
    rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in range(len(cu) - 1)])
    o_np = o.float().cpu().numpy()[rows]
    l_np = lse.cpu().numpy()[:, rows]
    assert np.isfinite(o_np).all() and np.isfinite(l_np).all(), f"{what}: non-finite"
    err_o = float(np.abs(o_np - o_ref[rows]).max())
    err_l = float(np.abs(l_np - l_ref[:, rows]).max())
    assert err_l <= LSE_TOL, f"{what}: max|dLSE| = {err_l:.3e} (O err {err_o:.3e})"
    assert err_o <= O_TOL, f"{what}: max|dO| = {err_o:.3e} (LSE err {err_l:.3e})"


LENS = [1, 127, 128, 129, 300, 0, 640, 5, 257]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_ragged_batch(fa, d, causal, dtype):
    q, k, v, cu = _packed(LENS, 4, 2, d, dtype, seed=600 + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, cu, scale, causal)
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, scale, causal)
    _check(o, lse, o_ref, l_ref, cu, f"d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("window", [(40, 40), (200, 0), (0, 0), (-1, 130)])
def test_windows(fa, d, causal, window):
    q, k, v, cu = _packed([700, 3, 260, 128], 2, 1, d, torch.bfloat16, seed=610 + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, cu, scale, causal, window)
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, scale, causal, *window)
    _check(o, lse, o_ref, l_ref, cu, f"d={d} causal={causal} window={window}")


@pytest.mark.parametrize("ctas", [1, 3])
@pytest.mark.parametrize("d", [128, 256])
def test_persistent_loop(fa, ctas, d):
    q, k, v, cu = _packed([900, 130, 1, 513, 256], 2, 2, d, torch.bfloat16, seed=620 + ctas)
    fa.fa_set_max_ctas(ctas)
    try:
        o, lse = _run(fa, q, k, v, cu, 0.08, True)
    finally:
        fa.fa_set_max_ctas(0)
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, 0.08, True)
    _check(o, lse, o_ref, l_ref, cu, f"ctas={ctas} d={d}")


@pytest.mark.parametrize("nseq,max_seqlen,H_kv", [
    (64, None, 2), (64, None, 1),   # the table's limit (H_kv 1: grouped heads packed)
    (65, None, 2),                  # one sequence more: pairs counted from each end
    (20, 5000, 1),                  # max_seqlen far above every length: empty pair groups
    (20, 70000, 2),                 # more than 256 units per problem: counted from each end
])
@pytest.mark.parametrize("ctas", [0, 5])
def test_causal_unit_table_and_fallback(fa, nseq, max_seqlen, H_kv, ctas):
    """Packed causal launches of the d <= 128 kernel with at most 64
    sequences and 256 units per problem take their units from a per-CTA
    table (groups of equal pair index, heaviest first, every other wave
    reversed); past either limit the pairs are counted from each sequence's
    end.  Both sides of both limits, on every SM and on 5 CTAs (many
    waves)."""
    g = torch.Generator().manual_seed(640 + nseq)
    lens = torch.randint(0, 700, (nseq,), generator=g).tolist()
    q, k, v, cu = _packed(lens, 2, H_kv, 128, torch.bfloat16, seed=641 + nseq)
    fa.fa_set_max_ctas(ctas)
    try:
        o, lse = _run(fa, q, k, v, cu, 0.09, True, max_seqlen=max_seqlen)
    finally:
        fa.fa_set_max_ctas(0)
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, 0.09, True)
    _check(o, lse, o_ref, l_ref, cu, f"nseq={nseq} max_seqlen={max_seqlen} H_kv={H_kv}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", [256, 333])
def test_equal_lengths_equal_the_batched_forward(fa, d, N):
    """Packing equal-length sequences gives the [B,H,N,d] forward bit for bit
    (same tiles, same arithmetic; padding keys are masked either way)."""
    q, k, v = make_random_qkv(3, 2, N, d, torch.bfloat16, seed=630 + N)
    o_b, l_b = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    pack = lambda t: t.permute(0, 2, 1, 3).reshape(3 * N, 2, d).contiguous()
    o_v, l_v = _run(fa, pack(q), pack(k), pack(v), [0, N, 2 * N, 3 * N], d ** -0.5, True)
    assert torch.equal(o_v, pack(o_b))
    assert torch.equal(l_v, l_b.permute(1, 0, 2).reshape(2, 3 * N))


def test_rows_outside_sequences_and_guards_untouched(fa):
    q, k, v, cu = _packed([200, 77], 2, 2, 128, torch.bfloat16, seed=640, extra_rows=50)
    total = q.shape[0]
    G = 256
    pattern = torch.tensor([0x7FC1], dtype=torch.int16).view(torch.bfloat16)
    obuf = pattern.repeat(q.numel() + 2 * G).cuda()
    lbuf = torch.full((2 * total + 2 * G,), -7.25, dtype=torch.float32, device="cuda")
    o = obuf[G:G + q.numel()].view(q.shape)
    lse = lbuf[G:G + 2 * total].view(2, total)
    _run(fa, q, k, v, cu, 0.1, False, out=o, lse=lse)
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, 0.1, False)
    _check(o, lse, o_ref, l_ref, cu, "guarded")
    tail = o[cu[-1]:].contiguous().view(torch.int16).cpu()
    assert (tail == 0x7FC1).all()
    assert (lse[:, cu[-1]:].cpu() == -7.25).all()
    og = torch.cat([obuf[:G], obuf[G + q.numel():]]).view(torch.int16).cpu()
    assert (og == 0x7FC1).all()
    lg = torch.cat([lbuf[:G], lbuf[G + 2 * total:]]).cpu()
    assert (lg == -7.25).all()


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("d", [64, 128])
def test_subset_of_sequences_matches_the_full_call(fa, causal, d):
    """A call over sequences b0 .. b1-1 only (cu_seqlens from entry b0 on,
    row offsets still those of the whole packed tensor, total unchanged)
    writes exactly those sequences' rows, bit for bit as the call over all
    sequences does, and nothing else."""
    lens = [300, 129, 700, 64, 1000, 3]
    H = 4
    q, k, v, cu = _packed(lens, H, H, d, torch.bfloat16, seed=2300 + d)
    total = cu[-1]
    o_full, l_full = _run(fa, q, k, v, cu, 0.1, causal)
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    for b0, b1 in ((1, 3), (0, 1), (2, 6), (5, 6)):
        o = torch.full((total, H, d), 7.0, dtype=torch.bfloat16, device="cuda")
        lse = torch.full((H, total), 7.0, dtype=torch.float32, device="cuda")
        fa.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_t[b0:b1 + 1], max(lens[b0:b1]),
                      scale=0.1, causal=causal, out=o, lse=lse)
        torch.cuda.synchronize()
        st, site = fa.fa_get_device_status(None)
        assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
        r0, r1 = cu[b0], cu[b1]
        assert torch.equal(o[r0:r1], o_full[r0:r1]), (b0, b1)
        assert torch.equal(lse[:, r0:r1], l_full[:, r0:r1]), (b0, b1)
        assert bool((o[:r0] == 7.0).all()) and bool((o[r1:] == 7.0).all()), (b0, b1)
        assert bool((lse[:, :r0] == 7.0).all()) and bool((lse[:, r1:] == 7.0).all()), (b0, b1)


def test_malformed_offsets_stay_in_bounds(fa):
    """Offsets past `total`, a decreasing pair and a sequence longer than
    max_seqlen are clamped by the kernels: the rows they still cover are
    correct and nothing outside the tensors is written."""
    total, H, d = 400, 2, 128
    g = torch.Generator().manual_seed(650)
    q, k, v = (torch.randn(total, H, d, generator=g).to(torch.bfloat16) for _ in range(3))
    # seq 0: rows [0, 300) cut to max_seqlen = 256 rows; seq 1: decreasing
    # offsets (empty); seq 2: rows [290, 350); seq 3: rows [350, 900) cut at
    # total -> [350, 400)
    cu = [0, 300, 290, 350, 900]
    G = 256
    pattern = torch.tensor([0x7FC1], dtype=torch.int16).view(torch.bfloat16)
    obuf = pattern.repeat(q.numel() + 2 * G).cuda()
    lbuf = torch.full((H * total + 2 * G,), -7.25, dtype=torch.float32, device="cuda")
    o = obuf[G:G + q.numel()].view(q.shape)
    lse = lbuf[G:G + H * total].view(H, total)
    _run(fa, q, k, v, cu, 0.1, True, out=o, lse=lse, max_seqlen=256)
    for (r0, r1, what) in ((0, 256, "first sequence, cut to max_seqlen"),
                           (290, 350, "third sequence"),
                           (350, 400, "last sequence, cut at total")):
        o_ref, l_ref = oracle.attention_varlen(q[r0:r1], k[r0:r1], v[r0:r1], [0, r1 - r0],
                                               0.1, True)
        _check(o[r0:r1], lse[:, r0:r1], o_ref, l_ref, [0, r1 - r0], what)
    assert (o[256:290].contiguous().view(torch.int16).cpu() == 0x7FC1).all()
    assert (lse[:, 256:290].cpu() == -7.25).all()
    og = torch.cat([obuf[:G], obuf[G + q.numel():]]).view(torch.int16).cpu()
    assert (og == 0x7FC1).all()
    lg = torch.cat([lbuf[:G], lbuf[G + H * total:]]).cpu()
    assert (lg == -7.25).all()


# ---------------------------------------------------------------- backward
def _bwd_check(fa, lens, H, H_kv, d, causal, window, seed):
    q, k, v, cu = _packed(lens, H, H_kv, d, torch.bfloat16, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    ms = max(lens)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd_varlen(qd, kd, vd, cu_t, ms, causal=causal, window=window)
    dq, dk, dv = fa.bwd_varlen(qd, kd, vd, o, lse, dod, cu_t, ms, causal=causal, window=window)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    scale = d ** -0.5
    for b, n in enumerate(lens):
        if n == 0:
            continue
        s0 = cu[b]
        view = lambda t: t[s0:s0 + n].permute(1, 0, 2).unsqueeze(0).contiguous()
        ref = oracle.attention_bwd(view(q), view(k), view(v), view(do), scale, causal, *window)
        got = [t[s0:s0 + n].permute(1, 0, 2).unsqueeze(0).float().cpu().numpy()
               for t in (dq, dk, dv)]
        for name, gt, r in zip(("dQ", "dK", "dV"), got, ref):
            err = float(np.abs(gt - r).max())
            bound = 2e-2 * float(np.abs(r).max()) + 1e-4
            assert err <= bound, f"seq {b} (n={n}) {name}: {err:.3e} > {bound:.3e}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_backward_ragged(fa, d, causal):
    _bwd_check(fa, [1, 127, 300, 0, 129, 513], 4, 2, d, causal, (-1, -1), seed=660 + d)


@pytest.mark.parametrize("window", [(40, 40), (200, 0)])
def test_backward_windows(fa, window):
    _bwd_check(fa, [700, 3, 260], 2, 2, 128, False, window, seed=670)


@pytest.mark.parametrize("ctas", [1, 4])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_backward_ragged_many_units_per_cta(fa, ctas, causal):
    """A small grid walks every (sequence, head) unit of a ragged batch,
    including the empty units of short and empty sequences."""
    fa.fa_set_max_ctas(ctas)
    try:
        _bwd_check(fa, [1, 127, 300, 0, 129, 513, 260], 4, 2, 128, causal, (-1, -1),
                   seed=690 + ctas)
    finally:
        fa.fa_set_max_ctas(0)


@pytest.mark.parametrize("nseq,H_kv", [(64, 2), (64, 1), (65, 2)])
@pytest.mark.parametrize("ctas", [0, 5])
def test_backward_unit_table_and_fallback(fa, nseq, H_kv, ctas):
    """Packed causal backward launches with at most 64 sequences order the
    units of both kernels from a per-CTA table (groups of equal tile index,
    heaviest first, every other wave reversed); with 65 sequences they keep
    the plain order.  On every SM and on 5 CTAs (many waves)."""
    g = torch.Generator().manual_seed(700 + nseq)
    lens = torch.randint(0, 400, (nseq,), generator=g).tolist()
    fa.fa_set_max_ctas(ctas)
    try:
        _bwd_check(fa, lens, 2, H_kv, 128, True, (-1, -1), seed=701 + nseq + H_kv)
    finally:
        fa.fa_set_max_ctas(0)


def test_backward_equal_lengths_equal_the_batched_backward(fa):
    """Equal-length packed sequences give fa_bwd's gradients bit for bit."""
    N, d = 256, 128
    q, k, v = make_random_qkv(2, 2, N, d, torch.bfloat16, seed=680)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(681)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=True)
    ref = fa.bwd(qd, kd, vd, o, lse, dod, causal=True)
    pack = lambda t: t.permute(0, 2, 1, 3).reshape(2 * N, 2, d).contiguous()
    cu_t = torch.tensor([0, N, 2 * N], dtype=torch.int32, device="cuda")
    lse_p = lse.permute(1, 0, 2).reshape(2, 2 * N).contiguous()
    got = fa.bwd_varlen(pack(qd), pack(kd), pack(vd), pack(o), lse_p, pack(dod), cu_t, N,
                        causal=True)
    torch.cuda.synchronize()
    for g_, r_ in zip(got, ref):
        assert torch.equal(g_, pack(r_))
