"""GPU parity of fa_fwd_varlen_qk (separate query and key sequences, used
lengths, bottom-right aligned masks) against the fp64 oracle's
attention_varlen_qk, element by element over every used query row.

Tolerances as for the plain forward: max |dO| <= 2e-2, max |dLSE| <= 1e-3 on
rows with at least one key; rows without a key must come out as exactly
O = 0 and LSE = -inf; query rows outside every sequence's used rows must
keep the sentinel values they held before the call.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_TOL = 1e-3
SENTINEL_O = 3.0
SENTINEL_L = 7.0


@pytest.fixture(scope="module")
def fa():
    from attention_forward_10_gb300 import build
    build.build()
    import attention_forward_10_gb300 as fa_mod
    fa_mod.fa_set_max_ctas(0)
    fa_mod.fa_set_wait_timeout_us(2_000_000)
    return fa_mod


def _offsets(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int64).tolist()


def _inputs(total_q, total_k, H, H_kv, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(total_q, H, d, generator=g).to(dtype)
    k = torch.randn(total_k, H_kv, d, generator=g).to(dtype)
    v = torch.randn(total_k, H_kv, d, generator=g).to(dtype)
    return q, k, v


def _run(fa, q, k, v, cu_q, cu_k, used_q, used_k, causal, window, scale):
    dev = "cuda"
    t32 = lambda x: None if x is None else torch.tensor(x, dtype=torch.int32, device=dev)  # noqa
    lq = [cu_q[i + 1] - cu_q[i] for i in range(len(cu_q) - 1)]
    lk = [cu_k[i + 1] - cu_k[i] for i in range(len(cu_k) - 1)]
    mq = max(used_q) if used_q is not None else max(lq)
    mk = max(used_k) if used_k is not None else max(lk)
    out = torch.full(q.shape, SENTINEL_O, dtype=q.dtype, device=dev)
    lse = torch.full((q.shape[1], q.shape[0]), SENTINEL_L, dtype=torch.float32, device=dev)
    o, l = fa.fwd_varlen_qk(q.to(dev), k.to(dev), v.to(dev), t32(cu_q), t32(cu_k), mq, mk,
                            seqused_q=t32(used_q), seqused_k=t32(used_k), scale=scale,
                            causal=causal, window=window, out=out, lse=lse)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    return o.float().cpu().numpy(), l.cpu().numpy()


def _check(o, lse, o_ref, l_ref, cu_q, used_q, what):
    B = len(cu_q) - 1
    nq = [used_q[b] if used_q is not None else cu_q[b + 1] - cu_q[b] for b in range(B)]
    rows = np.concatenate([np.arange(cu_q[b], cu_q[b] + nq[b]) for b in range(B)] +
                          [np.zeros(0, dtype=np.int64)]).astype(np.int64)
    empty = np.isneginf(l_ref[:, rows])            # [H, rows]: no admissible key
    lg = lse[:, rows]
    assert (np.isneginf(lg) == empty).all(), f"{what}: -inf LSE rows differ"
    og = o[rows].transpose(1, 0, 2)                # [H, rows, d]
    assert (og[empty] == 0).all(), f"{what}: rows without keys must have O = 0"
    if (~empty).any():
        err_l = float(np.abs(lg[~empty] - l_ref[:, rows][~empty]).max())
        err_o = float(np.abs(og[~empty] - o_ref[rows].transpose(1, 0, 2)[~empty]).max())
        assert err_o <= O_TOL and err_l <= LSE_TOL, (what, err_o, err_l)
    rest = np.setdiff1d(np.arange(o.shape[0]), rows)
    assert (o[rest] == SENTINEL_O).all() and (lse[:, rest] == SENTINEL_L).all(), \
        f"{what}: rows outside the used sequences were written"


CROSS = [
    # (query lengths, key lengths): cross-attention and decode shapes, a
    # prefill continuing a cache, fewer keys than queries, an empty query
    # sequence and a sequence without keys
    ([5, 1, 17, 0, 9, 300, 130], [12, 40, 17, 6, 3, 1000, 0]),
    ([1, 1, 1, 1, 64, 16], [2000, 1, 333, 129, 900, 4000]),
    ([700, 260], [200, 700]),
]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("case", range(len(CROSS)))
def test_separate_query_and_key_sequences(fa, d, causal, case):
    lq, lk = CROSS[case]
    cu_q, cu_k = _offsets(lq), _offsets(lk)
    q, k, v = _inputs(cu_q[-1] + 3, cu_k[-1] + 5, 4, 2, d, torch.bfloat16, seed=700 + case)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, cu_q, cu_k, None, None, causal, (-1, -1), scale)
    o_ref, l_ref = oracle.attention_varlen_qk(q, k, v, cu_q, cu_k, scale, causal)
    _check(o, lse, o_ref, l_ref, cu_q, None, f"case {case} d={d} causal={causal}")


@pytest.mark.parametrize("window", [(100, 0), (0, 50), (300, 300)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_windows_bottom_right(fa, window, dtype):
    lq, lk = [200, 1, 90, 513], [450, 700, 30, 513]
    cu_q, cu_k = _offsets(lq), _offsets(lk)
    q, k, v = _inputs(cu_q[-1], cu_k[-1], 2, 2, 128, dtype, seed=710)
    o, lse = _run(fa, q, k, v, cu_q, cu_k, None, None, False, window, 0.09)
    o_ref, l_ref = oracle.attention_varlen_qk(q, k, v, cu_q, cu_k, 0.09, False, *window)
    _check(o, lse, o_ref, l_ref, cu_q, None, f"window={window}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_kv_cache_used_lengths(fa, d, causal):
    """A KV cache with spare capacity: each sequence owns cap_k rows of K/V
    but only its first used_k take part; queries likewise (rows past used_q
    keep their sentinel)."""
    cap_q, cap_k = [8, 64, 3, 200], [1024, 512, 2048, 300]
    used_q, used_k = [3, 64, 0, 130], [1000, 1, 1500, 300]
    cu_q, cu_k = _offsets(cap_q), _offsets(cap_k)
    q, k, v = _inputs(cu_q[-1], cu_k[-1], 8, 1, d, torch.bfloat16, seed=720 + d)
    # cache rows past the used lengths hold values that would change the
    # result if they were read into the softmax
    for b in range(4):
        k[cu_k[b] + used_k[b]:cu_k[b + 1]] = 30.0
        v[cu_k[b] + used_k[b]:cu_k[b + 1]] = -50.0
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, cu_q, cu_k, used_q, used_k, causal, (-1, -1), scale)
    o_ref, l_ref = oracle.attention_varlen_qk(q, k, v, cu_q, cu_k, scale, causal,
                                              seqused_q=used_q, seqused_k=used_k)
    _check(o, lse, o_ref, l_ref, cu_q, used_q, f"d={d} causal={causal}")


def test_decode_gqa_many_heads(fa):
    """Decode-shaped: a few query rows per sequence against long caches with
    8 query heads per K/V head."""
    lq, lk = [1, 4, 16, 64, 2, 33], [8192, 3000, 5000, 8192, 777, 4096]
    cu_q, cu_k = _offsets(lq), _offsets(lk)
    q, k, v = _inputs(cu_q[-1], cu_k[-1], 16, 2, 128, torch.bfloat16, seed=730)
    o, lse = _run(fa, q, k, v, cu_q, cu_k, None, None, True, (-1, -1), 0.088)
    o_ref, l_ref = oracle.attention_varlen_qk(q, k, v, cu_q, cu_k, 0.088, True)
    _check(o, lse, o_ref, l_ref, cu_q, None, "decode gqa")


def test_no_key_rows_at_all(fa):
    """total_k = 0: every used query row has no key (O = 0, LSE = -inf)."""
    dev = "cuda"
    q = torch.randn(140, 2, 128).to(torch.bfloat16).to(dev)
    kd = torch.empty(1, 2, 128, dtype=torch.bfloat16, device=dev)
    cu_q = torch.tensor([0, 5, 140], dtype=torch.int32, device=dev)
    cu_k = torch.tensor([0, 0, 0], dtype=torch.int32, device=dev)
    out = torch.full(q.shape, SENTINEL_O, dtype=q.dtype, device=dev)
    lse = torch.full((2, 140), SENTINEL_L, dtype=torch.float32, device=dev)
    st = fa.fa_fwd_varlen_qk(q.data_ptr(), kd.data_ptr(), kd.data_ptr(), out.data_ptr(),
                             lse.data_ptr(), cu_q.data_ptr(), cu_k.data_ptr(), None, None, 2,
                             135, 0, 140, 0, 2, 2, 128, 0.1, 0, -1, -1, fa.FA_DTYPE_BF16, None)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, (st, site)
    assert (out == 0).all() and torch.isneginf(lse).all()


def test_equal_offsets_match_the_self_attention_call_bit_for_bit(fa):
    lens = [1, 127, 128, 129, 300, 0, 640]
    cu = _offsets(lens)
    q, k, v = _inputs(cu[-1], cu[-1], 4, 2, 128, torch.bfloat16, seed=740)
    o1, l1 = _run(fa, q, k, v, cu, cu, None, None, True, (-1, -1), 0.1)
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o2, l2 = fa.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_t, max(lens), scale=0.1, causal=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(o1, o2.float().cpu().numpy())
    np.testing.assert_array_equal(l1, l2.cpu().numpy())


def test_argument_errors(fa):
    z = torch.zeros(16, 1, 128, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 16], dtype=torch.int32, device="cuda")
    args = dict(q=z.data_ptr(), k=z.data_ptr(), v=z.data_ptr(), o=z.data_ptr(), lse=None,
                cu_seqlens_q=cu.data_ptr(), cu_seqlens_k=cu.data_ptr(), seqused_q=None,
                seqused_k=None, batch=1, max_seqlen_q=16, max_seqlen_k=16, total_q=16,
                total_k=16, H=1, H_kv=1, d=128, scale=0.1, causal=0, window_left=-1,
                window_right=-1, dtype=fa.FA_DTYPE_BF16, stream=None)
    for key, val, want in (("total_k", -1, fa.FA_ERR_INVALID_ARG),
                           ("max_seqlen_k", -1, fa.FA_ERR_INVALID_ARG),
                           ("max_seqlen_k", 1 << 30, fa.FA_ERR_INVALID_ARG),
                           ("cu_seqlens_k", None, fa.FA_ERR_INVALID_ARG),
                           ("seqused_k", cu.data_ptr() + 2, fa.FA_ERR_MISALIGNED),
                           ("d", 96, fa.FA_ERR_UNSUPPORTED)):
        bad = dict(args, **{key: val})
        assert fa.fa_fwd_varlen_qk(*bad.values()) == want, key
    torch.cuda.synchronize()


GQA_CASES = [
    # (H, H_kv): groups of 2, 4, 8 and 16 are packed into shared tiles, 32
    # is not
    (4, 2), (8, 2), (16, 2), (32, 2), (16, 1), (32, 1),
]


@pytest.mark.parametrize("pack", [1, 0], ids=["packed", "unpacked"])
@pytest.mark.parametrize("heads", GQA_CASES, ids=[f"H{h}_Hkv{k}" for h, k in GQA_CASES])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_grouped_query_packing(fa, pack, heads, d, causal):
    """Decode and prefill shapes with grouped query heads, with the packing
    of a group's heads into shared tiles on and off: both against the
    oracle (full and partial tiles, several tiles per sequence)."""
    H, H_kv = heads
    lq, lk = [1, 7, 40, 3, 300, 129], [2048, 700, 4000, 3, 300, 517]
    cu_q, cu_k = _offsets(lq), _offsets(lk)
    q, k, v = _inputs(cu_q[-1], cu_k[-1], H, H_kv, d, torch.bfloat16, seed=750 + H + d)
    fa.fa_set_gqa_pack(pack)
    try:
        o, lse = _run(fa, q, k, v, cu_q, cu_k, None, None, causal, (-1, -1), d ** -0.5)
    finally:
        fa.fa_set_gqa_pack(1)
    o_ref, l_ref = oracle.attention_varlen_qk(q, k, v, cu_q, cu_k, d ** -0.5, causal)
    _check(o, lse, o_ref, l_ref, cu_q, None, f"H={H}/{H_kv} d={d} pack={pack}")


def test_gqa_pack_setting_rejects_other_values(fa):
    assert fa.fa_set_gqa_pack(2) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_gqa_pack(-1) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_gqa_pack(1) == fa.FA_OK


# ---------------------------------------------------------------- backward
BWD_REL = 2e-2
BWD_FLOOR = 1e-4
SENTINEL_G = 5.0


def _bwd_case(fa, lens_q, lens_k, H, H_kv, d, causal, window, seed, used_q=None, used_k=None):
    """fa.bwd_varlen_qk against oracle.attention_bwd_qk sequence by sequence,
    on the used rows (a sequence without used queries or keys: its used rows
    of the other side must be exactly 0)."""
    cu_q, cu_k = _offsets(lens_q), _offsets(lens_k)
    total_q, total_k = cu_q[-1], cu_k[-1]
    q, k, v = _inputs(total_q, total_k, H, H_kv, d, torch.bfloat16, seed)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16)
    dev = "cuda"
    t32 = lambda x: None if x is None else torch.tensor(x, dtype=torch.int32, device=dev)  # noqa
    nq = used_q if used_q is not None else lens_q
    nk = used_k if used_k is not None else lens_k
    mq, mk = max(nq), max(nk)
    scale = d ** -0.5
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fwd_varlen_qk(qd, kd, vd, t32(cu_q), t32(cu_k), mq, mk, seqused_q=t32(used_q),
                              seqused_k=t32(used_k), scale=scale, causal=causal, window=window)
    dq, dk, dv = fa.bwd_varlen_qk(qd, kd, vd, o, lse, dod, t32(cu_q), t32(cu_k), mq, mk,
                                  seqused_q=t32(used_q), seqused_k=t32(used_k), scale=scale,
                                  causal=causal, window=window)
    torch.cuda.synchronize()
    st, site = fa.fa_get_device_status(None)
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)} at site {site}"
    dq, dk, dv = (t.float().cpu().numpy() for t in (dq, dk, dv))
    for b in range(len(lens_q)):
        q0, k0 = cu_q[b], cu_k[b]
        if nq[b] == 0 or nk[b] == 0:
            assert (dq[q0:q0 + nq[b]] == 0).all(), f"seq {b}: dQ of rows without keys"
            assert (dk[k0:k0 + nk[b]] == 0).all(), f"seq {b}: dK of keys without queries"
            assert (dv[k0:k0 + nk[b]] == 0).all(), f"seq {b}: dV of keys without queries"
            continue
        vq = lambda t: t[q0:q0 + nq[b]].permute(1, 0, 2).unsqueeze(0).contiguous()  # noqa
        vk = lambda t: t[k0:k0 + nk[b]].permute(1, 0, 2).unsqueeze(0).contiguous()  # noqa
        ref = oracle.attention_bwd_qk(vq(q), vk(k), vk(v), vq(do), scale, causal, *window)
        got = (dq[q0:q0 + nq[b]].transpose(1, 0, 2)[None], dk[k0:k0 + nk[b]].transpose(1, 0, 2)[None],
               dv[k0:k0 + nk[b]].transpose(1, 0, 2)[None])
        # the mask (bottom-right aligned): query rows without a key and keys
        # that no query sees have exactly zero gradients
        pos = np.arange(nq[b])[:, None] + (nk[b] - nq[b])
        j = np.arange(nk[b])[None, :]
        adm = np.ones((nq[b], nk[b]), dtype=bool)
        if causal:
            adm &= j <= pos
        if window[0] >= 0:
            adm &= j >= pos - window[0]
        if window[1] >= 0:
            adm &= j <= pos + window[1]
        idle = {"dQ": ~adm.any(1), "dK": ~adm.any(0), "dV": ~adm.any(0)}
        for name, g_, r in zip(("dQ", "dK", "dV"), got, ref):
            if r.size == 0:
                continue
            assert np.isfinite(g_).all(), f"seq {b} {name}: non-finite"
            err = float(np.abs(g_ - r).max())
            bound = BWD_REL * float(np.abs(r).max()) + BWD_FLOOR
            assert err <= bound, f"seq {b} (nq={nq[b]}, nk={nk[b]}) {name}: {err:.3e} > {bound:.3e}"
            assert (g_[:, :, idle[name]] == 0).all(), f"seq {b} {name}: rows without work must be 0"
    return q, k


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_backward_cross_attention(fa, d, causal):
    """Query and key sequences of different lengths (longer and shorter
    queries, one sequence without queries, a causal case with queries that
    see no key)."""
    _bwd_case(fa, [200, 1, 0, 300, 129], [130, 260, 40, 100, 500], 4, 2, d, causal, (-1, -1),
              seed=900 + d)


@pytest.mark.parametrize("window", [(40, 10), (0, 0), (300, 0)])
def test_backward_cross_attention_windows(fa, window):
    """Windows at bottom-right aligned positions; with a narrow window some
    keys are seen by no query and get dK = dV = 0."""
    _bwd_case(fa, [64, 300, 7], [400, 120, 260], 2, 2, 128, False, window, seed=910)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_backward_used_lengths(fa, causal):
    """Used lengths below the allocated rows (a padded batch): only the used
    rows take part."""
    _bwd_case(fa, [300, 200, 129], [260, 400, 129], 4, 1, 128, causal, (-1, -1), seed=920,
              used_q=[250, 1, 0], used_k=[100, 399, 129])


@pytest.mark.parametrize("ctas", [1, 3])
def test_backward_cross_attention_many_units_per_cta(fa, ctas):
    fa.fa_set_max_ctas(ctas)
    try:
        _bwd_case(fa, [200, 1, 300, 129], [130, 260, 100, 500], 4, 2, 128, True, (-1, -1),
                  seed=930 + ctas)
    finally:
        fa.fa_set_max_ctas(0)


def test_backward_equal_offsets_is_bwd_varlen(fa):
    """One offset array for queries and keys, no used lengths: bit for bit
    the gradients of fa_bwd_varlen."""
    lens = [300, 129, 1, 256]
    cu = _offsets(lens)
    q, k, v = _inputs(cu[-1], cu[-1], 4, 2, 128, torch.bfloat16, 940)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(941)).to(torch.bfloat16)
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    for causal in (False, True):
        o, lse = fa.fwd_varlen(qd, kd, vd, cu_t, max(lens), causal=causal)
        a = fa.bwd_varlen(qd, kd, vd, o, lse, dod, cu_t, max(lens), causal=causal)
        b = fa.bwd_varlen_qk(qd, kd, vd, o, lse, dod, cu_t, cu_t, max(lens), max(lens),
                             causal=causal)
        torch.cuda.synchronize()
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_backward_argument_errors(fa):
    q = torch.zeros(10, 2, 64, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 10], dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    base = [q.data_ptr()] * 9
    # a missing key offset array, a negative total, an over-long length
    assert fa.fa_bwd_varlen_qk(*base, cu.data_ptr(), 0, None, None, 1, 10, 10, 10, 10, 2, 2, 64,
                               0.1, 0, -1, -1, fa.FA_DTYPE_BF16, ws.data_ptr(), ws.numel(),
                               None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_varlen_qk(*base, cu.data_ptr(), cu.data_ptr(), None, None, 1, 10, 10, 10,
                               -1, 2, 2, 64, 0.1, 0, -1, -1, fa.FA_DTYPE_BF16, ws.data_ptr(),
                               ws.numel(), None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_varlen_qk(*base, cu.data_ptr(), cu.data_ptr(), None, None, 1, 10, 1 << 30,
                               10, 10, 2, 2, 64, 0.1, 0, -1, -1, fa.FA_DTYPE_BF16, ws.data_ptr(),
                               ws.numel(), None) == fa.FA_ERR_INVALID_ARG
    # nothing to do
    assert fa.fa_bwd_varlen_qk(*base, cu.data_ptr(), cu.data_ptr(), None, None, 0, 10, 10, 10,
                               10, 2, 2, 64, 0.1, 0, -1, -1, fa.FA_DTYPE_BF16, ws.data_ptr(),
                               ws.numel(), None) == fa.FA_OK
