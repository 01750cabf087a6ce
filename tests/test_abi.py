"""Host-only checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments with the documented status codes before
touching the GPU.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def fa():
    from attention_forward_10_gb300 import build
    build.build()
    import attention_forward_10_gb300 as fa_mod
    return fa_mod


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for n in ("fa_fwd", "fa_fwd_ext", "fa_status_string", "fa_get_device_status",
              "fa_set_wait_timeout_us", "fa_set_max_ctas", "fa_selftest_watchdog",
              "fa_num_sms"):
        assert n in names


def test_library_exports_every_declared_symbol(fa):
    lib = ctypes.CDLL(fa.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in fa.h but not exported"
    assert set(_declared_functions()) == set(fa.SIGNATURES)


def test_status_strings(fa):
    assert fa.fa_status_string(fa.FA_OK) == "FA_OK"
    assert fa.fa_status_string(fa.FA_ERR_MISALIGNED) == "FA_ERR_MISALIGNED"
    assert fa.fa_status_string(fa.FA_ERR_DEVICE_TIMEOUT) == "FA_ERR_DEVICE_TIMEOUT"
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


GOOD = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=2, N=256, d=128,
            scale=0.088, causal=0, dtype=1, stream=None)


def _call(fa, **kw):
    a = dict(GOOD)
    a.update(kw)
    return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                     a["d"], a["scale"], a["causal"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), 1), (dict(H=-3), 1), (dict(N=-1), 1),
    (dict(dtype=2), 1), (dict(dtype=-1), 1),
    (dict(causal=2), 1),
    (dict(scale=0.0), 1), (dict(scale=-0.5), 1), (dict(scale=float("nan")), 1),
    (dict(scale=float("inf")), 1),
    (dict(d=32), 2), (dict(d=96), 2), (dict(d=512), 2), (dict(d=0), 2),
    (dict(q=0), 1), (dict(k=0), 1), (dict(v=0), 1), (dict(o=0), 1),
    (dict(q=0x1008), 3), (dict(k=0x2004), 3), (dict(v=0x3002), 3), (dict(o=0x4001), 3),
    (dict(lse=0x5002), 3),
    (dict(B=1 << 16, H=1 << 16), 1),
])
def test_argument_errors(fa, kw, code):
    assert _call(fa, **kw) == code


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(N=0),
                                dict(N=0, q=0, k=0, v=0, o=0, lse=0)])
def test_empty_problem_is_a_noop(fa, kw):
    assert _call(fa, **kw) == fa.FA_OK


def test_setters_validate(fa):
    assert fa.fa_set_wait_timeout_us(0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_wait_timeout_us(2_000_000) == fa.FA_OK
    assert fa.fa_set_max_ctas(-1) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_max_ctas(0) == fa.FA_OK
    assert fa.fa_selftest_watchdog(0, None) == fa.FA_ERR_INVALID_ARG


def test_fwd_wrapper_rejects_cpu_tensors(fa):
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd(q, q, q)


def test_product_does_not_import_oracle():
    """The product package shares no code with the oracle."""
    pkg = os.path.join(ROOT, "attention_forward_10_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "attn_ref" not in text, f


def _call_ext(fa, H=4, H_kv=2, **kw):
    a = dict(GOOD)
    a.update(kw)
    return fa.fa_fwd_ext(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], H, H_kv, a["N"],
                         a["d"], a["scale"], a["causal"], -1, -1, a["dtype"], a["stream"])


@pytest.mark.parametrize("H,H_kv,code", [(4, 3, 1), (4, 0, 1), (4, -1, 1), (6, 4, 1),
                                         (4, 8, 1)])
def test_ext_head_grouping_errors(fa, H, H_kv, code):
    assert _call_ext(fa, H=H, H_kv=H_kv) == code


def test_ext_empty_is_noop(fa):
    assert _call_ext(fa, H=4, H_kv=2, N=0) == fa.FA_OK


# ------------------------------------------------------------- split-KV
def _ws_bytes(fa, B=1, H=2, N=1024, d=128, S=4):
    st, n = fa.fa_splitkv_workspace_bytes(B, H, N, d, 0, -1, -1, S)
    assert st == fa.FA_OK
    return n


def test_splitkv_workspace_size(fa):
    # 4 splits of 1024 keys (8 tiles of 128 -> 2 tiles each): 16-bit O
    # partials, then fp32 LSE partials at a 256-byte boundary
    assert _ws_bytes(fa) == 4 * 2 * 1024 * 128 * 2 + 4 * 2 * 1024 * 4
    # 3 splits of 8 tiles: 3 tiles per split -> still 3 splits
    assert _ws_bytes(fa, S=3) == 3 * 2 * 1024 * 128 * 2 + 3 * 2 * 1024 * 4
    # 7 requested of 8 tiles: 2 tiles per split -> 4 splits used
    assert _ws_bytes(fa, S=7) == _ws_bytes(fa, S=4)
    # more splits than tiles: one tile each
    assert _ws_bytes(fa, S=100) == _ws_bytes(fa, S=8)
    # d = 256 cuts 64-key tiles: 16 of them at N = 1024
    assert _ws_bytes(fa, d=256, S=16) == 16 * 2 * 1024 * 256 * 2 + 16 * 2 * 1024 * 4
    # odd sizes: the LSE part starts on a 256-byte boundary
    o_bytes = 2 * 1 * 3 * 200 * 64 * 2
    assert _ws_bytes(fa, B=1, H=3, N=200, d=64, S=2) == ((o_bytes + 255) // 256) * 256 \
        + 2 * 3 * 200 * 4
    # one split, or nothing to do: no workspace
    assert _ws_bytes(fa, S=1) == 0
    assert _ws_bytes(fa, N=100, S=4) == 0   # a single K/V tile
    assert _ws_bytes(fa, N=0, S=4) == 0


@pytest.mark.parametrize("args,code", [
    ((1, 2, 1024, 128, 0, -1, -1, -1), 1), ((-1, 2, 1024, 128, 0, -1, -1, 2), 1),
    ((1, 2, 1024, 96, 0, -1, -1, 2), 2), ((1, 2, 1024, 128, 2, -1, -1, 2), 1)])
def test_splitkv_workspace_size_errors(fa, args, code):
    assert fa.fa_splitkv_workspace_bytes(*args)[0] == code


def _call_split(fa, S=4, ws=0x100000, ws_bytes=None, **kw):
    a = dict(GOOD, N=1024, H=2)
    a.update(kw)
    if ws_bytes is None:
        ws_bytes = _ws_bytes(fa, a["B"], a["H"], a["N"], a["d"], S)
    return fa.fa_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                             a.get("H_kv", a["H"]), a["N"], a["d"], a["scale"], a["causal"],
                             -1, -1, a["dtype"], S, ws, ws_bytes, a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(S=-2, ws_bytes=1 << 30), 1),
    (dict(ws=0), 1),                     # splits used > 1 but no workspace
    (dict(ws_bytes=1024), 1),            # too small
    (dict(ws=0x100010), 3),              # not 256-byte aligned
    (dict(H_kv=3), 1), (dict(d=32, ws_bytes=1 << 30), 2), (dict(q=0x1008), 3),
    (dict(scale=0.0), 1),
])
def test_splitkv_argument_errors(fa, kw, code):
    assert _call_split(fa, **kw) == code


def test_splitkv_empty_is_noop(fa):
    assert _call_split(fa, N=0, ws=0, ws_bytes=0) == fa.FA_OK


# ----------------------------------------------- split-KV, fixed scratch
def _call_noalloc(fa, S, **kw):
    a = dict(GOOD, N=8192, H=8)
    a.update(kw)
    return fa.fa_fwd_splitkv_noalloc(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"],
                                     a["H"], a["H"], a["N"], a["d"], a["scale"], a["causal"],
                                     -1, -1, a["dtype"], S, a["stream"])


def test_noalloc_rejects_partials_beyond_the_scratch(fa):
    assert fa.fa_status_string(fa.FA_ERR_SCRATCH_LIMIT) == "FA_ERR_SCRATCH_LIMIT"
    # 8 splits of 8 heads x 8192 rows x (256 + 4) bytes = 136 MB > 32 MiB
    st, need = fa.fa_splitkv_workspace_bytes(1, 8, 8192, 128, 0, -1, -1, 8)
    assert st == fa.FA_OK and need > fa.FA_NOALLOC_SCRATCH_BYTES
    assert _call_noalloc(fa, 8) == fa.FA_ERR_SCRATCH_LIMIT


@pytest.mark.parametrize("kw,code", [(dict(S=-1), 1), (dict(S=2, d=32), 2),
                                     (dict(S=2, o=0x4001), 3), (dict(S=2, N=0), 0)])
def test_noalloc_argument_errors(fa, kw, code):
    S = kw.pop("S")
    assert _call_noalloc(fa, S, **kw) == code


# --------------------------------------------------- packed (varlen) batches
def _call_varlen(fa, cu=0x6000, batch=2, max_seqlen=300, total=500, H=4, H_kv=2, **kw):
    a = dict(GOOD)
    a.update(kw)
    return fa.fa_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], cu, batch, max_seqlen,
                            total, H, H_kv, a["d"], a["scale"], a["causal"], -1, -1,
                            a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(cu=0), 1), (dict(cu=0x6002), 3), (dict(total=-1), 1), (dict(batch=-1), 1),
    (dict(max_seqlen=-5), 1), (dict(H=4, H_kv=3), 1), (dict(d=96), 2), (dict(q=0x1008), 3),
    (dict(scale=float("nan")), 1),
])
def test_varlen_argument_errors(fa, kw, code):
    assert _call_varlen(fa, **kw) == code


@pytest.mark.parametrize("kw", [dict(batch=0), dict(total=0), dict(max_seqlen=0),
                                dict(batch=0, cu=0, q=0, k=0, v=0, o=0)])
def test_varlen_empty_is_noop(fa, kw):
    assert _call_varlen(fa, **kw) == fa.FA_OK


# ---------------------------------------------------------------- backward
def _call_bwd(fa, ws=0x100000, ws_bytes=1 << 30, **kw):
    a = dict(GOOD, H=2)
    a.update(kw)
    return fa.fa_bwd(a["q"], a["k"], a["v"], a.get("o", 0x7000), a.get("lse_", 0x8000),
                     a.get("do", 0x9000), a.get("dq", 0xA000), a.get("dk", 0xB000),
                     a.get("dv", 0xC000), ws, ws_bytes, a["B"], a["H"], a.get("H_kv", a["H"]),
                     a["N"], a["d"], a["scale"], a["causal"], -1, -1, a["dtype"], a["stream"])


def test_bwd_workspace_size(fa):
    st, n = fa.fa_bwd_workspace_bytes(2, 3, 300)
    assert st == fa.FA_OK and n == 2 * 2 * 3 * 384 * 4
    assert fa.fa_bwd_workspace_bytes(-1, 3, 300)[0] == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    (dict(d=256), 2), (dict(d=32), 2), (dict(ws=0), 1), (dict(ws_bytes=64), 1),
    (dict(ws=0x100010), 3), (dict(do=0), 1), (dict(o=0x7008), 3), (dict(lse_=0x8002), 3),
    (dict(dk=0xB004), 3), (dict(H_kv=3), 1), (dict(causal=3), 1),
])
def test_bwd_argument_errors(fa, kw, code):
    assert _call_bwd(fa, **kw) == code


def test_bwd_empty_is_noop(fa):
    assert _call_bwd(fa, N=0, ws=0, ws_bytes=0) == fa.FA_OK


# -------------------------------------------------------------------- FP8
def _call_fp8(fa, ws=0x100000, ws_bytes=1 << 30, dq=1.0, dk=1.0, dv=1.0, **kw):
    a = dict(GOOD, H=2)
    a.update(kw)
    return fa.fa_fwd_fp8(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                         a.get("H_kv", a["H"]), a["N"], a["d"], a["scale"], dq, dk, dv,
                         a["causal"], -1, -1, ws, ws_bytes, a["stream"])


def test_fp8_workspace_size(fa):
    st, n = fa.fa_fwd_fp8_workspace_bytes(2, 3, 300, 128)
    assert st == fa.FA_OK and n == 2 * 3 * 128 * 384
    assert fa.fa_fwd_fp8_workspace_bytes(2, 3, 300, 64)[0] == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), 2), (dict(d=256), 2), (dict(ws=0), 1), (dict(ws_bytes=16), 1),
    (dict(ws=0x100080), 3), (dict(dq=0.0), 1), (dict(dk=float("nan")), 1), (dict(dv=-1.0), 1),
    (dict(q=0x1008), 3), (dict(H_kv=3), 1),
])
def test_fp8_argument_errors(fa, kw, code):
    assert _call_fp8(fa, **kw) == code


def test_fp8_empty_is_noop(fa):
    assert _call_fp8(fa, N=0, ws=0, ws_bytes=0) == fa.FA_OK


def test_bwd_varlen_argument_errors(fa):
    args = dict(q=0x1000, k=0x2000, v=0x3000, o=0x7000, lse=0x8000, do=0x9000, dq=0xA000,
                dk=0xB000, dv=0xC000)
    base = [args[n] for n in ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv")]
    call = lambda cu, batch=2, ms=300, total=500, H=4, H_kv=2, d=128, ws=0x100000: \
        fa.fa_bwd_varlen(*base, cu, batch, ms, total, H, H_kv, d, 0.1, 0, -1, -1, 1, ws,
                         1 << 30, None)
    assert call(0) == fa.FA_ERR_INVALID_ARG              # no offsets
    assert call(0x6002) == fa.FA_ERR_MISALIGNED          # misaligned offsets
    assert call(0x6000, d=256) == fa.FA_ERR_UNSUPPORTED
    assert call(0x6000, H_kv=3) == fa.FA_ERR_INVALID_ARG
    assert call(0x6000, total=-1) == fa.FA_ERR_INVALID_ARG
    assert call(0x6000, ws=0x100010) == fa.FA_ERR_MISALIGNED
    assert call(0x6000, total=0) == fa.FA_OK             # empty
    assert call(0, batch=0) == fa.FA_OK


# ------------------------------------------------------------ host buffers
HOST = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=4, H_kv=2, N=512,
            d=128, scale=0.088, causal=0, wl=-1, wr=-1, dtype=1, ws=0x100000,
            ws_bytes=1 << 30, stream=None)


def _host(fa, **kw):
    a = dict(HOST)
    a.update(kw)
    return fa.fa_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["H_kv"],
                          a["N"], a["d"], a["scale"], a["causal"], a["wl"], a["wr"], a["dtype"],
                          a["ws"], a["ws_bytes"], a["stream"])


def _host_plan_bytes(B, H, H_kv, N, d, with_lse):
    """The documented default plan, restated: chunks of whole K/V-head
    groups, about 8 of them and each at least 4 MiB of input, up to 3
    staging slots; per slot Q, O, K, V (and LSE) each rounded up to 256 B."""
    a256 = lambda x: (x + 255) // 256 * 256
    groups, grp = B * H_kv, H // H_kv
    in_per_group = (grp + 2) * N * d * 2
    per = max(-(-groups // 8), -(-(4 << 20) // in_per_group))
    per = min(per, groups)
    chunks = -(-groups // per)
    slot = 2 * a256(per * grp * N * d * 2) + 2 * a256(per * N * d * 2) + \
        (a256(per * grp * N * 4) if with_lse else 0)
    return min(3, chunks) * slot


@pytest.mark.parametrize("shape", [(4, 16, 16, 2048, 128), (1, 7, 7, 128, 128),
                                   (2, 8, 2, 4096, 64), (1, 32, 32, 32768, 128),
                                   (3, 6, 1, 1000, 256), (1, 1, 1, 1, 64)])
@pytest.mark.parametrize("with_lse", [0, 1])
def test_host_workspace_size(fa, shape, with_lse):
    st, n = fa.fa_fwd_host_workspace_bytes(*shape, with_lse)
    assert st == fa.FA_OK
    assert n == _host_plan_bytes(*shape, with_lse)


@pytest.mark.parametrize("args,code", [
    ((1, 3, 2, 10, 128, 1), 1), ((1, 2, 2, 10, 96, 1), 2), ((-1, 2, 2, 10, 128, 1), 1),
    ((1, 2, 2, 10, 128, 2), 1)])
def test_host_workspace_size_errors(fa, args, code):
    assert fa.fa_fwd_host_workspace_bytes(*args)[0] == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(o=None), 1),
    (dict(ws=None), 1), (dict(d=96), 2), (dict(H=3), 1), (dict(scale=0.0), 1),
    (dict(causal=2), 1), (dict(dtype=5), 1), (dict(wl=-2), 1), (dict(wr=-7), 1),
    (dict(ws=0x100010), 3), (dict(ws_bytes=1024), 1)])
def test_host_argument_errors(fa, kw, code):
    assert _host(fa, **kw) == code


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0, H_kv=1), dict(N=0)])
def test_host_empty_is_noop(fa, kw):
    assert _host(fa, q=None, k=None, v=None, o=None, lse=None, ws=None, **kw) == fa.FA_OK


def test_host_wrapper_rejects_cuda_tensors(fa):
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd_host(q, q, q.to("meta"))
