"""C-ABI library checks that need no GPU.

The library must load, export every function include/saw_int4.h declares,
and reject bad arguments on the host before anything is launched.  Every
call below carries exactly one invalid argument that the host checks catch,
so no kernel is ever launched with these made-up pointers.
"""
import ctypes as C
import os
import re

import pytest

import bit_paged_kv_gb300 as saw
from bit_paged_kv_gb300 import build as saw_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "saw_int4.h")

A = 0x10000   # a 16-byte-aligned made-up address (never dereferenced)
B = 0x20000
MIS = 0x10008  # 8-byte aligned only


@pytest.fixture(scope="module")
def L():
    saw_build.build()
    return saw.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(saw_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert set(names) == set(saw.EXPORTS)
    for n in names:
        assert hasattr(L, n), n
    # the binding module exposes the same names
    for n in names:
        assert callable(getattr(saw, n))


def test_status_strings(L):
    for code, name in [(0, "SAW_OK"), (1, "SAW_ERR_INVALID_ARG"), (2, "SAW_ERR_UNSUPPORTED"),
                       (3, "SAW_ERR_CUDA"), (4, "SAW_ERR_DEVICE_INDEX"),
                       (5, "SAW_ERR_DEVICE_TIMEOUT"), (99, "SAW_ERR_UNKNOWN")]:
        assert saw.saw_status_string(code) == name


def test_cache_bytes(L):
    assert saw.saw_cache_bytes(1, 16, 1, 128) == 16 * 64 + 16 * 4 == 1088
    assert saw.saw_cache_bytes(2048, 16, 8, 128) == 2048 * 8 * 1088
    assert saw.saw_cache_bytes(10, 64, 8, 128) == 10 * 8 * 4352
    assert saw.saw_cache_bytes(0, 16, 8, 128) == 0
    assert saw.saw_cache_bytes(4, 16, -1, 128) == 0


def _append(L, **kw):
    a = dict(k=A, v=B, ks=1024, vs=1024, slots=A, T=4, hkv=8, d=128, kc=A, vc=B, pages=4, P=16,
             rk=1, rv=1, h=128, status=None, stream=None)
    a.update(kw)
    return L.saw_quantize_append(a["k"], a["v"], a["ks"], a["vs"], a["slots"], a["T"], a["hkv"],
                                 a["d"], a["kc"], a["vc"], a["pages"], a["P"], a["rk"], a["rv"],
                                 a["h"], a["status"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(d=96), saw.SAW_ERR_UNSUPPORTED),   # head_dim 64, 128, 256 only
    (dict(P=8), saw.SAW_ERR_UNSUPPORTED),
    (dict(h=3), saw.SAW_ERR_INVALID_ARG),
    (dict(h=256), saw.SAW_ERR_INVALID_ARG),
    (dict(h=8), saw.SAW_ERR_UNSUPPORTED),
    (dict(rk=2), saw.SAW_ERR_INVALID_ARG),
    (dict(k=None), saw.SAW_ERR_INVALID_ARG),
    (dict(slots=None), saw.SAW_ERR_INVALID_ARG),
    (dict(kc=None), saw.SAW_ERR_INVALID_ARG),
    (dict(vc=None), saw.SAW_ERR_INVALID_ARG),
    (dict(k=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(kc=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(ks=1000), saw.SAW_ERR_INVALID_ARG),
    (dict(vs=1020), saw.SAW_ERR_INVALID_ARG),
    (dict(T=-1), saw.SAW_ERR_INVALID_ARG),
    (dict(hkv=0), saw.SAW_ERR_INVALID_ARG),
    (dict(T=0), saw.SAW_OK),  # nothing to do: returns before any launch
])
def test_append_rejects_before_launch(L, kw, expect):
    assert _append(L, **kw) == expect


def _decode(L, **kw):
    a = dict(q=A, kc=A, vc=B, bt=A, mb=4, sl=B, B=2, maxlen=64, hq=32, hkv=8, d=128, pages=8,
             P=16, rk=1, rv=1, h=128, scale=0.0, out=A, ws=B, wsb=1 << 20, pps=0, status=None,
             stream=None)
    a.update(kw)
    return L.saw_paged_decode_int4(a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["sl"], a["B"],
                                   a["maxlen"], a["hq"], a["hkv"], a["d"], a["pages"], a["P"],
                                   a["rk"], a["rv"], a["h"], a["scale"], a["out"], a["ws"],
                                   a["wsb"], a["pps"], a["status"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(d=96), saw.SAW_ERR_UNSUPPORTED),
    (dict(P=128), saw.SAW_ERR_UNSUPPORTED),
    (dict(hq=12), saw.SAW_ERR_INVALID_ARG),
    (dict(hq=72), saw.SAW_ERR_UNSUPPORTED),        # 9 q-heads per kv-head
    (dict(h=48), saw.SAW_ERR_INVALID_ARG),
    (dict(rv=-1), saw.SAW_ERR_INVALID_ARG),
    (dict(scale=-1.0), saw.SAW_ERR_INVALID_ARG),
    (dict(scale=float("nan")), saw.SAW_ERR_INVALID_ARG),
    (dict(q=None), saw.SAW_ERR_INVALID_ARG),
    (dict(bt=None), saw.SAW_ERR_INVALID_ARG),
    (dict(sl=None), saw.SAW_ERR_INVALID_ARG),
    (dict(out=None), saw.SAW_ERR_INVALID_ARG),
    (dict(kc=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(out=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(mb=3), saw.SAW_ERR_INVALID_ARG),           # 3 * 16 < 64 tokens
    (dict(pps=1, ws=None), saw.SAW_ERR_INVALID_ARG),  # 4 splits need a workspace
    (dict(pps=1, wsb=16), saw.SAW_ERR_INVALID_ARG),
    (dict(pps=1, ws=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(B=-1), saw.SAW_ERR_INVALID_ARG),
    (dict(B=0), saw.SAW_OK),
])
def test_decode_rejects_before_launch(L, kw, expect):
    assert _decode(L, **kw) == expect


def test_plan_and_workspace(L):
    # forced split size: 4 pages of 16 tokens -> ceil(1000/16)=63 pages -> 16 splits
    s, pps = saw.saw_decode_plan(2, 8, 16, 1000, 4)
    assert (s, pps) == (16, 4)
    ws = saw.saw_decode_workspace_bytes(2, 32, 8, 128, 16, 1000, 4)
    # two counter words per (sequence, kv-head), rounded to 16 bytes, then partials
    assert ws == 2 * 8 * 8 + 2 * 32 * 16 * (128 + 2) * 4
    # one split -> no workspace
    assert saw.saw_decode_workspace_bytes(2, 32, 8, 128, 16, 64, 64) == 0
    # automatic plan: splits never shorter than 256 tokens, and cover the context
    s, pps = saw.saw_decode_plan(1, 8, 16, 32768, 0)
    assert pps * 16 >= 256 and s * pps * 16 >= 32768
    s, pps = saw.saw_decode_plan(256, 8, 16, 8192, 0)
    assert s * pps * 16 >= 8192
    assert saw.saw_decode_plan(1, 8, 64, 0, 0) == (1, 1)
    # many units (enough to fill every CTA slot unsplit on any GPU this targets):
    # splits of at least 4096 tokens, still covering the context
    for B, L_ in [(256, 8192), (128, 16384), (512, 32768)]:
        s, pps = saw.saw_decode_plan(B, 8, 16, L_, 0)
        assert pps * 16 >= min(4096, L_) and s * pps * 16 >= L_
    # few units: splits may go down to 1024 tokens to reach every SM
    s, pps = saw.saw_decode_plan(1, 8, 16, 32768, 0)
    assert 1024 <= pps * 16 < 4096 and s > 8
    # the workspace of an automatic head_dim-128 plan is that plan's partials
    w128 = saw.saw_decode_workspace_bytes(64, 32, 8, 128, 16, 16384, 0)
    s128, _ = saw.saw_decode_plan(64, 8, 16, 16384, 0)
    assert s128 > 1 and w128 == (64 * 8 * 8 + 15) // 16 * 16 + 64 * 32 * s128 * (128 + 2) * 4
    with pytest.raises(saw.SawError):
        saw.saw_decode_plan(1, 8, 12, 100, 0)
    # automatic splits are whole turns of the warps: a multiple of one 16-token
    # tile per warp of the chosen CTA shape (4, 8 or 16 warps), 16 for the
    # one-wave batch-1 plan
    for B, P, L_ in [(1, 16, 32768), (4, 16, 32768), (64, 16, 16384), (8, 64, 131072),
                     (1, 32, 65536), (256, 16, 8192)]:
        s, pps = saw.saw_decode_plan(B, 8, P, L_, 0)
        if s > 1:
            assert (pps * (P // 16)) % 4 == 0, (B, P, L_, s, pps)
    s, pps = saw.saw_decode_plan(1, 8, 16, 32768, 0)
    assert pps % 16 == 0 and s * pps * 16 >= 32768


def _step(L, **kw):
    a = dict(q=A, kn=B, vn=A, kc=A, vc=B, bt=A, mb=4, sl=B, B=2, maxlen=64, hq=32, hkv=8, d=128,
             pages=8, P=16, rk=1, rv=0, h=128, scale=0.0, out=A, ws=B, wsb=1 << 20, pps=0,
             flags=0, status=None, stream=None)
    a.update(kw)
    return L.saw_decode_step(a["q"], a["kn"], a["vn"], a["kc"], a["vc"], a["bt"], a["mb"],
                             a["sl"], a["B"], a["maxlen"], a["hq"], a["hkv"], a["d"], a["pages"],
                             a["P"], a["rk"], a["rv"], a["h"], a["scale"], a["out"], a["ws"],
                             a["wsb"], a["pps"], a["flags"], a["status"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(kn=None), saw.SAW_ERR_INVALID_ARG),
    (dict(vn=None), saw.SAW_ERR_INVALID_ARG),
    (dict(kn=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(kc=None), saw.SAW_ERR_INVALID_ARG),
    (dict(d=64), saw.SAW_ERR_UNSUPPORTED),
    (dict(hq=12), saw.SAW_ERR_INVALID_ARG),
    (dict(mb=3), saw.SAW_ERR_INVALID_ARG),
    (dict(flags=2), saw.SAW_ERR_INVALID_ARG),
    (dict(B=0), saw.SAW_OK),
])
def test_decode_step_rejects_before_launch(L, kw, expect):
    assert _step(L, **kw) == expect


def test_bf16_cache_bytes(L):
    assert saw.saw_bf16_cache_bytes(1, 16, 1, 128) == 16 * 128 * 2
    assert saw.saw_bf16_cache_bytes(10, 64, 8, 128) == 10 * 8 * 64 * 256
    assert saw.saw_bf16_cache_bytes(0, 16, 8, 128) == 0
    assert saw.saw_bf16_cache_bytes(4, 16, -1, 128) == 0


def _bf16_append(L, **kw):
    a = dict(k=A, v=B, ks=1024, vs=1024, slots=A, T=4, hkv=8, d=128, kc=A, vc=B, pages=8, P=16,
             status=None, stream=None)
    a.update(kw)
    return L.saw_bf16_append(a["k"], a["v"], a["ks"], a["vs"], a["slots"], a["T"], a["hkv"],
                             a["d"], a["kc"], a["vc"], a["pages"], a["P"], a["status"],
                             a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(d=64), saw.SAW_ERR_UNSUPPORTED),
    (dict(P=8), saw.SAW_ERR_UNSUPPORTED),
    (dict(T=-1), saw.SAW_ERR_INVALID_ARG),
    (dict(hkv=0), saw.SAW_ERR_INVALID_ARG),
    (dict(k=None), saw.SAW_ERR_INVALID_ARG),
    (dict(slots=None), saw.SAW_ERR_INVALID_ARG),
    (dict(vc=None), saw.SAW_ERR_INVALID_ARG),
    (dict(k=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(kc=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(ks=1000), saw.SAW_ERR_INVALID_ARG),     # shorter than Hkv * D
    (dict(vs=1028), saw.SAW_ERR_INVALID_ARG),     # not a multiple of 8
    (dict(T=0), saw.SAW_OK),
])
def test_bf16_append_rejects_before_launch(L, kw, expect):
    assert _bf16_append(L, **kw) == expect


def _bf16_decode(L, **kw):
    a = dict(q=A, kc=A, vc=B, bt=A, mb=512, sl=B, B=2, maxlen=8192, hq=32, hkv=8, d=128,
             pages=1024, P=16, scale=0.0, out=A, ws=B, wsb=1 << 24, status=None, stream=None)
    a.update(kw)
    return L.saw_paged_decode_bf16(a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["sl"], a["B"],
                                   a["maxlen"], a["hq"], a["hkv"], a["d"], a["pages"], a["P"],
                                   a["scale"], a["out"], a["ws"], a["wsb"], a["status"],
                                   a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(d=256), saw.SAW_ERR_UNSUPPORTED),
    (dict(P=128), saw.SAW_ERR_UNSUPPORTED),
    (dict(hq=12), saw.SAW_ERR_INVALID_ARG),
    (dict(hq=72), saw.SAW_ERR_UNSUPPORTED),
    (dict(scale=-1.0), saw.SAW_ERR_INVALID_ARG),
    (dict(scale=float("inf")), saw.SAW_ERR_INVALID_ARG),
    (dict(q=None), saw.SAW_ERR_INVALID_ARG),
    (dict(out=None), saw.SAW_ERR_INVALID_ARG),
    (dict(vc=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(mb=511), saw.SAW_ERR_INVALID_ARG),         # 511 * 16 < 8192 tokens
    (dict(ws=None), saw.SAW_ERR_INVALID_ARG),        # several splits need a workspace
    (dict(wsb=16), saw.SAW_ERR_INVALID_ARG),
    (dict(ws=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(B=-1), saw.SAW_ERR_INVALID_ARG),
    (dict(B=0), saw.SAW_OK),
])
def test_bf16_decode_rejects_before_launch(L, kw, expect):
    assert _bf16_decode(L, **kw) == expect


def test_bf16_workspace(L):
    # several splits at 8192 tokens: counters + partials per (seq, q-head, split)
    ws = saw.saw_decode_bf16_workspace_bytes(2, 32, 8, 128, 16, 8192)
    assert ws > 0 and (ws - 2 * 8 * 8) % (2 * 32 * (128 + 2) * 4) == 0
    splits = (ws - 2 * 8 * 8) // (2 * 32 * (128 + 2) * 4)
    assert 2 <= splits <= 8   # at least 1024 tokens per split
    # one split (short context) needs none
    assert saw.saw_decode_bf16_workspace_bytes(2, 32, 8, 128, 16, 512) == 0
    assert saw.saw_decode_bf16_workspace_bytes(2, 32, 8, 64, 16, 8192) == 0


def _prefill(L, **kw):
    a = dict(q=A, cu=B, kc=A, vc=B, bt=A, mb=64, sl=B, B=2, T=100, mq=64, maxlen=1024, hq=32,
             hkv=8, d=128, pages=128, P=16, rk=1, rv=1, h=128, scale=0.0, out=A, status=None,
             stream=None)
    a.update(kw)
    return L.saw_prefill_attn_int4(a["q"], a["cu"], a["kc"], a["vc"], a["bt"], a["mb"], a["sl"],
                                   a["B"], a["T"], a["mq"], a["maxlen"], a["hq"], a["hkv"],
                                   a["d"], a["pages"], a["P"], a["rk"], a["rv"], a["h"],
                                   a["scale"], a["out"], a["status"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(d=64), saw.SAW_ERR_UNSUPPORTED),
    (dict(P=8), saw.SAW_ERR_UNSUPPORTED),
    (dict(hq=12), saw.SAW_ERR_INVALID_ARG),
    (dict(h=48), saw.SAW_ERR_INVALID_ARG),
    (dict(rk=2), saw.SAW_ERR_INVALID_ARG),
    (dict(scale=-1.0), saw.SAW_ERR_INVALID_ARG),
    (dict(mq=2048), saw.SAW_ERR_INVALID_ARG),        # max_q_len above max_seq_len
    (dict(T=-1), saw.SAW_ERR_INVALID_ARG),
    (dict(q=None), saw.SAW_ERR_INVALID_ARG),
    (dict(cu=None), saw.SAW_ERR_INVALID_ARG),
    (dict(out=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(kc=MIS), saw.SAW_ERR_INVALID_ARG),
    (dict(mb=63), saw.SAW_ERR_INVALID_ARG),           # 63 * 16 < 1024 tokens
    (dict(B=0), saw.SAW_OK),
    (dict(T=0), saw.SAW_OK),
])
def test_prefill_rejects_before_launch(L, kw, expect):
    assert _prefill(L, **kw) == expect


# ---------------------------------------------------------------- format variants (*_ex)

def _append_ex(L, fmt, **kw):
    a = dict(k=A, v=B, ks=1024, vs=1024, slots=A, T=4, hkv=8, d=128, kc=A, vc=B, pages=4, P=16,
             rk=1, rv=1, h=128, status=None, stream=None)
    a.update(kw)
    return L.saw_quantize_append_ex(a["k"], a["v"], a["ks"], a["vs"], a["slots"], a["T"],
                                    a["hkv"], a["d"], a["kc"], a["vc"], a["pages"], a["P"],
                                    a["rk"], a["rv"], a["h"], fmt, a["status"], a["stream"])


def _decode_ex(L, fmt, **kw):
    a = dict(q=A, kc=A, vc=B, bt=A, mb=4, sl=B, B=2, maxlen=64, hq=32, hkv=8, d=128, pages=8,
             P=16, rk=1, rv=1, h=128, scale=0.0, out=A, ws=B, wsb=1 << 20, pps=0, status=None,
             stream=None)
    a.update(kw)
    return L.saw_paged_decode_int4_ex(a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["sl"],
                                      a["B"], a["maxlen"], a["hq"], a["hkv"], a["d"], a["pages"],
                                      a["P"], a["rk"], a["rv"], a["h"], a["scale"], a["out"],
                                      a["ws"], a["wsb"], a["pps"], fmt, a["status"], a["stream"])


def _step_ex(L, fmt, **kw):
    a = dict(q=A, kn=A, vn=B, kc=A, vc=B, bt=A, mb=4, sl=B, B=2, maxlen=64, hq=32, hkv=8, d=128,
             pages=8, P=16, rk=1, rv=1, h=128, scale=0.0, out=A, ws=B, wsb=1 << 20, pps=0,
             flags=0, status=None, stream=None)
    a.update(kw)
    return L.saw_decode_step_ex(a["q"], a["kn"], a["vn"], a["kc"], a["vc"], a["bt"], a["mb"],
                                a["sl"], a["B"], a["maxlen"], a["hq"], a["hkv"], a["d"],
                                a["pages"], a["P"], a["rk"], a["rv"], a["h"], a["scale"],
                                a["out"], a["ws"], a["wsb"], a["pps"], a["flags"], fmt,
                                a["status"], a["stream"])


def _prefill_ex(L, fmt, **kw):
    a = dict(q=A, cu=B, kc=A, vc=B, bt=A, mb=64, sl=B, B=2, T=100, mq=64, maxlen=1024, hq=32,
             hkv=8, d=128, pages=128, P=16, rk=1, rv=1, h=128, scale=0.0, out=A, status=None,
             stream=None)
    a.update(kw)
    return L.saw_prefill_attn_int4_ex(a["q"], a["cu"], a["kc"], a["vc"], a["bt"], a["mb"],
                                      a["sl"], a["B"], a["T"], a["mq"], a["maxlen"], a["hq"],
                                      a["hkv"], a["d"], a["pages"], a["P"], a["rk"], a["rv"],
                                      a["h"], a["scale"], a["out"], fmt, a["status"], a["stream"])


def _noalloc_ex(L, fmt, **kw):
    a = dict(q=A, kc=A, vc=B, bt=A, mb=4, sl=B, B=2, maxlen=64, hq=32, hkv=8, d=128, pages=8,
             P=16, rk=1, rv=1, h=128, scale=0.0, out=A, pps=0, status=None, stream=None)
    a.update(kw)
    return L.saw_paged_decode_int4_noalloc_ex(a["q"], a["kc"], a["vc"], a["bt"], a["mb"],
                                              a["sl"], a["B"], a["maxlen"], a["hq"], a["hkv"],
                                              a["d"], a["pages"], a["P"], a["rk"], a["rv"],
                                              a["h"], a["scale"], a["out"], a["pps"], fmt,
                                              a["status"], a["stream"])


EX_CALLS = [_append_ex, _decode_ex, _step_ex, _prefill_ex]


@pytest.mark.parametrize("fmt", [4, -1])
def test_noalloc_ex_rejects_unknown_format_bits_first(L, fmt):
    # refused before the scratch is looked up or cleared (B = 2, a real plan)
    assert _noalloc_ex(L, fmt) == saw.SAW_ERR_INVALID_ARG
    assert _noalloc_ex(L, 0, B=0) == saw.SAW_OK


@pytest.mark.parametrize("call", EX_CALLS)
@pytest.mark.parametrize("fmt", [4, 8, -1, 1 << 30])
def test_ex_rejects_unknown_format_bits(L, call, fmt):
    # B=0 / T=0 would otherwise return SAW_OK before any launch
    kw = dict(T=0) if call is _append_ex else dict(B=0)
    assert call(L, fmt, **kw) == saw.SAW_ERR_INVALID_ARG


@pytest.mark.parametrize("call", EX_CALLS)
@pytest.mark.parametrize("fmt", [0, saw.SAW_FMT_F16_INPUT, saw.SAW_FMT_BF16_META,
                                 saw.SAW_FMT_F16_INPUT | saw.SAW_FMT_BF16_META])
def test_ex_known_formats_keep_the_plain_checks(L, call, fmt):
    # the empty call succeeds without a launch, and the plain calls' argument
    # checks still apply under every format
    empty = dict(T=0) if call is _append_ex else dict(B=0)
    assert call(L, fmt, **empty) == saw.SAW_OK
    assert call(L, fmt, d=96) == saw.SAW_ERR_UNSUPPORTED
    assert call(L, fmt, kc=MIS) == saw.SAW_ERR_INVALID_ARG
    assert call(L, fmt, h=3) == saw.SAW_ERR_INVALID_ARG


def test_ex_step_and_prefill_stay_head_dim_128(L):
    for fmt in (saw.SAW_FMT_F16_INPUT, saw.SAW_FMT_BF16_META):
        assert _step_ex(L, fmt, d=64) == saw.SAW_ERR_UNSUPPORTED
        assert _prefill_ex(L, fmt, d=256) == saw.SAW_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw", [dict(q=None), dict(out=None), dict(kc=MIS), dict(mb=3),
                                dict(h=48), dict(hq=72), dict(scale=-1.0)])
def test_noalloc_checks_every_argument_before_touching_the_scratch(L, kw):
    # a plan with 4 splits (pps 1 over 64 tokens) needs the shared scratch:
    # the bad argument must be refused before the array is looked up or its
    # counters cleared.  Without a GPU the look-up itself would fail with
    # SAW_ERR_CUDA, so an argument error here shows that nothing ran first.
    s, _ = saw.saw_decode_plan(2, 8, 16, 64, 1)
    assert s > 1
    rc = _noalloc_ex(L, 0, pps=1, **kw)
    assert rc in (saw.SAW_ERR_INVALID_ARG, saw.SAW_ERR_UNSUPPORTED)
    assert rc != saw.SAW_ERR_CUDA
