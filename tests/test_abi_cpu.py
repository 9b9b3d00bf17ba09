"""The C-ABI library without a GPU: it builds, loads, exports every entry
point that include/paq8.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

from paged_attention_int8_gb300 import _lib, build as pkg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paq8.h")


@pytest.fixture(scope="module")
def lib():
    pkg_build.build()
    return _lib.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("pa_kv_store", "pa_paged_attention", "pa_workspace_size", "pa_check_status",
              "pa_status_string", "pa_auto_num_splits", "pa_last_error",
              "pa_merge_attn_states"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pa_\w+)", out))
    for name in _declared():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    for s in _lib.Status:
        assert lib.pa_status_string(int(s)).decode()


def test_workspace_size_formula(lib):
    # 256-byte header, plus fp32 [S, Hq, NS, D + 2] partials when splitting
    assert lib.pa_workspace_size(64, 32, 128, 1) == 256
    assert lib.pa_workspace_size(64, 32, 128, 16) == 256 + 64 * 32 * 16 * 130 * 4
    assert lib.pa_workspace_size(8, 32, 256, 0) == 256 + 8 * 32 * 16 * 258 * 4


def test_auto_splits_range(lib):
    for L in (1, 64, 511, 512, 513, 8192, 131072):
        ns = lib.pa_auto_num_splits(64, 8, 1, L)
        assert 1 <= ns <= 16
    assert lib.pa_auto_num_splits(8, 8, 1, 131072) == 16
    assert lib.pa_auto_num_splits(64, 8, 1, 8025) == 8
    assert lib.pa_auto_num_splits(132, 8, 1024, 16384) == 8   # capped by ~8192 units
    assert lib.pa_auto_num_splits(2, 2, 1, 100) == 1


def _store_args(**kw):
    a = dict(key=16, kstride=256, value=16, vstride=256, slots=16, n=4, hk=2, d=128,
             kc=16, ks=16, vc=16, vs=16, nb=4, bs=16, status=None, stream=None)
    a.update(kw)
    v = lambda x: ctypes.c_void_p(x) if x is not None else None  # noqa: E731
    return [v(a["key"]), a["kstride"], v(a["value"]), a["vstride"], v(a["slots"]), a["n"],
            a["hk"], a["d"], v(a["kc"]), v(a["ks"]), v(a["vc"]), v(a["vs"]), a["nb"], a["bs"],
            v(a["status"]), v(a["stream"])]


@pytest.mark.parametrize("kw,expect", [
    (dict(key=None), _lib.Status.INVALID_ARG),
    (dict(n=-1), _lib.Status.INVALID_ARG),
    (dict(d=96), _lib.Status.UNSUPPORTED),
    (dict(bs=8), _lib.Status.UNSUPPORTED),
    (dict(kstride=100), _lib.Status.INVALID_ARG),
    (dict(key=24), _lib.Status.INVALID_ARG),
    (dict(kc=8), _lib.Status.INVALID_ARG),
    (dict(nb=0), _lib.Status.INVALID_ARG),
    (dict(slots=20), _lib.Status.INVALID_ARG),   # slot_mapping not 8-byte aligned
])
def test_kv_store_rejects_bad_arguments(lib, kw, expect):
    assert lib.pa_kv_store(*_store_args(**kw)) == expect
    assert lib.pa_last_error().decode()


def test_kv_store_zero_tokens_is_a_no_op(lib):
    assert lib.pa_kv_store(*_store_args(n=0, key=None)) == _lib.Status.OK


def _attn_args(**kw):
    a = dict(q=16, kc=16, ks=16, vc=16, vs=16, cu=16, sl=16, bt=16, bts=8, S=2, T=2, hq=8,
             hk=2, d=128, nb=16, bs=16, mq=1, ms=100, scale=0.1, ns=1, out=16, lse=16, ws=16,
             wsb=256, flags=0, stream=None)
    a.update(kw)
    v = lambda x: ctypes.c_void_p(x) if x is not None else None  # noqa: E731
    return [v(a["q"]), v(a["kc"]), v(a["ks"]), v(a["vc"]), v(a["vs"]), v(a["cu"]), v(a["sl"]),
            v(a["bt"]), a["bts"], a["S"], a["T"], a["hq"], a["hk"], a["d"], a["nb"], a["bs"],
            a["mq"], a["ms"], ctypes.c_float(a["scale"]), a["ns"], v(a["out"]), v(a["lse"]),
            v(a["ws"]), a["wsb"], a["flags"], v(a["stream"])]


@pytest.mark.parametrize("kw,expect", [
    (dict(flags=2), _lib.Status.INVALID_ARG),              # unknown flag bit
    (dict(flags=_lib.ATTN_TEST_TIMEOUT, mq=4), _lib.Status.INVALID_ARG),  # decode path only
    (dict(flags=_lib.ATTN_TEST_TIMEOUT, hq=32, hk=2), _lib.Status.INVALID_ARG),
    (dict(ws=None), _lib.Status.INVALID_ARG),
    (dict(q=None), _lib.Status.INVALID_ARG),
    (dict(hq=7), _lib.Status.INVALID_ARG),
    (dict(hq=34, hk=2), _lib.Status.UNSUPPORTED),
    (dict(d=80), _lib.Status.UNSUPPORTED),
    (dict(bs=64), _lib.Status.UNSUPPORTED),
    (dict(mq=0), _lib.Status.INVALID_ARG),
    (dict(ns=17), _lib.Status.INVALID_ARG),
    (dict(ns=4, wsb=256), _lib.Status.INVALID_ARG),
    (dict(out=8), _lib.Status.INVALID_ARG),
    (dict(bts=0), _lib.Status.INVALID_ARG),
    (dict(nb=1 << 30), _lib.Status.UNSUPPORTED),
])
def test_paged_attention_rejects_bad_arguments(lib, kw, expect):
    assert lib.pa_paged_attention(*_attn_args(**kw)) == expect


def test_paged_attention_empty_batch_is_a_no_op(lib):
    assert lib.pa_paged_attention(*_attn_args(S=0, T=0, q=None)) == _lib.Status.OK


def _attn_ex_args(sinks=None, window=0, **kw):
    a = _attn_args(**kw)
    sk = ctypes.c_void_p(sinks) if sinks is not None else None
    return a[:20] + [sk, window] + a[20:]


@pytest.mark.parametrize("kw,expect", [
    (dict(window=-1), _lib.Status.INVALID_ARG),
    (dict(window=16, flags=_lib.ATTN_NON_CAUSAL), _lib.Status.INVALID_ARG),  # window is causal
    (dict(sinks=18), _lib.Status.INVALID_ARG),                               # not 4-byte aligned
    (dict(sinks=16, flags=4), _lib.Status.INVALID_ARG),
    (dict(window=8, q=None), _lib.Status.INVALID_ARG),
])
def test_paged_attention_ex_rejects_bad_arguments(lib, kw, expect):
    assert lib.pa_paged_attention_ex(*_attn_ex_args(**kw)) == expect
    assert lib.pa_last_error().decode()


def test_paged_attention_ex_empty_batch_is_a_no_op(lib):
    assert lib.pa_paged_attention_ex(*_attn_ex_args(S=0, T=0, q=None, window=4)) == _lib.Status.OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load()


def _merge_args(**kw):
    a = dict(oa=16, la=16, ob=32, lb=32, out=48, lse=64, rows=10, d=128, stream=None)
    a.update(kw)
    v = lambda x: ctypes.c_void_p(x) if x is not None else None  # noqa: E731
    return [v(a["oa"]), v(a["la"]), v(a["ob"]), v(a["lb"]), v(a["out"]), v(a["lse"]),
            a["rows"], a["d"], v(a["stream"])]


@pytest.mark.parametrize("kw,expect", [
    (dict(oa=None), _lib.Status.INVALID_ARG),
    (dict(out=None), _lib.Status.INVALID_ARG),
    (dict(rows=-1), _lib.Status.INVALID_ARG),
    (dict(d=96), _lib.Status.UNSUPPORTED),
    (dict(ob=40), _lib.Status.INVALID_ARG),   # not 16-byte aligned
    (dict(lse=66), _lib.Status.INVALID_ARG),  # not 4-byte aligned
])
def test_merge_attn_states_rejects_bad_arguments(lib, kw, expect):
    assert lib.pa_merge_attn_states(*_merge_args(**kw)) == expect
    assert lib.pa_last_error().decode()


def test_merge_attn_states_zero_rows_is_a_no_op(lib):
    assert lib.pa_merge_attn_states(*_merge_args(rows=0, oa=None)) == _lib.Status.OK


def test_bindings_mirror_the_boundary():
    # every compute entry point of the header has a binding of the same name
    import paged_attention_int8_gb300 as pkg
    for name in ("kv_store", "kv_store_norm_rope", "kv_store_f8v4", "paged_attention",
                 "paged_attention_f8v4", "paged_attention_noalloc",
                 "merge_attn_states", "workspace_size", "auto_num_splits", "check_status"):
        assert name in pkg.__all__ and callable(getattr(pkg, name))


def test_bindings_refuse_host_tensors():
    import torch
    q = torch.zeros((2, 4, 64), dtype=torch.bfloat16)
    kc = torch.zeros((2, 2, 16, 64), dtype=torch.int8)
    ks = torch.zeros((2, 2, 16, 2), dtype=torch.float16)
    vc = torch.zeros((2, 2, 64, 16), dtype=torch.int8)
    vs = torch.zeros((2, 2, 2, 16), dtype=torch.float16)
    cu = torch.tensor([0, 1, 2], dtype=torch.int32)
    sl = torch.tensor([5, 9], dtype=torch.int32)
    bt = torch.zeros((2, 1), dtype=torch.int32)
    for fn in (_lib.paged_attention, _lib.paged_attention_noalloc):
        with pytest.raises(ValueError):
            fn(q, kc, ks, vc, vs, cu, sl, bt, 1, 9)
    with pytest.raises(ValueError):
        _lib.merge_attn_states(q, sl.float(), q, sl.float())


def _fused_args(**kw):
    a = dict(key=16, kstride=256, value=16, vstride=256, slots=16, pos=16, n=4, hk=2, d=128,
             w=16, eps=1e-6, rope=16, maxpos=64, rot=128, inter=0, kc=16, ks=16, vc=16, vs=16,
             nb=4, bs=16, status=None, stream=None)
    a.update(kw)
    v = lambda x: ctypes.c_void_p(x) if x is not None else None  # noqa: E731
    return [v(a["key"]), a["kstride"], v(a["value"]), a["vstride"], v(a["slots"]), v(a["pos"]),
            a["n"], a["hk"], a["d"], v(a["w"]), ctypes.c_float(a["eps"]), v(a["rope"]),
            a["maxpos"], a["rot"], a["inter"], v(a["kc"]), v(a["ks"]), v(a["vc"]), v(a["vs"]),
            a["nb"], a["bs"], v(a["status"]), v(a["stream"])]


@pytest.mark.parametrize("kw,expect", [
    (dict(key=None), _lib.Status.INVALID_ARG),
    (dict(pos=None), _lib.Status.INVALID_ARG),        # a rotation needs positions
    (dict(rot=130), _lib.Status.INVALID_ARG),         # past head_dim
    (dict(rot=63), _lib.Status.INVALID_ARG),          # odd
    (dict(rot=0), _lib.Status.INVALID_ARG),
    (dict(rope=20), _lib.Status.INVALID_ARG),         # not 8-byte aligned
    (dict(maxpos=0), _lib.Status.INVALID_ARG),
    (dict(w=17), _lib.Status.INVALID_ARG),            # not 2-byte aligned
    (dict(d=96), _lib.Status.UNSUPPORTED),
    (dict(bs=8), _lib.Status.UNSUPPORTED),
    (dict(vstride=100), _lib.Status.INVALID_ARG),
])
def test_kv_store_norm_rope_rejects_bad_arguments(lib, kw, expect):
    assert lib.pa_kv_store_norm_rope(*_fused_args(**kw)) == expect
    assert lib.pa_last_error().decode()


def test_kv_store_norm_rope_zero_tokens_is_a_no_op(lib):
    assert lib.pa_kv_store_norm_rope(*_fused_args(n=0, key=None)) == _lib.Status.OK


def test_f8v4_entries_reject_bad_arguments(lib):
    args = _attn_ex_args()
    # pa_paged_attention_f8v4(q, k_cache, v_cache, v_scale, v_zero, ...): same tail as _ex
    f8 = lambda **kw: [v for v in _attn_ex_args(**kw)]  # noqa: E731
    base = f8()
    call = base[:2] + [base[3], base[4], ctypes.c_void_p(16)] + base[5:]
    assert len(call) == len(args)
    # no v_zero
    bad = base[:2] + [base[3], base[4], None] + base[5:]
    assert lib.pa_paged_attention_f8v4(*bad) == _lib.Status.INVALID_ARG
    # the same visibility checks as _ex: a window is causal only
    bad = f8(window=16, flags=_lib.ATTN_NON_CAUSAL)
    call = bad[:2] + [bad[3], bad[4], ctypes.c_void_p(16)] + bad[5:]
    assert lib.pa_paged_attention_f8v4(*call) == _lib.Status.INVALID_ARG
    # the store: a null zero array, an odd row stride
    st = _store_args()
    store = st[:8] + [st[8], st[10], st[11], ctypes.c_void_p(16)] + st[12:]
    assert lib.pa_kv_store_f8v4(*(store[:11] + [None] + store[12:])) == _lib.Status.INVALID_ARG
    odd = _store_args(kstride=260)
    store = odd[:8] + [odd[8], odd[10], odd[11], ctypes.c_void_p(16)] + odd[12:]
    assert lib.pa_kv_store_f8v4(*store) == _lib.Status.INVALID_ARG
