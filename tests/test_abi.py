"""The C-ABI library builds for sm_103a, loads, exports every declared entry
point, and refuses bad arguments before touching the GPU (no CUDA device needed)."""
import ctypes
import os
import re

import pytest

import head_attention_attn_gb300 as attn
from head_attention_attn_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return attn.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = declared_functions()
    assert set(names) == set(attn.EXPORTED)
    assert "attn_fwd" in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and nothing but the C ABI leaks out of the library
    out = os.popen(f"nm -D --defined-only {attn.library_path()}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(declared_functions()) <= exported
    assert not [s for s in exported if s.startswith("_ZN4attn")], "internal symbols are exported"


def test_version(lib):
    assert attn.version() == 100


def _call(**kw):
    args = dict(q_ptr=16, k_ptr=16, v_ptr=16, out_ptr=16, batch=1, q_heads=4, kv_heads=2, q_len=8, kv_len=8,
                head_dim=64, pos_offset=0, mask_mode=0, window=0, key_lens_ptr=None, scale=0.125,
                dtype=attn.ATTN_BF16, stream_handle=None)
    args.update(kw)
    return attn.attn_fwd_raw(**args)


@pytest.mark.parametrize("change,fragment", [
    (dict(batch=-1), "negative size"),
    (dict(q_len=-3), "negative size"),
    (dict(kv_len=-1), "negative size"),
    (dict(q_heads=0), "must be positive"),
    (dict(head_dim=0), "must be positive"),
    (dict(q_heads=3, kv_heads=2), "not a multiple"),
    (dict(mask_mode=4), "mask_mode"),
    (dict(mask_mode=-1), "mask_mode"),
    (dict(dtype=3), "dtype"),
    (dict(window=-1), "negative window"),
    (dict(pos_offset=-1), "negative pos_offset"),
    (dict(scale=float("nan")), "not finite"),
    (dict(scale=float("inf")), "not finite"),
    (dict(q_ptr=None), "null q"),
    (dict(out_ptr=None), "null q or out"),
    (dict(k_ptr=None), "null k"),
    (dict(q_ptr=18), "aligned"),
    (dict(out_ptr=24), "aligned"),
    (dict(dtype=attn.ATTN_F32, k_ptr=18), "aligned"),
    (dict(dtype=attn.ATTN_F16, v_ptr=24), "aligned"),
])
def test_invalid_arguments_are_refused_before_launch(lib, change, fragment):
    assert _call(**change) == attn.ATTN_ERR_INVALID_ARG
    assert fragment in attn.last_error()


@pytest.mark.parametrize("change", [dict(head_dim=32), dict(head_dim=96), dict(head_dim=256),
                                    dict(dtype=attn.ATTN_F16, head_dim=96),
                                    dict(dtype=attn.ATTN_F32, head_dim=257)])
def test_unsupported_head_dims(lib, change):
    assert _call(**change) == attn.ATTN_ERR_UNSUPPORTED
    assert "head_dim" in attn.last_error()


@pytest.mark.parametrize("change", [dict(batch=0), dict(q_len=0),
                                    dict(batch=0, q_ptr=None, k_ptr=None, v_ptr=None, out_ptr=None)])
def test_empty_problems_launch_nothing(lib, change):
    assert _call(**change) == attn.ATTN_OK
    assert attn.last_error() == ""


@pytest.mark.parametrize("change,fragment", [
    (dict(batch=-1), "negative size"),
    (dict(q_heads=3, kv_heads=2), "not a multiple"),
    (dict(mask_mode=4), "mask_mode"),
    (dict(dtype=3), "dtype"),
    (dict(out_ptr=None), "null q or out"),
    (dict(out_ptr=24), "aligned"),
])
def test_token_major_entry_checks_like_attn_fwd(lib, change, fragment):
    args = dict(q_ptr=16, k_ptr=16, v_ptr=16, out_ptr=16, batch=1, q_heads=4, kv_heads=2, q_len=8, kv_len=8,
                head_dim=64, pos_offset=0, mask_mode=0, window=0, key_lens_ptr=None, scale=0.125,
                dtype=attn.ATTN_BF16, stream_handle=None)
    args.update(change)
    a = list(args.values())
    a[14] = ctypes.c_float(a[14])
    assert lib.attn_fwd_out_token_major(*a) == attn.ATTN_ERR_INVALID_ARG
    assert fragment in attn.last_error()


@pytest.mark.parametrize("change,status", [
    (dict(m=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(num_pages=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(page_size=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(max_pages=1 << 20, page_size=1 << 12), attn.ATTN_ERR_INVALID_ARG),
    (dict(q_heads=6, kv_heads=4), attn.ATTN_ERR_INVALID_ARG),
    (dict(q_heads=12, kv_heads=4), attn.ATTN_ERR_UNSUPPORTED),
    (dict(head_dim=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=attn.ATTN_F32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(sliding=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(page_table=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(k_pool=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(kv_lens=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(k_pool=24), attn.ATTN_ERR_INVALID_ARG),
    (dict(page_table=18), attn.ATTN_ERR_INVALID_ARG),
    (dict(m=0), attn.ATTN_OK),
])
def test_decode_paged_arguments(lib, change, status):
    a = dict(q=16, k_pool=16, v_pool=16, page_table=16, out=16, m=2, q_heads=8, kv_heads=2, num_pages=4,
             page_size=16, max_pages=4, head_dim=128, kv_lens=16, sliding=0, scale=0.1, dtype=attn.ATTN_BF16)
    a.update(change)
    got = lib.attn_decode_paged(a["q"], a["k_pool"], a["v_pool"], a["page_table"], a["out"], a["m"], a["q_heads"],
                                a["kv_heads"], a["num_pages"], a["page_size"], a["max_pages"], a["head_dim"],
                                a["kv_lens"], a["sliding"], ctypes.c_float(a["scale"]), a["dtype"], None)
    assert got == status, attn.last_error()


def test_selftest_limit_is_checked(lib):
    assert lib.attn_selftest_timeout(0, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_timeout(2_000_000, None) == attn.ATTN_ERR_INVALID_ARG


def test_python_wrapper_rejects_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 2, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        attn.load(str(tmp_path / "libattn.so"))


def test_library_has_no_host_fallback_symbols(lib):
    # The product library never links the oracle.
    out = os.popen(f"nm -D {attn.library_path()}").read()
    assert "oracle" not in out
    assert isinstance(ctypes.CDLL(attn.library_path()), ctypes.CDLL)


def _caches_call(lib, noalloc=False, **kw):
    args = dict(q=16, kc=16, vc=16, out=16, m=2, hq=8, hkv=2, cap=64, d=128, lens=16, win=0, scale=0.1,
                dtype=attn.ATTN_BF16, stream=None)
    args.update(kw)
    entry = lib.attn_decode_caches_noalloc if noalloc else lib.attn_decode_caches
    return entry(args["q"], args["kc"], args["vc"], args["out"], args["m"], args["hq"], args["hkv"], args["cap"],
                 args["d"], args["lens"], args["win"], ctypes.c_float(args["scale"]), args["dtype"], args["stream"])


@pytest.mark.parametrize("change,status", [
    (dict(m=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(cap=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(hq=6, hkv=4), attn.ATTN_ERR_INVALID_ARG),
    (dict(win=-2), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(lens=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(kc=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=24), attn.ATTN_ERR_INVALID_ARG),
    (dict(kc=12), attn.ATTN_ERR_INVALID_ARG),
    (dict(dtype=attn.ATTN_F32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=3), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=attn.ATTN_F16, d=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(hq=6, hkv=2), attn.ATTN_ERR_UNSUPPORTED),
    (dict(m=0), attn.ATTN_OK),
])
@pytest.mark.parametrize("noalloc", [False, True])
def test_decode_caches_arguments(lib, change, status, noalloc):
    assert _caches_call(lib, noalloc=noalloc, **change) == status


def test_decode_caches_noalloc_refuses_more_items_than_its_table(lib):
    # ATTN_NOALLOC_MAX_ITEMS is 4096: the call is refused before anything is read or launched
    assert _caches_call(lib, noalloc=True, m=4097) == attn.ATTN_ERR_INVALID_ARG
    assert "fixed map table" in attn.last_error()


def _varlen_call(lib, **kw):
    args = dict(q=16, k=16, v=16, out=16, cu=16, batch=2, total=64, maxlen=40, hq=4, hkv=2, d=64, mode=0, win=0,
                scale=0.125, dtype=attn.ATTN_BF16, stream=None)
    args.update(kw)
    return lib.attn_fwd_varlen(args["q"], args["k"], args["v"], args["out"], args["cu"], args["batch"],
                               args["total"], args["maxlen"], args["hq"], args["hkv"], args["d"], args["mode"],
                               args["win"], ctypes.c_float(args["scale"]), args["dtype"], args["stream"])


@pytest.mark.parametrize("change,status", [
    (dict(batch=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(total=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(maxlen=65), attn.ATTN_ERR_INVALID_ARG),
    (dict(hq=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(mode=5), attn.ATTN_ERR_INVALID_ARG),
    (dict(win=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(cu=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(cu=18), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(out=40), attn.ATTN_ERR_INVALID_ARG),
    (dict(dtype=attn.ATTN_F32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(batch=0), attn.ATTN_OK),
    (dict(maxlen=0), attn.ATTN_OK),
])
def test_varlen_arguments(lib, change, status):
    assert _varlen_call(lib, **change) == status
    if status != attn.ATTN_OK:
        assert attn.last_error() != ""


def _prelude_call(lib, **kw):
    a = dict(qkv=16, qw=16, kw=16, cos=16, sin=16, npos=64, q=16, k=16, v=16, tokens=8, hq=4, hkv=2, d=128, pos=0,
             eps=1e-6, mode=1, clen=0, cap=0, dtype=attn.ATTN_BF16, stream=None)
    a.update(kw)
    return lib.attn_qkv_prelude(a["qkv"], a["qw"], a["kw"], a["cos"], a["sin"], a["npos"], a["q"], a["k"], a["v"],
                                a["tokens"], a["hq"], a["hkv"], a["d"], a["pos"], ctypes.c_float(a["eps"]), a["mode"],
                                a["clen"], a["cap"], a["dtype"], a["stream"])


@pytest.mark.parametrize("change,status", [
    (dict(tokens=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(hq=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(mode=4), attn.ATTN_ERR_INVALID_ARG),
    (dict(dtype=7), attn.ATTN_ERR_INVALID_ARG),
    (dict(dtype=attn.ATTN_F32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(eps=-1.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(eps=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(pos=60), attn.ATTN_ERR_INVALID_ARG),          # positions past the rope tables
    (dict(cap=10, clen=5), attn.ATTN_ERR_INVALID_ARG),  # cache slot past the capacity
    (dict(cos=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(sin=24), attn.ATTN_ERR_INVALID_ARG),
    (dict(qw=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(qkv=8), attn.ATTN_ERR_INVALID_ARG),
    (dict(v=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(tokens=0), attn.ATTN_OK),
    (dict(mode=0, cos=None, sin=None, qw=None, kw=None, npos=0, tokens=0), attn.ATTN_OK),
])
def test_prelude_arguments(lib, change, status):
    assert _prelude_call(lib, **change) == status
    if status != attn.ATTN_OK:
        assert attn.last_error() != ""


def _prelude_caches_call(lib, **kw):
    a = dict(qkv=16, qw=16, kw=16, cos=16, sin=16, npos=64, q=16, kc=16, vc=16, lens=16, m=4, hq=4, hkv=2, d=128,
             cap=32, eps=1e-6, mode=1, dtype=attn.ATTN_BF16, stream=None)
    a.update(kw)
    return lib.attn_qkv_prelude_caches(a["qkv"], a["qw"], a["kw"], a["cos"], a["sin"], a["npos"], a["q"], a["kc"],
                                       a["vc"], a["lens"], a["m"], a["hq"], a["hkv"], a["d"], a["cap"],
                                       ctypes.c_float(a["eps"]), a["mode"], a["dtype"], a["stream"])


@pytest.mark.parametrize("change,status", [
    (dict(m=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(cap=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(mode=9), attn.ATTN_ERR_INVALID_ARG),
    (dict(dtype=attn.ATTN_F32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(lens=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(kc=12), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=8), attn.ATTN_ERR_INVALID_ARG),
    (dict(cos=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(kw=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(m=0), attn.ATTN_OK),
])
def test_prelude_caches_arguments(lib, change, status):
    assert _prelude_caches_call(lib, **change) == status


def test_per_item_decode_wrappers_check_out_and_kv_lens():
    """A caller's out and kv_lens are checked before the library sees them: the kernels
    write m * Hq * D contiguous elements of q's type and read m contiguous lengths."""
    import torch
    from head_attention_attn_gb300._binding import _check_kv_lens, _decode_out
    q = torch.zeros(3, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="shape"):
        _decode_out(q, torch.zeros(3, 4, 32, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="shape"):
        _decode_out(q, torch.zeros(3, 4, 64, dtype=torch.float16))
    with pytest.raises(ValueError, match="contiguous"):
        _decode_out(q, torch.zeros(3, 64, 4, dtype=torch.bfloat16).transpose(1, 2))
    with pytest.raises(ValueError, match="CUDA"):
        _decode_out(q, torch.zeros(3, 4, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="m entries"):
        _check_kv_lens(torch.zeros(2, dtype=torch.int32), 3)
    with pytest.raises(ValueError, match="m entries"):
        _check_kv_lens(torch.zeros(3, dtype=torch.int64), 3)
    with pytest.raises(ValueError, match="contiguous"):
        _check_kv_lens(torch.zeros(6, dtype=torch.int32)[::2], 3)
    with pytest.raises(ValueError, match="CUDA"):
        _check_kv_lens(torch.zeros(3, dtype=torch.int32), 3)
