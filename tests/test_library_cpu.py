"""CPU checks of the C-ABI library: it builds for sm_103a, loads without a GPU
and exports every entry point that include/rpe_attn.h declares. No compute
call is made here (there is no GPU in this process)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "rpe_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(\w+)\s*\(", text)) - {"defined"})


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for required in ("rpe_build_bucket_ids", "rpe_attn_fwd", "swin_window_attn_fwd"):
        assert required in names


def test_library_builds_and_exports_every_declared_symbol():
    from vision_transformer_attention_gb300 import build, _lib
    path = build.build()
    handle = ctypes.CDLL(path)
    for name in _declared_symbols():
        assert hasattr(handle, name), name
    assert set(_declared_symbols()) == set(_lib.SIGNATURES)


def test_release_calls_without_gpu_have_nothing_to_free():
    from vision_transformer_attention_gb300 import _lib
    lib = _lib.lib()
    assert lib.rpe_release_stream(None) == _lib.RPE_OK
    assert lib.rpe_shutdown() == _lib.RPE_OK


def test_status_strings_without_gpu():
    from vision_transformer_attention_gb300 import _lib
    lib = _lib.lib()
    assert lib.rpe_status_string(0) == b"ok"
    assert b"invalid" in lib.rpe_status_string(1)


def test_host_argument_checks_reject_before_any_launch():
    # invalid arguments are refused on the host, so these calls need no GPU
    from vision_transformer_attention_gb300 import _lib
    lib = _lib.lib()
    nb = ctypes.c_int(0)
    fake = ctypes.c_void_p(1 << 20)
    assert lib.rpe_build_bucket_ids(0, 14, 0, 1.9, 3.8, 15.2, fake, None, ctypes.byref(nb), None) == 1
    assert lib.rpe_build_bucket_ids(14, 14, 4, 1.9, 3.8, 15.2, fake, None, ctypes.byref(nb), None) == 1
    assert lib.rpe_build_bucket_ids(14, 14, -1, 1.9, 3.8, 15.2, fake, None, ctypes.byref(nb), None) == 1
    assert lib.rpe_build_bucket_ids(14, 14, 0, 3.9, 3.8, 15.2, fake, None, ctypes.byref(nb), None) == 1
    # the N x N expansion needs N * N < 2^31 (a 256 x 256 grid without it is fine,
    # but needs a GPU); sides above 32768 are refused either way
    assert lib.rpe_build_bucket_ids(256, 256, 0, 1.9, 3.8, 15.2, fake, fake, ctypes.byref(nb),
                                    None) == 1
    assert lib.rpe_build_bucket_ids(32769, 1, 0, 1.9, 3.8, 15.2, fake, None, ctypes.byref(nb),
                                    None) == 1
    # an empty batch is invalid; more than 65536 tokens is unsupported
    assert lib.rpe_attn_fwd(fake, fake, fake, None, fake, None, fake, 49, 0, 1, 14, 14, 64, 1, 0,
                            fake, None) == 1
    assert lib.rpe_attn_fwd(fake, fake, fake, None, fake, None, fake, 49, 1, 1, 257, 256, 64, 1, 0,
                            fake, None) == 2
    # misaligned pointer
    bad = ctypes.c_void_p((1 << 20) + 4)
    assert lib.rpe_attn_fwd(bad, fake, fake, None, fake, None, fake, 49, 1, 1, 14, 14, 64, 1, 0,
                            fake, None) == 1
    # term bit set with a NULL table
    assert lib.rpe_attn_fwd(fake, fake, fake, None, None, None, fake, 49, 1, 1, 14, 14, 64, 1, 0,
                            fake, None) == 1
    # unsupported: too many buckets, bf16 with d != 64, Swin bf16 with M != 7
    assert lib.rpe_attn_fwd(fake, fake, fake, None, fake, None, fake, 129, 1, 1, 14, 14, 64, 1, 0,
                            fake, None) == 2
    assert lib.rpe_attn_fwd(fake, fake, fake, fake, fake, None, fake, 81, 1, 1, 14, 14, 64, 3, 0,
                            fake, None) == 2   # query term: 64 buckets at most in bf16
    assert lib.rpe_attn_fwd(fake, fake, fake, None, fake, None, fake, 257, 1, 1, 14, 14, 32, 1, 1,
                            fake, None) == 2   # fp32: 256 at most
    assert lib.rpe_attn_fwd(fake, fake, fake, None, fake, None, fake, 49, 1, 1, 14, 14, 32, 1, 0,
                            fake, None) == 2
    # Cross tables: an odd row count or (rows / 2)^2 joint ids above 64 are not
    # served; an unknown flag bit is invalid
    cross_k = _lib.RPE_TERM_K | _lib.RPE_TABLES_CROSS
    assert lib.rpe_attn_fwd(fake, fake, fake, None, fake, None, fake, 18, 1, 1, 14, 14, 64, cross_k,
                            0, fake, None) == 2
    assert lib.rpe_attn_fwd(fake, fake, fake, None, fake, None, fake, 13, 1, 1, 14, 14, 64, cross_k,
                            0, fake, None) == 2
    assert lib.rpe_attn_fwd(fake, fake, fake, None, fake, None, fake, 14, 1, 1, 14, 14, 64, 64,
                            0, fake, None) == 1
    # class token with Cross tables is not served
    cls_cross = cross_k | _lib.RPE_CLS_TOKEN
    assert lib.rpe_attn_fwd(fake, fake, fake, None, fake, None, fake, 14, 1, 1, 14, 14, 64,
                            cls_cross, 0, fake, None) == 2
    # bf16 bias mode needs d == 64 and at most 128 buckets
    assert lib.rpe_attn_bias_fwd(fake, fake, fake, fake, 1, fake, 50, _lib.RPE_CLS_TOKEN, 1, 1,
                                 14, 14, 32, 0, fake, None) == 2
    assert lib.rpe_attn_bias_fwd(fake, fake, fake, fake, 1, fake, 129, 0, 1, 1,
                                 14, 14, 64, 0, fake, None) == 2
    assert lib.rpe_attn_bias_fwd(fake, fake, fake, fake, 1, fake, 14, 2, 1, 1, 14, 14, 64, 0,
                                 fake, None) == 1
    assert lib.rpe_attn_bias_fwd(fake, fake, fake, fake, 1, fake, 18, _lib.RPE_TABLES_CROSS, 1, 1,
                                 14, 14, 64, 0, fake, None) == 2
    assert lib.swin_window_attn_fwd(fake, fake, fake, fake, 4, 3, 8, 32, 0, fake, None) == 2
    assert lib.swin_window_attn_fwd(fake, fake, fake, fake, 0, 3, 7, 32, 0, fake, None) == 1


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    from vision_transformer_attention_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.lib()
