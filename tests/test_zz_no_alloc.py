"""The no-allocation Swin entry point, called through the C ABI.

swin_window_attn_fwd_noalloc serves callers that must not allocate device
memory: code that may not call cudaMalloc once it runs (a pipeline whose
device memory is reserved up front by a pooling allocator, or one that runs
where allocation is not permitted). Its only scratch, the kernel's status
word, lives in a fixed device array inside the library instead of a buffer
the library allocates.

These tests check, on two calls in a row, that it returns exactly what the
regular swin_window_attn_fwd returns (the same kernel runs in both, so the
outputs are equal bit for bit) and agrees with the oracle; that every call
leaves its status word at zero, including a call made after the word was
set to a nonzero value by hand (each call clears it first, because the
array keeps the previous call's contents); and that shapes it does not serve
are refused. The file sorts last so that a run stopping at the first
failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from vision_transformer_attention_gb300 import _lib, api, workloads

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _status(lib):
    word = ctypes.c_uint(0xFFFFFFFF)
    rc = lib.swin_noalloc_status(ctypes.byref(word), 0)
    return rc, word.value


class _DeviceWord:
    """A one-element uint32 view of a device address, for torch.as_tensor."""

    def __init__(self, addr):
        self.__cuda_array_interface__ = {"shape": (1,), "typestr": "<u4", "data": (addr, False),
                                         "version": 3, "strides": None}


def _status_word_tensor(lib):
    addr = ctypes.c_void_p(0)
    assert lib.swin_noalloc_status_word(ctypes.byref(addr)) == _lib.RPE_OK
    assert addr.value
    return torch.as_tensor(_DeviceWord(addr.value), device="cuda")


def _call(lib, g, nw, heads, d, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.swin_window_attn_fwd_noalloc(_ptr(g["q"]), _ptr(g["k"]), _ptr(g["v"]),
                                            _ptr(g["table"]), nw, heads, 7, d, _ptr(out), stream)


@pytest.mark.parametrize("nw,heads,d", [(37, 3, 32), (5, 4, 64)])
def test_noalloc_matches_regular_entry_point_twice(nw, heads, d):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.lib()
    for call, seed in enumerate((11, 12)):
        inp = workloads.swin_inputs(nw, heads, 7, d, "bf16", table_std=2.0, seed=seed)
        g = {k: t.cuda() for k, t in inp.items()}
        ref = api.swin_window_attn_fwd(g["q"], g["k"], g["v"], g["table"], 7)
        out = torch.full_like(g["q"], float("nan"))
        rc = _call(lib, g, nw, heads, d, out)
        assert rc == _lib.RPE_OK, f"call {call}: status {rc}"
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}: differs from swin_window_attn_fwd"
        assert _status(lib) == (_lib.RPE_OK, 0), f"call {call}: status word set"
        if call == 0:
            want = oracle.swin_attention(inp["q"], inp["k"], inp["v"], inp["table"], 7)
            err = float(np.abs(out.float().cpu().numpy() - want).max())
            assert np.isfinite(err) and err <= TOL_BF16, f"max abs error vs oracle {err}"


def test_noalloc_clears_a_stale_status_word():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.lib()
    word = _status_word_tensor(lib)
    inp = workloads.swin_inputs(6, 3, 7, 32, "bf16", table_std=2.0, seed=13)
    g = {k: t.cuda() for k, t in inp.items()}
    ref = api.swin_window_attn_fwd(g["q"], g["k"], g["v"], g["table"], 7)
    for call in range(2):
        word.fill_(0x5A5A)  # what an earlier call could have left behind
        torch.cuda.synchronize()
        assert _status(lib) == (_lib.RPE_ERR_TIMEOUT, 0x5A5A)
        out = torch.empty_like(g["q"])
        assert _call(lib, g, 6, 3, 32, out) == _lib.RPE_OK
        torch.cuda.synchronize()
        assert _status(lib) == (_lib.RPE_OK, 0), f"call {call}: stale word not cleared"
        assert torch.equal(out, ref)
    # the reader's own clear
    word.fill_(3)
    cleared = ctypes.c_uint(0)
    assert lib.swin_noalloc_status(ctypes.byref(cleared), 1) == _lib.RPE_ERR_TIMEOUT
    assert cleared.value == 3
    assert _status(lib) == (_lib.RPE_OK, 0)


def test_noalloc_rejects_what_it_cannot_serve():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.lib()
    x = torch.zeros(1, 1, 64, 32, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(225, 1, device="cuda")
    # M = 8 is served by no bf16 kernel; 33 heads exceed the kernel's bias table
    assert lib.swin_window_attn_fwd_noalloc(_ptr(x), _ptr(x), _ptr(x), _ptr(t), 1, 1, 8, 32,
                                            _ptr(x), None) == _lib.RPE_ERR_UNSUPPORTED
    assert lib.swin_window_attn_fwd_noalloc(_ptr(x), _ptr(x), _ptr(x), _ptr(t), 1, 33, 7, 32,
                                            _ptr(x), None) == _lib.RPE_ERR_UNSUPPORTED
    assert lib.swin_window_attn_fwd_noalloc(None, _ptr(x), _ptr(x), _ptr(t), 1, 1, 7, 32,
                                            _ptr(x), None) == _lib.RPE_ERR_INVALID_ARG
