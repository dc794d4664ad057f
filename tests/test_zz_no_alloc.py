"""The no-allocation Swin entry point, called through the C ABI.

swin_window_attn_fwd_noalloc serves callers that must not allocate device
memory (allocation forbidden once a pipeline runs, memory reserved up front by
a pooling allocator): its kernel scratch is a fixed device array inside the
library. This test checks that two calls in a row give the same output as the
regular swin_window_attn_fwd on the same inputs, within the bf16 tolerance of
the other GPU tests, and that the second call is not disturbed by what the
first left in the shared array. It lives in its own file, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from vision_transformer_attention_gb300 import _lib, api, workloads

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("nw,heads,d", [(37, 3, 32), (5, 4, 64)])
def test_noalloc_matches_regular_entry_point_twice(nw, heads, d):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, seed in enumerate((11, 12)):
        inp = workloads.swin_inputs(nw, heads, 7, d, "bf16", table_std=2.0, seed=seed)
        g = {k: t.cuda() for k, t in inp.items()}
        ref = api.swin_window_attn_fwd(g["q"], g["k"], g["v"], g["table"], 7)
        out = torch.full_like(g["q"], float("nan"))
        rc = lib.swin_window_attn_fwd_noalloc(_ptr(g["q"]), _ptr(g["k"]), _ptr(g["v"]),
                                              _ptr(g["table"]), nw, heads, 7, d, _ptr(out),
                                              stream)
        assert rc == _lib.RPE_OK, f"call {call}: status {rc}"
        torch.cuda.synchronize()
        err = float((out.float() - ref.float()).abs().max())
        assert np.isfinite(err) and err <= TOL_BF16, f"call {call}: max abs diff {err}"


def test_noalloc_rejects_what_it_cannot_serve():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.lib()
    x = torch.zeros(1, 1, 64, 32, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(225, 1, device="cuda")
    # M = 8 is served by no bf16 kernel
    assert lib.swin_window_attn_fwd_noalloc(_ptr(x), _ptr(x), _ptr(x), _ptr(t), 1, 1, 8, 32,
                                            _ptr(x), None) == _lib.RPE_ERR_UNSUPPORTED
    assert lib.swin_window_attn_fwd_noalloc(None, _ptr(x), _ptr(x), _ptr(t), 1, 1, 7, 32,
                                            _ptr(x), None) == _lib.RPE_ERR_INVALID_ARG
