"""The gated FFN entry point that allocates nothing.

qws_q4k_ffn_gate_up_geglu_down_noalloc serves callers that may not allocate
device memory at call time and have no spare buffer to lend as workspace; it
keeps the intermediate vector in a fixed array inside the library.  Called
through the C ABI, it must give the same result as the workspace entry point
(within the FFN tolerance of the parity tests), on two calls in a row -- the
second call reuses the same array, so a stale intermediate would show up.
This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from quantized_weight_streaming_q4k_gb300 import _lib, build, ops, synth

pytestmark = pytest.mark.gpu


def _ptr(t):
    return C.c_void_p(t.data_ptr())


def test_ffn_noalloc_matches_workspace_entry_point():
    build.build()
    lib = _lib.lib()
    torch.cuda.set_device(0)
    H, I = 2560, 10240
    g = synth.rng(7000, 1)
    Wg = synth.q4_k_matrix(g, I, H)
    Wu = synth.q4_k_matrix(g, I, H)
    Wd = synth.q6_k_matrix(g, H, I)
    dWg, dWu, dWd = (torch.from_numpy(w).cuda() for w in (Wg, Wu, Wd))
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    ref_oracle = None
    for call, scale in enumerate((1.0, 0.37)):
        # a different input each call: a stale intermediate from the previous
        # call would change the result
        x = (synth.unit_rms_vector(g, H) * np.float32(scale)).astype(np.float32)
        dx = torch.from_numpy(x).cuda()
        y_ws = ops.q4k_ffn_gate_up_geglu_down(dWg, dWu, dWd, ops.Q6_K, dx, H, I)
        y = torch.full((H,), float("nan"), device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        st = lib.qws_q4k_ffn_gate_up_geglu_down_noalloc(_ptr(dWg), _ptr(dWu), _ptr(dWd),
                                                        ops.Q6_K, _ptr(dx), _ptr(y), H, I, stream)
        assert st == 0, lib.qws_last_error().decode()
        torch.cuda.synchronize()
        if call > 0:
            # the module is loaded by now: a call must not take device memory
            assert torch.cuda.mem_get_info()[0] == free_before, "the no-alloc call allocated"
        a = y.cpu().numpy().astype(np.float64)
        b = y_ws.cpu().numpy().astype(np.float64)
        ref_oracle = oracle.ffn(oracle.Q4_K, Wg, Wu, oracle.Q6_K, Wd, H, I, x)
        tol = np.maximum(1e-4 * np.abs(b), 1e-4 * ref_oracle["bound_y"])
        assert np.all(np.abs(a - b) <= tol), f"call {call}: noalloc differs from workspace path"
        # and both meet the FFN tolerance against the oracle
        err = np.abs(a - ref_oracle["y"])
        assert np.all((err <= 1e-4 * np.abs(ref_oracle["y"])) | (err <= 1e-4 * ref_oracle["bound_y"]))
    assert ops.device_error() == 0


def test_ffn_noalloc_rejects_sizes_beyond_its_scratch():
    build.build()
    lib = _lib.lib()
    A = C.c_void_p(0x10000)
    too_big = 20480 + 256
    st = lib.qws_q4k_ffn_gate_up_geglu_down_noalloc(A, A, A, ops.Q6_K, A, A, 2560, too_big, None)
    assert st == 2   # QWS_ERR_SHAPE, nothing enqueued
    assert "exceeds" in lib.qws_last_error().decode()
