"""Failure detection on the GPU without a GPU fault.

Every wait inside the library's kernels is bounded; when one gives up, the
kernel records a code, returns, and qws_device_error() reports it as
QWS_ERR_TIMEOUT.  qws_selftest_wait_timeout runs the two wait primitives the
kernels use -- the streaming engine's mbarrier wait and the decode chain's
stamped-word poll -- on something that never becomes ready (a flag nothing
sets), with a short limit.  The test checks the reported code, that the wait
gave up after its short limit rather than the ~1 s default, and that the
library keeps working in the same process afterwards.
"""
import ctypes as C
import time

import numpy as np
import pytest
import torch

import oracle
from quantized_weight_streaming_q4k_gb300 import _lib, build, ops, synth

pytestmark = pytest.mark.gpu

QWS_ERR_TIMEOUT = 7
CONSUMER_GAVE_UP = 1


@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier_wait", "stamped_poll"])
def test_bounded_wait_gives_up_and_library_recovers(kind):
    build.build()
    lib = _lib.lib()
    torch.cuda.set_device(0)
    assert ops.device_error() == 0
    word = torch.zeros(2, dtype=torch.float32, device="cuda")   # one 8-byte stamped word
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    limit = 2_000_000        # clock cycles: about a millisecond
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = lib.qws_selftest_wait_timeout(kind, limit, C.c_void_p(word.data_ptr()), stream)
    assert st == 0, lib.qws_last_error().decode()
    code = C.c_uint(0)
    st = lib.qws_device_error(C.byref(code))
    elapsed = time.perf_counter() - t0
    assert st == QWS_ERR_TIMEOUT
    assert code.value == CONSUMER_GAVE_UP
    assert elapsed < 0.5, f"the wait took {elapsed:.3f} s: the short limit was not honoured"
    # cleared by the read, and the context is still usable: a matvec is right
    assert ops.device_error() == 0
    rows, hidden = 300, 512
    g = synth.rng(7100, kind)
    W = synth.q4_k_matrix(g, rows, hidden)
    x = synth.normal_vector(g, hidden)
    y = ops.q4k_matvec(torch.from_numpy(W).cuda(), torch.from_numpy(x).cuda(), rows, hidden)
    torch.cuda.synchronize()
    ref, bound = oracle.matvec(oracle.Q4_K, W, rows, hidden, x)
    assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - ref) <= 1e-5 * bound)
    assert ops.device_error() == 0
