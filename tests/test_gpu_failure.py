"""Failure detection on the GPU without a fault: a bounded device-side wait that
runs out sets the library's status word, the host reads FP4Q_ERR_TIMEOUT, and
the context keeps working (a quantize afterwards is still bit-exact)."""
import time

import numpy as np
import pytest

from _helpers import dev_bf16, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import micro_scaled_fp4_gb300.fp4q as fq
    fq.load()
    return fq


def test_wait_that_runs_out_is_reported(fq, oracle):
    import torch
    fq.fp4q_device_status(reset=True)                             # start from a clean word
    assert fq.fp4q_device_status(reset=True) == 0
    t0 = time.time()
    fq.fp4q_check_wait_timeout(200_000_000)                      # 0.2 s limit
    word = fq.fp4q_device_status(reset=True)                      # synchronizes
    assert time.time() - t0 >= 0.15
    assert word == 1 << 31
    assert fq.fp4q_device_status() == 0                           # cleared by the reset
    # the same through the stream-scoped read
    fq.fp4q_check_wait_timeout(100_000_000)
    assert fq.fp4q_stream_status(reset=True) == 1 << 31          # waits for the current stream
    assert fq.fp4q_stream_status() == 0
    # the context is still usable
    from micro_scaled_fp4_gb300 import workloads as W
    x = W.activation_bf16(16, 256, seed=9)
    q, s = fq.mx_quantize(dev_bf16(x))
    qr, sr = oracle.mx_quantize(x)
    assert np.array_equal(host(q), qr) and np.array_equal(host(s), sr)


def test_wait_limit_is_validated(fq):
    with pytest.raises(fq.Fp4qError) as e:
        fq.fp4q_check_wait_timeout(0)
    assert e.value.status == 1
    with pytest.raises(fq.Fp4qError):
        fq.fp4q_check_wait_timeout(5_000_000_000)
