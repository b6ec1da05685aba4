"""The GEMMs' failure path on the GPU, without a fault: a probe kernel's one
pipeline wait (the same bounded mbarrier wait the GEMMs use) runs out on a
barrier nothing arrives on; agoq_device_status must then report the timeout
once, and the context must stay usable: a GEMM launched afterwards matches the
oracle and leaves the status clean."""
import time

import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_reports_timeout_then_context_is_usable(oracle):
    agoq.agoq_device_status()                       # start from a clean status word
    t0 = time.perf_counter()
    agoq.agoq_test_wait_timeout(2_000_000)          # about a millisecond at GB300 clocks
    with pytest.raises(agoq.AgoqError) as err:
        agoq.agoq_device_status()
    assert "timeout" in str(err.value).lower() or "7" in str(err.value)
    assert time.perf_counter() - t0 < 30.0
    agoq.agoq_device_status()                       # read and cleared: clean again

    M, N, K = 256, 512, 128
    dy, x = synthetic.wgrad_exact_sum_inputs_np(seed=5, M=M, N=N, K=K)
    xc, xs = oracle.quant_act(x.reshape(-1), 4)
    dw = agoq.agoq_wgrad_gemm_int4(G.dev_bf16(dy), G.dev(xc), G.dev(xs), M, N, K)
    agoq.agoq_device_status()
    # exact-sum operands: the binary64 product is the binary32 accumulator exactly
    exact = oracle.wgrad_gemm_int4_f64(dy, xc, xs, M, N, K).astype(np.float32)
    want = oracle.f32_to_bf16(exact)
    assert np.array_equal(G.host_bits_bf16(dw).reshape(M, N), want.reshape(M, N))
