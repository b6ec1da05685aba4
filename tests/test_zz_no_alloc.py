"""agoq_rmsnorm_backward_noalloc: the single-read RMSNorm backward for callers
that cannot allocate device memory where they call it (an operator hook that
must not touch its framework's allocator, code running while device memory is
reserved or accounted by someone else, a plain C caller without a device
allocator).  Its scratch is a static array inside the library instead of a
workspace argument, so the call allocates nothing.

The GPU test calls the entry point through the C ABI (ctypes, raw pointers)
twice in a row, on different inputs, and compares each result with the
workspace entry point agoq_rmsnorm_backward_ws on the same inputs: the same
kernels and the same partition of the rows, so dx, rstd and dw agree bit for
bit (zero tolerance, tighter than the oracle bounds the other RMSNorm tests
use).  The second call has fewer rows than the first, so it must not read what
the first call left in the shared array.  The file is named to be collected
last.
"""
import ctypes

import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic

SHAPE, NULL = 2, 1


def _inputs(T, H, bits, seed):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_t(4, T * H).astype(np.float32)).to(torch.bfloat16).cuda()
    codes, scales = agoq.agoq_quant_act(x, bits)
    dy = torch.from_numpy(rng.standard_normal(T * H).astype(np.float32)).to(torch.bfloat16).cuda()
    w = torch.from_numpy((1 + 0.1 * rng.standard_normal(H)).astype(np.float32)).to(
        torch.bfloat16).cuda()
    return codes, scales, dy, w


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    L = agoq.lib()
    H, bits, eps = 4096, 4, 1e-6
    for T, seed in ((2000, 1), (333, 2)):
        codes, scales, dy, w = _inputs(T, H, bits, seed)
        dx = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        rstd = torch.empty(T, dtype=torch.float32, device="cuda")
        dw = torch.empty(H, dtype=torch.float32, device="cuda")
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = L.agoq_rmsnorm_backward_noalloc(_p(codes), _p(scales), _p(dy), _p(w), T, H, bits,
                                             ctypes.c_float(eps), _p(dx), _p(rstd), _p(dw), st)
        assert rc == 0, agoq.lib().agoq_status_string(rc).decode()
        ws = torch.empty(agoq.agoq_rmsnorm_backward_workspace_bytes(H), dtype=torch.uint8,
                         device="cuda")
        rdx, rrstd, rdw = agoq.agoq_rmsnorm_backward_ws(codes, scales, dy, w, T, H, bits, eps, ws)
        torch.cuda.synchronize()
        assert torch.equal(dx, rdx), "dx, %d rows" % T
        assert torch.equal(rstd, rrstd), "rstd, %d rows" % T
        assert torch.equal(dw, rdw), "dw, %d rows" % T
        assert torch.isfinite(dw).all()


def test_noalloc_rejects_rows_beyond_its_scratch():
    """Argument checks return before any launch: rows longer than the static
    scratch holds, and a missing dw."""
    L = agoq.lib()
    fake = ctypes.c_void_p(1 << 40)
    args = (fake, fake, fake, fake, 8, 8192, 4, ctypes.c_float(1e-6), fake, fake, fake, None)
    assert L.agoq_rmsnorm_backward_noalloc(*args) == SHAPE
    args = (fake, fake, fake, fake, 8, 4096, 4, ctypes.c_float(1e-6), fake, fake, None, None)
    assert L.agoq_rmsnorm_backward_noalloc(*args) == NULL
    assert synthetic.DBCA_RMSNORM_SHAPE[1] <= 4096   # the workload's rows fit the scratch
