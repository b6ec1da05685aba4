"""GPU checks of the INT4-dequant-fused weight-gradient GEMM against the CPU
oracle's binary64 product of the dequantized operands.

Gates (the BF16 output cannot be compared with the unrounded product at 1e-3:
rounding any value to BF16 alone costs about 1.6e-3 relative Frobenius):
  * BF16 output vs bf16_rne(binary64 product): relative Frobenius <= 1e-3;
  * FP32-output variant vs the binary64 product: relative Frobenius <= 1e-3,
    and every entry within the binary32 summation bound K * 2^-23 * sum|terms|;
  * a one-hot dY makes dW rows exactly the dequantized X rows (bit-exact).
"""
import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _inputs(oracle, M, N, K, seed=4):
    dy, x = synthetic.wgrad_inputs_np(seed=seed, M=M, N=N, K=K)
    xc, xs = oracle.quant_act(x.reshape(-1), 4)
    return dy, xc, xs


def _bf16_round(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def _rel_frob(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def _abs_terms(oracle, dy, xc, xs, M, N, K):
    """sum_k |dY[k][m] * Xhat[k][n]| in binary64 (for the per-entry bound)."""
    dyv = np.abs((dy.astype(np.uint32) << 16).view(np.float32).astype(np.float64)).reshape(K, M)
    xh = oracle.dequant_act(xc, xs, K * N, 4)
    xhv = np.abs((xh.astype(np.uint32) << 16).view(np.float32).astype(np.float64)).reshape(K, N)
    return dyv.T @ xhv


# K a multiple of 128 runs the 128-deep instance, the other multiples of 64 the
# 64-deep one; M = 256 and 768 leave the second half of a 512-row pair tile empty,
# M = 128 and 384 also the second CTA's rows of a half; N = 128, 384, 640 end on a
# half-filled 256-column tile and (with N = 768) take the kernel that reads the
# scales without TMA (a scale row that is not a multiple of 16 bytes).
@pytest.mark.parametrize("M,N,K", [(256, 512, 64), (256, 512, 128), (512, 1024, 192),
                                   (768, 512, 320), (2560, 4096, 64), (512, 1024, 384),
                                   (768, 512, 640), (2560, 4096, 128),
                                   (128, 128, 64), (384, 640, 192), (128, 384, 128),
                                   (640, 768, 320), (1152, 1408, 256)])
def test_gemm_matches_fp64_product(oracle, M, N, K):
    dy, xc, xs = _inputs(oracle, M, N, K)
    dyd, xcd, xsd = G.dev_bf16(dy), G.dev(xc), G.dev(xs)
    dwg = G.Guarded(M * N * 2, torch.bfloat16)
    agoq.agoq_wgrad_gemm_int4(dyd, xcd, xsd, M, N, K, dwg.view)
    agoq.agoq_device_status()
    assert dwg.intact()
    ref = oracle.wgrad_gemm_int4_f64(dy, xc, xs, M, N, K)
    got = dwg.view.double().cpu().numpy().reshape(M, N)
    assert _rel_frob(got, _bf16_round(ref)) <= 1e-3
    f32 = agoq.agoq_wgrad_gemm_int4_f32out(dyd, xcd, xsd, M, N, K)
    agoq.agoq_device_status()
    got32 = f32.double().cpu().numpy()
    assert _rel_frob(got32, ref) <= 1e-3
    bound = K * 2.0 ** -23 * _abs_terms(oracle, dy, xc, xs, M, N, K) + 1e-30
    assert (np.abs(got32 - ref) <= bound).all()


def test_one_hot_rows_are_dequantized_rows(oracle):
    M, N, K = 512, 1024, 256
    _, xc, xs = _inputs(oracle, M, N, K, seed=9)
    rng = np.random.default_rng(10)
    pick = rng.integers(0, K, M)
    dy = np.zeros((K, M), np.uint16)
    dy[pick, np.arange(M)] = 0x3F80                     # 1.0
    dw = agoq.agoq_wgrad_gemm_int4(G.dev_bf16(dy), G.dev(xc), G.dev(xs), M, N, K)
    agoq.agoq_device_status()
    xhat = oracle.dequant_act(xc, xs, K * N, 4).reshape(K, N)
    assert np.array_equal(G.host_bits_bf16(dw).reshape(M, N), xhat[pick])


def test_repeatable_across_calls(oracle):
    M, N, K = 512, 1024, 128
    dy, xc, xs = _inputs(oracle, M, N, K, seed=12)
    args = (G.dev_bf16(dy), G.dev(xc), G.dev(xs), M, N, K)
    a = agoq.agoq_wgrad_gemm_int4(*args)
    b = agoq.agoq_wgrad_gemm_int4(*args)
    agoq.agoq_device_status()
    assert torch.equal(a, b)


def test_unaligned_scales_take_the_direct_path(oracle):
    """Scales 4 bytes off a 16-byte boundary (N a multiple of 512, which would
    otherwise load them by TMA): same results as the aligned call."""
    M, N, K = 512, 1024, 128
    dy, xc, xs = _inputs(oracle, M, N, K, seed=13)
    room = torch.zeros(xs.size + 4, dtype=torch.float32, device="cuda")
    xs_off = room[1:1 + xs.size]
    xs_off.copy_(G.dev(xs))
    assert xs_off.data_ptr() % 16 == 4
    args = (G.dev_bf16(dy), G.dev(xc))
    a = agoq.agoq_wgrad_gemm_int4_f32out(*args, G.dev(xs), M, N, K)
    b = agoq.agoq_wgrad_gemm_int4_f32out(*args, xs_off, M, N, K)
    agoq.agoq_device_status()
    assert torch.equal(a, b)


def test_output_16_byte_aligned_takes_the_narrow_stores(oracle):
    """An output 16 bytes off a 32-byte boundary is written with 16-byte stores
    instead of 32-byte ones: the same bits as a 32-byte-aligned output, for the
    BF16 and the FP32 result (two tile rows and columns, a partial last tile)."""
    M, N, K = 640, 384, 128
    dy, xc, xs = _inputs(oracle, M, N, K, seed=14)
    args = (G.dev_bf16(dy), G.dev(xc), G.dev(xs), M, N, K)
    for dtype, fn in ((torch.bfloat16, agoq.agoq_wgrad_gemm_int4),
                      (torch.float32, agoq.agoq_wgrad_gemm_int4_f32out)):
        esz = torch.empty(0, dtype=dtype).element_size()
        room = torch.zeros(M * N + 64 // esz, dtype=dtype, device="cuda")
        off = room[16 // esz:16 // esz + M * N].view(M, N)
        assert off.data_ptr() % 32 == 16
        want = fn(*args)
        fn(*args, off)
        agoq.agoq_device_status()
        assert torch.equal(off, want), str(dtype)
        assert not room[:16 // esz].any() and not room[16 // esz + M * N:].any()
