"""The precision-preserved all-reduce on the GPU path: a one-rank NCCL group
(127.0.0.1) runs the all-to-all, the library's reduce kernel and the
all-gather on device buffers; the result must equal the oracle's reduce of the
one gradient bit for bit (more ranks need more GPUs; the exchange pattern for
2 and 4 ranks is checked on CPU by test_allreduce_gloo.py)."""
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

from gradient_quantization_gb300 import synthetic
from gradient_quantization_gb300.allreduce import precision_preserved_allreduce

pytestmark = pytest.mark.gpu
BLOCK = 128


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture(scope="module")
def nccl_group():
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % _free_port(), rank=0,
                            world_size=1, device_id=torch.device("cuda", 0))
    yield
    dist.destroy_process_group()


def test_one_rank_allreduce_is_the_local_reduce(oracle, nccl_group):
    n = BLOCK * 1031
    vals = synthetic.reduce_shard_values_np(seed=61, W=1, n=n)[0]
    c, s = oracle.grad_accum_fp8(np.zeros(n, np.uint8), np.zeros(n // BLOCK, np.float32), vals)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    oc, os_ = precision_preserved_allreduce(torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(),
                                            naive_overflow_count=cnt)
    want_c, want_s, want_cnt = oracle.reduce_fp8_shards(c, s, 1, n)
    assert np.array_equal(oc.cpu().numpy(), want_c)
    assert np.array_equal(os_.cpu().numpy().view(np.uint32), want_s.view(np.uint32))
    assert int(cnt.item()) == want_cnt == 0
