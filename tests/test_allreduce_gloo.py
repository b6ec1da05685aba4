"""The precision-preserved all-reduce's exchange steps (all-to-all of FP8
shards, local reduce in rank order, all-gather) on CPU ranks over gloo
(127.0.0.1), world sizes 2 and 4, with the oracle's local reduce in place of
the device kernel.  Every rank must end with exactly the oracle's reduce of
the W full gradients (no block straddles a shard), and the summed naive
overflow count must equal the oracle's count over the whole gradient."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from gradient_quantization_gb300 import synthetic

BLOCK = 128


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_gradients(oracle, world, n, seed):
    """FP8 gradients (codes, scales) of every rank: the block quantization of
    seeded BF16 values, scaled up so that naive FP8 sums overflow somewhere."""
    vals = synthetic.reduce_shard_values_np(seed=seed, W=world, n=n)
    f = (vals.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** 14)
    vals = synthetic.bf16_bits_from_f32(f)
    out = []
    for r in range(world):
        c, s = oracle.grad_accum_fp8(np.zeros(n, np.uint8), np.zeros(n // BLOCK, np.float32), vals[r])
        out.append((c, s))
    return out


def _oracle_reduce(oracle):
    def red(shards, shard_scales, W, n, count):
        c, s, cnt = oracle.reduce_fp8_shards(shards.numpy(), shard_scales.numpy(), W, n,
                                             count_naive=count is not None)
        if count is not None:
            count += int(cnt)
        return torch.from_numpy(c), torch.from_numpy(s)
    return red


def _worker(rank, world, port, n, seed, q):
    import torch.distributed as dist
    from oracle import oracle
    from gradient_quantization_gb300.allreduce import precision_preserved_allreduce
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        c, s = _rank_gradients(oracle, world, n, seed)[rank]
        cnt = torch.zeros(1, dtype=torch.int64)
        oc, os_ = precision_preserved_allreduce(torch.from_numpy(c), torch.from_numpy(s),
                                                naive_overflow_count=cnt,
                                                local_reduce=_oracle_reduce(oracle))
        bad = None
        try:
            precision_preserved_allreduce(torch.from_numpy(c[:n - BLOCK]),
                                          torch.from_numpy(s[:n // BLOCK - 1]))
        except ValueError as e:
            bad = str(e)
        q.put((rank, oc.numpy().tobytes(), os_.numpy().tobytes(), int(cnt.item()), bad))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_allreduce_matches_oracle_reduce_of_all_ranks(oracle, world):
    n = world * BLOCK * 37
    seed = 40 + world
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, seed, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    grads = _rank_gradients(oracle, world, n, seed)
    want_c, want_s, want_cnt = oracle.reduce_fp8_shards(
        np.stack([g[0] for g in grads]), np.stack([g[1] for g in grads]), world, n)
    assert want_cnt > 0, "the inputs should make some naive FP8 sums overflow"
    for rank, c, s, cnt, bad in results:
        assert np.frombuffer(c, np.uint8).tobytes() == want_c.tobytes(), "codes on rank %d" % rank
        assert np.frombuffer(s, np.float32).view(np.uint32).tobytes() == \
            want_s.view(np.uint32).tobytes(), "scales on rank %d" % rank
        assert cnt == want_cnt
        assert bad is not None and "multiple" in bad
