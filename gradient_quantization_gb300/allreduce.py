"""QuanGrad's precision-preserved all-reduce of an FP8 block-scaled gradient
("AGoQ: Activation and Gradient Quantization for Memory-Efficient Distributed
Training of LLMs", section 2.B "Precision-Preserved All-Reduce", steps 1-3).

Every rank holds the whole gradient as E4M3 codes [n] with FP32 block scales
[n/128].  With W ranks and n a multiple of 128 W, the gradient is cut into W
shards of n/W elements (whole blocks):

  1. all-to-all: rank r receives shard r of every rank, stacked in rank order
     ([W][n/W] codes, [W][n/(128 W)] scales: the shard-major layout of the
     local reduce);
  2. local reduce: the W shards are dequantized, summed in binary32 in rank
     order and requantized with fresh block scales (agoq_reduce_fp8_shards,
     the library's kernel);
  3. all-gather: every rank receives every rank's reduced shard, in rank
     order, so all ranks end with the same reduced FP8 gradient.

Because no block straddles a shard, the result equals the local reduce of
the W full gradients.  The exchanges are torch.distributed collectives (NCCL
between GPUs); the arithmetic is the library's reduce kernel, or the
`local_reduce` callable given in its place.
"""
import torch
import torch.distributed as dist

from . import agoq

BLOCK = 128


def _device_reduce(shards, shard_scales, W, n, count):
    out, out_scales = agoq.agoq_reduce_fp8_shards(shards, shard_scales, W, n,
                                                  naive_overflow_count=count)
    return out, out_scales


def precision_preserved_allreduce(codes, scales, group=None, naive_overflow_count=None,
                                  local_reduce=None):
    """Precision-preserved all-reduce of this rank's FP8 gradient (codes uint8
    [n], scales float32 [n/128]) over `group`.  Returns the reduced (codes,
    scales), the same on every rank.

    naive_overflow_count: optional one-element int64 tensor (on the codes'
    device); it receives the number of elements, over the whole gradient,
    whose naive FP8 running sum left the E4M3 range (summed over ranks).
    local_reduce: callable (shards, shard_scales, W, n_shard, count) ->
    (codes, scales) used for step 2 instead of the library's kernel.
    """
    if codes.dtype != torch.uint8 or scales.dtype != torch.float32:
        raise TypeError("codes must be uint8 and scales float32")
    W = dist.get_world_size(group)
    n = codes.numel()
    if n % (BLOCK * W) or scales.numel() != n // BLOCK:
        raise ValueError("n must be a multiple of 128 * world size and scales hold n/128 values")
    ns = n // W
    dev = codes.device
    # 1. all-to-all: chunk j of the input goes to rank j; chunk i of the output
    # comes from rank i
    recv_c = torch.empty(W * ns, dtype=torch.uint8, device=dev)
    recv_s = torch.empty(W * (ns // BLOCK), dtype=torch.float32, device=dev)
    dist.all_to_all_single(recv_c, codes.reshape(-1).contiguous(), group=group)
    dist.all_to_all_single(recv_s, scales.reshape(-1).contiguous(), group=group)
    # 2. local reduce of the W shards, in rank order
    red = local_reduce if local_reduce is not None else _device_reduce
    if naive_overflow_count is not None:
        naive_overflow_count.zero_()
    red_c, red_s = red(recv_c, recv_s, W, ns, naive_overflow_count)
    # 3. all-gather of the reduced shards
    out_c = torch.empty(n, dtype=torch.uint8, device=dev)
    out_s = torch.empty(n // BLOCK, dtype=torch.float32, device=dev)
    dist.all_gather_into_tensor(out_c, red_c.reshape(-1).contiguous(), group=group)
    dist.all_gather_into_tensor(out_s, red_s.reshape(-1).contiguous(), group=group)
    if naive_overflow_count is not None:
        dist.all_reduce(naive_overflow_count, op=dist.ReduceOp.SUM, group=group)
    return out_c, out_s
