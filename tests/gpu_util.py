"""Helpers of the GPU tests: moving seeded inputs to the device, guard-banded
output buffers (sentinel margins that must survive a call), and block sampling."""
import numpy as np
import torch

GUARD = 4096          # bytes of sentinel before and after each guarded buffer
SENTINEL = 0xA5


def dev_bf16(bits_np):
    """uint16 BF16 bit patterns (numpy) -> torch.bfloat16 CUDA tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits_np).view(np.int16).reshape(-1))
    return t.view(torch.bfloat16).cuda()


def host_bits_bf16(t):
    """torch.bfloat16 tensor -> uint16 numpy bit patterns."""
    return t.detach().reshape(-1).view(torch.int16).cpu().numpy().view(np.uint16)


def dev(np_arr):
    return torch.from_numpy(np.ascontiguousarray(np_arr).reshape(-1)).cuda()


class Guarded:
    """A device buffer of `nbytes` with GUARD sentinel bytes on either side."""

    def __init__(self, nbytes, dtype):
        self.nbytes = nbytes
        itemsize = torch.empty((), dtype=dtype).element_size()
        assert GUARD % itemsize == 0 and nbytes % itemsize == 0
        self.raw = torch.full((nbytes + 2 * GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.view = self.raw[GUARD:GUARD + nbytes].view(dtype)

    def intact(self):
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == SENTINEL).all()) and bool((tail == SENTINEL).all())


def sample_blocks(nblocks, count, seed=0):
    """Sorted distinct block indices: the first, the last, and random ones."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(nblocks, size=min(count, nblocks), replace=False).tolist())
    pick.update({0, nblocks - 1})
    return np.array(sorted(pick), np.int64)


def gather_blocks(t, blocks, block_elems):
    """Rows `blocks` of a flat tensor viewed as [nblocks, block_elems] (on the host)."""
    idx = torch.from_numpy(blocks).to(t.device)
    return t.reshape(-1, block_elems).index_select(0, idx).cpu()
