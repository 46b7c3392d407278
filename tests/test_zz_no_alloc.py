"""The no-allocation sampling entry, through the C ABI on a GPU.

fs_top_k_top_p_sampling_noalloc serves callers that may not let a library allocate
device memory (an engine that has reserved nearly all of it, a pool that must see
every allocation, a decode step that must not risk an allocation's device-wide
synchronisation).  It keeps its row summaries in a fixed array built into the
library instead of a per-stream buffer.  It must give exactly the tokens, flags and
round counts of fs_top_k_top_p_sampling on the same inputs, seed and offset, on two
calls in a row (the second call finds the first call's contents in the array).

This file is collected last, so that a run stopping at the first failure has run
every other test before it; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from tests.helpers import ensure_built

P = ctypes.c_void_p
I32 = ctypes.c_int32
U64 = ctypes.c_uint64
ARGS = [P, I32, I32, P, I32, P, P, P, I32, U64, U64, P, P, P, P]


@pytest.mark.gpu
def test_noalloc_entry_matches_the_allocating_entry():
    import torch

    import workloads

    so = ctypes.CDLL(ensure_built())
    for name in ("fs_top_k_top_p_sampling", "fs_top_k_top_p_sampling_noalloc"):
        getattr(so, name).argtypes = ARGS
        getattr(so, name).restype = ctypes.c_int
    so.fs_last_error_string.restype = ctypes.c_char_p
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = workloads.config3(batch=16, with_logits=False)   # 16 rows of 151936, top_k 50, top_p 0.9
    B, V = w.probs.shape
    x = torch.from_numpy(w.probs).to(dev)
    k = torch.from_numpy(w.top_k).to(dev)
    p = torch.from_numpy(w.top_p).to(dev)
    stream = P(torch.cuda.current_stream(dev).cuda_stream)

    def run(name, order, offset):
        tok = torch.full((B,), -7, dtype=torch.int32, device=dev)
        val = torch.full((B,), 7, dtype=torch.uint8, device=dev)
        rnd = torch.full((B,), -7, dtype=torch.int32, device=dev)
        st = getattr(so, name)(P(x.data_ptr()), B, V, None, B, P(k.data_ptr()), P(p.data_ptr()), None, order,
                               1234, offset, P(tok.data_ptr()), P(val.data_ptr()), P(rnd.data_ptr()), stream)
        assert st == 0, (name, st, so.fs_last_error_string())
        torch.cuda.synchronize(dev)
        return tok.cpu().numpy(), val.cpu().numpy(), rnd.cpu().numpy()

    for order in (0, 1):          # top-k-first, joint: both keep their summaries in the fixed array
        for offset in (5, 6):     # two calls in a row on each entry
            ref = run("fs_top_k_top_p_sampling", order, offset)
            got = run("fs_top_k_top_p_sampling_noalloc", order, offset)
            for a, b in zip(ref, got):
                assert np.array_equal(a, b), (order, offset)
            assert got[1].all() and (got[0] >= 0).all() and (got[2] >= 1).all()


def test_noalloc_entry_rejects_batches_beyond_its_scratch():
    """Host-side check, before any CUDA call (runs without a GPU too)."""
    so = ctypes.CDLL(ensure_built())
    f = so.fs_top_k_top_p_sampling_noalloc
    f.argtypes = ARGS
    f.restype = ctypes.c_int
    so.fs_last_error_string.restype = ctypes.c_char_p
    fake = P(0x1000)   # never dereferenced: the size check comes first
    st = f(fake, 2048, 262144, None, 2048, fake, fake, None, 0, 1, 2, fake, fake, None, None)
    assert st == 2
    assert b"FS_NOALLOC_SCRATCH_BYTES" in so.fs_last_error_string()
