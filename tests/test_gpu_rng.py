"""Generator ownership ([explainer] RNG ownership: per-request seed / offset, a
device-resident offset for CUDA-graph replay), through the C ABI."""
import numpy as np
import pytest

import workloads
from oracle import dual_pivot
from tests.helpers import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ms():
    ensure_built()
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import min_sampling_gb300
    return min_sampling_gb300


def _u64(a):
    import torch
    return torch.from_numpy(np.asarray(a, dtype=np.uint64)).cuda()


def _rows():
    import torch
    w = workloads.config1()
    return w, torch.from_numpy(w.probs).cuda()


def test_scalar_state_matches_the_plain_entry(ms):
    import torch
    w, P = _rows()
    idx = torch.from_numpy(np.repeat(np.arange(4, dtype=np.int32), 64)).cuda()
    k = torch.from_numpy(w.top_k[idx.cpu().numpy()]).cuda()
    p = torch.from_numpy(w.top_p[idx.cpu().numpy()]).cuda()
    for order in ("joint", "top_k_first"):
        a = ms.top_k_top_p_sampling(P, k, p, None, order, idx, seed=77, offset=3)
        b = ms.top_k_top_p_sampling_rng(P, k, p, None, order, idx, seed=77, offset=3)
        c = ms.top_k_top_p_sampling_rng(P, k, p, None, order, idx, offsets=_u64(np.full(256, 3)), seed=77)
        od = _u64([1])
        d = ms.top_k_top_p_sampling_rng(P, k, p, None, order, idx, offset_dev=od, seed=77, offset=2)
        for x in (b, c, d):
            assert torch.equal(a[0], x[0]) and torch.equal(a[1], x[1])


def test_per_request_seeds_follow_the_request(ms):
    """With per-request seeds a request draws the same token wherever it sits in the
    batch, and that token is the oracle's run of the pages' algorithm on stream 0."""
    import torch
    w, P = _rows()
    rng = np.random.default_rng(5)
    n = 256
    src = rng.integers(0, 4, n).astype(np.int32)
    seeds = rng.integers(0, 2 ** 63, n, dtype=np.int64).astype(np.uint64)
    offs = rng.integers(0, 2 ** 40, n, dtype=np.int64).astype(np.uint64)
    k, p = w.top_k[src], w.top_p[src]
    t1, v1, r1 = ms.top_k_top_p_sampling_rng(P, torch.from_numpy(k).cuda(), torch.from_numpy(p).cuda(), None,
                                             "joint", torch.from_numpy(src).cuda(), seeds=_u64(seeds),
                                             offsets=_u64(offs), return_rounds=True)
    perm = rng.permutation(n)
    t2, v2 = ms.top_k_top_p_sampling_rng(P, torch.from_numpy(k[perm]).cuda(), torch.from_numpy(p[perm]).cuda(),
                                         None, "joint", torch.from_numpy(src[perm]).cuda(), seeds=_u64(seeds[perm]),
                                         offsets=_u64(offs[perm]))
    t1, t2 = t1.cpu().numpy(), t2.cpu().numpy()
    assert np.array_equal(t1[perm], t2)
    r1 = r1.cpu().numpy()
    agree = 0
    for b in range(n):
        ref = dual_pivot.sample_philox(w.probs[src[b]], int(k[b]), float(p[b]), None, "joint",
                                       seed=int(seeds[b]), offset=int(offs[b]), row=0)
        agree += int(ref[0] == t1[b] and ref[2] == r1[b])
    assert agree >= 0.99 * n, agree


def test_device_offset_advances_inside_a_captured_graph(ms):
    import torch
    w, P = _rows()
    idx = torch.from_numpy(np.repeat(np.arange(4, dtype=np.int32), 64)).cuda()
    k = torch.from_numpy(w.top_k[idx.cpu().numpy()]).cuda()
    p = torch.from_numpy(w.top_p[idx.cpu().numpy()]).cuda()
    od = _u64([10])
    ms.top_k_top_p_sampling_rng(P, k, p, None, "top_k_first", idx, offset_dev=od, seed=5)  # first-call setup
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        tok, valid = ms.top_k_top_p_sampling_rng(P, k, p, None, "top_k_first", idx, offset_dev=od, seed=5)
        ms.advance_offset(od, 1)
    od.copy_(_u64([10]))  # capture ran nothing; the replays start from offset 10
    got = []
    for _ in range(3):
        graph.replay()
        got.append(tok.clone())
    torch.cuda.synchronize()
    assert int(od.cpu().numpy()[0]) == 13
    for i in range(3):
        ref = ms.top_k_top_p_sampling(P, k, p, None, "top_k_first", idx, seed=5, offset=10 + i)
        assert torch.equal(got[i], ref[0])
    assert not torch.equal(got[0], got[1])
