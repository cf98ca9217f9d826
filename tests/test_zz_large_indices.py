"""Indices past 2^31 on the GPU: one layer of 2^31 + 4101 elements per
worker (a tiny layer before it shifts its offset), so the per-tensor index,
the fused [W][N] buffer (2^32 + 8208 halves) and the unit and tile counts all
leave the 32-bit range.  About 60 GB of device memory.

The oracle checks sampled elements (around 0, the layer edge, 2^31 and the
end), whole chunks' norms, the selection on the GPU's own norms, and the
update on the sampled elements; the five-call path must reproduce the
pipeline's reduced gradient bit for bit."""

import numpy as np
import pytest
import torch

import oracle
from gradient_aggregation_gb300 import fc

pytestmark = pytest.mark.gpu


def _u32(x):
    return np.ascontiguousarray(x).view(np.uint32)


def test_indices_past_2_31(fc_lib):
    W, chunk = 2, 1 << 20
    sizes = [3, (1 << 31) + 4101]
    N = sum(sizes)                                   # 2^31 + 4104
    loss_scale, lr, mu = 256.0, 0.01, 0.9
    dev = "cuda"
    gen = torch.Generator(device=dev)
    gen.manual_seed(20261202)
    grads = [[(torch.randn(n, generator=gen, device=dev) * 4.0).to(torch.float16)
              for n in sizes] for _ in range(W)]
    w0 = torch.randn(N, generator=gen, device=dev) * 0.05
    eng = fc.Engine(sizes, W, chunk, 1, 100, loss_scale, lr, mu, w0, keep_a=True)
    eng.step(grads)
    torch.cuda.synchronize()

    rng = np.random.default_rng(7)
    two31 = 1 << 31
    sample = np.unique(np.concatenate([
        np.arange(0, 16), np.arange(two31 - 16, two31 + 16), np.arange(N - 16, N),
        rng.integers(0, N, 2000)])).astype(np.int64)
    st = torch.from_numpy(sample).to(dev)
    in0 = st < sizes[0]
    x = np.empty((W, sample.size), np.float16)
    for w in range(W):
        v = torch.empty(sample.size, dtype=torch.float16, device=dev)
        v[in0] = grads[w][0][st[in0]]
        v[~in0] = grads[w][1][st[~in0] - sizes[0]]
        x[w] = v.cpu().numpy()

    # a2: sampled elements (residual 0 on the first step)
    a_s = eng.a[st].cpu().numpy()
    assert np.array_equal(_u32(a_s), _u32(oracle.tree_reduce(x, loss_scale)))

    # a3: whole chunks, including the one across 2^31 and the short last one
    C = fc.fc_num_chunks(N, chunk)
    norms = eng.norms.cpu().numpy()
    for c in (0, 1, C // 2, C - 2, C - 1):
        lo, hi = c * chunk, min(c * chunk + chunk, N)
        want = oracle.chunk_norms(eng.a[lo:hi].cpu().numpy(), chunk)[0]
        assert abs(float(norms[c]) - float(want)) <= 1e-6 * float(want), c

    # a4: the selection on the GPU's own norms
    k = oracle.keep_count(C, 1, 100)
    idx, mask, _, thr = oracle.chunk_select(norms, k, want_packed=False)
    assert np.array_equal(eng.idx.cpu().numpy(), idx)
    assert np.array_equal(eng.mask.cpu().numpy(), mask)
    assert _u32(eng.threshold.cpu().numpy())[0] == _u32(np.float32(thr))

    # a5: the update on the sampled elements (one element per "chunk")
    r = np.zeros(sample.size, np.float32)
    v = np.zeros(sample.size, np.float32)
    wt = w0[st].cpu().numpy().astype(np.float32)
    oracle.residual_sgd_update(a_s, mask[sample // chunk], 1, lr, mu, r, v, wt)
    for got, want in ((eng.residual, r), (eng.velocity, v), (eng.weights, wt)):
        assert np.array_equal(_u32(got[st].cpu().numpy()), _u32(want))
    del w0

    # a1 + a2 through the five calls: the fused buffer and its reduction
    fused = torch.empty(W * N, dtype=torch.float16, device=dev)
    assert fc.fc_fuse_pack(grads, fused) == [0, sizes[0]]
    for w in range(W):
        got = fused[w * N + st].cpu().numpy()
        assert np.array_equal(got.view(np.uint16), x[w].view(np.uint16))
    del grads
    a2 = torch.empty(N, dtype=torch.float32, device=dev)
    fc.fc_tree_reduce(fused, W, N, loss_scale, None, a2)
    torch.cuda.synchronize()
    assert torch.equal(a2.view(torch.int32), eng.a.view(torch.int32))
    del fused, a2, eng
    torch.cuda.empty_cache()
