"""moe_permute_noalloc: the permutation for callers that cannot allocate GPU
memory (a host framework owns every device allocation, a fixed memory budget,
or cudaMalloc's device-wide synchronisation is not allowed).  Its scratch is a
fixed device array inside the library, so it needs no layer and allocates
nothing.  Checked bit for bit against the oracle's permutation (and against
the layer's own permutation entry point, moe_debug_permute) on two calls in a
row; the second call finds the first call's contents in the shared scratch.
The cases cover the one-CTA path (N <= 128, up to E = 1024 and k = 32, whose
shared memory needs the raised per-device limit) and the multi-block path.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import numpy as np
import pytest
import torch

from helpers import need_gpu, small_spec
from oracle.native import layer as olayer
from routed_expert_layer_gemv_gb300 import capi
from routed_expert_layer_gemv_gb300.layer import MoELayer

pytestmark = pytest.mark.gpu


def _idx(N, E, k, seed):
    g = np.random.default_rng(seed)
    p = g.dirichlet(np.ones(E) * 0.3)
    return np.stack([np.sort(g.choice(E, k, replace=False, p=p)) for _ in range(N)]).astype(np.int32)


def _outs(N, E, k):
    return [torch.full((E,), -7, dtype=torch.int32, device="cuda"),
            torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
            torch.full((N * k,), -7, dtype=torch.int32, device="cuda"),
            torch.full((N * k,), -7, dtype=torch.int32, device="cuda")]


@pytest.mark.parametrize("E,k,Ns", [(128, 8, (4096, 1000)), (256, 8, (3000, 129)),
                                    (8, 2, (64, 5000)), (1024, 32, (200, 8192)),
                                    (1024, 32, (128, 37)), (256, 8, (1, 128))])
def test_noalloc_permute_matches_oracle_twice(E, k, Ns):
    need_gpu()
    L = MoELayer(small_spec(E=E, k=k, n_slots=E), max(Ns))
    for call, N in enumerate(Ns):
        idx_np = _idx(N, E, k, 100 * E + call)
        idx = torch.from_numpy(idx_np).cuda()
        got = _outs(N, E, k)
        capi.moe_permute_noalloc(idx, N, k, E, *got)
        lay = _outs(N, E, k)
        capi.moe_debug_permute(L.h, idx, N, *lay)
        torch.cuda.synchronize()
        counts, offsets, row_of, tok_of = olayer.permute(idx_np, E)
        want = [counts, offsets, row_of.reshape(-1), tok_of]
        for name, a, w in zip(("counts", "offsets", "row_of", "tok_of"), got, want):
            assert np.array_equal(a.cpu().numpy(), w), (name, E, k, N, call)
        for a, b in zip(got, lay):
            assert torch.equal(a.cpu(), b.cpu()), (E, k, N, call)
    L.close()


def test_noalloc_permute_rejects_sizes_beyond_its_scratch():
    need_gpu()
    N, E, k = 262144 // 8 + 1, 128, 8
    d = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.MoeError) as e:
        capi.moe_permute_noalloc(d, N, k, E, d, d, d, d)
    assert e.value.status == capi.MOE_ERR_ARG and "262144" in str(e.value)
    with pytest.raises(capi.MoeError):
        capi.moe_permute_noalloc(d, 4, 0, E, d, d, d, d)
    capi.moe_permute_noalloc(d, 0, k, E, d, d, d, d)      # N == 0: nothing to do
