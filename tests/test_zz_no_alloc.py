"""The allocation-free HSI pool selection (csa2_hier_pool_select_static).

It is for callers that cannot allocate device memory where they run the
selection (a runtime replaying a fixed memory plan, or host code holding only
raw device pointers): it keeps its scratch in a static device array of the
library instead of a caller workspace.  This test calls it through the C ABI
twice in a row, on different inputs, and checks each result against the
workspace-taking csa2_hier_pool_select on the same inputs; it also checks that
a request larger than the static array is refused.  It lives in a file that
pytest collects last and passes both alone and after the other tests."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def c2():
    import sparse_attention_fp4_csa2_gb300.build as b
    b.build()
    import sparse_attention_fp4_csa2_gb300 as c
    L = c.lib()
    P = ctypes.c_void_p
    L.csa2_hier_pool_select_static.argtypes = [P, P, ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(c.Params), P, P]
    L.csa2_hier_pool_select_static.restype = ctypes.c_int
    return c


def _static_call(c2, bs, nv, n_max, p, pool):
    st = c2.lib().csa2_hier_pool_select_static(
        ctypes.c_void_p(bs.data_ptr()), ctypes.c_void_p(nv.data_ptr()), bs.shape[0], n_max, ctypes.byref(p),
        ctypes.c_void_p(pool.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


@pytest.mark.parametrize("seed", [0])
def test_static_pool_select_matches_workspace_version_twice(c2, seed):
    cases = [(4, 200_000, [200_000, 150_001, 8, 77_777], 2048), (3, 40_000, [40_000, 39_999, 1], 512)]
    for i, (B, n_max, n_vis, nb) in enumerate(cases):
        g = torch.Generator(device="cuda").manual_seed(seed + i)
        nblk = (n_max + 7) // 8
        bs = torch.randn(B, nblk, device="cuda", generator=g)
        for b in range(B):
            bs[b, (n_vis[b] + 7) // 8:] = -float("inf")
        bs[0, 5:9] = 3.0                         # ties: the lower block wins
        nv = torch.tensor(n_vis, dtype=torch.int32, device="cuda")
        p = c2.Params.make(candidate_topk_blocks=nb)
        ref = torch.empty(B, nb, dtype=torch.int32, device="cuda")
        c2.hier_pool_select(bs, nv, n_max, p, ref, c2.workspace(c2.OP_POOL, B, n_max, p))
        ref_launches = c2.last_launch_count()
        got = torch.full((B, nb), -5, dtype=torch.int32, device="cuda")
        assert _static_call(c2, bs, nv, n_max, p, got) == 0
        assert c2.last_launch_count() == ref_launches > 0   # the same kernels, counted for this call
        assert c2.get_device_status() == 0
        assert torch.equal(got, ref), f"call {i}: static-scratch pool differs"


def test_static_pool_select_refuses_oversize(c2):
    B, n_max = 64, 1 << 22
    p = c2.Params.make()
    bs = torch.empty(1, device="cuda")
    nv = torch.empty(1, dtype=torch.int32, device="cuda")
    pool = torch.empty(1, dtype=torch.int32, device="cuda")
    st = c2.lib().csa2_hier_pool_select_static(
        ctypes.c_void_p(bs.data_ptr()), ctypes.c_void_p(nv.data_ptr()), B, n_max, ctypes.byref(p),
        ctypes.c_void_p(pool.data_ptr()), None)
    assert st == 3      # CSA2_ERR_WORKSPACE: more than the static scratch holds
    assert c2.last_launch_count() == 0
