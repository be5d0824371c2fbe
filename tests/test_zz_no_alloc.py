"""The router entry point that allocates nothing (moe_route_noalloc).

Some callers cannot call cudaMalloc: code inside another framework's memory
pool, services that forbid device allocation after start-up, or work being
captured into a CUDA graph. This test calls the no-allocation entry point
through the C ABI, twice in a row on different inputs, and checks each result
against the context-based moe_route on the same inputs. It is collected last
and creates everything it needs, so it passes alone in a fresh process and
after the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bec():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bounded_expert_cache_gb300 as m
    return m


def _noalloc(lib, x, xt, Wr, bias, k):
    T, H = x.shape
    E = Wr.shape[0]
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    wt = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    st = lib.moe_route_noalloc(C.c_void_p(x.data_ptr()), xt, T, H, E, k,
                               C.c_void_p(Wr.data_ptr()),
                               None if bias is None else C.c_void_p(bias.data_ptr()),
                               C.c_void_p(idx.data_ptr()), C.c_void_p(wt.data_ptr()),
                               C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.moe_last_error(None)
    return idx, wt


def _reference(bec, x, Wr, bias, k):
    T, H = x.shape
    E = Wr.shape[0]
    ctx = bec.Context(1, E, k, H, 128, 0, 0, min(E, 8), 0, 1, 0, 262144, T)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ctx.route(0, x, Wr, bias, idx, wt)
    torch.cuda.synchronize()
    ctx.close()
    return idx.cpu().numpy(), wt.cpu().numpy()


def test_noalloc_route_matches_context_route_twice(bec):
    from bounded_expert_cache_gb300 import _native as N
    lib = N.lib
    cases = []
    w = W.WORKLOADS["prefill"]  # hidden 2048, 256 experts, top-8, Zipf bias
    xb = W.activations(w, 0, 8)
    cases.append((torch.from_numpy(xb[:4].view(np.int16).copy()).view(torch.bfloat16).cuda(), N.BF16,
                  torch.from_numpy(W.router_weights(w, 0)).cuda(),
                  torch.from_numpy(W.router_bias(w, 0)).cuda(), w.top_k))
    t = W.WORKLOADS["tiny"]  # fp32 activations, 16 experts, top-2, no bias
    cases.append((torch.from_numpy(W.activations(t, 0)).cuda(), N.F32,
                  torch.from_numpy(W.router_weights(t, 0)).cuda(), None, t.top_k))
    refs = [_reference(bec, x, Wr, b, k) for (x, _, Wr, b, k) in cases]
    free_before = None
    for i, ((x, xt, Wr, b, k), (ridx, rw)) in enumerate(zip(cases, refs)):
        if i == 1:
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
        idx, wt = _noalloc(lib, x, xt, Wr, b, k)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), ridx), i
        assert np.allclose(wt.cpu().numpy(), rw, rtol=1e-5, atol=1e-7), i
    # the second call (after the one-time set-up) leaves device memory unchanged
    assert torch.cuda.mem_get_info()[0] == free_before


def test_noalloc_route_rejects_oversize(bec):
    from bounded_expert_cache_gb300 import _native as N
    x = torch.zeros((65, 32), device="cuda")
    Wr = torch.zeros((256, 32), device="cuda")
    idx = torch.empty((65, 8), dtype=torch.int32, device="cuda")
    wt = torch.empty((65, 8), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = N.lib.moe_route_noalloc(C.c_void_p(x.data_ptr()), N.F32, 65, 32, 256, 8,
                                 C.c_void_p(Wr.data_ptr()), None, C.c_void_p(idx.data_ptr()),
                                 C.c_void_p(wt.data_ptr()), C.c_void_p(s))
    assert st == 1
    x2 = torch.zeros((64, 32), device="cuda")
    Wr2 = torch.zeros((512, 32), device="cuda")  # 64 * 512 > 16384
    st = N.lib.moe_route_noalloc(C.c_void_p(x2.data_ptr()), N.F32, 64, 32, 512, 8,
                                 C.c_void_p(Wr2.data_ptr()), None, C.c_void_p(idx.data_ptr()),
                                 C.c_void_p(wt.data_ptr()), C.c_void_p(s))
    assert st == 1 and b"static scratch limit" in N.lib.moe_last_error(None)
