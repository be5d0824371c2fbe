"""The router entry point that allocates nothing (moe_route_noalloc).

Some callers cannot call cudaMalloc: code inside another framework's memory
pool, services that forbid device allocation after start-up, or work being
captured into a CUDA graph. This test calls the no-allocation entry point
through the C ABI, twice in a row on different inputs, and checks every
result against the CPU oracle's routing (top-k bit-exact, weights to fp32
rounding), including cases at the entry point's limits (T*E equal to the
8,192 logits its static scratch holds, T = 64). It is collected last and
creates everything it needs, so it passes alone in a fresh process and after
the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import workloads as W

from gpu_common import x_to_f64, x_to_torch

pytestmark = pytest.mark.gpu

MAX_LOGITS = 8192  # T*E limit of the static scratch, as declared in the header


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


def _case(name, T, E, H, k, token0=0):
    """Inputs of one call from a seeded workload recipe (router N(0, 0.02),
    activations as the workload draws them), resized to T x E x H."""
    w = W.with_changes(W.WORKLOADS[name], n_experts=E, hidden=H, top_k=k, tokens_per_step=T,
                       n_steps=max(1, (token0 + T + T - 1) // T))
    x = W.activations(w, 0, T, token0=token0)
    Wr = W.router_weights(w, 0)
    bias = W.router_bias(w, 0)
    return w, x, Wr, bias


def _check(lib, N, name, T, E, H, k, token0=0):
    w, x, Wr, bias = _case(name, T, E, H, k, token0)
    xt = N.BF16 if w.x_dtype == "bf16" else N.F32
    idx, wt = _noalloc(lib, x_to_torch(w, x), xt, torch.from_numpy(Wr).cuda(),
                       None if bias is None else torch.from_numpy(bias).cuda(), k)
    torch.cuda.synchronize()
    ridx, rw, _ = oracle.route(x_to_f64(w, x), Wr, bias, k)
    assert np.array_equal(idx.cpu().numpy(), ridx), (name, T, E)
    assert np.allclose(wt.cpu().numpy(), rw, rtol=1e-5, atol=1e-7), (name, T, E)


def test_noalloc_route_matches_oracle_twice(bec):
    from bounded_expert_cache_gb300 import _native as N
    lib = N.lib
    # the first call on this device also looks up the scratch array's address
    _check(lib, N, "prefill", 4, 256, 2048, 8)  # bf16, 256 experts top-8, Zipf bias
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    # the second call, on other inputs (fp32 activations, no bias)
    _check(lib, N, "tiny", 4, 16, 256, 2)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before  # nothing was allocated


@pytest.mark.parametrize("name,T,E,H,k", [
    ("decode", 32, 256, 2048, 8),   # bf16, T*E at the limit
    ("tiny", 32, 256, 512, 8),      # fp32, T*E at the limit
    ("decode", 8, 1024, 512, 16),   # bf16, the most experts and the largest k, T*E at the limit
    ("tiny", 8, 1024, 256, 16),     # fp32, same
    ("prefill", 64, 128, 1024, 8),  # bf16 with bias, the most tokens, T*E at the limit
    ("tiny", 64, 128, 256, 8),      # fp32, same
])
def test_noalloc_route_at_the_limits(bec, name, T, E, H, k):
    from bounded_expert_cache_gb300 import _native as N
    assert T * E == MAX_LOGITS
    # two calls in a row on different tokens: the shared scratch keeps the
    # first call's contents, which the second must not see
    _check(bec._native.lib, N, name, T, E, H, k)
    _check(bec._native.lib, N, name, T, E, H, k, token0=T)


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
    Wr2 = torch.zeros((129, 32), device="cuda")  # 64 * 129 > MAX_LOGITS
    st = N.lib.moe_route_noalloc(C.c_void_p(x2.data_ptr()), N.F32, 64, 32, 129, 8,
                                 C.c_void_p(Wr2.data_ptr()), None, C.c_void_p(idx.data_ptr()),
                                 C.c_void_p(wt.data_ptr()), C.c_void_p(s))
    assert st == 1 and b"static scratch limit" in N.lib.moe_last_error(None)
