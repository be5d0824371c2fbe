"""GPU parity of the decode path against the CPU oracle (through the C ABI).

Bit-exact: top-k indices, expert-major plans, page tables, slot generations,
hit/miss counters, staged slot bytes. Within tolerance (relative L2 <= 5e-3,
max |diff| <= 2e-2 * RMS): layer outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle.cache import SlotCache

from gpu_common import (ExpertCache, bind_all, make_context, oracle_route_rows, pinned_store,
                        tolerance_ok, x_to_f64, x_to_torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bec():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bounded_expert_cache_gb300 as m
    return m


def _route_gpu(bec, ctx, layer, x_t, Wr, bias, k):
    T = x_t.shape[0]
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ctx.route(layer, x_t, Wr, bias, idx, wt)
    torch.cuda.synchronize()
    ctx.check_device_errors()
    return idx.cpu().numpy(), wt.cpu().numpy()


@pytest.mark.parametrize("name,T", [("tiny", 4), ("decode", 1), ("decode", 4), ("mtp_decode", 4),
                                    ("prefill", 3)])
def test_route_matches_oracle(bec, name, T):
    w = W.WORKLOADS[name]
    ctx = make_context(bec, w, 1, max_tokens=T)
    n_tok = min(w.n_tokens, 12)
    Wr = W.router_weights(w, 0)
    bias = W.router_bias(w, 0)
    x = W.activations(w, 0, n_tok)
    Wr_t = torch.from_numpy(Wr).cuda()
    b_t = None if bias is None else torch.from_numpy(bias).cuda()
    for s in range(0, n_tok - T + 1, T):
        xs = x[s:s + T]
        idx, wt = _route_gpu(bec, ctx, 0, x_to_torch(w, xs), Wr_t, b_t, w.top_k)
        ridx, rw, _ = oracle.route(x_to_f64(w, xs), Wr, bias, w.top_k)
        assert np.array_equal(idx, ridx), (s, idx, ridx)
        assert np.allclose(wt, rw, rtol=1e-5, atol=1e-7)
    ctx.close()


def test_route_exact_ties_and_repair(bec):
    # duplicated router rows give exactly equal logits: the fast bounds cannot
    # order them, the exact repair must, with ties to the lower expert id
    E, H, k = 64, 256, 4
    rng = np.random.default_rng(5)
    Wr = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    for (a, b) in ((10, 3), (40, 41), (63, 0), (7, 22)):
        Wr[a] = Wr[b]
    x = rng.standard_normal((6, H)).astype(np.float32)
    x[5] = 0.0  # all logits zero -> experts 0..k-1
    ctx = bec.Context(1, E, k, H, 128, 0, 0, E, 0, 1, 0, 262144, 8)
    idx, wt = _route_gpu(bec, ctx, 0, torch.from_numpy(x).cuda(), torch.from_numpy(Wr).cuda(), None, k)
    ridx, rw, _ = oracle.route(x.astype(np.float64), Wr, None, k)
    assert np.array_equal(idx, ridx)
    assert idx[5].tolist() == [0, 1, 2, 3]
    assert np.allclose(wt, rw, rtol=1e-5, atol=1e-7)
    assert ctx.stats()["uncertified_repairs"] >= 1
    ctx.close()


def test_plan_matches_oracle(bec):
    rng = np.random.default_rng(7)
    for (T, E, k) in ((1, 256, 8), (4, 256, 8), (8, 16, 2), (64, 128, 8), (37, 1024, 16)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        wts = rng.random((T, k)).astype(np.float32)
        ctx = bec.Context(1, E, k, 256, 128, 0, 0, min(E, 8), 0, 1, 0, 262144, T)
        plan = bec.Plan(E, k, T)
        ctx.plan_union(torch.from_numpy(idx).cuda(), torch.from_numpy(wts).cuda(), T, plan)
        torch.cuda.synchronize()
        ref = oracle.plan_union(idx, wts.astype(np.float64), E)
        nu = int(plan.n_uniq.item())
        assert nu == len(ref["uniq"])
        assert plan.uniq[:nu].cpu().numpy().tolist() == ref["uniq"].tolist()
        for key in ("counts", "offsets"):
            assert np.array_equal(getattr(plan, key).cpu().numpy(), ref[key]), key
        A = T * k
        for key in ("perm_tok", "perm_rank", "inv"):
            assert np.array_equal(getattr(plan, key)[:A].cpu().numpy(), ref[key]), key
        assert np.array_equal(plan.perm_w[:A].cpu().numpy(), ref["perm_w"].astype(np.float32))
        ctx.close()


_ROUTES = {}


def _oracle_routes(w, layer, x64, Wr, bias):
    """The oracle's routing of every token of a layer's trace (per token, so
    the rows of one step are the step's routing), computed once per
    workload and layer."""
    key = (w, layer, x64.shape[0])
    if key not in _ROUTES:
        _ROUTES[key] = oracle_route_rows(x64, Wr, bias, w.top_k, range(x64.shape[0]))
    return _ROUTES[key]


def _run_trace(bec, w, layers, steps, ffn_steps, policy=None, seed=0, tile_bytes=262144,
               slots=None, preload=False, check_every_step=True, device_admit=False, stats_out=None,
               prefetch=0, decode_ffn=0):
    """Run layer_forward for every (step, layer) on the GPU and replay the
    same trace in the oracle; compare bit-exact state each step and outputs on
    ffn_steps. Returns the GPU outputs {(layer, step): y}."""
    T = w.tokens_per_step
    store = pinned_store(w, layers)
    pol = w.policy if policy is None else policy
    S = slots or w.slots
    ctx = make_context(bec, w, layers, policy=pol, slots=S, seed=seed, tile_bytes=tile_bytes,
                       device_admit=device_admit, decode_ffn=decode_ffn)
    keep = bind_all(ctx, w, layers, store)
    if prefetch:
        ctx.set_prefetch(prefetch)
    experts = ExpertCache(w)
    plan = bec.Plan(w.n_experts, w.top_k, T)
    idx_t = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt_t = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    y_t = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    outs = {}
    for l in range(layers):
        Wr = W.router_weights(w, l)
        bias = W.router_bias(w, l)
        Wr_t = torch.from_numpy(Wr).cuda()
        b_t = None if bias is None else torch.from_numpy(bias).cuda()
        x = W.activations(w, l, steps * T)
        all_idx, all_w = _oracle_routes(w, l, x_to_f64(w, x), Wr, bias)
        cache = SlotCache(w.n_experts, S, pol, seed=seed, layer=l, payload_bytes=w.payload_bytes)
        if preload:
            ctx.preload(l, list(range(w.n_experts)))
            cache.preload(range(w.n_experts))
        shared = experts.get(l, w.n_experts) if w.shared_inter else None
        pred = None
        for s in range(steps):
            xs = x[s * T:(s + 1) * T]
            ctx.layer_forward(l, x_to_torch(w, xs), Wr_t, b_t, idx_t, wt_t, plan, y_t)
            ctx.check_device_errors()
            y = y_t.cpu().numpy().copy()
            outs[(l, s)] = y
            x64 = x_to_f64(w, xs)
            ridx, rw = all_idx[s * T:(s + 1) * T], all_w[s * T:(s + 1) * T]
            rplan = oracle.plan_union(ridx, rw, w.n_experts)
            if prefetch and pred is not None:
                cache.prefetch(pred, prefetch)
            rec = cache.step(rplan["uniq"], rplan["counts"])
            if prefetch:
                # the decision is taken on fp32 weights on the device: it
                # must not sit on the threshold
                assert abs(rw[-1, 0] - 0.2) > 1e-5, (l, s)
                pred = oracle.prefetch_prediction(ridx, rw)
            assert np.array_equal(idx_t.cpu().numpy(), ridx), (l, s)
            if check_every_step or s == steps - 1:
                pt, gen = ctx.read_page_table(l)
                assert pt == rec["pt"], (l, s)
                assert gen == rec["gen"], (l, s)
            if s in ffn_steps:
                ref = oracle.moe_layer(x64, ridx, rw, lambda e: experts.get(l, e), shared)
                ok, rel, mx = tolerance_ok(y, ref)
                assert ok, (l, s, rel, mx)
                assert rel < 1e-4, (l, s, rel)  # fp32 path: far inside the bar
        st = ctx.stats(l)
        rs = cache.stats()
        for key in ("hits", "misses", "evictions", "materialized_bytes"):
            assert st[key] == rs[key], (l, key, st[key], rs[key])
        if prefetch:
            for key, v in cache.prefetch_stats().items():
                assert st["prefetch_" + key] == v, (l, key, st["prefetch_" + key], v)
            rs = dict(rs, **{"prefetch_" + key: v for key, v in cache.prefetch_stats().items()})
        if stats_out is not None:
            stats_out.append(rs)
    ctx.close()
    del keep
    return outs


MODES = [0, 1, 2]  # host admission; device admission + staging kernel; + read-through


@pytest.mark.parametrize("device_admit", MODES)
def test_layer_tiny_trace(bec, device_admit):
    w = W.with_changes(W.WORKLOADS["tiny"], n_steps=16)
    _run_trace(bec, w, 1, 16, set(range(16)), device_admit=device_admit)


@pytest.mark.parametrize("device_admit", MODES)
def test_layer_decode_full_size(bec, device_admit):
    w = W.WORKLOADS["decode"]
    _run_trace(bec, w, 2, 24, {0, 5, 23}, device_admit=device_admit)


@pytest.mark.parametrize("device_admit", MODES)
@pytest.mark.parametrize("policy,seed", [(0, 0), (1, 0), (1, 3)])
def test_layer_mtp_decode_q4(bec, policy, seed, device_admit):
    w = W.with_changes(W.WORKLOADS["mtp_decode"], slots=40)  # >= T*k, small enough to evict
    _run_trace(bec, w, 1, 14, {0, 13}, policy=policy, seed=seed, device_admit=device_admit)


@pytest.mark.parametrize("policy,seed,device_admit", [(0, 0, 0), (0, 0, 2), (1, 0, 1), (1, 3, 2)])
def test_layer_mtp_decode_at_its_configuration(bec, policy, seed, device_admit):
    # the MTP-batched decode workload as measured: Q4_0 experts, 4 tokens per
    # step through their expert-major union, 89 slots per layer (35% of 256),
    # LRU and seeded random; 4 layers x 32 steps with page tables,
    # generations and counters bit-exact every step and outputs on three steps
    w = W.with_changes(W.WORKLOADS["mtp_decode"], n_layers=4, n_steps=32)
    assert w.slots == 89 and w.tokens_per_step == 4
    stats = []
    _run_trace(bec, w, 4, 32, {0, 15, 31}, policy=policy, seed=seed, device_admit=device_admit,
               stats_out=stats)
    assert sum(r["evictions"] for r in stats) > 0  # the slots were full and refilled


# The decode FFN as one persistent launch with the tile-granular staging of a
# read-through miss's down plane (decode_ffn = 1): the same parity bar, in
# every admission mode, at one, four (MTP, Q4_0) and eight tokens, with small
# staging tiles (many ready counters per down plane) and the affine INT4
# format; outputs bitwise equal to the two-launch path.
@pytest.mark.parametrize("device_admit", MODES)
def test_fused_decode_ffn_trace(bec, device_admit):
    w = W.WORKLOADS["decode"]
    _run_trace(bec, w, 2, 24, {0, 5, 23}, device_admit=device_admit, decode_ffn=1)


@pytest.mark.parametrize("name,T,tile", [("mtp_decode", 4, 262144), ("decode", 8, 16000), ("decode", 1, 4096),
                                         ("i4_decode", 1, 262144), ("tiny", 4, 8192)])
def test_fused_decode_ffn_shapes_and_tiles(bec, name, T, tile):
    base = W.WORKLOADS[name]
    w = W.with_changes(base, tokens_per_step=T, n_layers=1, n_steps=10,
                       slots=min(base.n_experts, max(base.slots, base.top_k * T)))
    a = _run_trace(bec, w, 1, 10, {0, 9}, device_admit=2, tile_bytes=tile, decode_ffn=1)
    b = _run_trace(bec, w, 1, 10, set(), device_admit=2, tile_bytes=tile, check_every_step=False)
    for key in a:
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("mode", [1, 2])
def test_layer_decode_trace_with_prefetch(bec, mode):
    # confidence-gated prefetch with host admission on one-token steps (the
    # page's serial steps): before each step the previous step's top expert
    # (weight >= 0.20) is refreshed (mode 1) or probed (mode 2). Page tables,
    # generations and counters, prefetch counters included, bit-exact with
    # the oracle's replay; outputs within the bar on three steps
    w = W.with_changes(W.WORKLOADS["decode"], n_layers=2)
    stats = []
    _run_trace(bec, w, 2, 40, {0, 20, 39}, prefetch=mode, stats_out=stats)
    assert sum(r["prefetch_refreshes" if mode == 1 else "prefetch_probes"] for r in stats) > 10


@pytest.mark.parametrize("device_admit", [0, 2])
@pytest.mark.parametrize("T", [2, 3, 5, 8])
def test_layer_decode_token_counts(bec, T, device_admit):
    # decode steps of 2..8 tokens: the FFN kernels' four- and eight-token
    # groups, full (4, 8) and partial (2, 3, 5), with the union of up to T*k
    # experts in the slots
    w = W.with_changes(W.WORKLOADS["decode"], tokens_per_step=T, n_steps=6, slots=max(38, 8 * T))
    _run_trace(bec, w, 1, 6, {0, 3, 5}, device_admit=device_admit)


@pytest.mark.parametrize("device_admit", [0, 2])
@pytest.mark.parametrize("T", [1, 4])
def test_layer_at_maximum_experts_and_top_k(bec, T, device_admit):
    # the ABI's limits, 1,024 experts and top-16: the router's general
    # selection path (more than 256 experts), its block planner (more than 32
    # assignments at T = 4) and the admission warp reading the cache state
    w = W.with_changes(W.WORKLOADS["tiny"], n_experts=1024, top_k=16, tokens_per_step=T, n_steps=3,
                       slots=max(32, 16 * T))
    _run_trace(bec, w, 1, 3, {0, 2}, device_admit=device_admit)


def test_route_many_tokens_at_maximum_experts_and_top_k(bec):
    # the many-token router (T > 64: tiled logits, key folding, selection,
    # exact repair) at 1,024 experts and top-16
    w = W.with_changes(W.WORKLOADS["tiny"], n_experts=1024, top_k=16, tokens_per_step=100, n_steps=1,
                       slots=1024)
    T = w.tokens_per_step
    ctx = make_context(bec, w, 1, max_tokens=T)
    Wr = W.router_weights(w, 0)
    x = W.activations(w, 0, T)
    idx, wt = _route_gpu(bec, ctx, 0, x_to_torch(w, x), torch.from_numpy(Wr).cuda(), None, w.top_k)
    ridx, rw, _ = oracle.route(x_to_f64(w, x), Wr, None, w.top_k)
    assert np.array_equal(idx, ridx)
    assert np.allclose(wt, rw, rtol=1e-5, atol=1e-7)
    ctx.close()


@pytest.mark.parametrize("T", [1, 4, 100])
def test_route_reports_non_finite_input(bec, T):
    # a NaN in one token's activations leaves its routing undefined: the
    # router reports MOE_ERR_UNCERTIFIED (a decode step with on-device
    # admission through the last block's tail, or the many-token router)
    # and the next clean call matches the oracle
    w = W.with_changes(W.WORKLOADS["tiny"], tokens_per_step=T, n_steps=2)
    decode = T <= 8
    ctx = make_context(bec, w, 1, max_tokens=T, device_admit=2 if decode else 0)
    keep = bind_all(ctx, w, 1, pinned_store(w, 1)) if decode else None
    Wr = W.router_weights(w, 0)
    Wr_t = torch.from_numpy(Wr).cuda()
    x = W.activations(w, 0, 2 * T)
    bad = x[:T].copy()
    bad[0, 5] = np.nan
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    plan = bec.Plan(w.n_experts, w.top_k, T)
    y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")

    def call(xs):
        if decode:
            ctx.layer_forward(0, x_to_torch(w, xs), Wr_t, None, idx, wt, plan, y)
        else:
            ctx.route(0, x_to_torch(w, xs), Wr_t, None, idx, wt)

    call(bad)
    with pytest.raises(bec.MoeError) as ei:
        ctx.check_device_errors()
    assert ei.value.status == 6  # MOE_ERR_UNCERTIFIED
    good = x[T:]
    call(good)
    ctx.check_device_errors()
    ridx, rw, _ = oracle.route(x_to_f64(w, good), Wr, None, w.top_k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.allclose(wt.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)
    ctx.close()
    del keep


def test_calls_refuse_bad_token_counts(bec):
    # T = 0 and T > max_tokens are refused before any launch; the context
    # stays usable and the next valid step matches the oracle
    w = W.with_changes(W.WORKLOADS["tiny"], n_steps=2)
    T = w.tokens_per_step
    store = pinned_store(w, 1)
    ctx = make_context(bec, w, 1)
    keep = bind_all(ctx, w, 1, store)
    Wr = W.router_weights(w, 0)
    Wr_t = torch.from_numpy(Wr).cuda()
    plan = bec.Plan(w.n_experts, w.top_k, T)
    x = W.activations(w, 0, 2 * T)
    for bad in (0, T + 1):
        xb = x_to_torch(w, np.resize(x, (bad, w.hidden)))
        idx = torch.empty((max(bad, 1), w.top_k), dtype=torch.int32, device="cuda")
        wt = torch.empty((max(bad, 1), w.top_k), dtype=torch.float32, device="cuda")
        y = torch.empty((max(bad, 1), w.hidden), dtype=torch.float32, device="cuda")
        with pytest.raises(bec.MoeError):
            ctx.route(0, xb, Wr_t, None, idx, wt)
        with pytest.raises(bec.MoeError):
            ctx.layer_forward(0, xb, Wr_t, None, idx, wt, plan, y)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    xs = x[:T]
    ctx.layer_forward(0, x_to_torch(w, xs), Wr_t, None, idx, wt, plan, y)
    torch.cuda.synchronize()
    ctx.check_device_errors()
    x64 = x_to_f64(w, xs)
    ridx, rw, _ = oracle.route(x64, Wr, None, w.top_k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    experts = ExpertCache(w)
    ref = oracle.moe_layer(x64, ridx, rw, lambda e: experts.get(0, e),
                           experts.get(0, w.n_experts) if w.shared_inter else None)
    ok, rel, mx = tolerance_ok(y.cpu().numpy(), ref)
    assert ok, (rel, mx)
    st = ctx.stats(0)  # the refused calls counted nothing: one step from an empty cache
    assert st["misses"] == len(set(ridx.ravel().tolist()))
    assert st["hits"] + st["misses"] == T * w.top_k
    ctx.close()
    del keep


@pytest.mark.parametrize("device_admit", [1, 2])
def test_layer_decode_long_trace_device_admission(bec, device_admit):
    # the whole 128-step trace of one layer, cache state bit-exact every step
    w = W.WORKLOADS["decode"]
    _run_trace(bec, w, 1, 128, {127}, device_admit=device_admit)


def test_cache_transparency_bitwise(bec):
    # outputs must not depend on cache state, eviction policy, tile size or
    # where admission runs
    w = W.with_changes(W.WORKLOADS["decode"], n_layers=1)
    a = _run_trace(bec, w, 1, 8, set(), policy=0, check_every_step=False)
    b = _run_trace(bec, w, 1, 8, set(), policy=1, seed=4, check_every_step=False)
    c = _run_trace(bec, w, 1, 8, set(), slots=w.n_experts, preload=True, tile_bytes=4096,
                   check_every_step=False)
    d = _run_trace(bec, w, 1, 8, set(), policy=1, seed=2, check_every_step=False,
                   device_admit=True)
    e = _run_trace(bec, w, 1, 8, set(), slots=w.n_experts, preload=True, tile_bytes=8192,
                   check_every_step=False, device_admit=True)
    f = _run_trace(bec, w, 1, 8, set(), policy=1, seed=1, check_every_step=False,
                   device_admit=2)
    for key in a:
        for other in (b, c, d, e, f):
            assert np.array_equal(a[key], other[key]), key


def test_staged_slot_bytes_equal_store(bec):
    w = W.with_changes(W.WORKLOADS["decode"], n_layers=1)
    store = pinned_store(w, 1)
    for tile in (262144, 4096, 1000 * 16):
        ctx = make_context(bec, w, 1, tile_bytes=tile)
        bind_all(ctx, w, 1, store)
        plan = bec.Plan(w.n_experts, w.top_k, 1)
        idx = torch.tensor([[3, 9, 17, 100, 200, 255, 0, 1]], dtype=torch.int32, device="cuda")
        wt = torch.full((1, 8), 0.125, device="cuda")
        ctx.plan_union(idx, wt, 1, plan)
        ml = ctx.cache_admit(0, plan)
        ctx.stage_tiles(0, ml)
        torch.cuda.synchronize()
        tiles = oracle.tile_partition(w.hidden, w.inter, w.quant, tile)
        assert ctx.stats(0)["tiles_staged"] == 8 * len(tiles)
        assert ctx.stats(0)["bytes_staged"] == 8 * w.payload_bytes
        for e, s in zip(ml.expert, ml.slot):
            got = np.frombuffer(ctx.read_slot(0, s), dtype=np.uint8)
            assert np.array_equal(got, store[0, e].numpy()), (tile, e)
        ctx.close()


@pytest.mark.parametrize("device_admit", MODES)
def test_layer_affine_int4_trace(bec, device_admit):
    # the decode shapes with affine INT4 group-64 experts: routing, page
    # tables, counters and outputs against the oracle in every admission mode
    w = W.with_changes(W.WORKLOADS["i4_decode"], n_layers=2, n_steps=12)
    _run_trace(bec, w, 2, 12, {0, 5, 11}, device_admit=device_admit)


@pytest.mark.parametrize("device_admit", MODES)
def test_resident_slots_hold_store_payloads(bec, device_admit):
    # after decode steps with misses, every expert the page table marks
    # resident holds exactly its store payload, however it was materialised
    # (host copies, the staging kernel, or read-through by the FFN kernels)
    for name in ("decode", "i4_decode"):
        _check_resident_payloads(bec, W.with_changes(W.WORKLOADS[name], n_layers=1), device_admit)


def _check_resident_payloads(bec, w, device_admit):
    store = pinned_store(w, 1)
    ctx = make_context(bec, w, 1, device_admit=device_admit)
    keep = bind_all(ctx, w, 1, store)
    T = w.tokens_per_step
    plan = bec.Plan(w.n_experts, w.top_k, T)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    Wr = torch.from_numpy(W.router_weights(w, 0)).cuda()
    x = W.activations(w, 0, 24 * T)
    for s in range(24):
        ctx.layer_forward(0, x_to_torch(w, x[s * T:(s + 1) * T]), Wr, None, idx, wt, plan, y)
    ctx.check_device_errors()
    assert ctx.stats(0)["misses"] > w.slots  # slots were refilled
    pt, _ = ctx.read_page_table(0)
    resident = [(e, s) for e, s in enumerate(pt) if s >= 0]
    assert len(resident) == w.slots
    for e, s in resident:
        got = np.frombuffer(ctx.read_slot(0, s), dtype=np.uint8)
        assert np.array_equal(got, store[0, e].numpy()), (device_admit, e, s)
    ctx.close()
    del keep


@pytest.mark.parametrize("decode_ffn", [0, 1])
@pytest.mark.parametrize("device_admit", [1, 2])
def test_fail_closed_stale_generation_device_admission(bec, device_admit, decode_ffn):
    w = W.with_changes(W.WORKLOADS["tiny"], n_steps=2)
    store = pinned_store(w, 1)
    ctx = make_context(bec, w, 1, device_admit=device_admit, decode_ffn=decode_ffn)
    bind_all(ctx, w, 1, store)
    plan = bec.Plan(w.n_experts, w.top_k, 4)
    x = x_to_torch(w, W.activations(w, 0, 4))
    Wr = torch.from_numpy(W.router_weights(w, 0)).cuda()
    idx = torch.empty((4, 2), dtype=torch.int32, device="cuda")
    wt = torch.empty((4, 2), device="cuda")
    y = torch.empty((4, w.hidden), device="cuda")
    ctx.layer_forward(0, x, Wr, None, idx, wt, plan, y)
    ctx.check_device_errors()
    # the same step again: every expert now hits, so the FFN reads the slots
    # (a miss would be read from the store and never consult the slot)
    ctx.layer_forward(0, x, Wr, None, idx, wt, plan, y)
    ctx.check_device_errors()
    with pytest.raises(bec.MoeError):
        ctx.cache_admit(0, plan)  # host admission is refused on this context
    e0 = int(idx[0, 0].item())
    ctx.debug_corrupt_generation(0, e0)
    ctx.expert_ffn(0, x, plan, y)
    with pytest.raises(bec.MoeError) as ei:
        ctx.check_device_errors()
    assert ei.value.status == 4
    ctx.close()


def test_fail_closed_on_failed_staging_and_stale_generation(bec):
    w = W.with_changes(W.WORKLOADS["tiny"], n_steps=3)
    store = pinned_store(w, 1)
    ctx = make_context(bec, w, 1)
    bind_all(ctx, w, 1, store)
    plan = bec.Plan(w.n_experts, w.top_k, 4)
    x = x_to_torch(w, W.activations(w, 0, 4))
    Wr = torch.from_numpy(W.router_weights(w, 0)).cuda()
    idx = torch.empty((4, 2), dtype=torch.int32, device="cuda")
    wt = torch.empty((4, 2), device="cuda")
    y = torch.empty((4, w.hidden), device="cuda")
    ctx.route(0, x, Wr, None, idx, wt)
    ctx.plan_union(idx, wt, 4, plan)
    ml = ctx.cache_admit(0, plan)
    assert ml.misses > 1
    ctx.debug_fail_staging_after(1)
    with pytest.raises(bec.MoeError):
        ctx.stage_tiles(0, ml)
    ctx.expert_ffn(0, x, plan, y)
    with pytest.raises(bec.MoeError) as ei:
        ctx.check_device_errors()
    assert ei.value.status == 4  # MOE_ERR_STALE: unpublished slots were not read
    ctx.check_device_errors()  # cleared
    # a good staging publishes the slots; then corrupting one generation fails closed
    ctx.stage_tiles(0, ml)
    ctx.expert_ffn(0, x, plan, y)
    ctx.check_device_errors()
    ctx.debug_corrupt_generation(0, ml.expert[0])
    ctx.expert_ffn(0, x, plan, y)
    with pytest.raises(bec.MoeError) as ei:
        ctx.check_device_errors()
    assert ei.value.status == 4
    ctx.close()
