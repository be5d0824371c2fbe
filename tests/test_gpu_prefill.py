"""GPU parity of the many-token (prefill) path against the CPU oracle.

Routing for many tokens (tiled logits, certified selection, exact repair) and
the multi-block plan must be bit-exact; the grouped dequant-GEMM FFN (fp16
gate/up, bf16 down, fp32 accumulation in TMEM) must meet the output bar
(relative L2 <= 5e-3, max |diff| <= 2e-2 * RMS) on sampled tokens, which the
oracle routes and evaluates one by one.
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


@pytest.mark.parametrize("name,T", [("prefill", 200), ("tiny", 100), ("wide_prefill", 130)])
def test_route_many_tokens(bec, name, T):
    w = W.WORKLOADS[name]
    if name == "tiny":
        w = W.with_changes(w, n_steps=T // 4)
    ctx = make_context(bec, w, 1, slots=w.n_experts, max_tokens=T)
    Wr = W.router_weights(w, 0)
    bias = W.router_bias(w, 0)
    x = W.activations(w, 0, T)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    ctx.route(0, x_to_torch(w, x), torch.from_numpy(Wr).cuda(),
              None if bias is None else torch.from_numpy(bias).cuda(), idx, wt)
    ctx.check_device_errors()
    ridx, rw, _ = oracle.route(x_to_f64(w, x), Wr, bias, w.top_k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.allclose(wt.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)
    # the tensor-core filter's error model held for every candidate
    assert ctx.stats()["route_filter_fallbacks"] == 0
    ctx.close()


@pytest.mark.parametrize("E,k", [(16, 2), (64, 4), (256, 8), (1024, 16)])
def test_route_many_tokens_filter_ties_and_degenerate_tokens(bec, E, k):
    # bf16 tokens with H % 64 == 0 take the tensor-core filter: exact ties
    # (duplicated router rows and equal biases), an all-zero token (every
    # logit equal: every expert a candidate), a token of one large value, and
    # T = 150 (a ragged 128-token tile) must route as the oracle does, ties to
    # the lower expert id
    T = 150
    w = W.with_changes(W.WORKLOADS["tiny"], x_dtype="bf16", hidden=256, n_experts=E, top_k=k,
                       tokens_per_step=T, n_steps=1, slots=E)
    ctx = make_context(bec, w, 1, max_tokens=T)
    Wr = W.router_weights(w, 0)
    for (a, b) in ((E - 1, 0), (E // 2, E // 2 + 1), (3, 1)):
        Wr[a] = Wr[b]
    x = W.activations(w, 0, T)
    x[7] = 0                       # bf16 zero
    x[9] = 0
    x[9, 17] = 0x4480              # 1024.0
    bias = (np.arange(E) % 4 == 0).astype(np.float32) * np.float32(0.5)
    for b in (None, bias):
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
        ctx.route(0, x_to_torch(w, x), torch.from_numpy(Wr).cuda(),
                  None if b is None else torch.from_numpy(b).cuda(), idx, wt)
        ctx.check_device_errors()
        ridx, rw, _ = oracle.route(x_to_f64(w, x), Wr, b, k)
        assert np.array_equal(idx.cpu().numpy(), ridx)
        assert np.allclose(wt.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)
        assert idx[7].tolist() == (list(range(k)) if b is None else [e for e in range(E) if e % 4 == 0][:k])
    assert ctx.stats()["uncertified_repairs"] >= 2
    assert ctx.stats()["route_filter_fallbacks"] == 0
    ctx.close()


@pytest.mark.parametrize("E,k,H", [(100, 6, 64), (48, 4, 6144), (40, 4, 6208)])
def test_route_many_tokens_filter_shapes(bec, E, k, H):
    # the tensor-core filter at one K stage (H 64), at the largest hidden size
    # it takes (H 6,144: 96 stages, the refining kernel's activations at 192
    # KiB of shared memory) with an expert count that fills no 64-expert
    # tile, and just past it (H 6,208: the tiled CUDA-core router); routing
    # bit-exact against the oracle, T = 200 (a ragged tile)
    T = 200
    w = W.with_changes(W.WORKLOADS["tiny"], x_dtype="bf16", hidden=H, n_experts=E, top_k=k,
                       tokens_per_step=T, n_steps=1, slots=E)
    ctx = make_context(bec, w, 1, max_tokens=T)
    Wr = W.router_weights(w, 0)
    x = W.activations(w, 0, T)
    bias = (np.arange(E, dtype=np.float32) % 7) * np.float32(0.01)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ctx.route(0, x_to_torch(w, x), torch.from_numpy(Wr).cuda(), torch.from_numpy(bias).cuda(), idx, wt)
    ctx.check_device_errors()
    ridx, rw, _ = oracle.route(x_to_f64(w, x), Wr, bias, k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.allclose(wt.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)
    assert ctx.stats()["route_filter_fallbacks"] == 0
    ctx.close()


def test_plan_many_assignments(bec):
    rng = np.random.default_rng(11)
    for (T, E, k) in ((700, 256, 8), (333, 128, 8), (4096, 256, 8)):
        # Zipf-like skew: a few experts take most tokens
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        idx = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(T)]).astype(np.int32)
        wts = rng.random((T, k)).astype(np.float32)
        ctx = bec.Context(1, E, k, 256, 128, 0, 0, 8, 0, 1, 0, 262144, T)
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


def _prefill(bec, w, T, sample, device_admit=1, preload=True, slots=None, token0=0):
    """One prefill step of T tokens through layer_forward; returns (y, idx)
    and checks the sampled tokens against the oracle."""
    store = pinned_store(w, 1)
    S = slots or w.n_experts
    ctx = make_context(bec, w, 1, slots=S, max_tokens=T, device_admit=device_admit)
    keep = bind_all(ctx, w, 1, store)
    if preload:
        ctx.preload(0, list(range(w.n_experts)))
    Wr = W.router_weights(w, 0)
    bias = W.router_bias(w, 0)
    x = W.activations(w, 0, T, token0=token0)
    plan = bec.Plan(w.n_experts, w.top_k, T)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    ctx.layer_forward(0, x_to_torch(w, x), torch.from_numpy(Wr).cuda(),
                      None if bias is None else torch.from_numpy(bias).cuda(), idx, wt, plan, y)
    ctx.check_device_errors()
    yg = y.cpu().numpy().astype(np.float64)
    ig = idx.cpu().numpy()
    experts = ExpertCache(w)
    shared = experts.get(0, w.n_experts) if w.shared_inter else None
    refs, gots = [], []
    for t in sample:
        xt = x_to_f64(w, x[t:t + 1])
        ridx, rw, _ = oracle.route(xt, Wr, bias, w.top_k)
        assert np.array_equal(ig[t], ridx[0]), t
        refs.append(oracle.moe_layer(xt, ridx, rw, lambda e: experts.get(0, e), shared)[0])
        gots.append(yg[t])
    ok, rel, mx = tolerance_ok(np.stack(gots), np.stack(refs))
    assert ok, (rel, mx)
    ctx.close()
    del keep
    return yg, ig, rel


def test_prefill_tiny_shapes(bec):
    w = W.with_changes(W.WORKLOADS["tiny"], n_steps=16)
    _prefill(bec, w, 64, range(0, 64, 5))


def test_prefill_chunk_sampled(bec):
    w = W.WORKLOADS["prefill"]
    _prefill(bec, w, 512, [0, 1, 7, 100, 255, 256, 400, 511])


def test_prefill_full_chunk_4096_every_expert(bec):
    # the full 4096-token Zipf-skewed chunk: routing of all 4,096 tokens and
    # the expert-major plan bit-exact; the output within the bar on, for
    # every active expert, its first token, the first token of its last
    # 192-token tile and its last token (so every expert's partial tile is
    # read), plus every token of one heavy tile
    w = W.WORKLOADS["prefill"]
    T, E, k = 4096, w.n_experts, w.top_k
    store = pinned_store(w, 1)
    ctx = make_context(bec, w, 1, slots=E, max_tokens=T, device_admit=1)
    keep = bind_all(ctx, w, 1, store)
    ctx.preload(0, list(range(E)))
    Wr = W.router_weights(w, 0)
    bias = W.router_bias(w, 0)
    x = W.activations(w, 0, T)
    plan = bec.Plan(E, k, T)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    ctx.layer_forward(0, x_to_torch(w, x), torch.from_numpy(Wr).cuda(), torch.from_numpy(bias).cuda(),
                      idx, wt, plan, y)
    ctx.check_device_errors()
    yg = y.cpu().numpy().astype(np.float64)
    x64 = x_to_f64(w, x)
    ridx, rw = oracle_route_rows(x64, Wr, bias, k, range(T))
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.allclose(wt.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)
    assert ctx.stats()["route_filter_fallbacks"] == 0
    rplan = oracle.plan_union(ridx, rw, E)
    nu = int(plan.n_uniq.item())
    assert plan.uniq[:nu].cpu().numpy().tolist() == rplan["uniq"].tolist()
    for key in ("counts", "offsets"):
        assert np.array_equal(getattr(plan, key).cpu().numpy(), rplan[key]), key
    for key in ("perm_tok", "perm_rank", "inv"):
        assert np.array_equal(getattr(plan, key)[:T * k].cpu().numpy(), rplan[key]), key
    tile = 192  # tokens per GEMM tile
    sample = set()
    for e in rplan["uniq"].tolist():
        toks = rplan["perm_tok"][rplan["offsets"][e]:rplan["offsets"][e + 1]]
        sample.update((int(toks[0]), int(toks[(len(toks) - 1) // tile * tile]), int(toks[-1])))
    heavy = int(np.argmax(rplan["counts"]))
    toks = rplan["perm_tok"][rplan["offsets"][heavy]:rplan["offsets"][heavy + 1]]
    sample.update(int(t) for t in toks[tile:2 * tile])
    sample = sorted(sample)
    assert len(rplan["uniq"]) > 100 and len(sample) > 300
    experts = ExpertCache(w)
    shared = experts.get(0, E)
    refs = [oracle.moe_layer(x64[t:t + 1], ridx[t:t + 1], rw[t:t + 1], lambda e: experts.get(0, e),
                             shared)[0] for t in sample]
    ok, rel, mx = tolerance_ok(yg[sample], np.stack(refs))
    assert ok, (rel, mx)
    for t, ref in zip(sample, refs):  # every sampled token on its own
        ok, rel, mx = tolerance_ok(yg[t:t + 1], ref[None])
        assert ok, (t, rel, mx)
    ctx.close()
    del keep


def test_prefill_wide_shapes(bec):
    # hidden 2816, expert intermediate 704 (partial 128-row tiles), shared 2112
    w = W.WORKLOADS["wide_prefill"]
    _prefill(bec, w, 256, [0, 3, 128, 255])


def test_prefill_transparency_bitwise(bec):
    # preloaded cache vs cold cache filled by host tile staging vs on-device
    # staging: the same outputs, bit for bit
    w = W.WORKLOADS["prefill"]
    a, ia, _ = _prefill(bec, w, 256, [5], device_admit=1, preload=True)
    b, ib, _ = _prefill(bec, w, 256, [5], device_admit=0, preload=False)
    c, ic, _ = _prefill(bec, w, 256, [5], device_admit=1, preload=False)
    assert np.array_equal(ia, ib) and np.array_equal(ia, ic)
    assert np.array_equal(a, b) and np.array_equal(a, c)


def _check_waves(ml, union):
    """The wave schedule is valid: a fill that evicts an expert of the same
    step runs in a later wave than that expert, and n_waves covers them."""
    wave_of = {e: 0 for e in union}
    for e, v, wv in zip(ml.expert, ml.victim, ml.wave):
        if v in wave_of:
            assert wv > wave_of[v], (e, v, wv, wave_of[v])
        wave_of[e] = wv
    assert ml.n_waves == max(ml.wave) + 1


def test_prefill_waves_union_larger_than_slots(bec):
    # the long-prefill shapes with a cold 44-slot LRU cache: each chunk's
    # union is larger than the slots, so the step runs in compute waves.
    # Fills, page table, generations and counters match the oracle's replay;
    # the output matches an all-resident context bit for bit and the oracle
    # on sampled tokens.
    w = W.WORKLOADS["wide_prefill"]
    T, steps, E = 512, 2, w.n_experts
    store = pinned_store(w, 1)
    ctx = make_context(bec, w, 1, slots=w.slots, max_tokens=T, device_admit=0)
    res = make_context(bec, w, 1, slots=E, max_tokens=T, device_admit=0)
    keep = bind_all(ctx, w, 1, store) + bind_all(res, w, 1, store)
    res.preload(0, list(range(E)))
    cache = SlotCache(E, w.slots, w.policy, seed=0, layer=0, payload_bytes=w.payload_bytes)
    experts = ExpertCache(w)
    shared = experts.get(0, E) if w.shared_inter else None
    Wr = W.router_weights(w, 0)
    bias = W.router_bias(w, 0)
    Wr_t = torch.from_numpy(Wr).cuda()
    b_t = None if bias is None else torch.from_numpy(bias).cuda()
    x = W.activations(w, 0, steps * T)
    plan = bec.Plan(E, w.top_k, T)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    y_res = torch.empty_like(y)
    for s in range(steps):
        xs = x[s * T:(s + 1) * T]
        xt = x_to_torch(w, xs)
        ml = ctx.layer_forward(0, xt, Wr_t, b_t, idx, wt, plan, y)
        ctx.check_device_errors()
        ig = idx.cpu().numpy()
        res.layer_forward(0, xt, Wr_t, b_t, idx, wt, plan, y_res)
        res.check_device_errors()
        x64 = x_to_f64(w, xs)
        ridx, rw, _ = oracle.route(x64, Wr, bias, w.top_k)
        assert np.array_equal(ig, ridx), s
        rplan = oracle.plan_union(ridx, rw, E)
        rec = cache.step(rplan["uniq"], rplan["counts"])
        assert len(rplan["uniq"]) > w.slots and ml.n_waves > 1
        assert list(zip(ml.expert, ml.slot, ml.victim)) == [tuple(f) for f in rec["fills"]], s
        _check_waves(ml, set(int(e) for e in rplan["uniq"]))
        pt, gen = ctx.read_page_table(0)
        assert pt == rec["pt"] and gen == rec["gen"], s
        assert torch.equal(y, y_res), s
        yg = y.cpu().numpy().astype(np.float64)
        sample = [0, 200, T - 1] if s == 0 else [77]
        refs = [oracle.moe_layer(x64[t:t + 1], ridx[t:t + 1], rw[t:t + 1], lambda e: experts.get(0, e),
                                 shared)[0] for t in sample]
        ok, rel, mx = tolerance_ok(yg[sample], np.stack(refs))
        assert ok, (s, rel, mx)
    st, rs = ctx.stats(0), cache.stats()
    for key in ("hits", "misses", "evictions", "materialized_bytes"):
        assert st[key] == rs[key], (key, st[key], rs[key])
    ctx.close()
    res.close()
    del keep


@pytest.mark.parametrize("fills_before", ["wave1", "wave0_last_part"])
def test_prefill_waves_failed_staging_fails_closed(bec, fills_before):
    # a copy failure inside a later wave, or inside the last part of the
    # first wave (a wave's last quarter of fills, copied while its first
    # part would compute): the call fails, only waves whose copies all
    # landed publish their slots, and the experts whose payloads never landed
    # are refused (stale generation) when the next step reads them
    w = W.WORKLOADS["wide_prefill"]
    T, E = 256, w.n_experts
    store = pinned_store(w, 1)
    ctx = make_context(bec, w, 1, slots=w.slots, max_tokens=T, device_admit=0)
    keep = bind_all(ctx, w, 1, store)
    Wr_t = torch.from_numpy(W.router_weights(w, 0)).cuda()
    bias = W.router_bias(w, 0)
    b_t = None if bias is None else torch.from_numpy(bias).cuda()
    xt = x_to_torch(w, W.activations(w, 0, T))
    plan = bec.Plan(E, w.top_k, T)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    tiles = len(oracle.tile_partition(w.hidden, w.inter, w.quant))
    # a cold step's wave 0 fills all 44 slots: 33 fills in its first part, 11 in its last
    first_part = w.slots - max(1, w.slots // 4)
    ctx.debug_fail_staging_after((w.slots if fills_before == "wave1" else first_part) * tiles + 3)
    with pytest.raises(bec.MoeError):
        ctx.layer_forward(0, xt, Wr_t, b_t, idx, wt, plan, y)
    ctx.check_device_errors()  # nothing was read from an unpublished slot
    ctx.layer_forward(0, xt, Wr_t, b_t, idx, wt, plan, y)
    with pytest.raises(bec.MoeError) as ei:
        ctx.check_device_errors()
    assert ei.value.status == 4  # MOE_ERR_STALE
    ctx.close()
    del keep


def test_prefill_gemm_wait_runs_out_and_context_recovers(bec):
    # a bounded device wait that runs out, without a fault: the first CTA of
    # the next gate/up GEMM issues no copy for its first ring stage and every
    # wait is limited to ~1 ms, so its consumers' wait on that stage expires.
    # The kernel drains what it issued and returns; the call reports
    # MOE_ERR_TIMEOUT, and the next step on the same context matches the
    # oracle.
    w = W.with_changes(W.WORKLOADS["tiny"], n_steps=32)
    T = 64
    store = pinned_store(w, 1)
    ctx = make_context(bec, w, 1, slots=w.n_experts, max_tokens=T, device_admit=1)
    keep = bind_all(ctx, w, 1, store)
    ctx.preload(0, list(range(w.n_experts)))
    Wr = W.router_weights(w, 0)
    Wr_t = torch.from_numpy(Wr).cuda()
    x = W.activations(w, 0, 2 * T)
    plan = bec.Plan(w.n_experts, w.top_k, T)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    ctx.debug_prefill_wait_timeout(2_000_000, 0)
    ctx.layer_forward(0, x_to_torch(w, x[:T]), Wr_t, None, idx, wt, plan, y)
    with pytest.raises(bec.MoeError) as ei:
        ctx.check_device_errors()
    assert ei.value.status == 5  # MOE_ERR_TIMEOUT
    good = x[T:]
    ctx.layer_forward(0, x_to_torch(w, good), Wr_t, None, idx, wt, plan, y)
    ctx.check_device_errors()
    x64 = x_to_f64(w, good)
    ridx, rw, _ = oracle.route(x64, Wr, None, w.top_k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    experts = ExpertCache(w)
    ref = oracle.moe_layer(x64, ridx, rw, lambda e: experts.get(0, e), None)
    ok, rel, mx = tolerance_ok(y.cpu().numpy(), ref)
    assert ok, (rel, mx)
    ctx.close()
    del keep


def test_prefill_waves_with_prefetch(bec):
    # confidence-gated prefetch ("Paging the Experts" §3.3, during prefill)
    # on the long-prefill shapes with a cold 44-slot LRU cache: each chunk's
    # union is larger than the slots, so its later waves can evict the
    # previous chunk's predicted expert, which the next chunk then loads
    # speculatively before its routing. Fills, page tables, generations,
    # demand and prefetch counters match the oracle's replay; the output is
    # bit for bit the all-resident context's.
    w = W.WORKLOADS["wide_prefill"]
    T, steps, E = 256, 4, w.n_experts
    store = pinned_store(w, 1)
    ctx = make_context(bec, w, 1, slots=w.slots, max_tokens=T, device_admit=0)
    res = make_context(bec, w, 1, slots=E, max_tokens=T, device_admit=0)
    keep = bind_all(ctx, w, 1, store) + bind_all(res, w, 1, store)
    res.preload(0, list(range(E)))
    ctx.set_prefetch(bec.PREFETCH_REFRESH)
    cache = SlotCache(E, w.slots, w.policy, seed=0, layer=0, payload_bytes=w.payload_bytes)
    experts = ExpertCache(w)
    shared = experts.get(0, E)
    Wr = W.router_weights(w, 0)
    Wr_t = torch.from_numpy(Wr).cuda()
    x = W.activations(w, 0, steps * T)
    x64 = x_to_f64(w, x)
    all_idx, all_w = oracle_route_rows(x64, Wr, None, w.top_k, range(steps * T))
    plan = bec.Plan(E, w.top_k, T)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, w.top_k), dtype=torch.float32, device="cuda")
    y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    y_res = torch.empty_like(y)
    pred, actions = None, []
    for s in range(steps):
        xt = x_to_torch(w, x[s * T:(s + 1) * T])
        ml = ctx.layer_forward(0, xt, Wr_t, None, idx, wt, plan, y)
        ctx.check_device_errors()
        res.layer_forward(0, xt, Wr_t, None, idx, wt, plan, y_res)
        res.check_device_errors()
        ridx, rw = all_idx[s * T:(s + 1) * T], all_w[s * T:(s + 1) * T]
        assert np.array_equal(idx.cpu().numpy(), ridx), s
        rplan = oracle.plan_union(ridx, rw, E)
        if pred is not None:
            actions.append(cache.prefetch(pred, oracle.PREFETCH_REFRESH)["action"])
        rec = cache.step(rplan["uniq"], rplan["counts"])
        assert abs(rw[-1, 0] - 0.2) > 1e-5, s  # the fp32 decision is well posed
        pred = oracle.prefetch_prediction(ridx, rw)
        assert list(zip(ml.expert, ml.slot, ml.victim)) == [tuple(f) for f in rec["fills"]], s
        pt, gen = ctx.read_page_table(0)
        assert pt == rec["pt"] and gen == rec["gen"], s
        assert torch.equal(y, y_res), s
        yg = y.cpu().numpy().astype(np.float64)
        sample = [0, T // 2, T - 1]
        refs = [oracle.moe_layer(x64[s * T + t:s * T + t + 1], ridx[t:t + 1], rw[t:t + 1],
                                 lambda e: experts.get(0, e), shared)[0] for t in sample]
        ok, rel, mx = tolerance_ok(yg[sample], np.stack(refs))
        assert ok, (s, rel, mx)
    assert "load" in actions  # a prediction evicted by a later wave was loaded
    st, rs, pf = ctx.stats(0), cache.stats(), cache.prefetch_stats()
    for key in ("hits", "misses", "evictions", "materialized_bytes"):
        assert st[key] == rs[key], (key, st[key], rs[key])
    for key, v in pf.items():
        assert st["prefetch_" + key] == v, (key, st["prefetch_" + key], v)
    ctx.close()
    res.close()
    del keep
