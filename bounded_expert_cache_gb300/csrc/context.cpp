// Context, cache admission, miss staging and the C ABI entry points.
//
// "MawForge" §IV-C: the worker allocates compact per-layer slot tensors; the
// slot count follows from the cache bytes and the per-slot expert size; a
// miss materialises the expert block into an available slot and updates the
// route-to-slot metadata. "Nanite for Experts" §5.4: experts are copied as
// 256 KiB virtual tiles rotating over three streams, and persistent device
// page-table entries carry generations; §3.2: an invalid slot or generation
// fails closed; §3.4: asynchronous copies need pinned host memory and
// non-default streams. "Paging the Experts" §3.2: entries are pinned while
// their layer is evaluated; §4.2: materialised bytes = misses x payload.
//
// Device state per layer: slot pool [S][slot_stride], page table pt[E]
// (slot or -1), pt_gen[E] (generation the entry expects) and gen[S]
// (generation of the slot's content). Admission writes pt/pt_gen; staging
// writes gen only after every tile of the step has landed, so a kernel that
// runs without the staging (or after a failed one) sees gen != pt_gen and
// reads nothing from that slot.
#include <algorithm>
#include <cstdio>
#include <cstring>

#include "internal.h"
#include "prefill.h"

namespace {

thread_local std::string g_create_err;

#define CK(call)                                                                   \
  do {                                                                             \
    cudaError_t e_ = (call);                                                       \
    if (e_ != cudaSuccess) {                                                       \
      ctx->err = std::string(#call) + ": " + cudaGetErrorString(e_);               \
      return MOE_ERR_CUDA;                                                         \
    }                                                                              \
  } while (0)

moe_status_t fail(moe_ctx_t* ctx, moe_status_t st, const std::string& msg) {
  if (ctx) ctx->err = msg;
  return st;
}

bool valid_layer(const moe_ctx_t* ctx, int32_t layer) {
  return layer >= 0 && layer < ctx->cfg.n_layers;
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

cudaEvent_t timing_event(moe_ctx_t* ctx) {
  if (!ctx->ev_pool.empty()) {
    cudaEvent_t e = ctx->ev_pool.back();
    ctx->ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Fold finished timed launches into the per-kind totals and recycle events.
cudaError_t resolve_timing(moe_ctx_t* ctx) {
  for (auto& r : ctx->timed) {
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e != cudaSuccess) return e;
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, r.a, r.b);
    if (e != cudaSuccess) return e;
    ctx->kt_ms[r.kind] += ms;
    ctx->kt_n[r.kind] += 1;
    ctx->ev_pool.push_back(r.a);
    ctx->ev_pool.push_back(r.b);
  }
  ctx->timed.clear();
  return cudaSuccess;
}

}  // namespace

namespace moe {

void set_thread_error(const std::string& msg) { g_create_err = msg; }

ExpertGeom expert_geom(int32_t H, int32_t I, int32_t quant) {
  ExpertGeom g;
  g.H = H;
  g.I = I;
  g.quant = quant;
  const int32_t rows[3] = {I, I, H};
  const int32_t ks[3] = {H, H, I};
  int64_t off = 0;
  for (int m = 0; m < 3; ++m) {
    const int64_t n = static_cast<int64_t>(rows[m]) * ks[m];
    g.qbytes[m] = quant == MOE_Q8_0 ? n : n / 2;
    g.sbytes[m] = n / 32 * 2;
    g.qoff[m] = off;
    off += g.qbytes[m];
    g.soff[m] = off;
    off += g.sbytes[m];
  }
  g.bytes = off;
  return g;
}

}  // namespace moe

extern "C" const char* moe_last_error(const moe_ctx_t* ctx) {
  return ctx ? ctx->err.c_str() : g_create_err.c_str();
}

extern "C" void moe_destroy(moe_ctx_t* ctx) {
  if (!ctx) return;
  for (auto s : ctx->streams)
    if (s) cudaStreamSynchronize(s);
  cudaDeviceSynchronize();
  for (auto s : ctx->slots) moe_slots_destroy(s);
  for (auto e : ctx->ev_stage)
    if (e) cudaEventDestroy(e);
  for (auto e : ctx->ev_stage_b)
    if (e) cudaEventDestroy(e);
  for (auto e : ctx->ev_prefetch)
    if (e) cudaEventDestroy(e);
  for (auto& r : ctx->timed) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : ctx->ev_pool) cudaEventDestroy(e);
  if (ctx->ev_compute) cudaEventDestroy(ctx->ev_compute);
  for (auto s : ctx->streams)
    if (s) cudaStreamDestroy(s);
  cudaFree(ctx->d_pool);
  cudaFree(ctx->d_pt);
  cudaFree(ctx->d_ptgen);
  cudaFree(ctx->d_gen);
  cudaFree(ctx->d_keys);
  cudaFree(ctx->d_ticket);
  cudaFree(ctx->d_repairs);
  cudaFree(ctx->d_h);
  cudaFree(ctx->d_err);
  cudaFree(ctx->d_units);
  cudaFree(ctx->d_owner);
  cudaFree(ctx->d_sgen);
  cudaFree(ctx->d_last);
  cudaFree(ctx->d_tick);
  cudaFree(ctx->d_rng);
  cudaFree(ctx->d_stats);
  cudaFree(ctx->d_fills);
  cudaFree(ctx->d_done);
  cudaFree(ctx->d_ffn_ticket);
  cudaFree(ctx->d_fsync);
  cudaFree(ctx->d_x16);
  cudaFree(ctx->d_hp);
  cudaFree(ctx->d_yp);
  cudaFree(ctx->d_items0);
  cudaFree(ctx->d_items1);
  cudaFree(ctx->d_nitems);
  cudaFree(ctx->d_plan_local);
  cudaFree(ctx->d_norms);
  cudaFree(ctx->d_flags);
  cudaFree(ctx->d_wsplit);
  cudaFree(ctx->d_lpart);
  cudaFreeHost(ctx->h_units);
  cudaFreeHost(ctx->h_pt);
  cudaFreeHost(ctx->h_ptgen);
  cudaFreeHost(ctx->h_gen);
  cudaFreeHost(ctx->h_err);
  cudaFreeHost(ctx->h_union);
  delete ctx;
}

extern "C" moe_status_t moe_create(const moe_config_t* cfg, moe_ctx_t** out) {
  if (!out) return MOE_ERR_ARG;
  *out = nullptr;
  if (!cfg) {
    g_create_err = "moe_create: cfg is NULL";
    return MOE_ERR_ARG;
  }
  const moe_config_t& c = *cfg;
  std::string why;
  if (c.n_layers < 1) why = "n_layers < 1";
  else if (c.n_experts < 1 || c.n_experts > 1024) why = "n_experts outside 1..1024";
  else if (c.top_k < 1 || c.top_k > 16 || c.top_k > c.n_experts) why = "top_k outside 1..min(16, E)";
  else if (c.hidden < 32 || c.hidden % 32) why = "hidden not a positive multiple of 32";
  else if (c.inter < 32 || c.inter % 32) why = "inter not a positive multiple of 32";
  else if (c.shared_inter < 0 || c.shared_inter % 32) why = "shared_inter not a multiple of 32";
  else if (c.quant != MOE_Q8_0 && c.quant != MOE_Q4_0 && c.quant != MOE_I4_G64) why = "unknown quant";
  else if (c.quant == MOE_I4_G64 && (c.hidden % 64 || c.inter % 64 || c.shared_inter % 64))
    why = "I4_G64 needs hidden, inter and shared_inter multiples of 64";
  else if (c.slots_per_layer < 1 || c.slots_per_layer > c.n_experts) why = "slots_per_layer outside 1..E";
  else if (c.policy != MOE_LRU && c.policy != MOE_RANDOM) why = "unknown policy";
  else if (c.n_streams < 1 || c.n_streams > 8) why = "n_streams outside 1..8";
  else if (c.tile_bytes < 16 || c.tile_bytes % 16) why = "tile_bytes not a positive multiple of 16";
  else if (c.max_tokens < 1) why = "max_tokens < 1";
  else if (c.admit_on_device < 0 || c.admit_on_device > 2) why = "admit_on_device must be 0, 1 or 2";
  else if (c.decode_ffn < 0 || c.decode_ffn > 1) why = "decode_ffn must be 0 or 1";
  if (!why.empty()) {
    g_create_err = "moe_create: " + why;
    return MOE_ERR_ARG;
  }
  auto* ctx = new moe_ctx();
  ctx->cfg = c;
  moe_status_t st = MOE_OK;
  auto bail = [&](moe_status_t s) {
    g_create_err = ctx->err;
    moe_destroy(ctx);
    return s;
  };
#define CKC(call)                                                                  \
  do {                                                                             \
    cudaError_t e_ = (call);                                                       \
    if (e_ != cudaSuccess) {                                                       \
      ctx->err = std::string("moe_create: ") + #call + ": " + cudaGetErrorString(e_); \
      return bail(MOE_ERR_CUDA);                                                   \
    }                                                                              \
  } while (0)
  CKC(cudaGetDevice(&ctx->device));
  CKC(cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device));
  const int L = c.n_layers, E = c.n_experts, S = c.slots_per_layer;
  ctx->geom = moe::expert_geom(c.hidden, c.inter, c.quant);
  if (c.shared_inter > 0) ctx->sgeom = moe::expert_geom(c.hidden, c.shared_inter, c.quant);
  ctx->slot_stride = round_up(ctx->geom.bytes, 256);
  const size_t pool = static_cast<size_t>(L) * S * ctx->slot_stride + 256;
  CKC(cudaMalloc(&ctx->d_pool, pool));
  CKC(cudaMalloc(&ctx->d_pt, sizeof(int32_t) * L * E));
  CKC(cudaMalloc(&ctx->d_ptgen, sizeof(uint32_t) * L * E));
  CKC(cudaMalloc(&ctx->d_gen, sizeof(uint32_t) * L * S));
  CKC(cudaMemset(ctx->d_pt, 0xFF, sizeof(int32_t) * L * E));
  CKC(cudaMemset(ctx->d_ptgen, 0, sizeof(uint32_t) * L * E));
  CKC(cudaMemset(ctx->d_gen, 0, sizeof(uint32_t) * L * S));
  CKC(cudaHostAlloc(&ctx->h_pt, sizeof(int32_t) * L * E, cudaHostAllocDefault));
  CKC(cudaHostAlloc(&ctx->h_ptgen, sizeof(uint32_t) * L * E, cudaHostAllocDefault));
  CKC(cudaHostAlloc(&ctx->h_gen, sizeof(uint32_t) * L * S, cudaHostAllocDefault));
  std::fill(ctx->h_pt, ctx->h_pt + L * E, -1);
  std::fill(ctx->h_ptgen, ctx->h_ptgen + L * E, 0u);
  std::fill(ctx->h_gen, ctx->h_gen + L * S, 0u);
  const size_t te = static_cast<size_t>(c.max_tokens) * E;
  CKC(cudaMalloc(&ctx->d_keys, sizeof(unsigned long long) * 3 * te));
  CKC(cudaMalloc(&ctx->d_ticket, sizeof(unsigned int)));
  CKC(cudaMemset(ctx->d_ticket, 0, sizeof(unsigned int)));
  CKC(cudaMalloc(&ctx->d_repairs, sizeof(unsigned long long) * 2 * L));
  CKC(cudaMemset(ctx->d_repairs, 0, sizeof(unsigned long long) * 2 * L));
  ctx->ldh = static_cast<int32_t>(round_up(std::max(c.inter, c.shared_inter), 32));
  const int tdec = std::min(c.max_tokens, 8);
  CKC(cudaMalloc(&ctx->d_h, sizeof(float) * static_cast<size_t>(tdec * c.top_k + tdec) * ctx->ldh));
  CKC(cudaMalloc(&ctx->d_err, sizeof(uint32_t)));
  CKC(cudaMemset(ctx->d_err, 0, sizeof(uint32_t)));
  CKC(cudaHostAlloc(&ctx->h_err, sizeof(uint32_t), cudaHostAllocDefault));
  // uniq [E], counts [E], n_uniq, spare, then the prefetch prediction of the
  // step (expert, weight bits)
  CKC(cudaHostAlloc(&ctx->h_union, sizeof(int32_t) * (2 * E + 4), cudaHostAllocDefault));
  ctx->max_units = std::min(E, c.max_tokens * c.top_k) + 1;
  // room for one unit table and one fill list per compute wave (a wave
  // holds at least one unit; fills <= units)
  // a step's unit tables: at most 1.5 tables per unit (a wave is split only
  // when it has two fills or more), each at most 8 ints of header and padding
  // beyond 4 ints per unit and 2 per fill
  const size_t unit_ints = moe::kUnitHeader + 32 * static_cast<size_t>(ctx->max_units);
  ctx->unit_ints = unit_ints;
  CKC(cudaMalloc(&ctx->d_units, sizeof(int32_t) * unit_ints));
  CKC(cudaMemset(ctx->d_units, 0, sizeof(int32_t) * unit_ints));
  CKC(cudaHostAlloc(&ctx->h_units, sizeof(int32_t) * unit_ints, cudaHostAllocDefault));
  if (c.max_tokens > 8) {
    // prefill scratch: expert-major activations, h, weighted rows, work items
    ctx->prefill = true;
    const int64_t rows = static_cast<int64_t>(c.max_tokens) * (c.top_k + 1);
    ctx->ldh_p = static_cast<int>(round_up(std::max(c.inter, c.shared_inter), 64));
    const int64_t mtiles = (rows + moe::kPrefillTok - 1) / moe::kPrefillTok +
                           std::min<int64_t>(E, static_cast<int64_t>(c.max_tokens) * c.top_k) + 1;
    ctx->max_items0 = static_cast<int>(mtiles * ((std::max(c.inter, c.shared_inter) + 127) / 128));
    ctx->max_items1 = static_cast<int>(mtiles * ((c.hidden + 127) / 128));
    CKC(cudaMalloc(&ctx->d_x16, sizeof(uint16_t) * rows * c.hidden));
    CKC(cudaMalloc(&ctx->d_hp, sizeof(uint16_t) * rows * ctx->ldh_p));
    CKC(cudaMalloc(&ctx->d_yp, sizeof(float) * rows * c.hidden));
    CKC(cudaMalloc(&ctx->d_items0, sizeof(int32_t) * 4 * ctx->max_items0));
    CKC(cudaMalloc(&ctx->d_items1, sizeof(int32_t) * 4 * ctx->max_items1));
    CKC(cudaMalloc(&ctx->d_nitems, sizeof(int32_t) * 2));
    CKC(cudaMalloc(&ctx->d_plan_local,
                   sizeof(int32_t) * moe::plan_blocks(c.max_tokens * c.top_k) * static_cast<int64_t>(E)));
    CKC(cudaMalloc(&ctx->d_norms, sizeof(float) * (c.max_tokens + E)));
    CKC(cudaMalloc(&ctx->d_flags, sizeof(int32_t) * c.max_tokens));
    CKC(cudaMalloc(&ctx->d_lpart, sizeof(float2) * 4 * static_cast<size_t>(c.max_tokens) * E));
    if (c.hidden % 64 == 0) CKC(cudaMalloc(&ctx->d_wsplit, moe::router_split_bytes(E, c.hidden)));
  }
  ctx->dev_admit = c.admit_on_device >= 1;
  ctx->read_through = c.admit_on_device == 2;
  CKC(cudaMalloc(&ctx->d_ffn_ticket, sizeof(unsigned int)));
  CKC(cudaMemset(ctx->d_ffn_ticket, 0, sizeof(unsigned int)));
  {
    // counters of the fused decode FFN: end ticket, abort flag, gate/up
    // items done, one per tile of each unit's down plane
    ctx->fused_units = std::min(E, std::min(c.max_tokens, 8) * c.top_k) + 1;
    const int64_t dn = ctx->geom.qbytes[2] + ctx->geom.sbytes[2];
    ctx->fused_tiles = static_cast<int>((dn + c.tile_bytes - 1) / c.tile_bytes);
    const size_t n = 3 + static_cast<size_t>(ctx->fused_units) * ctx->fused_tiles;
    CKC(cudaMalloc(&ctx->d_fsync, sizeof(unsigned int) * n));
    CKC(cudaMemset(ctx->d_fsync, 0, sizeof(unsigned int) * n));
  }
  if (ctx->dev_admit) {
    ctx->max_fills = std::min(E, c.max_tokens * c.top_k);
    CKC(cudaMalloc(&ctx->d_owner, sizeof(int32_t) * L * S));
    CKC(cudaMemset(ctx->d_owner, 0xFF, sizeof(int32_t) * L * S));
    CKC(cudaMalloc(&ctx->d_sgen, sizeof(uint32_t) * L * S));
    CKC(cudaMemset(ctx->d_sgen, 0, sizeof(uint32_t) * L * S));
    CKC(cudaMalloc(&ctx->d_last, sizeof(unsigned long long) * L * S));
    CKC(cudaMemset(ctx->d_last, 0, sizeof(unsigned long long) * L * S));
    CKC(cudaMalloc(&ctx->d_tick, sizeof(unsigned long long) * L));
    CKC(cudaMemset(ctx->d_tick, 0, sizeof(unsigned long long) * L));
    CKC(cudaMalloc(&ctx->d_rng, sizeof(unsigned long long) * L));
    std::vector<unsigned long long> rng(L);
    for (int l = 0; l < L; ++l) rng[l] = c.seed ^ (static_cast<unsigned long long>(l) * 0x9E3779B97F4A7C15ull);
    CKC(cudaMemcpy(ctx->d_rng, rng.data(), sizeof(unsigned long long) * L, cudaMemcpyHostToDevice));
    CKC(cudaMalloc(&ctx->d_stats, sizeof(long long) * L * moe::kStatCount));
    CKC(cudaMemset(ctx->d_stats, 0, sizeof(long long) * L * moe::kStatCount));
    CKC(cudaMalloc(&ctx->d_fills, sizeof(int32_t) * (1 + 2 * ctx->max_fills)));
    CKC(cudaMemset(ctx->d_fills, 0, sizeof(int32_t) * (1 + 2 * ctx->max_fills)));
    CKC(cudaMalloc(&ctx->d_done, sizeof(unsigned int) * ctx->max_fills));
    CKC(cudaMemset(ctx->d_done, 0, sizeof(unsigned int) * ctx->max_fills));
  }
  ctx->streams.assign(c.n_streams, nullptr);
  ctx->ev_stage.assign(c.n_streams, nullptr);
  ctx->ev_stage_b.assign(c.n_streams, nullptr);
  ctx->ev_prefetch.assign(c.n_streams, nullptr);
  for (int i = 0; i < c.n_streams; ++i) {
    CKC(cudaStreamCreateWithFlags(&ctx->streams[i], cudaStreamNonBlocking));
    CKC(cudaEventCreateWithFlags(&ctx->ev_stage[i], cudaEventDisableTiming));
    CKC(cudaEventCreateWithFlags(&ctx->ev_stage_b[i], cudaEventDisableTiming));
    CKC(cudaEventCreateWithFlags(&ctx->ev_prefetch[i], cudaEventDisableTiming));
  }
  ctx->pred.assign(L, -1);
  CKC(cudaEventCreateWithFlags(&ctx->ev_compute, cudaEventDisableTiming));
  ctx->shared.assign(L, nullptr);
  ctx->tiles_staged.assign(L, 0);
  ctx->bytes_staged.assign(L, 0);
  for (int l = 0; l < L; ++l) {
    moe_slots_t* s = nullptr;
    st = moe_slots_create(E, S, c.policy, c.seed, l, ctx->geom.bytes, &s);
    if (st != MOE_OK) {
      ctx->err = "moe_create: slot manager";
      return bail(st);
    }
    ctx->slots.push_back(s);
  }
  CKC(cudaDeviceSynchronize());
#undef CKC
  *out = ctx;
  return MOE_OK;
}

extern "C" int64_t moe_payload_bytes(const moe_ctx_t* ctx) { return ctx ? ctx->geom.bytes : 0; }
extern "C" int64_t moe_shared_payload_bytes(const moe_ctx_t* ctx) {
  return ctx && ctx->cfg.shared_inter > 0 ? ctx->sgeom.bytes : 0;
}

extern "C" moe_status_t moe_bind_store(moe_ctx_t* ctx, const void* store, size_t bytes) {
  if (!ctx) return MOE_ERR_ARG;
  const size_t want = static_cast<size_t>(ctx->cfg.n_layers) * ctx->cfg.n_experts * ctx->geom.bytes;
  if (!store || bytes != want)
    return fail(ctx, MOE_ERR_ARG, "moe_bind_store: size must be L*E*payload = " + std::to_string(want));
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, store);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return fail(ctx, MOE_ERR_ARG, "moe_bind_store: store is not page-locked host memory");
  }
  void* dev = nullptr;
  e = cudaHostGetDevicePointer(&dev, const_cast<void*>(store), 0);
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (ctx->dev_admit)
      return fail(ctx, MOE_ERR_ARG, "moe_bind_store: store has no device mapping (on-device staging needs one)");
    dev = nullptr;
  }
  if (dev) {
    // touch every page once from the device (one load per page), so that no
    // decode step pays the first-access cost of a page of the store
    uint32_t* sink = nullptr;
    e = cudaMalloc(&sink, sizeof(uint32_t));
    if (e == cudaSuccess) e = moe::launch_touch_pages(static_cast<const uint8_t*>(dev), bytes, ctx->num_sms, sink,
                                                      ctx->streams[0]);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->streams[0]);
    if (sink) cudaFree(sink);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(ctx, MOE_ERR_CUDA, std::string("moe_bind_store: ") + cudaGetErrorString(e));
    }
  }
  ctx->store = static_cast<const uint8_t*>(store);
  ctx->store_dev = static_cast<const uint8_t*>(dev);
  ctx->store_bytes = bytes;
  return MOE_OK;
}

extern "C" moe_status_t moe_bind_shared(moe_ctx_t* ctx, int32_t layer, const void* dev_shared) {
  if (!ctx) return MOE_ERR_ARG;
  if (!valid_layer(ctx, layer)) return fail(ctx, MOE_ERR_ARG, "moe_bind_shared: bad layer");
  if (ctx->cfg.shared_inter == 0) return fail(ctx, MOE_ERR_ARG, "moe_bind_shared: no shared expert configured");
  if (!dev_shared || reinterpret_cast<uintptr_t>(dev_shared) % 16)
    return fail(ctx, MOE_ERR_ARG, "moe_bind_shared: pointer must be non-null and 16-byte aligned");
  ctx->shared[layer] = static_cast<const uint8_t*>(dev_shared);
  return MOE_OK;
}

// ------------------------------------------------------------ routing
static moe::DevCacheLayer dev_cache(moe_ctx_t* ctx, int32_t layer) {
  const size_t E = ctx->cfg.n_experts, S = ctx->cfg.slots_per_layer;
  moe::DevCacheLayer c{};
  c.pt = ctx->d_pt + layer * E;
  c.ptgen = ctx->d_ptgen + layer * E;
  c.owner = ctx->d_owner + layer * S;
  c.sgen = ctx->d_sgen + layer * S;
  c.last = ctx->d_last + layer * S;
  c.tick = ctx->d_tick + layer;
  c.rng = ctx->d_rng + layer;
  c.stats = ctx->d_stats + layer * moe::kStatCount;
  return c;
}

static moe_status_t route_impl(moe_ctx_t* ctx, int32_t layer, const void* x, int32_t xt, int32_t T,
                               const float* w_router, const float* bias, int32_t* topk_idx,
                               float* topk_w, const moe_plan_t* plan, cudaStream_t st,
                               bool admit = false) {
  if (!valid_layer(ctx, layer)) return fail(ctx, MOE_ERR_ARG, "route: bad layer");
  if (T < 1 || T > ctx->cfg.max_tokens) return fail(ctx, MOE_ERR_ARG, "route: T outside 1..max_tokens");
  if (xt != MOE_F32 && xt != MOE_BF16) return fail(ctx, MOE_ERR_ARG, "route: bad activation dtype");
  if (!x || !w_router || !topk_idx || !topk_w) return fail(ctx, MOE_ERR_ARG, "route: null pointer");
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(w_router) % 16)
    return fail(ctx, MOE_ERR_ARG, "route: x and w_router must be 16-byte aligned");
  if (plan && plan->capacity < T * ctx->cfg.top_k)
    return fail(ctx, MOE_ERR_ARG, "route: plan capacity < T*k");
  if (T > 64 && !ctx->d_norms) return fail(ctx, MOE_ERR_ARG, "route: T > 64 needs max_tokens > 8");
  moe::RouteArgs a{};
  a.x = x;
  a.xt = xt;
  a.T = T;
  a.H = ctx->cfg.hidden;
  a.E = ctx->cfg.n_experts;
  a.k = ctx->cfg.top_k;
  a.w = w_router;
  a.bias = bias;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.keys = ctx->d_keys;
  a.ticket = ctx->d_ticket;
  a.repairs = ctx->d_repairs + 2 * layer;
  a.err = ctx->d_err;
  if (plan) a.plan = *plan;
  if (admit) {
    a.admit.enabled = 1;
    a.admit.read_through = (ctx->read_through && T <= 8) ? 1 : 0;
    a.admit.E = ctx->cfg.n_experts;
    a.admit.S = ctx->cfg.slots_per_layer;
    a.admit.policy = ctx->cfg.policy;
    a.admit.has_shared = ctx->cfg.shared_inter > 0 ? 1 : 0;
    a.admit.T = T;
    a.admit.payload = ctx->geom.bytes;
    a.admit.c = dev_cache(ctx, layer);
    a.admit.fills = ctx->d_fills;
    a.admit.units = ctx->d_units;
    a.admit.done = ctx->d_done;
    a.admit.max_fills = ctx->max_fills;
    ctx->dev_state_used = true;
  }
  moe_ctx::TimedLaunch r{MOE_KT_ROUTE, nullptr, nullptr};
  if (ctx->timing) {
    r.a = timing_event(ctx);
    r.b = timing_event(ctx);
    CK(cudaEventRecord(r.a, st));
  }
  if (T > 64) {
    // many tokens: tiled logits, per-token selection, exact repair; the plan
    // and admission run as their own launches
    a.plan = moe_plan_t{};
    a.admit.enabled = 0;
    CK(moe::launch_route_large(a, ctx->d_norms, ctx->d_flags, ctx->d_lpart, ctx->d_wsplit, ctx->num_sms, st));
  } else {
    CK(moe::launch_route(a, ctx->num_sms, st));
  }
  if (ctx->timing) {
    CK(cudaEventRecord(r.b, st));
    ctx->timed.push_back(r);
  }
  return MOE_OK;
}

extern "C" moe_status_t moe_route(moe_ctx_t* ctx, int32_t layer, const void* x, int32_t xt, int32_t T,
                                  const float* w_router, const float* bias, int32_t* topk_idx,
                                  float* topk_w, moe_stream_t stream) {
  if (!ctx) return MOE_ERR_ARG;
  return route_impl(ctx, layer, x, xt, T, w_router, bias, topk_idx, topk_w, nullptr,
                    reinterpret_cast<cudaStream_t>(stream));
}

static bool plan_ok(const moe_plan_t* p) {
  return p && p->counts && p->offsets && p->uniq && p->n_uniq && p->perm_tok && p->perm_rank &&
         p->perm_w && p->inv;
}

extern "C" moe_status_t moe_plan_union(moe_ctx_t* ctx, const int32_t* topk_idx, const float* topk_w,
                                       int32_t T, const moe_plan_t* plan, moe_stream_t stream) {
  if (!ctx) return MOE_ERR_ARG;
  if (!plan_ok(plan) || !topk_idx || !topk_w) return fail(ctx, MOE_ERR_ARG, "plan: null pointer");
  if (T < 1 || T > ctx->cfg.max_tokens) return fail(ctx, MOE_ERR_ARG, "plan: T outside 1..max_tokens");
  if (plan->capacity < T * ctx->cfg.top_k) return fail(ctx, MOE_ERR_ARG, "plan: capacity < T*k");
  moe::PlanArgs a{};
  a.idx = topk_idx;
  a.w = topk_w;
  a.T = T;
  a.k = ctx->cfg.top_k;
  a.E = ctx->cfg.n_experts;
  a.plan = *plan;
  a.err = ctx->d_err;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool large = T * ctx->cfg.top_k > 256;
  if (large && !ctx->d_plan_local) return fail(ctx, MOE_ERR_ARG, "plan: T*k > 256 needs max_tokens > 8");
  moe_ctx::TimedLaunch r{MOE_KT_PLAN, nullptr, nullptr};
  if (ctx->timing) {
    r.a = timing_event(ctx);
    r.b = timing_event(ctx);
    CK(cudaEventRecord(r.a, st));
  }
  if (large)
    CK(moe::launch_plan_large(a, ctx->d_plan_local, st));
  else
    CK(moe::launch_plan(a, st));
  if (ctx->timing) {
    CK(cudaEventRecord(r.b, st));
    ctx->timed.push_back(r);
  }
  return MOE_OK;
}

// ------------------------------------------------------------ cache
static void publish_page_table_host(moe_ctx_t* ctx, int32_t layer) {
  const int E = ctx->cfg.n_experts, S = ctx->cfg.slots_per_layer;
  const moe_slots* s = ctx->slots[layer];
  const int32_t* pt = moe::slots_pt(s);
  const uint32_t* gen = moe::slots_gen(s);
  int32_t* hpt = ctx->h_pt + static_cast<size_t>(layer) * E;
  uint32_t* hpg = ctx->h_ptgen + static_cast<size_t>(layer) * E;
  for (int e = 0; e < E; ++e) {
    hpt[e] = pt[e];
    hpg[e] = pt[e] >= 0 ? gen[pt[e]] : 0u;
  }
  (void)S;
}

// Compute waves of one step, each in two parts: part 0 holds the wave's
// resident units and its first fills, part 1 its last fills (a quarter, at
// least one, when the wave has two fills or more; else nothing). Part 0 is
// computed while part 1's copies are still on the host link; a wave's fills
// never evict its own units, so those copies touch no slot part 0 reads.
// Part j of wave w has its unit table at int offset off[2w+j] of the unit
// buffer and the list of its fills [n, (slot, generation) x n] at offset
// pub[2w+j], with n_units[2w+j] units; fill i of the miss list belongs to
// part part[i] and leaves its slot at generation fill_gen[i].
struct WavePlan {
  std::vector<int32_t> off, pub, n_units;
  std::vector<uint32_t> fill_gen;
  std::vector<int8_t> part;
};

// Host admission of one step. With `waves` null a union larger than the
// slots is refused; otherwise (the prefill path) the step may run in compute
// waves, described by *waves. Each unit carries the slot and the generation it holds
// during its wave: a slot can change hands inside the step, so they come
// from replaying the fill list over the state before the step, not from the
// final page table.
static moe_status_t admit_host(moe_ctx_t* ctx, int32_t layer, const moe_plan_t* plan, moe_miss_list_t* misses,
                               cudaStream_t st, WavePlan* waves) {
  const int E = ctx->cfg.n_experts, S = ctx->cfg.slots_per_layer;
  int32_t* hu = ctx->h_union;
  CK(cudaMemcpyAsync(hu + 2 * E, plan->n_uniq, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  CK(cudaMemcpyAsync(hu, plan->uniq, sizeof(int32_t) * E, cudaMemcpyDeviceToHost, st));
  CK(cudaMemcpyAsync(hu + E, plan->counts, sizeof(int32_t) * E, cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  const int32_t nu = hu[2 * E];
  if (nu < 0 || nu > E) return fail(ctx, MOE_ERR_STATE, "admit: plan holds no valid union");
  if (nu > S && !waves)
    return fail(ctx, MOE_ERR_CAPACITY,
                "admit: the step's union is larger than the slots; only moe_layer_forward on the "
                "prefill path (T > 8) runs such a step, in compute waves");
  moe_slots* sl = ctx->slots[layer];
  std::vector<int32_t> slot_of(E, -1), wave_of(E, 0);
  std::vector<uint32_t> gen_of(E, 0u);
  std::vector<uint32_t> g(moe::slots_gen(sl), moe::slots_gen(sl) + S);
  for (int i = 0; i < nu; ++i) {
    const int e = hu[i];
    if (e < 0 || e >= E) return fail(ctx, MOE_ERR_STATE, "admit: union entry out of range");
    slot_of[e] = moe::slots_pt(sl)[e];
    if (slot_of[e] >= 0) gen_of[e] = g[slot_of[e]];
  }
  moe_status_t s = moe::slots_step(sl, hu, nu, hu + E, misses, &ctx->err);
  if (s != MOE_OK) return s;
  if (waves) waves->fill_gen.assign(misses->n, 0u);
  for (int i = 0; i < misses->n; ++i) {
    const int e = misses->expert[i], slot = misses->slot[i];
    slot_of[e] = slot;
    gen_of[e] = ++g[slot];
    wave_of[e] = misses->wave[i];
    if (waves) waves->fill_gen[i] = gen_of[e];
  }
  publish_page_table_host(ctx, layer);
  const size_t off = static_cast<size_t>(layer) * E;
  CK(cudaMemcpyAsync(ctx->d_pt + off, ctx->h_pt + off, sizeof(int32_t) * E, cudaMemcpyHostToDevice, st));
  CK(cudaMemcpyAsync(ctx->d_ptgen + off, ctx->h_ptgen + off, sizeof(uint32_t) * E,
                     cudaMemcpyHostToDevice, st));
  // unit tables: per wave, its routed experts in union order; the shared
  // expert runs in wave 0
  std::vector<int32_t> p0_of(E, 0);
  int p0 = 0;
  for (int e = 0; e < E; ++e) {
    p0_of[e] = p0;
    p0 += hu[E + e];
  }
  const int n_waves = std::max(1, misses->n_waves);
  const int n_parts = waves ? 2 : 1;
  // part of each expert (1: among the last fills of its wave)
  std::vector<int8_t> part_of(E, 0);
  if (waves) {
    waves->off.assign(2 * n_waves, 0);
    waves->pub.assign(2 * n_waves, 0);
    waves->n_units.assign(2 * n_waves, 0);
    waves->part.assign(misses->n, 0);
    std::vector<int> nf_w(n_waves, 0), seen(n_waves, 0);
    for (int i = 0; i < misses->n; ++i) ++nf_w[misses->wave[i]];
    for (int i = 0; i < misses->n; ++i) {
      const int w = misses->wave[i];
      const int n_last = nf_w[w] >= 2 ? std::max(1, nf_w[w] / 4) : 0;
      const int8_t pt = seen[w]++ >= nf_w[w] - n_last ? 1 : 0;
      waves->part[i] = pt;
      part_of[misses->expert[i]] = pt;
    }
  }
  int32_t* ut = ctx->h_units;
  size_t at = 0;
  for (int w = 0; w < n_waves; ++w) {
    for (int pt = 0; pt < n_parts; ++pt) {
      // size the table (and its fill list) before writing it
      int need_units = (w == 0 && pt == 0 && ctx->cfg.shared_inter > 0) ? 1 : 0, need_fills = 0;
      for (int i = 0; i < nu; ++i) need_units += wave_of[hu[i]] == w && part_of[hu[i]] == pt;
      if (waves)
        for (int i = 0; i < misses->n; ++i) need_fills += misses->wave[i] == w && waves->part[i] == pt;
      const size_t need = moe::kUnitHeader + moe::kUnitInts * static_cast<size_t>(need_units) +
                          (waves ? static_cast<size_t>((1 + 2 * need_fills + 3) / 4 * 4) : 0);
      if (at + need > ctx->unit_ints) return fail(ctx, MOE_ERR_STATE, "admit: unit tables overflow their buffer");
      if (waves) waves->off[n_parts * w + pt] = static_cast<int32_t>(at);
      int32_t* tab = ut + at;
      int n_tab = 0;
      for (int i = 0; i < nu; ++i) {
        const int e = hu[i];
        if (wave_of[e] != w || part_of[e] != pt) continue;
        int32_t* U = tab + moe::kUnitHeader + moe::kUnitInts * n_tab++;
        U[0] = slot_of[e];
        U[1] = p0_of[e];
        U[2] = hu[E + e];
        U[3] = static_cast<int32_t>(gen_of[e]);
      }
      if (w == 0 && pt == 0 && ctx->cfg.shared_inter > 0) {
        int32_t* U = tab + moe::kUnitHeader + moe::kUnitInts * n_tab++;
        U[0] = -1;
        U[1] = -1;
        U[2] = p0 / ctx->cfg.top_k;  // tokens of the step
        U[3] = 0;
      }
      tab[0] = n_tab;
      at += moe::kUnitHeader + moe::kUnitInts * n_tab;
      if (waves) {
        waves->n_units[n_parts * w + pt] = n_tab;
        waves->pub[n_parts * w + pt] = static_cast<int32_t>(at);
        int32_t* pl = ut + at;
        int nf = 0;
        for (int i = 0; i < misses->n; ++i) {
          if (misses->wave[i] != w || waves->part[i] != pt) continue;
          pl[1 + 2 * nf] = misses->slot[i];
          pl[2 + 2 * nf] = static_cast<int32_t>(waves->fill_gen[i]);
          ++nf;
        }
        pl[0] = nf;
        at += (1 + 2 * nf + 3) / 4 * 4;  // keep the next table 16-byte aligned
      }
    }
  }
  CK(cudaMemcpyAsync(ctx->d_units, ut, sizeof(int32_t) * at, cudaMemcpyHostToDevice, st));
  return MOE_OK;
}

extern "C" moe_status_t moe_cache_admit(moe_ctx_t* ctx, int32_t layer, const moe_plan_t* plan,
                                        moe_miss_list_t* misses, moe_stream_t stream) {
  if (!ctx) return MOE_ERR_ARG;
  if (!valid_layer(ctx, layer)) return fail(ctx, MOE_ERR_ARG, "admit: bad layer");
  if (!plan_ok(plan) || !misses) return fail(ctx, MOE_ERR_ARG, "admit: null pointer");
  if (ctx->dev_admit)
    return fail(ctx, MOE_ERR_STATE, "admit: this context admits on the device (moe_layer_forward)");
  return admit_host(ctx, layer, plan, misses, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

// Host->device copies of the fills of compute wave `wave` (all fills if
// wave < 0; with `part`, only fills i with part[i] == which), after the
// compute enqueued so far on `cst` when `after_compute`; their completion is
// recorded in `evs` (one event per copy stream), and `cst` waits for it when
// `join`. *n_out (if given) receives the number of fills copied. The payload is cut into tiles of at most tile_bytes per matrix
// (the accounting unit, and the point where the failure hook cuts); the
// consecutive tiles of one fill go out as one copy, and fills rotate over
// the copy streams: a copy costs microseconds of submission, which 256 KiB
// copies would turn into the bound on the host link. The slots' new
// generations are published by the caller.
static moe_status_t stage_fills(moe_ctx_t* ctx, int32_t layer, const moe_miss_list_t* misses, int wave,
                                const int8_t* part, int which, cudaStream_t cst, bool after_compute,
                                std::vector<cudaEvent_t>& evs, bool join, int* n_out = nullptr) {
  const int E = ctx->cfg.n_experts, S = ctx->cfg.slots_per_layer;
  const int ns = static_cast<int>(ctx->streams.size());
  auto chosen = [&](int i) {
    return (wave < 0 || misses->wave[i] == wave) && (!part || part[i] == which);
  };
  int n = 0;
  for (int i = 0; i < misses->n; ++i) n += chosen(i);
  if (n_out) *n_out = n;
  if (n == 0) return MOE_OK;
  // slots are overwritten only after the compute enqueued so far
  if (after_compute) {
    CK(cudaEventRecord(ctx->ev_compute, cst));
    for (int i = 0; i < ns; ++i) CK(cudaStreamWaitEvent(ctx->streams[i], ctx->ev_compute, 0));
  }
  const moe::ExpertGeom& g = ctx->geom;
  const int64_t tile = ctx->cfg.tile_bytes;
  int64_t issued = 0, bytes = 0, copies = 0;
  bool injected = false;
  for (int i = 0; i < misses->n && !injected; ++i) {
    if (!chosen(i)) continue;
    const int e = misses->expert[i], slot = misses->slot[i];
    if (e < 0 || e >= E || slot < 0 || slot >= S) return fail(ctx, MOE_ERR_ARG, "stage: fill out of range");
    const uint8_t* src = ctx->store + (static_cast<size_t>(layer) * E + e) * g.bytes;
    uint8_t* dst = ctx->d_pool + (static_cast<size_t>(layer) * S + slot) * ctx->slot_stride;
    cudaStream_t cs = ctx->streams[copies % ns];
    int64_t run0 = 0, run_len = 0;  // pending run of consecutive tiles
    for (int m = 0; m < 3 && !injected; ++m) {
      const int64_t mo = g.qoff[m], mb = g.qbytes[m] + g.sbytes[m];
      for (int64_t o = 0; o < mb; o += tile) {
        if (ctx->fail_after_tiles >= 0 && issued == ctx->fail_after_tiles) {
          injected = true;
          break;
        }
        const int64_t len = std::min(tile, mb - o);
        if (run_len > 0 && run0 + run_len != mo + o) {
          CK(cudaMemcpyAsync(dst + run0, src + run0, static_cast<size_t>(run_len), cudaMemcpyHostToDevice, cs));
          run_len = 0;
        }
        if (run_len == 0) run0 = mo + o;
        run_len += len;
        ++issued;
        bytes += len;
      }
    }
    if (run_len > 0)
      CK(cudaMemcpyAsync(dst + run0, src + run0, static_cast<size_t>(run_len), cudaMemcpyHostToDevice, cs));
    ++copies;
  }
  for (int i = 0; i < ns; ++i) {
    CK(cudaEventRecord(evs[i], ctx->streams[i]));
    if (join) CK(cudaStreamWaitEvent(cst, evs[i], 0));
  }
  ctx->tiles_staged[layer] += issued;
  ctx->bytes_staged[layer] += bytes;
  if (injected) {
    ctx->fail_after_tiles = -1;
    return fail(ctx, MOE_ERR_CUDA, "stage: injected copy failure (test hook); slots not published");
  }
  if (ctx->fail_after_tiles >= 0) ctx->fail_after_tiles -= static_cast<int32_t>(issued);
  return MOE_OK;
}

extern "C" moe_status_t moe_stage_tiles(moe_ctx_t* ctx, int32_t layer, const moe_miss_list_t* misses,
                                        moe_stream_t compute_stream) {
  if (!ctx) return MOE_ERR_ARG;
  if (!valid_layer(ctx, layer) || !misses || misses->layer != layer)
    return fail(ctx, MOE_ERR_ARG, "stage: bad layer or miss list");
  if (misses->n > 0 && !ctx->store) return fail(ctx, MOE_ERR_STATE, "stage: no store bound");
  if (ctx->dev_admit)
    return fail(ctx, MOE_ERR_STATE, "stage: this context stages on the device (moe_layer_forward)");
  if (misses->n_waves > 1)
    return fail(ctx, MOE_ERR_STATE, "stage: a step in compute waves is staged by moe_layer_forward");
  cudaStream_t cst = reinterpret_cast<cudaStream_t>(compute_stream);
  const int S = ctx->cfg.slots_per_layer;
  if (misses->n == 0) return MOE_OK;
  moe_status_t s = stage_fills(ctx, layer, misses, -1, nullptr, 0, cst, true, ctx->ev_stage, true);
  if (s != MOE_OK) return s;
  // publish the new generations of the filled slots
  const uint32_t* gen = moe::slots_gen(ctx->slots[layer]);
  uint32_t* hg = ctx->h_gen + static_cast<size_t>(layer) * S;
  for (int i = 0; i < misses->n; ++i) hg[misses->slot[i]] = gen[misses->slot[i]];
  CK(cudaMemcpyAsync(ctx->d_gen + static_cast<size_t>(layer) * S, hg, sizeof(uint32_t) * S,
                     cudaMemcpyHostToDevice, cst));
  return MOE_OK;
}

extern "C" moe_status_t moe_cache_evict(moe_ctx_t* ctx, int32_t layer, int32_t expert) {
  if (!ctx) return MOE_ERR_ARG;
  if (!valid_layer(ctx, layer)) return fail(ctx, MOE_ERR_ARG, "evict: bad layer");
  CK(cudaDeviceSynchronize());
  if (ctx->dev_admit) {
    if (expert < 0 || expert >= ctx->cfg.n_experts) return fail(ctx, MOE_ERR_ARG, "evict: bad expert");
    moe::DevCacheLayer c = dev_cache(ctx, layer);
    int32_t slot = -1;
    CK(cudaMemcpy(&slot, c.pt + expert, sizeof(int32_t), cudaMemcpyDeviceToHost));
    if (slot < 0) return MOE_OK;
    const int32_t none = -1;
    long long ev = 0;
    CK(cudaMemcpy(c.pt + expert, &none, sizeof(int32_t), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(c.owner + slot, &none, sizeof(int32_t), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(&ev, c.stats + moe::kStatEvictions, sizeof(long long), cudaMemcpyDeviceToHost));
    ++ev;
    CK(cudaMemcpy(c.stats + moe::kStatEvictions, &ev, sizeof(long long), cudaMemcpyHostToDevice));
    return MOE_OK;
  }
  moe_status_t s = moe::slots_evict(ctx->slots[layer], expert, &ctx->err);
  if (s != MOE_OK) return s;
  publish_page_table_host(ctx, layer);
  const size_t off = static_cast<size_t>(layer) * ctx->cfg.n_experts;
  CK(cudaMemcpy(ctx->d_pt + off, ctx->h_pt + off, sizeof(int32_t) * ctx->cfg.n_experts,
                cudaMemcpyHostToDevice));
  CK(cudaMemcpy(ctx->d_ptgen + off, ctx->h_ptgen + off, sizeof(uint32_t) * ctx->cfg.n_experts,
                cudaMemcpyHostToDevice));
  return MOE_OK;
}

extern "C" moe_status_t moe_cache_preload(moe_ctx_t* ctx, int32_t layer, const int32_t* experts,
                                          int32_t n) {
  if (!ctx) return MOE_ERR_ARG;
  if (!valid_layer(ctx, layer) || n < 0 || (n > 0 && !experts))
    return fail(ctx, MOE_ERR_ARG, "preload: bad arguments");
  if (!ctx->store) return fail(ctx, MOE_ERR_STATE, "preload: no store bound");
  if (ctx->dev_admit && ctx->dev_state_used)
    return fail(ctx, MOE_ERR_STATE, "preload: on-device admission already ran on this context");
  CK(cudaDeviceSynchronize());
  std::vector<int32_t> filled, fslots;
  moe_status_t s = moe::slots_preload(ctx->slots[layer], experts, n, &filled, &fslots, &ctx->err);
  if (s != MOE_OK) return s;
  const int E = ctx->cfg.n_experts, S = ctx->cfg.slots_per_layer;
  for (size_t i = 0; i < filled.size(); ++i) {
    const uint8_t* src = ctx->store + (static_cast<size_t>(layer) * E + filled[i]) * ctx->geom.bytes;
    uint8_t* dst = ctx->d_pool + (static_cast<size_t>(layer) * S + fslots[i]) * ctx->slot_stride;
    CK(cudaMemcpy(dst, src, ctx->geom.bytes, cudaMemcpyHostToDevice));
  }
  publish_page_table_host(ctx, layer);
  const uint32_t* gen = moe::slots_gen(ctx->slots[layer]);
  uint32_t* hg = ctx->h_gen + static_cast<size_t>(layer) * S;
  for (int i = 0; i < S; ++i) hg[i] = gen[i];
  const size_t off = static_cast<size_t>(layer) * E;
  CK(cudaMemcpy(ctx->d_pt + off, ctx->h_pt + off, sizeof(int32_t) * E, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(ctx->d_ptgen + off, ctx->h_ptgen + off, sizeof(uint32_t) * E, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(ctx->d_gen + static_cast<size_t>(layer) * S, hg, sizeof(uint32_t) * S,
                cudaMemcpyHostToDevice));
  if (ctx->dev_admit) {
    // the device-side cache state starts from the host manager's
    moe::DevCacheLayer c = dev_cache(ctx, layer);
    const moe_slots* sl = ctx->slots[layer];
    std::vector<unsigned long long> last(moe::slots_last(sl), moe::slots_last(sl) + S);
    const unsigned long long tick = moe::slots_tick(sl);
    CK(cudaMemcpy(c.owner, moe::slots_owner(sl), sizeof(int32_t) * S, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(c.sgen, moe::slots_gen(sl), sizeof(uint32_t) * S, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(c.last, last.data(), sizeof(unsigned long long) * S, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(c.tick, &tick, sizeof(unsigned long long), cudaMemcpyHostToDevice));
  }
  return MOE_OK;
}

// Checks and arguments of the prefill FFN over the unit table at d_units.
static moe_status_t prefill_setup(moe_ctx_t* ctx, int32_t layer, const void* x, int32_t xt, int32_t T,
                                  const moe_plan_t* plan, float* y, moe::PrefillArgs* out) {
  const moe_config_t& c = ctx->cfg;
  const int E = c.n_experts, S = c.slots_per_layer;
  if (!ctx->prefill) return fail(ctx, MOE_ERR_ARG, "ffn: the prefill path needs max_tokens > 8");
  if (c.quant != MOE_Q8_0) return fail(ctx, MOE_ERR_ARG, "ffn: the prefill path reads Q8_0 experts");
  if (c.hidden % 128 || c.inter % 64 || c.shared_inter % 64 || E > 1023)
    return fail(ctx, MOE_ERR_ARG, "ffn: the prefill path needs H % 128 == 0, I and I_s multiples of 64 and E <= 1023");
  moe::PrefillArgs& p = *out;
  p = moe::PrefillArgs{};
  p.x = x;
  p.xt = xt;
  p.T = T;
  p.k = c.top_k;
  p.H = c.hidden;
  p.I = c.inter;
  p.Is = c.shared_inter;
  p.S = S;
  p.units = ctx->d_units;
  p.plan = *plan;
  p.pool = ctx->d_pool + static_cast<size_t>(layer) * S * ctx->slot_stride;
  p.slot_stride = ctx->slot_stride;
  p.shared = ctx->shared[layer];
  p.g = ctx->geom;
  p.gs = ctx->sgeom;
  p.x16 = reinterpret_cast<__half*>(ctx->d_x16);
  p.h = ctx->d_hp;
  p.ldh = ctx->ldh_p;
  p.yp = ctx->d_yp;
  p.y = y;
  p.items0 = ctx->d_items0;
  p.items1 = ctx->d_items1;
  p.n_items0 = ctx->d_nitems;
  p.n_items1 = ctx->d_nitems + 1;
  p.max_items0 = ctx->max_items0;
  p.max_items1 = ctx->max_items1;
  p.n_sm = ctx->num_sms;
  p.err = ctx->d_err;
  p.gen = ctx->d_gen + static_cast<size_t>(layer) * S;
  return MOE_OK;
}

// Enqueues the parts p.parts of the prefill FFN (timed when enabled).
static moe_status_t prefill_run(moe_ctx_t* ctx, moe::PrefillArgs& p, cudaStream_t st) {
  const bool timed = ctx->timing && (p.parts & moe::kPartGemm);
  p.wait_cycles = 0;
  p.skip_ring = -1;
  if ((p.parts & moe::kPartGemm) && ctx->dbg_skip_ring >= 0) {  // one-shot test hook
    p.wait_cycles = ctx->dbg_wait_cycles;
    p.skip_ring = ctx->dbg_skip_ring;
    ctx->dbg_wait_cycles = 0;
    ctx->dbg_skip_ring = -1;
  }
  for (int i = 0; i < 4; ++i) p.ev[i] = timed ? timing_event(ctx) : nullptr;
  CK(moe::prefill_ffn(p, st));
  if (timed) {
    ctx->timed.push_back({MOE_KT_GATEUP, p.ev[0], p.ev[1]});
    ctx->timed.push_back({MOE_KT_DOWN, p.ev[2], p.ev[3]});
    if (ctx->timed.size() > 16384) CK(resolve_timing(ctx));
  }
  return MOE_OK;
}

// ------------------------------------------------------------ FFN
extern "C" moe_status_t moe_expert_ffn(moe_ctx_t* ctx, int32_t layer, const void* x, int32_t xt,
                                       int32_t T, const moe_plan_t* plan, float* y, int32_t mode,
                                       moe_stream_t stream) {
  if (!ctx) return MOE_ERR_ARG;
  if (!valid_layer(ctx, layer)) return fail(ctx, MOE_ERR_ARG, "ffn: bad layer");
  if (!plan_ok(plan) || !x || !y) return fail(ctx, MOE_ERR_ARG, "ffn: null pointer");
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(y) % 16)
    return fail(ctx, MOE_ERR_ARG, "ffn: x and y must be 16-byte aligned");
  if (T < 1 || T > ctx->cfg.max_tokens) return fail(ctx, MOE_ERR_ARG, "ffn: T outside 1..max_tokens");
  if (xt != MOE_F32 && xt != MOE_BF16) return fail(ctx, MOE_ERR_ARG, "ffn: bad activation dtype");
  if (plan->capacity < T * ctx->cfg.top_k) return fail(ctx, MOE_ERR_ARG, "ffn: plan capacity < T*k");
  if (ctx->cfg.shared_inter > 0 && !ctx->shared[layer])
    return fail(ctx, MOE_ERR_STATE, "ffn: shared expert of this layer not bound");
  if (mode == MOE_MODE_AUTO) mode = T <= 8 ? MOE_MODE_DECODE : MOE_MODE_PREFILL;
  const int E = ctx->cfg.n_experts, S = ctx->cfg.slots_per_layer;
  if (mode == MOE_MODE_PREFILL) {
    moe::PrefillArgs p{};
    moe_status_t s = prefill_setup(ctx, layer, x, xt, T, plan, y, &p);
    if (s != MOE_OK) return s;
    p.parts = moe::kPartAll;
    return prefill_run(ctx, p, reinterpret_cast<cudaStream_t>(stream));
  }
  if (mode != MOE_MODE_DECODE || T > 8) return fail(ctx, MOE_ERR_ARG, "ffn: decode mode needs T <= 8");
  moe::FfnArgs a{};
  a.x = x;
  a.xt = xt;
  a.T = T;
  a.H = ctx->cfg.hidden;
  a.I = ctx->cfg.inter;
  a.Is = ctx->cfg.shared_inter;
  a.k = ctx->cfg.top_k;
  a.E = E;
  a.quant = ctx->cfg.quant;
  a.pool = ctx->d_pool + static_cast<size_t>(layer) * S * ctx->slot_stride;
  a.slot_stride = ctx->slot_stride;
  a.units = ctx->d_units;
  a.gen = ctx->d_gen + static_cast<size_t>(layer) * S;
  if (ctx->read_through) {
    if (!ctx->store_dev) return fail(ctx, MOE_ERR_STATE, "ffn: no store bound");
    a.store = ctx->store_dev + static_cast<size_t>(layer) * E * ctx->geom.bytes;
    a.payload = ctx->geom.bytes;
    a.sgen = ctx->d_sgen + static_cast<size_t>(layer) * S;
    a.ticket = ctx->d_ffn_ticket;
    a.stats = ctx->d_stats + static_cast<size_t>(layer) * moe::kStatCount;
    a.tiles_per_expert = 0;
    for (int m = 0; m < 3; ++m)
      a.tiles_per_expert += static_cast<int>((ctx->geom.qbytes[m] + ctx->geom.sbytes[m] +
                                              ctx->cfg.tile_bytes - 1) / ctx->cfg.tile_bytes);
  }
  a.S = S;
  a.shared = ctx->shared[layer];
  a.g = ctx->geom;
  a.gs = ctx->sgeom;
  a.plan = *plan;
  a.h = ctx->d_h;
  a.ldh = ctx->ldh;
  a.y = y;
  a.err = ctx->d_err;
  if (ctx->cfg.decode_ffn == 0) {
    // two launches: gate/up + SwiGLU, then down + combine
    if (ctx->timing) {
      for (int i = 0; i < 4; ++i) a.ev[i] = timing_event(ctx);
    }
    CK(moe::launch_ffn_decode(a, ctx->num_sms, reinterpret_cast<cudaStream_t>(stream)));
    if (ctx->timing) {
      ctx->timed.push_back({MOE_KT_GATEUP, a.ev[0], a.ev[1]});
      ctx->timed.push_back({MOE_KT_DOWN, a.ev[2], a.ev[3]});
      if (ctx->timed.size() > 16384) CK(resolve_timing(ctx));
    }
    return MOE_OK;
  }
  if (ctx->timing) {
    for (int i = 0; i < 2; ++i) a.ev[i] = timing_event(ctx);
  }
  // one persistent launch: gate/up, down and the misses' down-plane tiles
  moe::FusedLaunch fl{};
  fl.sync = ctx->d_fsync;
  fl.max_units = ctx->fused_units;
  fl.max_tiles = ctx->fused_tiles;
  fl.tile_bytes = ctx->cfg.tile_bytes;
  fl.wait_cycles = moe::kFusedWaitCycles;
  fl.grid = ctx->num_sms;
  fl.pdl = true;
  CK(moe::launch_ffn_decode_fused(a, fl, reinterpret_cast<cudaStream_t>(stream)));
  if (ctx->timing) {
    ctx->timed.push_back({MOE_KT_FFN, a.ev[0], a.ev[1]});
    if (ctx->timed.size() > 16384) CK(resolve_timing(ctx));
  }
  return MOE_OK;
}

extern "C" moe_status_t moe_layer_forward(moe_ctx_t* ctx, int32_t layer, const void* x, int32_t xt,
                                          int32_t T, const float* w_router, const float* bias,
                                          int32_t* topk_idx, float* topk_w, const moe_plan_t* plan,
                                          float* y, moe_miss_list_t* misses, moe_stream_t stream) {
  if (!ctx) return MOE_ERR_ARG;
  if (!plan_ok(plan)) return fail(ctx, MOE_ERR_ARG, "layer_forward: plan has a null array");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (ctx->dev_admit) {
    // route + plan + admission in one launch, then staging and the FFN; no
    // host synchronisation (the step can be captured in a CUDA graph)
    if (!ctx->store_dev) return fail(ctx, MOE_ERR_STATE, "layer_forward: no store bound");
    moe_status_t s = route_impl(ctx, layer, x, xt, T, w_router, bias, topk_idx, topk_w, plan, st, true);
    if (s != MOE_OK) return s;
    if (T > 64) {
      // many tokens: the plan and the admission are separate launches
      s = moe_plan_union(ctx, topk_idx, topk_w, T, plan, stream);
      if (s != MOE_OK) return s;
      moe::AdmitArgs ad{};
      ad.enabled = 1;
      ad.read_through = 0;
      ad.E = ctx->cfg.n_experts;
      ad.S = ctx->cfg.slots_per_layer;
      ad.policy = ctx->cfg.policy;
      ad.has_shared = ctx->cfg.shared_inter > 0 ? 1 : 0;
      ad.T = T;
      ad.payload = ctx->geom.bytes;
      ad.c = dev_cache(ctx, layer);
      ad.fills = ctx->d_fills;
      ad.units = ctx->d_units;
      ad.done = ctx->d_done;
      ad.max_fills = ctx->max_fills;
      ctx->dev_state_used = true;
      CK(moe::launch_admit(ad, *plan, std::min(ctx->cfg.n_experts, T * ctx->cfg.top_k), ctx->d_err, st));
    }
    if (ctx->read_through && T <= 8)  // misses are materialised by the FFN as it reads them
      return moe_expert_ffn(ctx, layer, x, xt, T, plan, y, MOE_MODE_AUTO, stream);
    const moe::ExpertGeom& g = ctx->geom;
    moe::StageArgs sa{};
    const size_t E = ctx->cfg.n_experts, S = ctx->cfg.slots_per_layer;
    sa.store = ctx->store_dev + static_cast<size_t>(layer) * E * g.bytes;
    sa.pool = ctx->d_pool + static_cast<size_t>(layer) * S * ctx->slot_stride;
    sa.slot_stride = ctx->slot_stride;
    sa.payload = g.bytes;
    sa.fills = ctx->d_fills;
    sa.done = ctx->d_done;
    sa.sgen = ctx->d_sgen + static_cast<size_t>(layer) * S;
    sa.gen = ctx->d_gen + static_cast<size_t>(layer) * S;
    sa.stats = ctx->d_stats + static_cast<size_t>(layer) * moe::kStatCount;
    sa.tile_bytes = ctx->cfg.tile_bytes;
    sa.tiles_per_expert = 0;
    sa.chunks_per_expert = 0;
    for (int m = 0; m < 3; ++m) {
      sa.mat_off[m] = g.qoff[m];
      sa.mat_bytes[m] = g.qbytes[m] + g.sbytes[m];
      sa.tiles_per_expert += static_cast<int>((sa.mat_bytes[m] + sa.tile_bytes - 1) / sa.tile_bytes);
      sa.chunks[m] = static_cast<int>((sa.mat_bytes[m] + moe::kStageChunkBytes - 1) / moe::kStageChunkBytes);
      sa.chunks_per_expert += sa.chunks[m];
    }
    sa.max_fills = std::min(ctx->max_fills, std::min(T * ctx->cfg.top_k, ctx->cfg.n_experts));
    sa.grid = 4 * ctx->num_sms;
    if (ctx->timing) {
      moe_ctx::TimedLaunch r{MOE_KT_STAGE, timing_event(ctx), timing_event(ctx)};
      CK(cudaEventRecord(r.a, st));
      CK(moe::launch_stage_copy(sa, st));
      CK(cudaEventRecord(r.b, st));
      ctx->timed.push_back(r);
    } else {
      CK(moe::launch_stage_copy(sa, st));
    }
    return moe_expert_ffn(ctx, layer, x, xt, T, plan, y, MOE_MODE_AUTO, stream);
  }
  // confidence-gated prefetch of the layer's prediction from its previous
  // step: a load goes out on the staging streams now, overlapping this
  // step's routing and admission
  int pf_slot = -1;
  uint32_t pf_gen = 0;
  if (ctx->prefetch_mode != MOE_PREFETCH_OFF && ctx->pred[layer] >= 0) {
    if (!ctx->store) return fail(ctx, MOE_ERR_STATE, "layer_forward: no store bound");
    int32_t action = 0;
    moe_miss_list_t fl{};
    moe_status_t ps = moe::slots_prefetch(ctx->slots[layer], ctx->pred[layer], ctx->prefetch_mode, &action, &fl,
                                          &ctx->err);
    ctx->pred[layer] = -1;
    if (ps != MOE_OK) return ps;
    if (action == MOE_PREFETCH_LOADED) {
      ps = stage_fills(ctx, layer, &fl, -1, nullptr, 0, st, true, ctx->ev_prefetch, false);
      if (ps != MOE_OK) return ps;
      pf_slot = fl.slot[0];
      pf_gen = moe::slots_gen(ctx->slots[layer])[pf_slot];
    }
  }
  moe_status_t s = route_impl(ctx, layer, x, xt, T, w_router, bias, topk_idx, topk_w, plan, st);
  if (s != MOE_OK) return s;
  if (T > 64) {
    s = moe_plan_union(ctx, topk_idx, topk_w, T, plan, stream);
    if (s != MOE_OK) return s;
  }
  const int E_ = ctx->cfg.n_experts, k_ = ctx->cfg.top_k;
  int32_t* hpred = ctx->h_union + 2 * E_ + 2;
  if (ctx->prefetch_mode != MOE_PREFETCH_OFF) {
    // the next step's prediction: the last token's rank-0 expert and weight
    // (read back with the union, before the admission's synchronisation)
    CK(cudaMemcpyAsync(hpred, topk_idx + static_cast<size_t>(T - 1) * k_, sizeof(int32_t),
                       cudaMemcpyDeviceToHost, st));
    CK(cudaMemcpyAsync(hpred + 1, topk_w + static_cast<size_t>(T - 1) * k_, sizeof(float),
                       cudaMemcpyDeviceToHost, st));
  }
  // after the admission: record the prediction; the prefetched slot's
  // generation is published once its copy has landed (before any copy or
  // compute of this step that could touch or read that slot)
  auto after_admit = [&]() -> moe_status_t {
    if (ctx->prefetch_mode != MOE_PREFETCH_OFF) {
      float wgt;
      std::memcpy(&wgt, hpred + 1, sizeof(float));
      ctx->pred[layer] = (hpred[0] >= 0 && hpred[0] < E_ && wgt >= ctx->prefetch_threshold) ? hpred[0] : -1;
    }
    if (pf_slot >= 0) {
      const int S_ = ctx->cfg.slots_per_layer;
      for (auto e : ctx->ev_prefetch) CK(cudaStreamWaitEvent(st, e, 0));
      // (the host mirror may change again within this call, in a later
      // compute wave, before a copy from it would run)
      ctx->h_gen[static_cast<size_t>(layer) * S_ + pf_slot] = pf_gen;
      CK(moe::launch_set_word(ctx->d_gen + static_cast<size_t>(layer) * S_ + pf_slot, pf_gen, st));
    }
    return MOE_OK;
  };
  moe_miss_list_t local{};
  moe_miss_list_t* ml = misses ? misses : &local;
  if (T <= 8) {
    s = moe_cache_admit(ctx, layer, plan, ml, stream);
    if (s != MOE_OK) return s;
    if ((s = after_admit()) != MOE_OK) return s;
    s = moe_stage_tiles(ctx, layer, ml, stream);
    if (s != MOE_OK) return s;
    return moe_expert_ffn(ctx, layer, x, xt, T, plan, y, MOE_MODE_AUTO, stream);
  }
  // prefill: the step may run in compute waves
  if (!ctx->store) return fail(ctx, MOE_ERR_STATE, "layer_forward: no store bound");
  if (ctx->cfg.shared_inter > 0 && !ctx->shared[layer])
    return fail(ctx, MOE_ERR_STATE, "layer_forward: shared expert of this layer not bound");
  moe::PrefillArgs p{};
  s = prefill_setup(ctx, layer, x, xt, T, plan, y, &p);
  if (s != MOE_OK) return s;
  WavePlan wp;
  s = admit_host(ctx, layer, plan, ml, st, &wp);
  if (s != MOE_OK) return s;
  if ((s = after_admit()) != MOE_OK) return s;
  const int S = ctx->cfg.slots_per_layer;
  uint32_t* hg = ctx->h_gen + static_cast<size_t>(layer) * S;
  p.parts = moe::kPartGather;
  if ((s = prefill_run(ctx, p, st)) != MOE_OK) return s;
  const int n_waves = static_cast<int>(wp.off.size()) / 2;
  for (int w = 0; w < n_waves; ++w) {
    // both parts' copies go out now (part 1's behind part 0's on the same
    // streams, with no new wait on the compute): part 0 is computed while
    // part 1 is still on the host link
    int nf[2] = {0, 0};
    s = stage_fills(ctx, layer, ml, w, wp.part.data(), 0, st, true, ctx->ev_stage, false, &nf[0]);
    if (s != MOE_OK) return s;
    // (part 1 waits for the compute itself if part 0 copied nothing)
    s = stage_fills(ctx, layer, ml, w, wp.part.data(), 1, st, nf[0] == 0, ctx->ev_stage_b, false, &nf[1]);
    if (s != MOE_OK) return s;
    for (int pt = 0; pt < 2; ++pt) {
      const int sw = 2 * w + pt;
      if (wp.n_units[sw] == 0) continue;
      if (nf[pt] > 0)
        for (auto e : pt == 0 ? ctx->ev_stage : ctx->ev_stage_b) CK(cudaStreamWaitEvent(st, e, 0));
      // the part's slots hold their new payloads: publish their generations
      // on the device (from the part's fill list) and in the host mirror
      p.parts = moe::kPartGemm;
      p.units = ctx->d_units + wp.off[sw];
      p.publish_gen = ctx->d_gen + static_cast<size_t>(layer) * S;
      p.publish_list = ctx->d_units + wp.pub[sw];
      if ((s = prefill_run(ctx, p, st)) != MOE_OK) return s;
      for (int i = 0; i < ml->n; ++i)
        if (ml->wave[i] == w && wp.part[i] == pt) hg[ml->slot[i]] = wp.fill_gen[i];
    }
  }
  p.parts = moe::kPartCombine;
  p.publish_gen = nullptr;
  return prefill_run(ctx, p, st);
}

extern "C" moe_status_t moe_check_device_errors(moe_ctx_t* ctx, moe_stream_t stream) {
  if (!ctx) return MOE_ERR_ARG;
  CK(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  CK(cudaMemcpy(ctx->h_err, ctx->d_err, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  const uint32_t e = *ctx->h_err;
  if (e == 0) return MOE_OK;
  CK(cudaMemset(ctx->d_err, 0, sizeof(uint32_t)));
  if (e & MOE_DEVERR_STALE)
    return fail(ctx, MOE_ERR_STALE, "device: an expert's page-table entry or slot generation was invalid");
  if (e & MOE_DEVERR_TIMEOUT) return fail(ctx, MOE_ERR_TIMEOUT, "device: a bounded wait ran out");
  if (e & MOE_DEVERR_CAPACITY)
    return fail(ctx, MOE_ERR_CAPACITY, "device: a step's union did not fit the slots; it was not admitted");
  if (e & MOE_DEVERR_NONFINITE)
    return fail(ctx, MOE_ERR_UNCERTIFIED, "device: non-finite router input; routing undefined");
  return fail(ctx, MOE_ERR_ARG, "device: expert id out of range in a plan input");
}

// ------------------------------------------------------------ inspection
extern "C" moe_status_t moe_get_stats(const moe_ctx_t* cctx, int32_t layer, moe_stats_t* out) {
  moe_ctx_t* ctx = const_cast<moe_ctx_t*>(cctx);
  if (!ctx || !out) return MOE_ERR_ARG;
  if (layer != -1 && !valid_layer(ctx, layer)) return fail(ctx, MOE_ERR_ARG, "stats: bad layer");
  const int L = ctx->cfg.n_layers;
  std::vector<unsigned long long> rep(2 * static_cast<size_t>(L));
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(rep.data(), ctx->d_repairs, sizeof(unsigned long long) * 2 * L, cudaMemcpyDeviceToHost));
  std::vector<long long> ds;
  if (ctx->dev_admit) {
    ds.resize(static_cast<size_t>(L) * moe::kStatCount);
    CK(cudaMemcpy(ds.data(), ctx->d_stats, sizeof(long long) * ds.size(), cudaMemcpyDeviceToHost));
  }
  moe_stats_t t{};
  for (int l = 0; l < L; ++l) {
    if (layer != -1 && l != layer) continue;
    moe_stats_t s = moe::slots_stats(ctx->slots[l]);
    if (ctx->dev_admit) {
      const long long* d = ds.data() + static_cast<size_t>(l) * moe::kStatCount;
      s.steps = d[moe::kStatSteps];
      s.hits = d[moe::kStatHits];
      s.misses = d[moe::kStatMisses];
      s.evictions += d[moe::kStatEvictions];
      s.materialized_bytes = d[moe::kStatMaterialized];
      t.tiles_staged += d[moe::kStatTiles];
      t.bytes_staged += d[moe::kStatBytes];
    }
    t.steps += s.steps;
    t.hits += s.hits;
    t.misses += s.misses;
    t.evictions += s.evictions;
    t.materialized_bytes += s.materialized_bytes;
    t.tiles_staged += ctx->tiles_staged[l];
    t.bytes_staged += ctx->bytes_staged[l];
    t.uncertified_repairs += static_cast<int64_t>(rep[2 * l]);
    t.route_filter_fallbacks += static_cast<int64_t>(rep[2 * l + 1]);
    t.prefetch_loads += s.prefetch_loads;
    t.prefetch_useful += s.prefetch_useful;
    t.prefetch_wasted += s.prefetch_wasted;
    t.prefetch_refreshes += s.prefetch_refreshes;
    t.prefetch_probes += s.prefetch_probes;
    t.prefetch_bytes += s.prefetch_bytes;
  }
  *out = t;
  return MOE_OK;
}

extern "C" moe_status_t moe_read_page_table(moe_ctx_t* ctx, int32_t layer, int32_t* host_pt,
                                            uint32_t* host_gen) {
  if (!ctx) return MOE_ERR_ARG;
  if (!valid_layer(ctx, layer)) return fail(ctx, MOE_ERR_ARG, "read_page_table: bad layer");
  CK(cudaDeviceSynchronize());
  const int E = ctx->cfg.n_experts, S = ctx->cfg.slots_per_layer;
  if (host_pt)
    CK(cudaMemcpy(host_pt, ctx->d_pt + static_cast<size_t>(layer) * E, sizeof(int32_t) * E,
                  cudaMemcpyDeviceToHost));
  if (host_gen)
    CK(cudaMemcpy(host_gen, ctx->d_gen + static_cast<size_t>(layer) * S, sizeof(uint32_t) * S,
                  cudaMemcpyDeviceToHost));
  return MOE_OK;
}

extern "C" moe_status_t moe_read_slot(moe_ctx_t* ctx, int32_t layer, int32_t slot, void* host_out,
                                      size_t bytes) {
  if (!ctx) return MOE_ERR_ARG;
  if (!valid_layer(ctx, layer) || slot < 0 || slot >= ctx->cfg.slots_per_layer || !host_out ||
      bytes > static_cast<size_t>(ctx->geom.bytes))
    return fail(ctx, MOE_ERR_ARG, "read_slot: bad arguments");
  CK(cudaDeviceSynchronize());
  const uint8_t* src =
      ctx->d_pool + (static_cast<size_t>(layer) * ctx->cfg.slots_per_layer + slot) * ctx->slot_stride;
  CK(cudaMemcpy(host_out, src, bytes, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

extern "C" moe_status_t moe_debug_fail_staging_after(moe_ctx_t* ctx, int32_t fail_after_tiles) {
  if (!ctx) return MOE_ERR_ARG;
  ctx->fail_after_tiles = fail_after_tiles < 0 ? -1 : fail_after_tiles;
  return MOE_OK;
}

extern "C" moe_status_t moe_debug_corrupt_generation(moe_ctx_t* ctx, int32_t layer, int32_t expert) {
  if (!ctx) return MOE_ERR_ARG;
  if (!valid_layer(ctx, layer) || expert < 0 || expert >= ctx->cfg.n_experts)
    return fail(ctx, MOE_ERR_ARG, "corrupt_generation: bad arguments");
  CK(cudaDeviceSynchronize());
  // the slot's published generation no longer matches the page-table entry,
  // as if its content had been replaced behind the table's back
  const size_t E = ctx->cfg.n_experts, S = ctx->cfg.slots_per_layer;
  int32_t slot = -1;
  CK(cudaMemcpy(&slot, ctx->d_pt + layer * E + expert, sizeof(int32_t), cudaMemcpyDeviceToHost));
  if (slot < 0) return fail(ctx, MOE_ERR_ARG, "corrupt_generation: expert not resident");
  uint32_t g = 0;
  CK(cudaMemcpy(&g, ctx->d_gen + layer * S + slot, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  g += 0x10000u;
  CK(cudaMemcpy(ctx->d_gen + layer * S + slot, &g, sizeof(uint32_t), cudaMemcpyHostToDevice));
  return MOE_OK;
}

extern "C" moe_status_t moe_set_prefetch(moe_ctx_t* ctx, int32_t mode, float threshold) {
  if (!ctx) return MOE_ERR_ARG;
  if (mode != MOE_PREFETCH_OFF && mode != MOE_PREFETCH_REFRESH && mode != MOE_PREFETCH_PRESERVE)
    return fail(ctx, MOE_ERR_ARG, "set_prefetch: bad mode");
  if (!(threshold >= 0.f && threshold <= 1.f)) return fail(ctx, MOE_ERR_ARG, "set_prefetch: threshold outside [0, 1]");
  if (ctx->dev_admit && mode != MOE_PREFETCH_OFF)
    return fail(ctx, MOE_ERR_STATE, "set_prefetch: prefetch runs with host admission only");
  ctx->prefetch_mode = mode;
  ctx->prefetch_threshold = threshold;
  std::fill(ctx->pred.begin(), ctx->pred.end(), -1);
  return MOE_OK;
}

extern "C" moe_status_t moe_debug_prefill_wait_timeout(moe_ctx_t* ctx, int64_t wait_cycles, int32_t skip_ring) {
  if (!ctx) return MOE_ERR_ARG;
  if (skip_ring < -1 || wait_cycles < 0)
    return fail(ctx, MOE_ERR_ARG, "debug_prefill_wait_timeout: bad arguments");
  ctx->dbg_skip_ring = skip_ring;
  ctx->dbg_wait_cycles = skip_ring >= 0 ? wait_cycles : 0;
  return MOE_OK;
}

extern "C" moe_status_t moe_set_kernel_timing(moe_ctx_t* ctx, int32_t enable) {
  if (!ctx) return MOE_ERR_ARG;
  ctx->timing = enable != 0;
  return MOE_OK;
}

extern "C" moe_status_t moe_get_kernel_times(moe_ctx_t* ctx, double* ms, int64_t* launches) {
  if (!ctx) return MOE_ERR_ARG;
  CK(resolve_timing(ctx));
  for (int k = 0; k < MOE_KT_COUNT; ++k) {
    if (ms) ms[k] = ctx->kt_ms[k];
    if (launches) launches[k] = ctx->kt_n[k];
    ctx->kt_ms[k] = 0.0;
    ctx->kt_n[k] = 0;
  }
  return MOE_OK;
}
