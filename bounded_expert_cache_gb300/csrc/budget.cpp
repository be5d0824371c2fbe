// Static budget check before serving.
//
// "MawForge" §IV-D: the static lower bound L(p, n) = C + E(p) + K(n) of the
// runtime footprint F(p, n) = L(p, n) + O (resident common tensors, expert
// cache at cache percentage p, KV cache at context n, runtime overhead);
// rows whose lower bound already exceeds the serving target are rejected.
// The expert-cache budget is p of every layer's expert bytes: the §V-C
// static minima of one model at 50% and 65% cache differ by exactly 15% of
// its total expert bytes.
#include "internal.h"

namespace {

constexpr int64_t kPpm = 1000000;

// a * b, or false if it leaves int64 (a, b >= 0)
bool mul_ok(int64_t a, int64_t b, int64_t* r) {
  return !__builtin_mul_overflow(a, b, r);
}
bool add_ok(int64_t a, int64_t b, int64_t* r) {
  return !__builtin_add_overflow(a, b, r);
}

}  // namespace

extern "C" moe_status_t moe_static_budget(int32_t n_layers, int32_t n_experts, int64_t payload_bytes,
                                          int64_t cache_ppm, int64_t common_bytes, int64_t kv_bytes_per_token,
                                          int64_t context, int64_t overhead_bytes, int64_t target_bytes,
                                          moe_budget_t* out) {
  if (!out || n_layers < 0 || n_experts < 0 || payload_bytes < 0 || cache_ppm < 0 || cache_ppm > kPpm ||
      common_bytes < 0 || kv_bytes_per_token < 0 || context < 0 || overhead_bytes < 0 || target_bytes < 0)
    return MOE_ERR_ARG;
  // E(p) = floor(layers * experts * payload * ppm / 10^6), exact in 128 bits
  int64_t total = 0;
  if (!mul_ok(static_cast<int64_t>(n_layers) * n_experts, payload_bytes, &total)) return MOE_ERR_ARG;
  const unsigned __int128 e = static_cast<unsigned __int128>(total) * static_cast<uint64_t>(cache_ppm) / kPpm;
  int64_t kv = 0, lower = 0, foot = 0;
  if (!mul_ok(kv_bytes_per_token, context, &kv)) return MOE_ERR_ARG;
  if (!add_ok(common_bytes, static_cast<int64_t>(e), &lower) || !add_ok(lower, kv, &lower) ||
      !add_ok(lower, overhead_bytes, &foot))
    return MOE_ERR_ARG;
  out->common_bytes = common_bytes;
  out->expert_bytes = static_cast<int64_t>(e);
  out->kv_bytes = kv;
  out->overhead_bytes = overhead_bytes;
  out->lower_bound = lower;
  out->footprint = foot;
  out->slots_per_layer = static_cast<int32_t>(static_cast<int64_t>(n_experts) * cache_ppm / kPpm);
  out->accepted = lower <= target_bytes ? 1 : 0;
  return MOE_OK;
}
