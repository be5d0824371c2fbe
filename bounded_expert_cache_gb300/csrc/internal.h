// Library-internal declarations shared by the host (.cpp) and device (.cu)
// translation units of libmoecache. Not part of the public ABI.
#pragma once

#include <algorithm>
#include <cstdint>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/moecache.h"

// Device error bits, OR-ed into the context's error word by kernels.
enum : uint32_t {
  MOE_DEVERR_STALE = 1u,       // unit whose slot is absent or of another generation
  MOE_DEVERR_TIMEOUT = 2u,     // a bounded wait ran out
  MOE_DEVERR_NONFINITE = 4u,   // router input or weight not finite
  MOE_DEVERR_BADIDX = 8u,      // expert id out of range in a plan input
  MOE_DEVERR_CAPACITY = 16u,   // on-device admission: union larger than the slots allow
};

namespace moe {

moe_slots* slots_new(int32_t E, int32_t S, int32_t policy, uint64_t seed, int32_t layer,
                     int64_t payload);
moe_status_t slots_step(moe_slots* s, const int32_t* uniq, int32_t n_uniq, const int32_t* counts,
                        moe_miss_list_t* out, std::string* err);
moe_status_t slots_preload(moe_slots* s, const int32_t* experts, int32_t n,
                           std::vector<int32_t>* filled, std::vector<int32_t>* filled_slots,
                           std::string* err);
moe_status_t slots_evict(moe_slots* s, int32_t e, std::string* err);
moe_status_t slots_prefetch(moe_slots* s, int32_t e, int32_t mode, int32_t* action, moe_miss_list_t* fill,
                            std::string* err);
const int32_t* slots_pt(const moe_slots* s);
const int32_t* slots_owner(const moe_slots* s);
const uint64_t* slots_last(const moe_slots* s);
uint64_t slots_tick(const moe_slots* s);
uint64_t slots_rng(const moe_slots* s);
const uint32_t* slots_gen(const moe_slots* s);
moe_stats_t slots_stats(const moe_slots* s);

// Geometry of one expert payload in the split-plane layout.
struct ExpertGeom {
  int32_t H = 0, I = 0, quant = 0;
  int64_t qbytes[3] = {0, 0, 0};  // quant-plane bytes of gate, up, down
  int64_t sbytes[3] = {0, 0, 0};  // scale-plane bytes
  int64_t qoff[3] = {0, 0, 0};    // quant-plane offsets within the payload
  int64_t soff[3] = {0, 0, 0};    // scale-plane offsets
  int64_t bytes = 0;              // payload bytes
};
ExpertGeom expert_geom(int32_t H, int32_t I, int32_t quant);

// Per-layer cache state kept on the device when admission runs on the GPU.
struct DevCacheLayer {
  int32_t* pt;                 // [E] expert -> slot or -1
  uint32_t* ptgen;             // [E] generation the entry expects
  int32_t* owner;              // [S] slot -> expert or -1
  uint32_t* sgen;              // [S] fill count of the slot (the manager's generation)
  unsigned long long* last;    // [S] tick of the slot's last access
  unsigned long long* tick;    // [1]
  unsigned long long* rng;     // [1] SplitMix64 state
  long long* stats;            // [8] see kStat*
};
enum { kStatSteps = 0, kStatHits, kStatMisses, kStatEvictions, kStatMaterialized, kStatTiles,
       kStatBytes, kStatCount = 8 };

// Unit table read by the FFN kernels: int32 [kUnitHeader + 4 * max_units]:
// count (then padding to 16 bytes), then per unit {slot, p0 (first
// expert-major assignment, -1: shared), M (tokens), generation the slot must
// hold}. slot -1 is the shared expert; slot <= -2 marks a miss that the FFN
// materialises while reading it (slot -2 - s, and the 4th field holds the
// expert id instead of a generation). Routed units come first, in union order.
constexpr int kUnitHeader = 4;
constexpr int kUnitInts = 4;

// On-device admission, run by the router's last block after the plan.
struct AdmitArgs {
  int enabled;
  int read_through;  // misses are materialised by the FFN while it reads them
  int E, S, policy, has_shared, T;
  long long payload;
  DevCacheLayer c;
  int32_t* fills;      // [1 + 2 * max_fills]: n, then (expert, slot) pairs
  int32_t* units;      // unit table
  unsigned int* done;  // [max_fills] tiles copied per fill
  int max_fills;
};

// Arguments of the router launch.
struct RouteArgs {
  const void* x;
  int32_t xt, T, H, E, k;
  const float* w;
  const float* bias;
  int32_t* topk_idx;
  float* topk_w;
  unsigned long long* keys;  // [3][T][E] scratch: logit, lower, upper keys
  unsigned int* ticket; // last-block counter, zero between launches
  unsigned long long* repairs;  // counters of the layer: [0] repaired tokens, [1] filter fallbacks
  uint32_t* err;
  // optional fused plan (plan.counts == nullptr: none)
  moe_plan_t plan;
  // optional fused admission (requires the fused plan)
  AdmitArgs admit;
};
cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t st);

struct PlanArgs {
  const int32_t* idx;
  const float* w;
  int32_t T, k, E;
  moe_plan_t plan;
  uint32_t* err;
};
cudaError_t launch_plan(const PlanArgs& a, cudaStream_t st);
// Many-token routing (any T): norms [T + E] and flags [T] are scratch; part
// holds up to 4 * T * E (hi, lo) pairs of split-K partials (or T * E
// approximate logits). wsplit (router_split_bytes(E, H), or nullptr): the
// router weights' bf16 parts, which enable the tensor-core filter for bf16
// activations with H % 64 == 0.
size_t router_split_bytes(int E, int H);
cudaError_t launch_route_large(const RouteArgs& a, float* norms, int* flags, float2* part, uint16_t* wsplit,
                               int num_sms, cudaStream_t st);
// Multi-block plan for any T*k: local is scratch [plan_blocks(T*k)][E].
int plan_blocks(int A);
cudaError_t launch_plan_large(const PlanArgs& a, int* local, cudaStream_t st);
// On-device admission of one step as its own launch (one warp).
cudaError_t launch_admit(const AdmitArgs& A, const moe_plan_t& P, int max_units, uint32_t* err,
                         cudaStream_t st);

// Message returned by moe_last_error(NULL) on this thread.
void set_thread_error(const std::string& msg);

// Device-driven staging of the fills listed by on-device admission: copy
// each filled expert's tiles from the pinned store (read over the host link)
// into its slot, then publish the slot's generation.
struct StageArgs {
  const uint8_t* store;      // pinned host store of the layer: [E][payload]
  uint8_t* pool;             // slot pool of the layer
  int64_t slot_stride, payload;
  const int32_t* fills;      // from admission
  unsigned int* done;        // [max_fills]
  const uint32_t* sgen;      // [S] manager generations
  uint32_t* gen;             // [S] published generations
  long long* stats;          // [kStatCount]
  int64_t mat_off[3], mat_bytes[3];
  int64_t tile_bytes;
  int tiles_per_expert;      // 256 KiB tiles of one expert (accounting unit)
  int chunks[3];             // copy chunks per matrix
  int chunks_per_expert;
  int max_fills;
  int grid;                  // persistent CTAs (a few per SM)
};
constexpr int64_t kStageChunkBytes = 32768;  // one CTA's copy: 256 threads x 8 x 16 B
cudaError_t launch_stage_copy(const StageArgs& a, cudaStream_t st);
cudaError_t launch_set_word(uint32_t* dst, uint32_t v, cudaStream_t st);
// One load per kTouchPage bytes of a bound store (its device mapping), at bind time.
constexpr size_t kTouchPage = 4096;
cudaError_t launch_touch_pages(const uint8_t* dev_store, size_t bytes, int sms, uint32_t* sink, cudaStream_t st);

// Arguments of the decode FFN launches.
struct FfnArgs {
  const void* x;
  int32_t xt, T, H, I, Is, k, E, quant;
  uint8_t* pool;              // slot pool of the layer (written by read-through misses)
  int64_t slot_stride;
  const int32_t* units;       // unit table of this step
  uint32_t* gen;              // [S] published slot generations
  int32_t S;
  // read-through materialisation of misses (store == nullptr: off)
  const uint8_t* store;       // device alias of the layer's pinned store [E][payload]
  int64_t payload;
  const uint32_t* sgen;       // [S] manager generations, published at the end
  unsigned int* ticket;       // last-block counter of the down kernel
  long long* stats;           // [kStatCount] of the layer
  int tiles_per_expert;
  const uint8_t* shared;      // shared payload or nullptr
  ExpertGeom g, gs;           // routed and shared geometry
  moe_plan_t plan;
  float* h;                   // scratch [(T*k + T)][ldh]
  int32_t ldh;
  float* y;                   // [T][H]
  uint32_t* err;
  cudaEvent_t ev[4];          // optional timing events around gate/up and down
};
cudaError_t launch_ffn_decode(const FfnArgs& a, int num_sms, cudaStream_t st);

// The fused decode FFN (one persistent cooperative launch): its counters
// (zero between launches; the kernel clears them) and launch shape.
struct FusedLaunch {
  unsigned int* sync;   // [3 + max_units * max_tiles]
  int max_units;        // unit-table capacity
  int max_tiles;        // tiles of one down plane
  int64_t tile_bytes;   // staging tile
  long long wait_cycles;
  int grid;             // CTAs (one per SM)
  bool pdl;             // with programmatic stream serialisation
};
cudaError_t launch_ffn_decode_fused(const FfnArgs& a, const FusedLaunch& fl, cudaStream_t st);
constexpr long long kFusedWaitCycles = 4000000000ll;  // about 2 s at the SM clock

}  // namespace moe

struct moe_ctx {
  moe_config_t cfg{};
  int device = 0;
  int num_sms = 0;
  moe::ExpertGeom geom, sgeom;
  int64_t slot_stride = 0;
  uint8_t* d_pool = nullptr;     // [L][S][slot_stride] (+ tail)
  int32_t* d_pt = nullptr;       // [L][E]
  uint32_t* d_ptgen = nullptr;   // [L][E]
  uint32_t* d_gen = nullptr;     // [L][S]
  int32_t* h_pt = nullptr;       // pinned mirrors
  uint32_t* h_ptgen = nullptr;
  uint32_t* h_gen = nullptr;
  std::vector<moe_slots*> slots;
  const uint8_t* store = nullptr;
  const uint8_t* store_dev = nullptr;  // device alias of the pinned store
  size_t store_bytes = 0;
  std::vector<const uint8_t*> shared;
  // scratch
  unsigned long long* d_keys = nullptr;
  unsigned int* d_ticket = nullptr;
  unsigned long long* d_repairs = nullptr;  // [L][2]: repaired tokens, filter fallbacks
  float* d_h = nullptr;
  int32_t ldh = 0;
  uint32_t* d_err = nullptr;
  uint32_t* h_err = nullptr;
  int32_t* h_union = nullptr;  // pinned: uniq [E], counts [E], n_uniq
  int32_t* d_units = nullptr;  // unit table (device)
  int32_t* h_units = nullptr;  // pinned staging of the unit table (host admission)
  int32_t max_units = 0;
  // on-device admission
  bool dev_admit = false;
  bool dev_state_used = false;
  int32_t* d_owner = nullptr;             // [L][S]
  uint32_t* d_sgen = nullptr;             // [L][S]
  unsigned long long* d_last = nullptr;   // [L][S]
  unsigned long long* d_tick = nullptr;   // [L]
  unsigned long long* d_rng = nullptr;    // [L]
  long long* d_stats = nullptr;           // [L][kStatCount]
  int32_t* d_fills = nullptr;             // [1 + 2 * max_fills]
  unsigned int* d_done = nullptr;         // [max_fills]
  int32_t max_fills = 0;
  bool read_through = false;              // misses materialised by the FFN
  unsigned int* d_ffn_ticket = nullptr;
  unsigned int* d_fsync = nullptr;        // counters of the fused decode FFN
  int fused_units = 0, fused_tiles = 0;
  // prefill path (max_tokens > 8)
  bool prefill = false;
  uint16_t* d_x16 = nullptr;               // fp16 [rows][H]
  uint16_t* d_hp = nullptr;                // bf16 [rows][ldh_p]
  float* d_yp = nullptr;                   // fp32 [rows][H]
  int32_t* d_items0 = nullptr;
  int32_t* d_items1 = nullptr;
  int32_t* d_nitems = nullptr;             // [2]
  int max_items0 = 0, max_items1 = 0, ldh_p = 0;
  int32_t* d_plan_local = nullptr;         // multi-block plan scratch
  float* d_norms = nullptr;                // many-token router scratch
  uint16_t* d_wsplit = nullptr;            // bf16 parts of the router weights (H % 64 == 0)
  int32_t* d_flags = nullptr;
  float2* d_lpart = nullptr;               // split-K logit partials [4][T][E]
  std::vector<cudaStream_t> streams;
  std::vector<cudaEvent_t> ev_stage, ev_stage_b;  // copies of a wave's two parts
  cudaEvent_t ev_compute = nullptr;
  size_t unit_ints = 0;  // capacity of the unit-table buffer
  int32_t prefetch_mode = 0;      // moe_prefetch_mode_t (host admission only)
  float prefetch_threshold = 0.2f;
  std::vector<int32_t> pred;      // [L] expert to prefetch before the layer's next step, or -1
  std::vector<cudaEvent_t> ev_prefetch;  // the prefetch copy, one per staging stream
  long long dbg_wait_cycles = 0;  // test hook of the next prefill gate/up GEMM
  int32_t dbg_skip_ring = -1;
  int32_t fail_after_tiles = -1;
  // kernel timing
  struct TimedLaunch {
    int kind;
    cudaEvent_t a, b;
  };
  bool timing = false;
  std::vector<TimedLaunch> timed;
  std::vector<cudaEvent_t> ev_pool;
  double kt_ms[MOE_KT_COUNT] = {};
  int64_t kt_n[MOE_KT_COUNT] = {};
  std::vector<int64_t> tiles_staged, bytes_staged;
  std::string err;
};
