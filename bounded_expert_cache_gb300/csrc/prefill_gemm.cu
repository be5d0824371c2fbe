// Prefill expert FFN: grouped dequant-GEMM on the 5th-generation tensor cores.
//
// "Paging the Experts" §3.1 (gate, up, down projections), "Nanite for
// Experts" §1 (eight routed + one shared expert per token), §5.3 (one
// schedule per unique expert, expert-major), §5.5 (merge into the original
// positions), §12 (keep the quantised operators; one expert-major operator
// over the resident experts).
//
// For a prefill chunk every unit (an expert of the union, or the shared
// expert) owns a contiguous block of expert-major rows: its tokens'
// activations (gathered once, fp16) and later its SwiGLU outputs h (bf16).
// The weights are the MMA's A operand (M side) and the tokens its B operand
// (N side), so a weight tile is dequantised once for up to 192 tokens:
//   gate/up: G = Wg[128 rows] x X^T and U = Wu[the same rows] x X^T, two
//            MMAs per K slice on one token tile -> SwiGLU in the epilogue
//            -> h[n tokens][128 columns]  (fp16 operands: x exact, d*q
//            rounded to fp16)
//   down:    D = Wd[128 rows] x h^T -> fp32 rows (bf16 operands: h and d*q
//            rounded to bf16; h may exceed the fp16 range); the combine
//            applies the routing weights
// The dequantised A tiles never touch shared memory: they are written to
// tensor memory with tcgen05.st and the MMA reads A from there, so shared
// memory holds only the TMA ring (token tile and raw Q8_0 rows).
// A persistent CTA of 14 warps walks the work items (unit, token tile,
// weight tile) of the launch:
//   warp 0      TMA, two copies per stage: the token tile (64 K, 128-byte
//               swizzle; one box for a whole tile, 32-row boxes for a
//               partial one) and the raw Q8_0 rows of the weight tile(s)
//               (64-byte swizzle), addressed in the slot pool through a 4-D
//               tensor map (bytes, rows, matrix, slot)
//   warp 1      allocates TMEM and issues tcgen05.mma (M 128, N <= 192,
//               K 16, A from TMEM, B from a shared-memory descriptor);
//               gate/up: one accumulator pair (G, U); down: two
//               accumulators so the epilogue overlaps the next item
//   warps 2..9  dequantise (block scales prefetched into registers) and
//               store to the A stage of their TMEM lane group
//   warps 10-13 epilogue (tcgen05.ld)
// Every wait is bounded; a wait that runs out sets an error bit and every
// role leaves its loop; in-flight copies and MMAs are drained before TMEM
// is released.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "prefill.h"
#include "tc.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kMaxStages = 8;
constexpr int kTok = kPrefillTok;  // tokens per item (MMA N at most)
constexpr int kWR = 128;           // weight rows per tile (MMA M)
constexpr int kBK = 64;            // K per stage
constexpr int kThreadsG = 448;
constexpr int kDqWarps = 8, kEpWarps = 4;
constexpr int kEpTid0 = 64 + 32 * kDqWarps;   // first epilogue thread
constexpr uint32_t kBBytes = kTok * kBK * 2;  // 24 KiB of tokens
constexpr uint32_t kAcc = 2 * kTok;           // TMEM columns of the accumulators
constexpr int kGeoCap = 96;                   // items per CTA kept in shared memory
constexpr int kSP = kWR + 8;                  // bf16 per transpose row (gate/up epilogue)
constexpr int kPF = 4;                        // stages of block scales prefetched
static_assert(kBBytes % 1024 == 0 && kTok % 32 == 0, "stage alignment");

// Per-phase shape: weight tiles per item (gate + up, or down), raw quant
// bytes per stage, A stages in TMEM (each tiles x 32 columns), accumulator
// buffers.
template <int PHASE> struct Shape {
  static constexpr int kTiles = PHASE == 0 ? 2 : 1;
  static constexpr uint32_t kQBytes = kTiles * kWR * kBK;
  static constexpr uint32_t kStageBytes = kBBytes + kQBytes;
  static constexpr int kAStages = PHASE == 0 ? 2 : 4;
  static constexpr uint32_t kAStride = 32u * kTiles;  // TMEM columns per A stage
  static constexpr int kAccBufs = PHASE == 0 ? 1 : 2;
  static constexpr uint32_t kEpiBytes = PHASE == 0 ? static_cast<uint32_t>(kTok) * kSP * 2 : 0u;
  static_assert(kAcc + kAStages * kAStride <= 512, "TMEM columns");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
};


__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ uint32_t hsub_hmul(uint32_t v, uint32_t magic, uint32_t d2) {
  uint32_t r;
  asm("{ .reg .b32 t; sub.rn.f16x2 t, %1, %2; mul.rn.f16x2 %0, t, %3; }" : "=r"(r) : "r"(v), "r"(magic), "r"(d2));
  return r;
}

// 16 Q8_0 codes times the block scale, rounded to fp16: the biased byte
// q+128 becomes the mantissa of 1024 (exact), 1152 is subtracted (exact)
// and the product with d is rounded once.
__device__ __forceinline__ void dq16_f16(uint4 raw, uint32_t d2, uint4& o0, uint4& o1) {
  const uint32_t w[4] = {raw.x ^ 0x80808080u, raw.y ^ 0x80808080u, raw.z ^ 0x80808080u, raw.w ^ 0x80808080u};
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r[2 * i] = hsub_hmul(__byte_perm(w[i], 0x64646464u, 0x4140), 0x64806480u, d2);
    r[2 * i + 1] = hsub_hmul(__byte_perm(w[i], 0x64646464u, 0x4342), 0x64806480u, d2);
  }
  o0 = make_uint4(r[0], r[1], r[2], r[3]);
  o1 = make_uint4(r[4], r[5], r[6], r[7]);
}

// The same 16 codes as bf16 of the exact fp32 product d*q (one rounding):
// the biased byte becomes the mantissa of 2^23 (exact), 2^23+128 is
// subtracted and the product formed in fp32, two lanes per instruction.
__device__ __forceinline__ void dq16_bf16(uint4 raw, float d, uint4& o0, uint4& o1) {
  const uint32_t w[4] = {raw.x ^ 0x80808080u, raw.y ^ 0x80808080u, raw.z ^ 0x80808080u, raw.w ^ 0x80808080u};
  unsigned long long dd, bias;
  asm("mov.b64 %0, {%1, %1};" : "=l"(dd) : "f"(d));
  asm("mov.b64 %0, {%1, %1};" : "=l"(bias) : "f"(8388736.0f));
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t lo = __byte_perm(w[i], 0x4B000000u, 0x7540u | (2 * h));
      const uint32_t hi = __byte_perm(w[i], 0x4B000000u, 0x7540u | (2 * h + 1));
      unsigned long long v;
      asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(lo), "r"(hi));
      asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(v) : "l"(v), "l"(bias));
      asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(v) : "l"(v), "l"(dd));
      float f0, f1;
      asm("mov.b64 {%0, %1}, %2;" : "=f"(f0), "=f"(f1) : "l"(v));
      __nv_bfloat162 p = __floats2bfloat162_rn(f0, f1);
      r[2 * i + h] = *reinterpret_cast<uint32_t*>(&p);
    }
  }
  o0 = make_uint4(r[0], r[1], r[2], r[3]);
  o1 = make_uint4(r[4], r[5], r[6], r[7]);
}

// silu(g) * u = g * u / (1 + e^-g); the reciprocal of an infinite
// denominator is 0, so very negative g gives 0.
__device__ __forceinline__ float silu_mul(float g, float u) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + __expf(-g)));
  return g * r * u;
}

// Geometry of one work item, derived identically by every role.
struct ItemGeo {
  int m0, n0, slot, p0, ntok, K, nrows, flags;  // flags: 1 shared, 2 stale
};

template <int PHASE>
__device__ __forceinline__ ItemGeo item_geo(const GemmArgs& a, int bid) {
  ItemGeo g;
  const int4 t = __ldg(reinterpret_cast<const int4*>(a.items) + bid);
  g.m0 = t.y;
  g.n0 = t.z;
  const int4 U = __ldg(reinterpret_cast<const int4*>(a.units + kUnitHeader) + t.x);
  const bool shared = U.x == -1;
  g.slot = U.x >= 0 ? U.x : (U.x <= -2 ? -2 - U.x : 0);
  g.p0 = shared ? a.rows_routed : U.y;
  g.ntok = min(kTok, U.z - g.m0);
  g.K = PHASE == 0 ? a.H : (shared ? a.Is : a.I);
  // weight rows of the tile inside the matrix (gate/up rows run to I or I_s)
  g.nrows = PHASE == 0 ? min(kWR, (shared ? a.Is : a.I) - g.n0) : kWR;
  // fail closed: a routed expert is used only if its slot holds the
  // generation its page-table entry expects
  const bool stale =
      !shared && (g.slot >= a.S || (U.x >= 0 && __ldg(a.gen + g.slot) != static_cast<uint32_t>(U.w)));
  g.flags = (shared ? 1 : 0) | (stale ? 2 : 0);
  return g;
}

// The CTA's items are decoded once into shared memory at launch (the i-th
// item of CTA b is b + i*gridDim.x); items past the table's capacity are
// decoded on the fly.
template <int PHASE>
__device__ __forceinline__ ItemGeo geo_of(const GemmArgs& a, const ItemGeo* table, int i) {
  if (i < kGeoCap) return table[i];
  return item_geo<PHASE>(a, blockIdx.x + i * gridDim.x);
}

// First item at or after i that is not stale (my_items if none).
template <int PHASE>
__device__ __forceinline__ int next_live(const GemmArgs& a, const ItemGeo* table, int i, int my_items) {
  while (i < my_items && (geo_of<PHASE>(a, table, i).flags & 2)) ++i;
  return i;
}

// Block-scale word (the two fp16 scales of one stage) of this thread's
// weight row: gate/up: tile t is the gate (0) or up (1) plane; down: the
// down plane. Rows past the matrix read as 0.
template <int PHASE>
__device__ __forceinline__ const uint32_t* scale_row(const GemmArgs& a, const ItemGeo& g, int t, int r) {
  if (r >= g.nrows) return nullptr;
  const uint8_t* wbase = (g.flags & 1) ? a.shared : a.pool + static_cast<int64_t>(g.slot) * a.slot_stride;
  const int64_t* soff = (g.flags & 1) ? a.s_soff : a.r_soff;
  const int64_t plane = PHASE == 0 ? soff[t] : soff[2];
  return reinterpret_cast<const uint32_t*>(wbase + plane + static_cast<int64_t>(g.n0 + r) * (g.K / 16));
}

template <int PHASE>  // 0: gate/up + SwiGLU, 1: down
__global__ void __launch_bounds__(kThreadsG, 1) gemm_kernel(const __grid_constant__ CUtensorMap map_b32,
                                                            const __grid_constant__ CUtensorMap map_bt,
                                                            const __grid_constant__ CUtensorMap map_q,
                                                            const __grid_constant__ CUtensorMap map_sq,
                                                            GemmArgs a) {
  using Sh = Shape<PHASE>;
  constexpr int kAStages = Sh::kAStages;
  extern __shared__ unsigned char smraw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  // smem ring: full (TMA bytes), sfree (the MMA's commit + the 8 dequant
  // warps); TMEM A ring: aready (8 dequant warps), afree (the MMA's
  // commit); accumulators: accf (commit), acce (4 epilogue warps)
  __shared__ uint64_t bar_full[kMaxStages], bar_sfree[kMaxStages];
  __shared__ uint64_t bar_aready[4], bar_afree[4];
  __shared__ uint64_t bar_accf[2], bar_acce[2], bar_drain;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_abort;
  __shared__ ItemGeo s_geo[kGeoCap];
  volatile int* abort_flag = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kStages = a.stages;
  const uint32_t sbase = su32(sm);
  const uint32_t sepi = sbase + static_cast<uint32_t>(kStages) * Sh::kStageBytes;
  const int n_items = __ldg(a.n_items);
  const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  for (int i = tid; i < my_items && i < kGeoCap; i += kThreadsG)
    s_geo[i] = item_geo<PHASE>(a, blockIdx.x + i * gridDim.x);
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(su32(&bar_full[s]), 1);
      mbar_init(su32(&bar_sfree[s]), 1 + kDqWarps);
    }
    for (int j = 0; j < kAStages; ++j) {
      mbar_init(su32(&bar_aready[j]), kDqWarps);
      mbar_init(su32(&bar_afree[j]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(su32(&bar_accf[b]), 1);
      mbar_init(su32(&bar_acce[b]), kEpWarps);
    }
    mbar_init(su32(&bar_drain), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_holder)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = tmem_holder;

  if (warp == 0) {
    // ---------------- producer (one thread): per stage the token tile and
    // the raw quant rows (gate/up: rows [n0, n0+128) of the gate and of the
    // up plane in one box; down: rows [n0, n0+128))
    if (lane == 0) {
      uint32_t ring = 0;
      RingPos rp;
      for (int i = 0; i < my_items && !*abort_flag; ++i) {
        const ItemGeo g = geo_of<PHASE>(a, s_geo, i);
        if (g.flags & 2) continue;
        const int nkb = g.K / kBK;
        const bool whole = g.ntok == kTok;
        const int nbox = (g.ntok + 31) / 32;
        const uint32_t bytes = (whole ? kBBytes : static_cast<uint32_t>(nbox) * 4096u) + Sh::kQBytes;
        const CUtensorMap* mq = (g.flags & 1) ? &map_sq : &map_q;
        const int zs = (g.flags & 1) ? 0 : g.slot;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++ring, rp.next(kStages)) {
          const int s = rp.s;
          if (ring >= static_cast<uint32_t>(kStages) &&
              !(ok = mbar_wait(su32(&bar_sfree[s]), rp.ph ^ 1u, abort_flag, a.err, a.wait_cycles)))
            break;
          if (static_cast<int>(ring) == a.skip_ring && blockIdx.x == 0) continue;  // test hook: nothing issued
          const uint32_t st = sbase + s * Sh::kStageBytes, fb = su32(&bar_full[s]);
          mbar_expect_tx(fb, bytes);
          if (whole)
            tma2d(st, &map_bt, fb, kb * kBK, g.p0 + g.m0);
          else
            for (int bx = 0; bx < nbox; ++bx) tma2d(st + bx * 4096u, &map_b32, fb, kb * kBK, g.p0 + g.m0 + bx * 32);
          tma4d(st + kBBytes, mq, fb, kb * kBK, g.n0, 0, zs);
        }
        if (!ok) break;
      }
      // drain: the last copies into each stage complete before exit
      const uint32_t n = ring < static_cast<uint32_t>(kStages) ? ring : static_cast<uint32_t>(kStages);
      for (uint32_t j = 0; j < n; ++j) {
        const uint32_t r = ring - 1 - j;
        if (static_cast<int>(r) == a.skip_ring && blockIdx.x == 0) continue;  // no copy in flight
        mbar_drain(su32(&bar_full[r % kStages]), (r / kStages) & 1u, a.err, a.wait_cycles);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer. It waits only on aready: the dequantising
    // warps arrive there after they observed the stage's full barrier, so the
    // token tile of the stage has landed as well.
    if (lane == 0) {
      uint32_t ring = 0, acc_i = 0;
      int s = 0, j = 0;
      uint32_t aph = 0;
      const uint32_t fmt = PHASE == 0 ? 0u : 1u;  // f16 : bf16
      const uint64_t bd0 = sdesc(sbase);          // B descriptor of stage 0; + 16-byte units
      for (int i = 0; i < my_items && !*abort_flag; ++i) {
        const ItemGeo g = geo_of<PHASE>(a, s_geo, i);
        if (g.flags & 2) continue;
        const int nkb = g.K / kBK;
        const uint32_t n = static_cast<uint32_t>((g.ntok + 15) & ~15);
        const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((n >> 3) << 17) | ((kWR >> 4) << 24);
        const uint32_t buf = Sh::kAccBufs == 2 ? (acc_i & 1u) : 0u;
        const uint32_t cph = Sh::kAccBufs == 2 ? ((acc_i >> 1) & 1u) : (acc_i & 1u);
        if (acc_i >= static_cast<uint32_t>(Sh::kAccBufs) &&
            !mbar_wait(su32(&bar_acce[buf]), cph ^ 1u, abort_flag, a.err, a.wait_cycles))
          break;
        asm volatile("tcgen05.fence::after_thread_sync;");
        const uint32_t dt = tmem + buf * static_cast<uint32_t>(kTok);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!(ok = mbar_wait(su32(&bar_aready[j]), aph, abort_flag, a.err, a.wait_cycles))) break;
          asm volatile("tcgen05.fence::after_thread_sync;");
          const uint64_t bd = bd0 + static_cast<uint64_t>((static_cast<uint32_t>(s) * Sh::kStageBytes) >> 4);
          const uint32_t at = tmem + kAcc + Sh::kAStride * static_cast<uint32_t>(j);
          const uint32_t acc0 = kb > 0 ? 1u : 0u;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            umma_ts(dt, at + 8 * k, bd + 2 * k, idesc, k > 0 ? 1u : acc0);
            if (PHASE == 0) umma_ts(dt + kTok, at + 32 + 8 * k, bd + 2 * k, idesc, k > 0 ? 1u : acc0);  // up rows into U
          }
          umma_commit(su32(&bar_sfree[s]));
          umma_commit(su32(&bar_afree[j]));
          ++ring;
          if (++s == kStages) s = 0;
          if (++j == kAStages) {
            j = 0;
            aph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(su32(&bar_accf[buf]));
        ++acc_i;
      }
      // drain: every MMA issued here has completed before TMEM is released
      umma_commit(su32(&bar_drain));
      mbar_drain(su32(&bar_drain), 0, a.err, a.wait_cycles);
      (void)ring;
    }
  } else if (warp < 2 + kDqWarps) {
    // ---------------- dequantisation: warp w owns TMEM lanes 32*(w%4) ..
    // +31; gate/up: warps 2..5 the gate tile, 6..9 the up tile, both blocks
    // of a stage; down: one tile, warps 2..5 the first block, 6..9 the
    // second. Block scales run kPF stages ahead in registers, across items.
    const int sp = warp & 3, sub = (warp - 2) >> 2;
    const int r = sp * 32 + lane;  // weight row within a tile
    const uint32_t lane_base = static_cast<uint32_t>(sp * 32) << 16;
    const uint32_t swz = static_cast<uint32_t>((r >> 1) & 3);  // 64-byte swizzle phase of row r
    const uint32_t qrow = kBBytes + static_cast<uint32_t>((PHASE == 0 ? sub * kWR : 0) + r) * kBK;
    // prefetch cursor (item pi, stage pk)
    int pi = next_live<PHASE>(a, s_geo, 0, my_items), pk = 0, pnkb = 1;
    const uint32_t* prow = nullptr;
    if (pi < my_items) {
      const ItemGeo g = geo_of<PHASE>(a, s_geo, pi);
      pnkb = g.K / kBK;
      prow = scale_row<PHASE>(a, g, sub, r);
    }
    uint32_t sc[kPF];
#pragma unroll
    for (int u = 0; u < kPF; ++u) {
      sc[u] = (pi < my_items && prow) ? __ldg(prow + pk) : 0u;
      if (pi < my_items && ++pk == pnkb) {
        pi = next_live<PHASE>(a, s_geo, pi + 1, my_items);
        pk = 0;
        if (pi < my_items) {
          const ItemGeo g = geo_of<PHASE>(a, s_geo, pi);
          pnkb = g.K / kBK;
          prow = scale_row<PHASE>(a, g, sub, r);
        }
      }
    }
    // consumer cursor (item ci, stage kb)
    int ci = next_live<PHASE>(a, s_geo, 0, my_items), kb = 0, nkb = 1;
    if (ci < my_items) nkb = geo_of<PHASE>(a, s_geo, ci).K / kBK;
    RingPos rp, ap;
    uint32_t ring = 0;
    bool ok = true;
    while (ci < my_items && ok && !*abort_flag) {
#pragma unroll
      for (int u = 0; u < kPF; ++u) {
        if (ci >= my_items) break;
        const uint32_t scw = sc[u];
        sc[u] = (pi < my_items && prow) ? __ldg(prow + pk) : 0u;
        if (pi < my_items && ++pk == pnkb) {
          pi = next_live<PHASE>(a, s_geo, pi + 1, my_items);
          pk = 0;
          if (pi < my_items) {
            const ItemGeo g = geo_of<PHASE>(a, s_geo, pi);
            pnkb = g.K / kBK;
            prow = scale_row<PHASE>(a, g, sub, r);
          }
        }
        const int s = rp.s, j = ap.s;
        if (!(ok = mbar_wait(su32(&bar_full[s]), rp.ph, abort_flag, a.err, a.wait_cycles))) break;
        const uint32_t sq = sbase + s * Sh::kStageBytes + qrow;
        uint32_t out[32];
        if (PHASE == 0) {
          // both blocks of the stage: chunks 0,1 (scale lo) and 2,3 (scale hi)
          const uint32_t lo = scw & 0xFFFFu, hi = scw >> 16;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 raw = lds128(sq + ((static_cast<uint32_t>(c) ^ swz) << 4));
            const uint32_t h = c < 2 ? lo : hi;
            uint4 o0, o1;
            dq16_f16(raw, h | (h << 16), o0, o1);
            out[8 * c] = o0.x, out[8 * c + 1] = o0.y, out[8 * c + 2] = o0.z, out[8 * c + 3] = o0.w;
            out[8 * c + 4] = o1.x, out[8 * c + 5] = o1.y, out[8 * c + 6] = o1.z, out[8 * c + 7] = o1.w;
          }
        } else {
          const uint32_t h = sub ? (scw >> 16) : (scw & 0xFFFFu);
          const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint4 raw = lds128(sq + ((static_cast<uint32_t>(2 * sub + c) ^ swz) << 4));
            uint4 o0, o1;
            dq16_bf16(raw, d, o0, o1);
            out[8 * c] = o0.x, out[8 * c + 1] = o0.y, out[8 * c + 2] = o0.z, out[8 * c + 3] = o0.w;
            out[8 * c + 4] = o1.x, out[8 * c + 5] = o1.y, out[8 * c + 6] = o1.z, out[8 * c + 7] = o1.w;
          }
        }
        // the stage's quant rows have been read
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&bar_sfree[s]));
        if (ring >= static_cast<uint32_t>(kAStages) &&
            !(ok = mbar_wait(su32(&bar_afree[j]), ap.ph ^ 1u, abort_flag, a.err, a.wait_cycles)))
          break;
        asm volatile("tcgen05.fence::after_thread_sync;");
        const uint32_t ta = tmem + lane_base + kAcc + Sh::kAStride * j;
        if (PHASE == 0) {
          tmem_st16(ta + 32u * sub, out);
          tmem_st16(ta + 32u * sub + 16u, out + 16);
        } else {
          tmem_st16(ta + 16u * sub, out);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;");
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&bar_aready[j]));
        ++ring;
        rp.next(kStages);
        ap.next(kAStages);
        if (++kb == nkb) {
          ci = next_live<PHASE>(a, s_geo, ci + 1, my_items);
          kb = 0;
          if (ci < my_items) nkb = geo_of<PHASE>(a, s_geo, ci).K / kBK;
        }
      }
    }
  } else {
    // ---------------- epilogue: warp w reads TMEM lanes 32*(w%4) .. +31
    const int sp = warp & 3;
    const int r = sp * 32 + lane;  // weight row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(sp * 32) << 16;
    // The four epilogue warps meet at named barriers inside an item, so they
    // decide together whether to take it: by its accumulator barrier alone
    // (a completed phase is seen by all of them), never by the abort flag,
    // which one warp could read before and another after it was raised.
    uint32_t acc_i = 0;
    for (int i = 0; i < my_items; ++i) {
      const ItemGeo g = geo_of<PHASE>(a, s_geo, i);
      if (g.flags & 2) {
        if (tid == kEpTid0) atomicOr(a.err, MOE_DEVERR_STALE);
        continue;
      }
      const uint32_t buf = Sh::kAccBufs == 2 ? (acc_i & 1u) : 0u;
      const uint32_t aph = Sh::kAccBufs == 2 ? ((acc_i >> 1) & 1u) : (acc_i & 1u);
      if (!mbar_wait(su32(&bar_accf[buf]), aph, abort_flag, a.err, a.wait_cycles)) break;
      asm volatile("tcgen05.fence::after_thread_sync;");
      const int nch = (g.ntok + 31) / 32;
      const uint32_t tb = tmem + lane_base + buf * static_cast<uint32_t>(kTok);
      const int64_t prow0 = static_cast<int64_t>(g.p0) + g.m0;
      if (PHASE == 0) {
        // lane r holds G and U of weight row n0 + r: h column n0 + r. The
        // whole tile's h goes to a transpose buffer first, so that the one
        // accumulator pair is released to the next item's MMAs before the
        // rows of h are written, 16 bytes at a time
        const int et = tid - kEpTid0;  // 0..127
        for (int ch = 0; ch < nch; ++ch) {
          uint32_t gv[32], uv[32];
          tmem_ld32(tb + ch * 32, gv);
          tmem_ld32(tb + kTok + ch * 32, uv);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const __nv_bfloat16 hb = __float2bfloat16_rn(silu_mul(__uint_as_float(gv[j]), __uint_as_float(uv[j])));
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(sepi + ((ch * 32 + j) * kSP + r) * 2),
                         "h"(*reinterpret_cast<const unsigned short*>(&hb))
                         : "memory");
          }
        }
        asm volatile("tcgen05.fence::before_thread_sync;");
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&bar_acce[buf]));  // the accumulators have been read
        epi_sync();
        // tokens x 128 columns of bf16, 16 bytes a piece
        for (int ch = 0; ch < nch; ++ch) {
#pragma unroll
          for (int rep = 0; rep < 4; ++rep) {
            const int piece = et + 128 * rep, j = piece >> 4, part = piece & 15;
            const int tok = ch * 32 + j;
            if (tok < g.ntok && part * 8 < g.nrows) {
              const uint4 w = lds128(sepi + ((ch * 32 + j) * kSP + part * 8) * 2);
              *reinterpret_cast<uint4*>(a.h + (prow0 + tok) * a.ldh + g.n0 + part * 8) = w;
            }
          }
        }
        epi_sync();
      } else {
        for (int ch = 0; ch < nch; ++ch) {
          uint32_t v[32];
          tmem_ld32(tb + ch * 32, v);
          float* dst = a.yp + (prow0 + ch * 32) * a.H + g.n0 + r;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (ch * 32 + j < g.ntok) dst[static_cast<int64_t>(j) * a.H] = __uint_as_float(v[j]);
        }
      }
      if (PHASE != 0) {
        asm volatile("tcgen05.fence::before_thread_sync;");
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&bar_acce[buf]));
      }
      ++acc_i;
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
}

template <int PHASE>
size_t smem_bytes(int stages) {
  return static_cast<size_t>(stages) * Shape<PHASE>::kStageBytes + Shape<PHASE>::kEpiBytes + 1024;
}

}  // namespace

// Pipeline stages that fit in shared memory beside the epilogue buffer.
int gemm_stages(int phase) {
  const size_t limit = 227 * 1024 - sizeof(ItemGeo) * kGeoCap - 512;  // static shared memory
  const size_t fixed = phase == 0 ? smem_bytes<0>(0) : smem_bytes<1>(0);
  const size_t per = phase == 0 ? Shape<0>::kStageBytes : Shape<1>::kStageBytes;
  const int n = static_cast<int>((limit - fixed) / per);
  return n < 2 ? 0 : (n > kMaxStages ? kMaxStages : n);
}

size_t gemm_smem_bytes(int phase, int stages) { return phase == 0 ? smem_bytes<0>(stages) : smem_bytes<1>(stages); }

cudaError_t launch_gemm(int phase, const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t st) {
  const int smem = static_cast<int>(gemm_smem_bytes(phase, a.stages));
  cudaError_t e;
  if (phase == 0) {
    e = cudaFuncSetAttribute(gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gemm_kernel<0><<<grid, kThreadsG, smem, st>>>(m.b32, m.btile, m.q, m.sq, a);
  } else {
    e = cudaFuncSetAttribute(gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gemm_kernel<1><<<grid, kThreadsG, smem, st>>>(m.b32, m.btile, m.q, m.sq, a);
  }
  return cudaGetLastError();
}

}  // namespace moe
