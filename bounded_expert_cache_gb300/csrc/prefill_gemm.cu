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
//   gate/up: D[128 x n] = [64 gate rows | the same 64 up rows] x X^T
//            -> SwiGLU -> h[n tokens][64 columns]   (fp16 operands: x exact,
//            d*q rounded to fp16)
//   down:    D[128 x n] = [128 down rows] x h^T -> fp32 rows (bf16
//            operands: h and d*q rounded to bf16; h may exceed the fp16
//            range); the combine applies the routing weights
// The dequantised A tile never touches shared memory: it is written to
// tensor memory with tcgen05.st and the MMA reads A from there, so shared
// memory holds only the TMA ring (token tile, raw Q8_0 rows, block scales).
// A persistent CTA of 14 warps walks the work items (unit, token tile,
// weight tile) of the launch:
//   warp 0      TMA, two copies per stage: the token tile (64 K, 128-byte
//               swizzle; one box for a whole tile, 32-row boxes for a
//               partial one) and the raw Q8_0 rows of the weight tile
//               (64-byte swizzle) addressed in the slot pool through a 4-D
//               tensor map (bytes, rows, matrix, slot); once per item, a
//               bulk copy of the tile's block scales into a double buffer
//   warp 1      allocates TMEM (two 128-lane x 192-column fp32
//               accumulators and four 32-column A stages) and issues
//               tcgen05.mma (M 128, N <= 192, K 16, A from TMEM, B from a
//               shared-memory descriptor)
//   warps 2..9  dequantise one Q8_0 block (32 weights) of one row per stage
//               each and store it to the A stage of their TMEM lane group
//   warps 10-13 epilogue of one accumulator (tcgen05.ld) while the MMAs of
//               the next item fill the other
// Every wait is bounded; a wait that runs out sets an error bit and every
// role leaves its loop; in-flight copies and MMAs are drained before TMEM
// is released.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "prefill.h"

namespace moe {
namespace {

constexpr int kMaxStages = 8;
constexpr int kTok = kPrefillTok;  // tokens per item (MMA N at most)
constexpr int kWR = 128;           // weight rows per item (MMA M)
constexpr int kBK = 64;            // K per stage
constexpr int kAStages = 4;        // A stages in TMEM (32 columns each)
constexpr uint32_t kAcol0 = 2 * kTok;  // first A column (after two accumulators)
constexpr int kThreadsG = 448;
constexpr int kDqWarps = 8, kEpWarps = 4;
constexpr int kEpTid0 = 64 + 32 * kDqWarps;   // first epilogue thread
constexpr uint32_t kBBytes = kTok * kBK * 2;  // 24 KiB of tokens
constexpr uint32_t kQBytes = kWR * kBK;       // 8 KiB raw int8
constexpr uint32_t kStageBytes = kBBytes + kQBytes;
constexpr uint32_t kEpiBytes = 16384;   // epilogue exchange + transpose
constexpr int kGeoCap = 96;             // items per CTA kept in shared memory
constexpr int kXP = 20;                 // floats per exchange row
constexpr int kSP = 72;                 // bf16 per transpose row
static_assert(kAcol0 + kAStages * 32 <= 512, "TMEM columns");
static_assert(kBBytes % 1024 == 0 && kTok % 32 == 0, "stage alignment");
constexpr long long kWaitCycles = 4000000000ll;  // about 2 s at the SM clock

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t b, uint32_t c) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(c));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(b), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a phase of an mbarrier. False if it ran out (about 2 s;
// this raises the CTA's abort flag) or if another role has aborted. The
// clock and the flag are read once per 16 probes.
__device__ __forceinline__ bool mbar_wait(uint32_t b, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* err) {
  if (mbar_try(b, parity)) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try(b, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      atomicOr(err, MOE_DEVERR_TIMEOUT);
      return false;
    }
  }
}
// Position in a ring of n stages: stage index and the parity of its phase.
struct RingPos {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};
// Bounded wait that ignores the abort flag (draining before exit).
__device__ __forceinline__ void mbar_drain(uint32_t b, uint32_t parity, uint32_t* err) {
  const long long t0 = clock64();
  while (!mbar_try(b, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(err, MOE_DEVERR_TIMEOUT);
      return;
    }
  }
}
__device__ __forceinline__ void tma2d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          dst),
      "l"(m), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          dst),
      "l"(m), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma4d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y, int z,
                                      int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(
          dst),
      "l"(m), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// D (TMEM) += A (TMEM) * B (shared-memory descriptor)
__device__ __forceinline__ void umma_ts(uint32_t dt, uint32_t at, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(dt),
      "r"(at), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tmem_st16(uint32_t ta, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          ta),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t ta, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(ta));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
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
  int m0, n0, slot, p0, ntok, K, shared, stale;
};

template <int PHASE>
__device__ __forceinline__ ItemGeo item_geo(const GemmArgs& a, int bid) {
  ItemGeo g;
  const int4 t = __ldg(reinterpret_cast<const int4*>(a.items) + bid);
  g.m0 = t.y;
  g.n0 = t.z;
  const int4 U = __ldg(reinterpret_cast<const int4*>(a.units + kUnitHeader) + t.x);
  g.shared = U.x == -1;
  g.slot = U.x >= 0 ? U.x : (U.x <= -2 ? -2 - U.x : 0);
  g.p0 = g.shared ? a.rows_routed : U.y;
  g.ntok = min(kTok, U.z - g.m0);
  g.K = PHASE == 0 ? a.H : (g.shared ? a.Is : a.I);
  // fail closed: a routed expert is used only if its slot holds the
  // generation its page-table entry expects
  g.stale = !g.shared && (g.slot >= a.S || (U.x >= 0 && __ldg(a.gen + g.slot) != static_cast<uint32_t>(U.w)));
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

template <int PHASE>  // 0: gate/up + SwiGLU, 1: down
__global__ void __launch_bounds__(kThreadsG, 1) gemm_kernel(const __grid_constant__ CUtensorMap map_b32,
                                                            const __grid_constant__ CUtensorMap map_bt,
                                                            const __grid_constant__ CUtensorMap map_q,
                                                            const __grid_constant__ CUtensorMap map_sq,
                                                            GemmArgs a) {
  extern __shared__ unsigned char smraw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  // smem ring: full (TMA bytes), sfree (the MMA's commit + the 8 dequant
  // warps); item scales: scf (bulk-copy bytes), sce (8 dequant warps); TMEM
  // A ring: aready (8 dequant warps), afree (the MMA's commit);
  // accumulators: accf (commit), acce (4 epilogue warps)
  __shared__ uint64_t bar_full[kMaxStages], bar_sfree[kMaxStages], bar_scf[2], bar_sce[2];
  __shared__ uint64_t bar_aready[kAStages], bar_afree[kAStages];
  __shared__ uint64_t bar_accf[2], bar_acce[2], bar_drain;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_abort;
  __shared__ ItemGeo s_geo[kGeoCap];
  volatile int* abort_flag = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kStages = a.stages;
  const uint32_t sbase = su32(sm);
  const uint32_t sscale = sbase + static_cast<uint32_t>(kStages) * kStageBytes;  // 2 item-scale buffers
  const uint32_t sepi = sscale + 2u * static_cast<uint32_t>(a.sc_bytes);
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(su32(&bar_scf[b]), 1);
      mbar_init(su32(&bar_sce[b]), kDqWarps);
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
    // ---------------- producer (one thread): per item the block scales of
    // the weight tile (fp16 [rows][K/32]: gate rows then up rows, or the down
    // rows) by bulk copy; per stage the token tile and the raw quant rows
    if (lane == 0) {
      uint32_t ring = 0, it = 0;
      RingPos rp;
      for (int i = 0; i < my_items && !*abort_flag; ++i) {
        const ItemGeo g = geo_of<PHASE>(a, s_geo, i);
        if (g.stale) continue;
        const int nkb = g.K / kBK;
        const bool whole = g.ntok == kTok;
        const int nbox = (g.ntok + 31) / 32;
        const uint32_t bytes = (whole ? kBBytes : static_cast<uint32_t>(nbox) * 4096u) + kQBytes;
        const uint8_t* wbase = g.shared ? a.shared : a.pool + static_cast<int64_t>(g.slot) * a.slot_stride;
        const int64_t* soff = g.shared ? a.s_soff : a.r_soff;
        const int64_t pitch = g.K / 16;  // bytes per scale row
        const uint32_t sb = it & 1u;
        if (it >= 2 && !mbar_wait(su32(&bar_sce[sb]), ((it >> 1) & 1u) ^ 1u, abort_flag, a.err)) break;
        const uint32_t sdst = sscale + sb * static_cast<uint32_t>(a.sc_bytes), scb = su32(&bar_scf[sb]);
        mbar_expect_tx(scb, static_cast<uint32_t>(kWR * pitch));
        if (PHASE == 0) {
          bulk_g2s(sdst, wbase + soff[0] + g.n0 * pitch, static_cast<uint32_t>(64 * pitch), scb);
          bulk_g2s(sdst + static_cast<uint32_t>(64 * pitch), wbase + soff[1] + g.n0 * pitch,
                   static_cast<uint32_t>(64 * pitch), scb);
        } else {
          bulk_g2s(sdst, wbase + soff[2] + g.n0 * pitch, static_cast<uint32_t>(kWR * pitch), scb);
        }
        ++it;
        const CUtensorMap* mq = g.shared ? &map_sq : &map_q;
        const int zs = g.shared ? 0 : g.slot;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++ring, rp.next(kStages)) {
          const int s = rp.s;
          if (ring >= static_cast<uint32_t>(kStages) &&
              !(ok = mbar_wait(su32(&bar_sfree[s]), rp.ph ^ 1u, abort_flag, a.err)))
            break;
          const uint32_t st = sbase + s * kStageBytes, fb = su32(&bar_full[s]);
          mbar_expect_tx(fb, bytes);
          if (whole)
            tma2d(st, &map_bt, fb, kb * kBK, g.p0 + g.m0);
          else
            for (int bx = 0; bx < nbox; ++bx) tma2d(st + bx * 4096u, &map_b32, fb, kb * kBK, g.p0 + g.m0 + bx * 32);
          // gate/up: rows [n0, n0+64) of the gate and of the up plane in one
          // box; down: rows [n0, n0+128)
          tma4d(st + kBBytes, mq, fb, kb * kBK, g.n0, 0, zs);
        }
        if (!ok) break;
      }
      // drain: the last copies into each stage and scale buffer complete
      const uint32_t n = ring < static_cast<uint32_t>(kStages) ? ring : static_cast<uint32_t>(kStages);
      for (uint32_t j = 0; j < n; ++j) {
        const uint32_t r = ring - 1 - j;
        mbar_drain(su32(&bar_full[r % kStages]), (r / kStages) & 1u, a.err);
      }
      for (uint32_t j = 0; j < (it < 2u ? it : 2u); ++j) {
        const uint32_t q = it - 1 - j;
        mbar_drain(su32(&bar_scf[q & 1u]), (q >> 1) & 1u, a.err);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      uint32_t ring = 0, acc_i = 0;
      RingPos rp, ap;
      const uint32_t fmt = PHASE == 0 ? 0u : 1u;  // f16 : bf16
      for (int i = 0; i < my_items && !*abort_flag; ++i) {
        const ItemGeo g = geo_of<PHASE>(a, s_geo, i);
        if (g.stale) continue;
        const int nkb = g.K / kBK;
        const uint32_t n = static_cast<uint32_t>((g.ntok + 15) & ~15);
        const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((n >> 3) << 17) | ((kWR >> 4) << 24);
        const uint32_t buf = acc_i & 1u, aph = (acc_i >> 1) & 1u;
        if (acc_i >= 2 && !mbar_wait(su32(&bar_acce[buf]), aph ^ 1u, abort_flag, a.err)) break;
        asm volatile("tcgen05.fence::after_thread_sync;");
        const uint32_t dt = tmem + buf * static_cast<uint32_t>(kTok);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++ring, rp.next(kStages), ap.next(kAStages)) {
          const int s = rp.s, j = ap.s;
          if (!(ok = mbar_wait(su32(&bar_full[s]), rp.ph, abort_flag, a.err))) break;
          if (!(ok = mbar_wait(su32(&bar_aready[j]), ap.ph, abort_flag, a.err))) break;
          asm volatile("tcgen05.fence::after_thread_sync;");
          const uint32_t sb = sbase + s * kStageBytes, at = tmem + kAcol0 + 32u * j;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_ts(dt, at + 8 * k, sdesc(sb + 32 * k), idesc, (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit(su32(&bar_sfree[s]));
          umma_commit(su32(&bar_afree[j]));
        }
        if (!ok) break;
        umma_commit(su32(&bar_accf[buf]));
        ++acc_i;
      }
      // drain: every MMA issued here has completed before TMEM is released
      umma_commit(su32(&bar_drain));
      mbar_drain(su32(&bar_drain), 0, a.err);
    }
  } else if (warp < 2 + kDqWarps) {
    // ---------------- dequantisation: warp w owns TMEM lanes 32*(w%4) ..
    // +31 (its weight rows) and one of the stage's two Q8_0 blocks
    const int sp = warp & 3, half = (warp - 2) >> 2;
    const int r = sp * 32 + lane;  // weight row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(sp * 32) << 16;
    const uint32_t swz = static_cast<uint32_t>((r >> 1) & 3);  // 64-byte swizzle phase of row r
    uint32_t ring = 0, it = 0;
    RingPos rp, ap;
    for (int i = 0; i < my_items && !*abort_flag; ++i) {
      const ItemGeo g = geo_of<PHASE>(a, s_geo, i);
      if (g.stale) continue;
      const int nkb = g.K / kBK;
      const uint32_t sb = it & 1u;
      if (!mbar_wait(su32(&bar_scf[sb]), (it >> 1) & 1u, abort_flag, a.err)) break;
      ++it;
      // this row's block scales; block 2*kb + half in stage kb
      const uint32_t srow = sscale + sb * static_cast<uint32_t>(a.sc_bytes) + r * (g.K / 16) + half * 2;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb, ++ring, rp.next(kStages), ap.next(kAStages)) {
        const int s = rp.s, j = ap.s;
        if (!(ok = mbar_wait(su32(&bar_full[s]), rp.ph, abort_flag, a.err))) break;
        const uint32_t sq = sbase + s * kStageBytes + kBBytes + r * kBK;
        uint32_t h;
        asm volatile("ld.shared.u16 %0, [%1];" : "=r"(h) : "r"(srow + kb * 4));
        const uint4 raw0 = lds128(sq + (((2 * half) ^ swz) << 4));
        const uint4 raw1 = lds128(sq + (((2 * half + 1) ^ swz) << 4));
        uint32_t out[16];
        {
          uint4 o0, o1, o2, o3;
          if (PHASE == 0) {
            dq16_f16(raw0, h | (h << 16), o0, o1);
            dq16_f16(raw1, h | (h << 16), o2, o3);
          } else {
            const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
            dq16_bf16(raw0, d, o0, o1);
            dq16_bf16(raw1, d, o2, o3);
          }
          out[0] = o0.x, out[1] = o0.y, out[2] = o0.z, out[3] = o0.w;
          out[4] = o1.x, out[5] = o1.y, out[6] = o1.z, out[7] = o1.w;
          out[8] = o2.x, out[9] = o2.y, out[10] = o2.z, out[11] = o2.w;
          out[12] = o3.x, out[13] = o3.y, out[14] = o3.z, out[15] = o3.w;
        }
        // the stage's quant rows and scales have been read
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&bar_sfree[s]));
        if (ring >= static_cast<uint32_t>(kAStages) &&
            !(ok = mbar_wait(su32(&bar_afree[j]), ap.ph ^ 1u, abort_flag, a.err)))
          break;
        asm volatile("tcgen05.fence::after_thread_sync;");
        tmem_st16(tmem + lane_base + kAcol0 + 32u * j + 16u * half, out);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;");
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&bar_aready[j]));
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(su32(&bar_sce[sb]));  // done with the item's scales
    }
  } else {
    // ---------------- epilogue: warp w reads TMEM lanes 32*(w%4) .. +31
    const int sp = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(sp * 32) << 16;
    uint32_t acc_i = 0;
    for (int i = 0; i < my_items && !*abort_flag; ++i) {
      const ItemGeo g = geo_of<PHASE>(a, s_geo, i);
      if (g.stale) {
        if (tid == kEpTid0) atomicOr(a.err, MOE_DEVERR_STALE);
        continue;
      }
      const uint32_t buf = acc_i & 1u, aph = (acc_i >> 1) & 1u;
      if (!mbar_wait(su32(&bar_accf[buf]), aph, abort_flag, a.err)) break;
      asm volatile("tcgen05.fence::after_thread_sync;");
      const int nch = (g.ntok + 31) / 32;
      const uint32_t tb = tmem + lane_base + buf * static_cast<uint32_t>(kTok);
      const int64_t prow0 = static_cast<int64_t>(g.p0) + g.m0;
      if (PHASE == 0) {
        // lanes 0..63 hold gate rows, 64..127 the same up rows; in each chunk
        // of 32 tokens the gate warps finish tokens 0..15, the up warps 16..31
        const bool gate = sp < 2;
        const int rr = (sp & 1) * 32 + lane;  // h column within the tile
        const uint32_t xg = sepi, xu = sepi + 64 * kXP * 4, sh = sepi + 2 * 64 * kXP * 4;
        const int et = tid - kEpTid0;  // 0..127
        const uint32_t mine = (gate ? xg : xu) + rr * kXP * 4;
        const uint32_t other = (gate ? xu : xg) + rr * kXP * 4;
        const int tok0 = gate ? 0 : 16;
        for (int ch = 0; ch < nch; ++ch) {
          uint32_t v[32];
          tmem_ld32(tb + ch * 32, v);
          uint32_t send[16];  // gate warps pass tokens 16..31, up warps 0..15
#pragma unroll
          for (int j = 0; j < 16; ++j) send[j] = gate ? v[16 + j] : v[j];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            sts128(mine + q * 16, make_uint4(send[4 * q], send[4 * q + 1], send[4 * q + 2], send[4 * q + 3]));
          epi_sync();
          float o[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 w = lds128(other + q * 16);
            o[4 * q] = __uint_as_float(w.x);
            o[4 * q + 1] = __uint_as_float(w.y);
            o[4 * q + 2] = __uint_as_float(w.z);
            o[4 * q + 3] = __uint_as_float(w.w);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float gg = gate ? __uint_as_float(v[j]) : o[j];
            const float uu = gate ? o[j] : __uint_as_float(v[16 + j]);
            const __nv_bfloat16 hb = __float2bfloat16_rn(silu_mul(gg, uu));
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(sh + ((tok0 + j) * kSP + rr) * 2),
                         "h"(*reinterpret_cast<const unsigned short*>(&hb))
                         : "memory");
          }
          epi_sync();
          // 32 tokens x 64 columns of bf16: 256 pieces of 16 bytes
#pragma unroll
          for (int rep = 0; rep < 2; ++rep) {
            const int piece = et + 128 * rep, j = piece >> 3, part = piece & 7;
            const int tok = ch * 32 + j;
            if (tok < g.ntok) {
              const uint4 w = lds128(sh + (j * kSP + part * 8) * 2);
              *reinterpret_cast<uint4*>(a.h + (prow0 + tok) * a.ldh + g.n0 + part * 8) = w;
            }
          }
        }
      } else {
        const int r = sp * 32 + lane;  // output column n0 + r
        for (int ch = 0; ch < nch; ++ch) {
          uint32_t v[32];
          tmem_ld32(tb + ch * 32, v);
          float* dst = a.yp + (prow0 + ch * 32) * a.H + g.n0 + r;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (ch * 32 + j < g.ntok) dst[static_cast<int64_t>(j) * a.H] = __uint_as_float(v[j]);
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;");
      __syncwarp();
      if (lane == 0) mbar_arrive(su32(&bar_acce[buf]));
      ++acc_i;
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
}

}  // namespace

// Shared memory of one item-scale buffer: 128 weight rows x K/32 fp16.
int gemm_scale_bytes(int K) { return ((kWR * (K / 16)) + 1023) / 1024 * 1024; }

// Pipeline stages that fit in shared memory beside the item-scale buffers
// and the epilogue buffers.
int gemm_stages(int K) {
  const size_t limit = 227 * 1024 - sizeof(ItemGeo) * kGeoCap - 512;  // static shared memory
  const size_t fixed = 2 * static_cast<size_t>(gemm_scale_bytes(K)) + kEpiBytes + 1024;
  const int n = static_cast<int>((limit - fixed) / kStageBytes);
  return n < 2 ? 0 : (n > kMaxStages ? kMaxStages : n);
}

size_t gemm_smem_bytes(int stages, int K) {
  return static_cast<size_t>(stages) * kStageBytes + 2 * static_cast<size_t>(gemm_scale_bytes(K)) + kEpiBytes +
         1024;
}

cudaError_t launch_gemm(int phase, const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t st) {
  const int smem = static_cast<int>(gemm_smem_bytes(a.stages, a.kmax));
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
