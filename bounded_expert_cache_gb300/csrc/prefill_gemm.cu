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
// Two grouped GEMMs run over (unit, 128-row tile, 256-column tile) work
// items:
//   gate/up: [rows x H] * [(64..128 gate rows | same up rows) x H]^T -> SwiGLU
//            -> h (bf16)   (fp16 operands: x exact, d*q rounded to fp16)
//   down:    [rows x I] * [256 down rows x I]^T * combine weight -> fp32 rows
//            (bf16 operands: h and d*q rounded to bf16, h may exceed fp16)
// A CTA of 10 warps handles one work item:
//   warp 0      TMA: the activation tile (128 rows x 64, 128-byte swizzle)
//               and the raw Q8_0 quant rows of the weight tile, addressed in
//               the slot pool through a 3-D tensor map (bytes, rows, slot)
//   warp 1      allocates the TMEM accumulator (128 lanes x 256 fp32
//               columns) and issues tcgen05.mma (M 128, N 256, K 16) from
//               shared-memory descriptors; commits release the stage
//   warps 2..9  dequantise: int8 * fp16 block scale -> fp16/bf16, written in
//               the same 128-byte-swizzled K-major layout the MMA reads; then
//               the epilogue (tcgen05.ld of the accumulator rows)
// A 3-stage mbarrier ring overlaps TMA, dequantisation and MMA. Every wait
// is bounded; a wait that runs out sets an error bit and the CTA leaves
// without touching the results.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "prefill.h"

namespace moe {
namespace {

constexpr int kMaxStages = 4;
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kThreadsG = 320;  // 10 warps
constexpr int kDqWarps = 8;
constexpr uint32_t kABytes = kBM * kBK * 2;    // 16 KiB
constexpr uint32_t kBqBytes = kBN * kBK;       // 16 KiB of int8
constexpr uint32_t kB16Bytes = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kStageBytes = kABytes + kBqBytes + kB16Bytes;
constexpr long long kWaitCycles = 4000000000ll;  // about 2 s at the SM clock

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t c) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(c));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
// Bounded wait on a phase of an mbarrier; false if it ran out (about 2 s).
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > kWaitCycles) return false;
  }
}
__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          su32(dst)),
      "l"(m), "r"(su32(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma3d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          su32(dst)),
      "l"(m), "r"(su32(bar)), "r"(x), "r"(y), "r"(z)
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
__device__ __forceinline__ void umma(uint32_t dt, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(dt),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
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

__device__ __forceinline__ uint32_t pack2(float a, float b, bool fp16) {
  if (fp16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Work item of a GEMM: unit, first row within the unit, first weight row.
struct Item {
  int u, m0, n0;
};

__device__ __forceinline__ bool item_of(const GemmArgs& a, int bid, Item& it) {
  const int n_items = __ldg(a.n_items);
  if (bid >= n_items) return false;
  const int4 t = __ldg(reinterpret_cast<const int4*>(a.items) + bid);
  it.u = t.x;
  it.m0 = t.y;
  it.n0 = t.z;
  return true;
}

template <int PHASE>  // 0: gate/up + SwiGLU, 1: down + combine weight
__global__ void __launch_bounds__(kThreadsG, 1) gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                                                            const __grid_constant__ CUtensorMap map_q0,
                                                            const __grid_constant__ CUtensorMap map_q1,
                                                            const __grid_constant__ CUtensorMap map_sq0,
                                                            const __grid_constant__ CUtensorMap map_sq1,
                                                            GemmArgs a) {
  extern __shared__ unsigned char smraw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_full[kMaxStages], bar_ready[kMaxStages], bar_empty[kMaxStages], bar_acc;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  Item it;
  if (!item_of(a, blockIdx.x, it)) return;
  // unit geometry
  const int4 U = __ldg(reinterpret_cast<const int4*>(a.units + kUnitHeader) + it.u);
  const bool shared = U.x == -1;
  const int slot = U.x >= 0 ? U.x : (U.x <= -2 ? -2 - U.x : 0);
  const int p0 = shared ? a.rows_routed : U.y;
  const int M = U.z;
  // fail closed: a routed expert is used only if its slot holds the
  // generation its page-table entry expects
  if (!shared && (slot >= a.S || (U.x >= 0 && __ldg(a.gen + slot) != static_cast<uint32_t>(U.w)))) {
    if (threadIdx.x == 0) atomicOr(a.err, MOE_DEVERR_STALE);
    return;
  }
  const int K = PHASE == 0 ? a.H : (shared ? a.Is : a.I);
  const int n_rows_b = PHASE == 0 ? (shared ? a.Is : a.I) : a.H;  // weight rows of the matrix
  const int nkb = K / kBK;
  const int halfN = kBN / 2;
  // scale planes (fp16 [rows][K/32]) of the weight tile's matrix(es)
  const uint8_t* wbase = shared ? a.shared : a.pool + static_cast<int64_t>(slot) * a.slot_stride;
  const int64_t soff0 = shared ? a.s_soff[PHASE == 0 ? 0 : 2] : a.r_soff[PHASE == 0 ? 0 : 2];
  const int64_t soff1 = shared ? a.s_soff[1] : a.r_soff[1];
  const __half* sc0 = reinterpret_cast<const __half*>(wbase + soff0);
  const __half* sc1 = reinterpret_cast<const __half*>(wbase + soff1);
  const int kStages = a.stages;
  // the tile's block scales (fp16 [256 rows][K/32]) sit after the stages
  __half* s_scale = reinterpret_cast<__half*>(sm + static_cast<size_t>(kStages) * kStageBytes);
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_ready[s], kDqWarps);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_acc, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_holder)),
                 "r"(256));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = tmem_holder;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      const uint32_t bytes = kABytes + kBqBytes;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kStages;
        const uint32_t round = kb / kStages;
        if (kb >= kStages && !mbar_wait(&bar_empty[s], (round - 1) & 1)) {
          atomicOr(a.err, MOE_DEVERR_TIMEOUT);
          s_abort = 1;
          break;
        }
        unsigned char* st = sm + s * kStageBytes;
        mbar_expect_tx(&bar_full[s], bytes);
        tma2d(st, &map_a, &bar_full[s], kb * kBK, p0 + it.m0);
        if (PHASE == 0) {
          // gate rows [n0, n0+128) then up rows [n0, n0+128) of the quant planes
          if (shared) {
            tma3d(st + kABytes, &map_sq0, &bar_full[s], kb * kBK, it.n0, 0);
            tma3d(st + kABytes + halfN * kBK, &map_sq1, &bar_full[s], kb * kBK, it.n0, 0);
          } else {
            tma3d(st + kABytes, &map_q0, &bar_full[s], kb * kBK, it.n0, slot);
            tma3d(st + kABytes + halfN * kBK, &map_q1, &bar_full[s], kb * kBK, it.n0, slot);
          }
        } else {
          if (shared)
            tma3d(st + kABytes, &map_sq0, &bar_full[s], kb * kBK, it.n0, 0);
          else
            tma3d(st + kABytes, &map_q0, &bar_full[s], kb * kBK, it.n0, slot);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = (1u << 4) | ((PHASE == 0 ? 0u : 1u) << 7) | ((PHASE == 0 ? 0u : 1u) << 10) |
                             ((static_cast<uint32_t>(kBN) >> 3) << 17) | ((static_cast<uint32_t>(kBM) >> 4) << 24);
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int s = kb % kStages;
        const uint32_t round = kb / kStages;
        ok = mbar_wait(&bar_ready[s], round & 1);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;");
        unsigned char* st = sm + s * kStageBytes;
        const uint32_t sa = su32(st), sb = su32(st + kABytes + kBqBytes);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          umma(tmem, sdesc(sa + 32 * k), sdesc(sb + 32 * k), idesc, (kb > 0 || k > 0) ? 1u : 0u);
        umma_commit(&bar_empty[s]);
      }
      if (!ok) {
        atomicOr(a.err, MOE_DEVERR_TIMEOUT);
        s_abort = 1;
      }
      umma_commit(&bar_acc);
    }
  } else {
    // ---------------- dequantisation: 256 rows x 8 chunks of 8 weights per stage
    const int dt = tid - 64;  // 0..255
    {
      // the tile's scale rows: gate rows then up rows (or 256 down rows),
      // each row K/32 halves, contiguous in the plane; rows past the matrix
      // get scale 0
      const int spr = K / 32;
      const int rows_half = PHASE == 0 ? halfN : kBN;
      for (int m = 0; m < (PHASE == 0 ? 2 : 1); ++m) {
        const __half* src = (m == 0 ? sc0 : sc1) + static_cast<int64_t>(it.n0) * spr;
        __half* dst = s_scale + m * halfN * spr;
        const int valid_rows = max(0, min(rows_half, n_rows_b - it.n0));
        const int nvalid = valid_rows * spr, ntot = rows_half * spr;
        for (int i = dt; i < ntot; i += 256) dst[i] = i < nvalid ? __ldg(src + i) : __float2half(0.f);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");  // dequant warps only
    }
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % kStages;
      const uint32_t round = kb / kStages;
      bool ok = mbar_wait(&bar_full[s], round & 1);
      if (!ok) {
        if (lane == 0) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      unsigned char* st = sm + s * kStageBytes;
      const int8_t* q8 = reinterpret_cast<const int8_t*>(st + kABytes);
      unsigned char* b16 = st + kABytes + kBqBytes;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int item = dt + j * 256;
        const int r = item >> 3, c = item & 7;
        const float d = __half2float(s_scale[r * (K / 32) + kb * 2 + (c >> 2)]);
        const uint2 raw = *reinterpret_cast<const uint2*>(q8 + r * kBK + c * 8);
        const uint32_t lo = raw.x ^ 0x80808080u, hi = raw.y ^ 0x80808080u;
        float f[8];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          f[b] = (__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7540u | b)) - 8388736.0f) * d;
          f[4 + b] = (__uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7540u | b)) - 8388736.0f) * d;
        }
      const uint4 w = make_uint4(pack2(f[0], f[1], PHASE == 0), pack2(f[2], f[3], PHASE == 0),
                                   pack2(f[4], f[5], PHASE == 0), pack2(f[6], f[7], PHASE == 0));
        const uint32_t off = (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(b16 + off) = w;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ready[s]);
    }
    // ---------------- epilogue: warps 2..5 own TMEM lane groups (warp % 4)
    if (warp < 6) {
      const bool ok = mbar_wait(&bar_acc, 0);
      asm volatile("tcgen05.fence::after_thread_sync;");
      const int lg = warp & 3;  // lanes 32*lg .. 32*lg+31
      const int row = lg * 32 + lane;
      const bool live = ok && !s_abort && it.m0 + row < M;
      const int64_t prow = static_cast<int64_t>(p0) + it.m0 + row;
      const uint32_t tl = tmem + (static_cast<uint32_t>(lg * 32) << 16);
      if (PHASE == 0) {
        const int Iu = shared ? a.Is : a.I;
        for (int c = 0; c < halfN / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tl + c * 32, g);
          tmem_ld32(tl + halfN + c * 32, u);
          if (live) {
            uint32_t o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
              const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
              const float h0 = g0 / (1.f + expf(-g0)) * u0, h1 = g1 / (1.f + expf(-g1)) * u1;
              o[j] = pack2(h0, h1, false);
            }
            const int col = it.n0 + c * 32;
            if (col + 32 <= Iu) {
              uint4* dst = reinterpret_cast<uint4*>(a.h + prow * a.ldh + col);
#pragma unroll
              for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            } else {
              uint16_t* dst = reinterpret_cast<uint16_t*>(a.h + prow * a.ldh);
              for (int j = 0; j < 32 && col + j < Iu; ++j)
                dst[col + j] = static_cast<uint16_t>(j & 1 ? o[j >> 1] >> 16 : o[j >> 1] & 0xFFFFu);
            }
          }
        }
      } else {
        const float wgt = live ? (shared ? 1.f : __ldg(a.perm_w + prow)) : 0.f;
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tl + c * 32, v);
          const int col = it.n0 + c * 32;
          if (live && col < a.H) {
            float4* dst = reinterpret_cast<float4*>(a.yp + prow * a.H + col);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(wgt * __uint_as_float(v[4 * q]), wgt * __uint_as_float(v[4 * q + 1]),
                                   wgt * __uint_as_float(v[4 * q + 2]), wgt * __uint_as_float(v[4 * q + 3]));
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256));
}

}  // namespace

// Stages that fit beside the tile's scales (K/32 halves per weight row).
int gemm_stages(int K) {
  const size_t limit = 227 * 1024, scales = static_cast<size_t>(kBN) * (K / 32) * 2;
  const int n = static_cast<int>((limit - scales - 1024 - 256) / kStageBytes);
  return n < 2 ? 0 : (n > kMaxStages ? kMaxStages : n);
}

size_t gemm_smem_bytes(int stages, int K) {
  return static_cast<size_t>(stages) * kStageBytes + static_cast<size_t>(kBN) * (K / 32) * 2 + 1024;
}

cudaError_t launch_gemm(int phase, const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t st) {
  const int smem = static_cast<int>(gemm_smem_bytes(a.stages, a.kmax));
  cudaError_t e;
  if (phase == 0) {
    e = cudaFuncSetAttribute(gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gemm_kernel<0><<<grid, kThreadsG, smem, st>>>(m.a, m.q0, m.q1, m.sq0, m.sq1, a);
  } else {
    e = cudaFuncSetAttribute(gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gemm_kernel<1><<<grid, kThreadsG, smem, st>>>(m.a, m.q0, m.q1, m.sq0, m.sq1, a);
  }
  return cudaGetLastError();
}

}  // namespace moe
