// Decode-path expert FFN: fused dequantise + SwiGLU + down projection +
// shared expert + weighted combine for a few tokens per step.
//
// "Paging the Experts" §3.1: gate, up and down projections per expert.
// "Nanite for Experts" §1: eight routed experts plus one shared expert per
// token; §5.5: results merge into their original positions; §12: one
// expert-major operator consumes routed positions and page-table entries of
// many resident experts; §3.2: an invalid slot or generation is never read.
//
// Both phases stream weights straight from the slots with coalesced 16-byte
// loads (a warp covers 512 contiguous bytes of a row per instruction) and
// keep the activations in shared memory in a bank-conflict-free swizzled
// layout, reused across the rows a warp holds. Dequantisation is exact in
// fp32: a Q8_0 byte q becomes the float 2^23 + (q + 128) by one byte
// permute, and one subtraction leaves q; a Q4_0 nibble likewise gives q - 8.
// Each 16- or 32-weight chunk is dotted in fp32 and scaled once by its fp16
// block scale.
//
// Phase 1 (gate/up): one warp item = (unit, 2 rows): rows r, r+1 of the gate
// and up matrices of one unit (a routed expert of the union, or the shared
// expert), for every token routed to it; writes h = silu(g) * u in fp32 to
// scratch, indexed by expert-major assignment (routed) or token (shared).
// Phase 2 (down + combine): a block owns 8 output rows; warp items = (unit,
// 2 rows); each item's partial sums (already weighted by the combine weight)
// go to shared memory and are added in unit order, so the output does not
// depend on scheduling and is identical whatever the cache state.
#include <cuda_fp16.h>

#include "internal.h"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerItem = 2;   // rows per warp item
constexpr int kDownRows = 8;      // output rows per phase-2 block

// Swizzled position of element k in an fp32 row whose length is a multiple
// of 32: the four 16-byte quads of each 16-float chunk c are rotated by
// XOR with (c >> 1) & 3, so eight lanes reading quad j of eight consecutive
// chunks hit eight distinct 16-byte bank groups.
__device__ __forceinline__ int swz(int k) {
  const int c = k >> 4, j = (k >> 2) & 3;
  return (c << 4) | ((j ^ ((c >> 1) & 3)) << 2) | (k & 3);
}

__device__ __forceinline__ void load_chunk16(const float* row, int c, float* v) {
  const int s = (c >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 q = *reinterpret_cast<const float4*>(row + (c << 4) + ((j ^ s) << 2));
    v[4 * j + 0] = q.x;
    v[4 * j + 1] = q.y;
    v[4 * j + 2] = q.z;
    v[4 * j + 3] = q.w;
  }
}

template <int XT>
__device__ __forceinline__ float load_act(const void* x, size_t i) {
  if (XT == MOE_BF16) {
    const uint16_t b = static_cast<const uint16_t*>(x)[i];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  } else {
    return static_cast<const float*>(x)[i];
  }
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float ld_scale(const uint8_t* p) {
  const unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(p));
  return __half2float(__ushort_as_half(b));
}

// Loads from a miss's source: the pinned store, read over the host link.
__device__ __forceinline__ uint4 ld_host(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ unsigned short ld_scale_host_bits(const uint8_t* p) {
  return __ldcs(reinterpret_cast<const unsigned short*>(p));
}

// A miss's scales reach its slot from the loads the dot products make: the
// lane whose chunk opens a 32-weight block (every Q4_0 chunk, even Q8_0
// chunks) stores that block's fp16 scale, so no copy waits on its own load.
template <int Q>
__device__ __forceinline__ bool owns_scale(int c) {
  return Q != MOE_Q8_0 || (c & 1) == 0;
}

// q (Q8_0 byte) -> float, exact: bits 0x4B0000uu = 2^23 + uu with uu = q + 128.
__device__ __forceinline__ float q8_to_f(uint32_t biased, int b) {
  return __uint_as_float(__byte_perm(biased, 0x4B000000u, 0x7540u | b)) - 8388736.0f;
}
// nibble n (0..15) in byte b of w -> n - 8, exact.
__device__ __forceinline__ float q4_to_f(uint32_t nib, int b) {
  return __uint_as_float(__byte_perm(nib, 0x4B000000u, 0x7540u | b)) - 8388616.0f;
}

// Dot of one 16-byte Q8_0 chunk (16 weights) with 16 activations.
__device__ __forceinline__ float dot_q8(const uint4 w, const float* x) {
  const uint32_t ws[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u,
                          w.w ^ 0x80808080u};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int b = 0; b < 4; ++b) s = fmaf(q8_to_f(ws[i], b), x[4 * i + b], s);
  return s;
}

// Dot of one 16-byte Q4_0 block (32 weights) with activations: xl for
// elements 0..15 (low nibbles), xh for 16..31 (high nibbles).
__device__ __forceinline__ float dot_q4(const uint4 w, const float* xl, const float* xh) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = ws[i] & 0x0F0F0F0Fu, hi = (ws[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      s = fmaf(q4_to_f(lo, b), xl[4 * i + b], s);
      s = fmaf(q4_to_f(hi, b), xh[4 * i + b], s);
    }
  }
  return s;
}

struct UnitRef {
  const uint8_t* base;  // payload
  int64_t qoff[3];      // quant-plane offsets of gate, up, down
  int64_t soff[3];      // scale-plane offsets
  int M;                // tokens of the unit
  int p0;               // first expert-major assignment (routed) or -1 (shared)
  int slot;             // slot (routed) or -1 (shared)
  uint32_t egen;        // generation the slot must hold
  bool miss;            // materialised by this step: read from the store, write to dst
  uint8_t* dst;         // slot payload being filled (miss only)
};

// Unit u of the step's unit table: routed experts of the union (in union
// order) then the shared expert. Only the entry is read here; the slot's
// generation is checked by unit_ok, issued alongside the weight loads.
__device__ __forceinline__ UnitRef resolve_unit(const FfnArgs& a, int u) {
  const int4 d = __ldg(reinterpret_cast<const int4*>(a.units + kUnitHeader) + u);
  UnitRef r;
  r.miss = d.x <= -2;
  r.slot = r.miss ? -2 - d.x : d.x;
  r.p0 = d.y;
  r.M = d.z;
  r.egen = static_cast<uint32_t>(d.w);
  const bool routed = r.slot >= 0;
  const bool in_range = r.slot < a.S && (!r.miss || (a.store && d.w >= 0 && d.w < a.E));
  // an out-of-range slot or a missing shared payload points at slot 0 (always
  // mapped) and is refused by unit_ok, so no load leaves the pool
  const int64_t slot_off = static_cast<int64_t>(routed && in_range ? r.slot : 0) * a.slot_stride;
  if (r.miss && in_range) {
    r.base = a.store + static_cast<int64_t>(d.w) * a.payload;
    r.dst = a.pool + slot_off;
  } else {
    r.base = routed ? a.pool + slot_off : (a.shared ? a.shared : a.pool);
    r.dst = nullptr;
    r.miss = false;
    if (d.x <= -2) r.slot = a.S;  // refused below
  }
#pragma unroll
  for (int m = 0; m < 3; ++m) {
    r.qoff[m] = routed ? a.g.qoff[m] : a.gs.qoff[m];
    r.soff[m] = routed ? a.g.soff[m] : a.gs.soff[m];
  }
  return r;
}

// A routed unit is usable only if its slot holds the generation the page
// table expects (every tile of its last fill has landed); the shared expert
// always is.
__device__ __forceinline__ bool unit_ok(const FfnArgs& a, const UnitRef& U) {
  if (U.miss) return true;
  if (U.slot < 0) return a.shared != nullptr;
  return U.slot < a.S && __ldg(a.gen + U.slot) == U.egen;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------------ phase 1
template <int Q, int TM, int XT>
__global__ void __launch_bounds__(kThreads) gateup_kernel(FfnArgs a) {
  extern __shared__ float xs[];  // [T][H] swizzled
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, T = a.T;
  // x is the layer's input, complete once the router has passed its wait
  for (int i = tid; i < T * H; i += kThreads) {
    const int t = i / H, k = i - t * H;
    xs[t * H + swz(k)] = load_act<XT>(a.x, i);
  }
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const int n_units = __ldg(a.units);
  const int nu = n_units - (a.shared ? 1 : 0);  // routed units
  const int per_routed = a.I / kRowsPerItem;
  const int per_shared = a.shared ? a.Is / kRowsPerItem : 0;
  const int items = nu * per_routed + per_shared;
  const int rowbytes = Q == MOE_Q8_0 ? H : H / 2;
  const int nch = rowbytes / 16;
  const int sc_row = (H / 32) * 2;  // scale bytes per row
  for (int it = blockIdx.x * kWarps + warp; it < items; it += gridDim.x * kWarps) {
    int u, r0;
    if (it < nu * per_routed) {
      u = it / per_routed;
      r0 = (it - u * per_routed) * kRowsPerItem;
    } else {
      u = nu;
      r0 = (it - nu * per_routed) * kRowsPerItem;
    }
    const UnitRef U = resolve_unit(a, u);
    const bool ok = unit_ok(a, U);
    const uint8_t* q[2 * kRowsPerItem];
    const uint8_t* s[2 * kRowsPerItem];
#pragma unroll
    for (int r = 0; r < kRowsPerItem; ++r) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        q[m * kRowsPerItem + r] = U.base + U.qoff[m] + static_cast<int64_t>(r0 + r) * rowbytes;
        s[m * kRowsPerItem + r] = U.base + U.soff[m] + static_cast<int64_t>(r0 + r) * sc_row;
      }
    }
    for (int m0 = 0; m0 < U.M; m0 += TM) {
      const int mcount = min(TM, U.M - m0);
      int tok[TM];
#pragma unroll
      for (int m = 0; m < TM; ++m)
        tok[m] = (m < mcount) ? (U.p0 >= 0 ? __ldg(a.plan.perm_tok + U.p0 + m0 + m) : m0 + m) : 0;
      float acc[2 * kRowsPerItem][TM];
#pragma unroll
      for (int r = 0; r < 2 * kRowsPerItem; ++r)
#pragma unroll
        for (int m = 0; m < TM; ++m) acc[r][m] = 0.f;
#pragma unroll 2
      for (int c = lane; c < nch; c += 32) {
        uint4 w[2 * kRowsPerItem];
        float d[2 * kRowsPerItem];
        if (U.miss) {
          unsigned short sb[2 * kRowsPerItem];
#pragma unroll
          for (int r = 0; r < 2 * kRowsPerItem; ++r) {
            w[r] = ld_host(q[r] + c * 16);
            sb[r] = ld_scale_host_bits(s[r] + (Q == MOE_Q8_0 ? (c >> 1) : c) * 2);
          }
#pragma unroll
          for (int r = 0; r < 2 * kRowsPerItem; ++r) d[r] = __half2float(__ushort_as_half(sb[r]));
          if (m0 == 0) {
#pragma unroll
            for (int r = 0; r < 2 * kRowsPerItem; ++r) {
              *reinterpret_cast<uint4*>(U.dst + (q[r] - U.base) + c * 16) = w[r];
              if (owns_scale<Q>(c))
                *reinterpret_cast<unsigned short*>(U.dst + (s[r] - U.base) + (Q == MOE_Q8_0 ? (c >> 1) : c) * 2) = sb[r];
            }
          }
        } else {
#pragma unroll
          for (int r = 0; r < 2 * kRowsPerItem; ++r) {
            w[r] = ldg_stream(q[r] + c * 16);
            d[r] = ld_scale(s[r] + (Q == MOE_Q8_0 ? (c >> 1) : c) * 2);
          }
        }
#pragma unroll
        for (int m = 0; m < TM; ++m) {
          if (m < mcount) {
            const float* xr = xs + tok[m] * H;
            if (Q == MOE_Q8_0) {
              float xv[16];
              load_chunk16(xr, c, xv);
#pragma unroll
              for (int r = 0; r < 2 * kRowsPerItem; ++r)
                acc[r][m] = fmaf(d[r], dot_q8(w[r], xv), acc[r][m]);
            } else {
              float xl[16], xh[16];
              load_chunk16(xr, 2 * c, xl);
              load_chunk16(xr, 2 * c + 1, xh);
#pragma unroll
              for (int r = 0; r < 2 * kRowsPerItem; ++r)
                acc[r][m] = fmaf(d[r], dot_q4(w[r], xl, xh), acc[r][m]);
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2 * kRowsPerItem; ++r)
#pragma unroll
        for (int m = 0; m < TM; ++m)
#pragma unroll
          for (int off = 16; off; off >>= 1)
            acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);
      if (!ok) {
        if (lane == 0) atomicOr(a.err, MOE_DEVERR_STALE);
        break;
      }
      if (lane == 0) {
#pragma unroll
        for (int m = 0; m < TM; ++m) {
          if (m < mcount) {
            const int hrow = U.p0 >= 0 ? U.p0 + m0 + m : a.T * a.k + m0 + m;
#pragma unroll
            for (int r = 0; r < kRowsPerItem; ++r)
              a.h[static_cast<int64_t>(hrow) * a.ldh + r0 + r] =
                  silu(acc[r][m]) * acc[kRowsPerItem + r][m];
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------ phase 2
template <int Q, int TM>
__global__ void __launch_bounds__(kThreads) down_kernel(FfnArgs a) {
  extern __shared__ float sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, A = a.T * a.k;
  const int nrows = A + (a.shared ? T : 0);
  const int ldh = a.ldh;
  float* hs = sm;                                   // [nrows][ldh] swizzled
  float* part = sm + static_cast<size_t>(nrows) * ldh;  // [items][2][TM]
  pdl_wait();
  pdl_trigger();
  for (int i = tid; i < nrows * ldh; i += kThreads) {
    const int p = i / ldh, k = i - p * ldh;
    hs[p * ldh + swz(k)] = __ldcg(a.h + i);
  }
  __syncthreads();
  const int units = __ldg(a.units);
  const int o0 = blockIdx.x * kDownRows;
  constexpr int kPairs = kDownRows / kRowsPerItem;
  const int items = units * kPairs;
  for (int it = warp; it < items; it += kWarps) {
    const int u = it / kPairs, rp = it - u * kPairs;
    const UnitRef U = resolve_unit(a, u);
    const bool ok = unit_ok(a, U);
    float acc[kRowsPerItem][TM];
#pragma unroll
    for (int r = 0; r < kRowsPerItem; ++r)
#pragma unroll
      for (int m = 0; m < TM; ++m) acc[r][m] = 0.f;
    {
      const int K = U.p0 >= 0 ? a.I : a.Is;
      const int rowbytes = Q == MOE_Q8_0 ? K : K / 2;
      const int nch = rowbytes / 16;
      const int sc_row = (K / 32) * 2;
      const uint8_t* q[kRowsPerItem];
      const uint8_t* s[kRowsPerItem];
      bool rv[kRowsPerItem];
#pragma unroll
      for (int r = 0; r < kRowsPerItem; ++r) {
        const int o = o0 + rp * kRowsPerItem + r;
        rv[r] = o < a.H;
        q[r] = U.base + U.qoff[2] + static_cast<int64_t>(rv[r] ? o : 0) * rowbytes;
        s[r] = U.base + U.soff[2] + static_cast<int64_t>(rv[r] ? o : 0) * sc_row;
      }
      for (int m0 = 0; m0 < U.M; m0 += TM) {
        const int mcount = min(TM, U.M - m0);
        int tok[TM], hrow[TM];
        float wt[TM];
#pragma unroll
        for (int m = 0; m < TM; ++m) {
          if (m < mcount) {
            if (U.p0 >= 0) {
              hrow[m] = U.p0 + m0 + m;
              tok[m] = __ldg(a.plan.perm_tok + hrow[m]);
              wt[m] = __ldg(a.plan.perm_w + hrow[m]);
            } else {
              hrow[m] = A + m0 + m;
              tok[m] = m0 + m;
              wt[m] = 1.0f;
            }
          } else {
            hrow[m] = 0;
            tok[m] = 0;
            wt[m] = 0.f;
          }
        }
        float pm[kRowsPerItem][TM];
#pragma unroll
        for (int r = 0; r < kRowsPerItem; ++r)
#pragma unroll
          for (int m = 0; m < TM; ++m) pm[r][m] = 0.f;
#pragma unroll 2
        for (int c = lane; c < nch; c += 32) {
          uint4 w[kRowsPerItem];
          float d[kRowsPerItem];
          if (U.miss) {
            unsigned short sb[kRowsPerItem];
#pragma unroll
            for (int r = 0; r < kRowsPerItem; ++r) {
              w[r] = rv[r] ? ld_host(q[r] + c * 16) : make_uint4(0, 0, 0, 0);
              sb[r] = rv[r] ? ld_scale_host_bits(s[r] + (Q == MOE_Q8_0 ? (c >> 1) : c) * 2) : 0;
            }
#pragma unroll
            for (int r = 0; r < kRowsPerItem; ++r) {
              d[r] = __half2float(__ushort_as_half(sb[r]));
              if (rv[r] && m0 == 0) {
                *reinterpret_cast<uint4*>(U.dst + (q[r] - U.base) + c * 16) = w[r];
                if (owns_scale<Q>(c))
                  *reinterpret_cast<unsigned short*>(U.dst + (s[r] - U.base) + (Q == MOE_Q8_0 ? (c >> 1) : c) * 2) = sb[r];
              }
            }
          } else {
#pragma unroll
            for (int r = 0; r < kRowsPerItem; ++r) {
              w[r] = rv[r] ? ldg_stream(q[r] + c * 16) : make_uint4(0, 0, 0, 0);
              d[r] = rv[r] ? ld_scale(s[r] + (Q == MOE_Q8_0 ? (c >> 1) : c) * 2) : 0.f;
            }
          }
#pragma unroll
          for (int m = 0; m < TM; ++m) {
            if (m < mcount) {
              const float* hr = hs + hrow[m] * ldh;
              if (Q == MOE_Q8_0) {
                float hv[16];
                load_chunk16(hr, c, hv);
#pragma unroll
                for (int r = 0; r < kRowsPerItem; ++r) pm[r][m] = fmaf(d[r], dot_q8(w[r], hv), pm[r][m]);
              } else {
                float hl[16], hh[16];
                load_chunk16(hr, 2 * c, hl);
                load_chunk16(hr, 2 * c + 1, hh);
#pragma unroll
                for (int r = 0; r < kRowsPerItem; ++r)
                  pm[r][m] = fmaf(d[r], dot_q4(w[r], hl, hh), pm[r][m]);
              }
            }
          }
        }
        if (!ok) break;
        // weight by the combine weight, accumulate per token (T <= TM)
#pragma unroll
        for (int m = 0; m < TM; ++m) {
          if (m < mcount) {
#pragma unroll
            for (int t = 0; t < TM; ++t)
              if (t == tok[m])
#pragma unroll
                for (int r = 0; r < kRowsPerItem; ++r) acc[r][t] = fmaf(wt[m], pm[r][m], acc[r][t]);
          }
        }
      }
    }
    if (!ok) {
      if (lane == 0) atomicOr(a.err, MOE_DEVERR_STALE);
#pragma unroll
      for (int r = 0; r < kRowsPerItem; ++r)
#pragma unroll
        for (int m = 0; m < TM; ++m) acc[r][m] = 0.f;
    }
#pragma unroll
    for (int r = 0; r < kRowsPerItem; ++r)
#pragma unroll
      for (int m = 0; m < TM; ++m)
#pragma unroll
        for (int off = 16; off; off >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < kRowsPerItem; ++r)
#pragma unroll
        for (int m = 0; m < TM; ++m) part[(it * kRowsPerItem + r) * TM + m] = acc[r][m];
    }
  }
  __syncthreads();
  // y[t][o] = sum over units in order
  for (int i = tid; i < kDownRows * T; i += kThreads) {
    const int r = i / T, t = i - r * T;
    const int o = o0 + r;
    if (o >= a.H) continue;
    const int rp = r / kRowsPerItem, rr = r - rp * kRowsPerItem;
    float v = 0.f;
    for (int u = 0; u < units; ++u) v += part[((u * kPairs + rp) * kRowsPerItem + rr) * TM + t];
    a.y[static_cast<int64_t>(t) * a.H + o] = v;
  }
  if (a.store) {
    // read-through: once every block has written its rows, the misses' slots
    // are complete; the last block publishes their generations
    __shared__ unsigned int s_ticket;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_ticket = atomicAdd(a.ticket, 1u);
    __syncthreads();
    if (s_ticket == gridDim.x - 1) {
      __threadfence();
      int nmiss = 0;
      for (int u = tid; u < units; u += kThreads) {
        const int sl = __ldg(a.units + kUnitHeader + kUnitInts * u);
        if (sl <= -2 && -2 - sl < a.S) {
          a.gen[-2 - sl] = __ldcg(a.sgen + (-2 - sl));
          ++nmiss;
        }
      }
      for (int off = 16; off; off >>= 1) nmiss += __shfl_xor_sync(0xffffffffu, nmiss, off);
      if (lane == 0 && nmiss) {
        atomicAdd(reinterpret_cast<unsigned long long*>(a.stats + kStatTiles),
                  static_cast<unsigned long long>(nmiss) * a.tiles_per_expert);
        atomicAdd(reinterpret_cast<unsigned long long*>(a.stats + kStatBytes),
                  static_cast<unsigned long long>(nmiss) * a.payload);
      }
      if (tid == 0) *a.ticket = 0u;
    }
  }
}

template <int Q, int TM>
cudaError_t launch_tm(const FfnArgs& a, int num_sms, cudaStream_t st) {
  const size_t smem1 = sizeof(float) * static_cast<size_t>(a.T) * a.H;
  const int A = a.T * a.k;
  const int nrows = A + (a.shared ? a.T : 0);
  const int max_units = std::min(a.E, A) + (a.shared ? 1 : 0);
  const size_t smem2 = sizeof(float) * (static_cast<size_t>(nrows) * a.ldh +
                                        static_cast<size_t>(max_units) * kDownRows * TM);
  if (smem1 > 220 * 1024 || smem2 > 220 * 1024) return cudaErrorInvalidValue;
  cudaError_t err;
  if (a.xt == MOE_BF16) {
    err = cudaFuncSetAttribute(gateup_kernel<Q, TM, MOE_BF16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem1));
    if (err != cudaSuccess) return err;
  } else {
    err = cudaFuncSetAttribute(gateup_kernel<Q, TM, MOE_F32>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem1));
    if (err != cudaSuccess) return err;
  }
  err = cudaFuncSetAttribute(down_kernel<Q, TM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem2));
  if (err != cudaSuccess) return err;
  const int items1 = max_units * (std::max(a.I, a.Is) / kRowsPerItem);
  const int grid1 = std::max(1, std::min((items1 + kWarps - 1) / kWarps, num_sms * 2));
  if (a.ev[0]) cudaEventRecord(a.ev[0], st);
  err = a.xt == MOE_BF16 ? pdl_launch(gateup_kernel<Q, TM, MOE_BF16>, dim3(grid1), dim3(kThreads), smem1, st, a)
                         : pdl_launch(gateup_kernel<Q, TM, MOE_F32>, dim3(grid1), dim3(kThreads), smem1, st, a);
  if (err == cudaSuccess) err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (a.ev[1]) cudaEventRecord(a.ev[1], st);
  const int grid2 = (a.H + kDownRows - 1) / kDownRows;
  if (a.ev[2]) cudaEventRecord(a.ev[2], st);
  err = pdl_launch(down_kernel<Q, TM>, dim3(grid2), dim3(kThreads), smem2, st, a);
  if (a.ev[3]) cudaEventRecord(a.ev[3], st);
  return err != cudaSuccess ? err : cudaGetLastError();
}

template <int Q>
cudaError_t launch_q(const FfnArgs& a, int num_sms, cudaStream_t st) {
  if (a.T <= 1) return launch_tm<Q, 1>(a, num_sms, st);
  if (a.T <= 4) return launch_tm<Q, 4>(a, num_sms, st);
  return launch_tm<Q, 8>(a, num_sms, st);
}

}  // namespace

cudaError_t launch_ffn_decode(const FfnArgs& a, int num_sms, cudaStream_t st) {
  if (a.T < 1 || a.T > 8) return cudaErrorInvalidValue;
  if (a.quant == MOE_Q8_0) return launch_q<MOE_Q8_0>(a, num_sms, st);
  return launch_q<MOE_Q4_0>(a, num_sms, st);
}

}  // namespace moe
