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
// Phase 1 (gate/up): one warp item = (unit, rows): row r (one token) or rows
// r, r+1 (several tokens) of the gate and up matrices of one unit (a routed
// expert of the union, or the shared expert), for every token routed to it;
// writes h = silu(g) * u in fp32 to scratch, indexed by expert-major
// assignment (routed) or token (shared).
// Phase 2 (down + combine): one block per SM owns an even run of output rows
// (about H / SMs); warp items = (unit, 2 rows), loaded in batches; each
// item's partial sums (already weighted by the combine weight) go to shared
// memory and are added in unit order, so the output does not depend on
// scheduling and is identical whatever the cache state.
#include <cuda_fp16.h>

#include <mutex>

#include "internal.h"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerItem = 2;   // rows per warp item

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

// Loads from a miss's source: the pinned store, read over the host link.
__device__ __forceinline__ uint4 ld_host(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

// Block metadata of the 16-byte chunk c of a row: Q8_0 the fp16 scale of
// its 32-weight block (chunks 2j and 2j+1 share one), Q4_0 the fp16 scale of
// its block (one per chunk), I4_G64 the bf16 (scale, bias) pair of its
// 64-weight group (chunks 2j and 2j+1), loaded as one 32-bit word.
template <int Q>
__device__ __forceinline__ int meta_off(int c) {
  return Q == MOE_Q4_0 ? 2 * c : (Q == MOE_Q8_0 ? 2 * (c >> 1) : 4 * (c >> 1));
}
template <int Q>
__device__ __forceinline__ uint32_t ld_meta(const uint8_t* row, int c) {
  const uint8_t* p = row + meta_off<Q>(c);
  return Q == MOE_I4_G64 ? __ldg(reinterpret_cast<const uint32_t*>(p))
                         : static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p)));
}
template <int Q>
__device__ __forceinline__ uint32_t ld_meta_host(const uint8_t* row, int c) {
  const uint8_t* p = row + meta_off<Q>(c);
  return Q == MOE_I4_G64 ? __ldcs(reinterpret_cast<const uint32_t*>(p))
                         : static_cast<uint32_t>(__ldcs(reinterpret_cast<const unsigned short*>(p)));
}
// A miss's metadata reaches its slot from the loads the dot products make:
// the lane whose chunk opens a block (every Q4_0 chunk, even chunks of the
// others) stores it, so no copy waits on its own load.
template <int Q>
__device__ __forceinline__ void st_meta(uint8_t* row, int c, uint32_t v) {
  if (Q != MOE_Q4_0 && (c & 1)) return;
  uint8_t* p = row + meta_off<Q>(c);
  if (Q == MOE_I4_G64)
    *reinterpret_cast<uint32_t*>(p) = v;
  else
    *reinterpret_cast<unsigned short*>(p) = static_cast<unsigned short>(v);
}
template <int Q>
__device__ __forceinline__ float meta_scale(uint32_t v) {
  return Q == MOE_I4_G64 ? __uint_as_float(v << 16) : __half2float(__ushort_as_half(static_cast<unsigned short>(v)));
}
template <int Q>
__device__ __forceinline__ float meta_bias(uint32_t v) {
  return Q == MOE_I4_G64 ? __uint_as_float(v & 0xFFFF0000u) : 0.f;
}

// Packed pairs of fp32 (Blackwell's f32x2 add and FMA).
__device__ __forceinline__ unsigned long long f2pack(uint32_t a, uint32_t b) {
  unsigned long long v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(a), "r"(b));
  return v;
}
__device__ __forceinline__ unsigned long long f2packf(float a, float b) {
  unsigned long long v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(a), "f"(b));
  return v;
}
__device__ __forceinline__ float f2sum(unsigned long long v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return a + b;
}
__device__ __forceinline__ unsigned long long f2sub(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2fma(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Dot of one 16-byte Q8_0 chunk (16 weights) with 16 activations. A biased
// byte u = q + 128 becomes the float 2^23 + u by one byte permute; a packed
// subtraction of 2^23 + 128 leaves q exactly, two weights at a time, and
// packed FMAs accumulate even and odd positions separately.
__device__ __forceinline__ float dot_q8(const uint4 w, const float* x) {
  const uint32_t ws[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u,
                          w.w ^ 0x80808080u};
  const unsigned long long bias = f2packf(8388736.0f, 8388736.0f);
  unsigned long long s = 0ull;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const unsigned long long q = f2sub(f2pack(__byte_perm(ws[i], 0x4B000000u, 0x7540u | (2 * h)),
                                                __byte_perm(ws[i], 0x4B000000u, 0x7540u | (2 * h + 1))),
                                         bias);
      s = f2fma(q, f2packf(x[4 * i + 2 * h], x[4 * i + 2 * h + 1]), s);
    }
  return f2sum(s);
}

// Dot of one 16-byte Q4_0 block (32 weights) with activations: xl for
// elements 0..15 (low nibbles), xh for 16..31 (high nibbles); a nibble n
// becomes 2^23 + n, and the packed subtraction of 2^23 + 8 leaves n - 8.
__device__ __forceinline__ float dot_q4(const uint4 w, const float* xl, const float* xh) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  const unsigned long long bias = f2packf(8388616.0f, 8388616.0f);
  unsigned long long s = 0ull;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = ws[i] & 0x0F0F0F0Fu, hi = (ws[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const unsigned long long ql = f2sub(f2pack(__byte_perm(lo, 0x4B000000u, 0x7540u | (2 * h)),
                                                 __byte_perm(lo, 0x4B000000u, 0x7540u | (2 * h + 1))),
                                          bias);
      const unsigned long long qh = f2sub(f2pack(__byte_perm(hi, 0x4B000000u, 0x7540u | (2 * h)),
                                                 __byte_perm(hi, 0x4B000000u, 0x7540u | (2 * h + 1))),
                                          bias);
      s = f2fma(ql, f2packf(xl[4 * i + 2 * h], xl[4 * i + 2 * h + 1]), s);
      s = f2fma(qh, f2packf(xh[4 * i + 2 * h], xh[4 * i + 2 * h + 1]), s);
    }
  }
  return f2sum(s);
}

// Dot of one 16-byte I4_G64 chunk (32 weights, half a group) with its
// activations (xl elements 0..15, xh 16..31): byte j holds elements 2j (low
// nibble) and 2j+1 (high nibble); a nibble n becomes 2^23 + n and the packed
// subtraction of 2^23 leaves n. Returns sum(q * x); the caller adds
// scale * that + bias * sum(x).
__device__ __forceinline__ float dot_u4(const uint4 w, const float* xl, const float* xh) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  const unsigned long long bias = f2packf(8388608.0f, 8388608.0f);
  unsigned long long s = 0ull;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = ws[i] & 0x0F0F0F0Fu, hi = (ws[i] >> 4) & 0x0F0F0F0Fu;
    const float* x8 = i < 2 ? xl + 8 * i : xh + 8 * (i - 2);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const unsigned long long q = f2sub(f2pack(__byte_perm(lo, 0x4B000000u, 0x7540u | b),
                                                __byte_perm(hi, 0x4B000000u, 0x7540u | b)),
                                         bias);
      s = f2fma(q, f2packf(x8[2 * b], x8[2 * b + 1]), s);
    }
  }
  return f2sum(s);
}

__device__ __forceinline__ float sum32(const float* xl, const float* xh) {
  unsigned long long s = 0ull;
  const unsigned long long one = f2packf(1.0f, 1.0f);
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    s = f2fma(f2packf(xl[j], xl[j + 1]), one, s);
    s = f2fma(f2packf(xh[j], xh[j + 1]), one, s);
  }
  return f2sum(s);
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
// Rows per gate/up warp item and blocks per SM the launch asks for. One
// token: one gate and one up row per item, four blocks per SM (64
// registers a thread, a few spilled): twice the warps of two-row items, 13.6
// against 16.6 us a launch on the decode workload (16.0 at three blocks per
// SM). Q4_0 groups of up to four tokens: one row pair, whose nibbles are
// unpacked once per chunk for every token of the group; two blocks per SM.
// Other groups: two rows, two blocks per SM for four tokens (at most 128
// registers, a few spilled), as many blocks as fit for eight.
template <int Q, int TM>
struct GateupRows {
  static constexpr bool kQ4Shared = Q == MOE_Q4_0 && TM > 1 && TM <= 4;
  static constexpr int R = (TM == 1 || kQ4Shared) ? 1 : 2;
  static constexpr int kMinBlocks = TM == 1 ? 4 : (TM == 4 ? 2 : 1);
};
template <int Q, int TM, int XT>
__global__ void __launch_bounds__(kThreads, GateupRows<Q, TM>::kMinBlocks) gateup_kernel(FfnArgs a) {
  extern __shared__ float xs[];  // [T][H] swizzled
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, T = a.T;
  constexpr int RG = GateupRows<Q, TM>::R;  // gate rows (and as many up rows) per warp item
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
  const int per_routed = a.I / RG;
  const int per_shared = a.shared ? a.Is / RG : 0;
  const int items = nu * per_routed + per_shared;
  const int rowbytes = Q == MOE_Q8_0 ? H : H / 2;
  const int nch = rowbytes / 16;
  const int sc_row = (H / 32) * 2;  // scale bytes per row
  for (int it = blockIdx.x * kWarps + warp; it < items; it += gridDim.x * kWarps) {
    int u, r0;
    if (it < nu * per_routed) {
      u = it / per_routed;
      r0 = (it - u * per_routed) * RG;
    } else {
      u = nu;
      r0 = (it - nu * per_routed) * RG;
    }
    const UnitRef U = resolve_unit(a, u);
    const bool ok = unit_ok(a, U);
    const uint8_t* q[2 * RG];
    const uint8_t* s[2 * RG];
#pragma unroll
    for (int r = 0; r < RG; ++r) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        q[m * RG + r] = U.base + U.qoff[m] + static_cast<int64_t>(r0 + r) * rowbytes;
        s[m * RG + r] = U.base + U.soff[m] + static_cast<int64_t>(r0 + r) * sc_row;
      }
    }
    for (int m0 = 0; m0 < U.M; m0 += TM) {
      const int mcount = min(TM, U.M - m0);
      int tok[TM];
#pragma unroll
      for (int m = 0; m < TM; ++m)
        tok[m] = (m < mcount) ? (U.p0 >= 0 ? __ldg(a.plan.perm_tok + U.p0 + m0 + m) : m0 + m) : 0;
      float acc[2 * RG][TM];
#pragma unroll
      for (int r = 0; r < 2 * RG; ++r)
#pragma unroll
        for (int m = 0; m < TM; ++m) acc[r][m] = 0.f;
#pragma unroll(GateupRows<Q, TM>::kQ4Shared ? 1 : 2)
      for (int c = lane; c < nch; c += 32) {
        uint4 w[2 * RG];
        uint32_t mb[2 * RG];
        if (U.miss) {
#pragma unroll
          for (int r = 0; r < 2 * RG; ++r) {
            w[r] = ld_host(q[r] + c * 16);
            mb[r] = ld_meta_host<Q>(s[r], c);
          }
          if (m0 == 0) {
#pragma unroll
            for (int r = 0; r < 2 * RG; ++r) {
              *reinterpret_cast<uint4*>(U.dst + (q[r] - U.base) + c * 16) = w[r];
              st_meta<Q>(U.dst + (s[r] - U.base), c, mb[r]);
            }
          }
        } else {
#pragma unroll
          for (int r = 0; r < 2 * RG; ++r) {
            w[r] = ldg_stream(q[r] + c * 16);
            mb[r] = ld_meta<Q>(s[r], c);
          }
        }
        float d[2 * RG];
#pragma unroll
        for (int r = 0; r < 2 * RG; ++r) d[r] = meta_scale<Q>(mb[r]);
        if constexpr (GateupRows<Q, TM>::kQ4Shared) {
          // the chunk's 32 nibbles of each row unpacked once (as dot_q4
          // does) for every token of the group; each token's products are
          // then summed in dot_q4's order, so the sums are bitwise dot_q4's
          const unsigned long long bias = f2packf(8388616.0f, 8388616.0f);
          unsigned long long qp[2 * RG][16];
#pragma unroll
          for (int r = 0; r < 2 * RG; ++r) {
            const uint32_t ws[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t lo = ws[i] & 0x0F0F0F0Fu, hi = (ws[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                qp[r][4 * i + 2 * h] = f2sub(f2pack(__byte_perm(lo, 0x4B000000u, 0x7540u | (2 * h)),
                                                    __byte_perm(lo, 0x4B000000u, 0x7540u | (2 * h + 1))),
                                             bias);
                qp[r][4 * i + 2 * h + 1] = f2sub(f2pack(__byte_perm(hi, 0x4B000000u, 0x7540u | (2 * h)),
                                                        __byte_perm(hi, 0x4B000000u, 0x7540u | (2 * h + 1))),
                                                 bias);
              }
            }
          }
#pragma unroll
          for (int m = 0; m < TM; ++m) {
            if (m < mcount) {
              const float* xr = xs + tok[m] * H;
              float xl[16], xh[16];
              load_chunk16(xr, 2 * c, xl);
              load_chunk16(xr, 2 * c + 1, xh);
#pragma unroll
              for (int r = 0; r < 2 * RG; ++r) {
                unsigned long long sp = 0ull;
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    sp = f2fma(qp[r][4 * i + 2 * h], f2packf(xl[4 * i + 2 * h], xl[4 * i + 2 * h + 1]), sp);
                    sp = f2fma(qp[r][4 * i + 2 * h + 1], f2packf(xh[4 * i + 2 * h], xh[4 * i + 2 * h + 1]), sp);
                  }
                acc[r][m] = fmaf(d[r], f2sum(sp), acc[r][m]);
              }
            }
          }
        } else {
#pragma unroll
          for (int m = 0; m < TM; ++m) {
            if (m < mcount) {
              const float* xr = xs + tok[m] * H;
              if (Q == MOE_Q8_0) {
                float xv[16];
                load_chunk16(xr, c, xv);
#pragma unroll
                for (int r = 0; r < 2 * RG; ++r)
                  acc[r][m] = fmaf(d[r], dot_q8(w[r], xv), acc[r][m]);
              } else if (Q == MOE_Q4_0) {
                float xl[16], xh[16];
                load_chunk16(xr, 2 * c, xl);
                load_chunk16(xr, 2 * c + 1, xh);
#pragma unroll
                for (int r = 0; r < 2 * RG; ++r)
                  acc[r][m] = fmaf(d[r], dot_q4(w[r], xl, xh), acc[r][m]);
              } else {
                float xl[16], xh[16];
                load_chunk16(xr, 2 * c, xl);
                load_chunk16(xr, 2 * c + 1, xh);
                const float xsum = sum32(xl, xh);
#pragma unroll
                for (int r = 0; r < 2 * RG; ++r)
                  acc[r][m] = fmaf(d[r], dot_u4(w[r], xl, xh), fmaf(meta_bias<Q>(mb[r]), xsum, acc[r][m]));
              }
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2 * RG; ++r)
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
            for (int r = 0; r < RG; ++r)
              a.h[static_cast<int64_t>(hrow) * a.ldh + r0 + r] =
                  silu(acc[r][m]) * acc[RG + r][m];
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------ phase 2
// One block per SM, 16 warps: block b owns output rows [b*rpb, b*rpb + rpb)
// (rpb even, about H / SMs) of every unit. The prologue stages, in one round
// of loads, the h rows (swizzled), the unit table (resolved) and the
// permutation's tokens and weights; each warp then takes its items (unit,
// row pair) in batches whose weight loads are all in flight at once.
constexpr int kDownThreads = 512;
constexpr int kDownWarps = kDownThreads / 32;

struct DUnit {
  const uint8_t* base;  // payload to read
  uint8_t* dst;         // slot being filled (read-through miss) or nullptr
  int M, p0, slot;      // slot: routed slot (S if refused), -1 shared
  uint32_t egen;
  int miss, pad;
};

// Shared-memory layout of the down kernel.
struct DownSmem {
  size_t part, perm, units, total;
};
__host__ __device__ inline DownSmem down_smem(int nrows, int ldh, int cap, int rpb, int TM, int A) {
  DownSmem L{};
  L.part = (static_cast<size_t>(nrows) * ldh * sizeof(float) + 15) & ~size_t(15);
  L.perm = L.part + ((static_cast<size_t>(cap) * rpb * TM * sizeof(float) + 15) & ~size_t(15));
  L.units = L.perm + ((static_cast<size_t>(A) * 8 + 15) & ~size_t(15));
  L.total = L.units + sizeof(DUnit) * static_cast<size_t>(cap);
  return L;
}

template <int TM>
struct DownBatch {
  static constexpr int B = TM == 1 ? 4 : (TM <= 4 ? 2 : 1);
};

template <int Q, int TM>
__global__ void __launch_bounds__(kDownThreads, 1) down_kernel(FfnArgs a, int rpb) {
  extern __shared__ __align__(16) float sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, A = a.T * a.k;
  const int nrows = A + (a.shared ? T : 0);
  const int ldh = a.ldh;
  const int cap = min(a.E, A) + (a.shared ? 1 : 0);
  const DownSmem L = down_smem(nrows, ldh, cap, rpb, TM, A);
  float* hs = sm;                                                        // [nrows][ldh] swizzled
  float* part = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(sm) + L.part);  // [units][rpb][TM]
  int* ptok = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(sm) + L.perm);
  float* pw = reinterpret_cast<float*>(ptok + A);
  DUnit* su = reinterpret_cast<DUnit*>(reinterpret_cast<unsigned char*>(sm) + L.units);
  pdl_wait();
  pdl_trigger();
  const int units = __ldg(a.units);
  // prologue, one round of loads: the unit table's capacity (entries past
  // the count are never used), the permutation, the h rows
  for (int u = tid; u < cap; u += kDownThreads) {
    const UnitRef U = resolve_unit(a, u);
    DUnit r;
    r.base = U.base;
    r.dst = U.miss ? U.dst : nullptr;
    r.M = U.M;
    r.p0 = U.p0;
    r.slot = U.slot;
    r.egen = U.egen;
    r.miss = U.miss ? 1 : 0;
    r.pad = 0;
    su[u] = r;
  }
  for (int i = tid; i < A; i += kDownThreads) {
    ptok[i] = __ldg(a.plan.perm_tok + i);
    pw[i] = __ldg(a.plan.perm_w + i);
  }
  {
    constexpr int kU = 8;
    const int n = nrows * ldh;
    for (int i0 = tid * 4; i0 < n; i0 += kDownThreads * 4 * kU) {
      float4 v[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int i = i0 + j * kDownThreads * 4;
        if (i < n) v[j] = __ldcg(reinterpret_cast<const float4*>(a.h + i));
      }
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int i = i0 + j * kDownThreads * 4;
        if (i < n) {
          const int p = i / ldh, kk = i - p * ldh;
          *reinterpret_cast<float4*>(hs + p * ldh + swz(kk)) = v[j];
        }
      }
    }
  }
  __syncthreads();
  const int o0 = blockIdx.x * rpb;
  const int pairs = rpb / kRowsPerItem;
  const int items = units * pairs;
  constexpr int B = DownBatch<TM>::B;
  for (int j0 = warp; j0 < items; j0 += kDownWarps * B) {
    // the first chunk of every row of the batch, and the slots'
    // generations, all in flight before the first is used
    uint4 w[B][kRowsPerItem];
    uint32_t sb[B][kRowsPerItem];
    uint32_t gb[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      gb[b] = 0u;
#pragma unroll
      for (int r = 0; r < kRowsPerItem; ++r) {
        w[b][r] = make_uint4(0, 0, 0, 0);
        sb[b][r] = 0;
      }
      const int it = j0 + b * kDownWarps;
      if (it >= items) continue;
      const int u = it / pairs, rp = it - u * pairs;
      const DUnit U = su[u];
      const bool routed = U.p0 >= 0;
      gb[b] = (!U.miss && routed && U.slot < a.S) ? __ldg(a.gen + U.slot) : 0u;
      const int K = routed ? a.I : a.Is;
      const int rowbytes = Q == MOE_Q8_0 ? K : K / 2;
      const int64_t qo = routed ? a.g.qoff[2] : a.gs.qoff[2];
      const int64_t so = routed ? a.g.soff[2] : a.gs.soff[2];
      if (lane < rowbytes / 16) {
#pragma unroll
        for (int r = 0; r < kRowsPerItem; ++r) {
          const int o = o0 + rp * kRowsPerItem + r;
          if (o >= a.H) continue;
          const uint8_t* qp = U.base + qo + static_cast<int64_t>(o) * rowbytes + lane * 16;
          const uint8_t* srow = U.base + so + static_cast<int64_t>(o) * (K / 16);
          if (U.miss) {
            w[b][r] = ld_host(qp);
            sb[b][r] = ld_meta_host<Q>(srow, lane);
          } else {
            w[b][r] = ldg_stream(qp);
            sb[b][r] = ld_meta<Q>(srow, lane);
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int it = j0 + b * kDownWarps;
      if (it >= items) break;
      const int u = it / pairs, rp = it - u * pairs;
      const DUnit U = su[u];
      const bool routed = U.p0 >= 0;
      const int K = routed ? a.I : a.Is;
      const int rowbytes = Q == MOE_Q8_0 ? K : K / 2;
      const int nch = rowbytes / 16;
      const int sc_row = (K / 32) * 2;
      const int64_t qo = routed ? a.g.qoff[2] : a.gs.qoff[2];
      const int64_t so = routed ? a.g.soff[2] : a.gs.soff[2];
      const int mcount = U.M;  // <= T <= TM
      int tok[TM], hrow[TM];
      float wt[TM];
#pragma unroll
      for (int m = 0; m < TM; ++m) {
        if (m < mcount) {
          hrow[m] = routed ? U.p0 + m : A + m;
          tok[m] = routed ? ptok[hrow[m]] : m;
          wt[m] = routed ? pw[hrow[m]] : 1.0f;
        } else {
          hrow[m] = 0;
          tok[m] = 0;
          wt[m] = 0.f;
        }
      }
      const uint8_t* q[kRowsPerItem];
      const uint8_t* sp0[kRowsPerItem];
      bool rv[kRowsPerItem];
#pragma unroll
      for (int r = 0; r < kRowsPerItem; ++r) {
        const int o = o0 + rp * kRowsPerItem + r;
        rv[r] = o < a.H;
        q[r] = U.base + qo + static_cast<int64_t>(rv[r] ? o : 0) * rowbytes;
        sp0[r] = U.base + so + static_cast<int64_t>(rv[r] ? o : 0) * sc_row;
      }
      float pm[kRowsPerItem][TM];
#pragma unroll
      for (int r = 0; r < kRowsPerItem; ++r)
#pragma unroll
        for (int m = 0; m < TM; ++m) pm[r][m] = 0.f;
      for (int c = lane; c < nch; c += 32) {
        uint4 wv[kRowsPerItem];
        uint32_t sv[kRowsPerItem];
        if (c == lane) {
#pragma unroll
          for (int r = 0; r < kRowsPerItem; ++r) {
            wv[r] = w[b][r];
            sv[r] = sb[b][r];
          }
        } else {
#pragma unroll
          for (int r = 0; r < kRowsPerItem; ++r) {
            const uint8_t* qp = q[r] + c * 16;
            wv[r] = !rv[r] ? make_uint4(0, 0, 0, 0) : (U.miss ? ld_host(qp) : ldg_stream(qp));
            sv[r] = !rv[r] ? 0u : (U.miss ? ld_meta_host<Q>(sp0[r], c) : ld_meta<Q>(sp0[r], c));
          }
        }
        if (U.miss) {
#pragma unroll
          for (int r = 0; r < kRowsPerItem; ++r) {
            if (!rv[r]) continue;
            *reinterpret_cast<uint4*>(U.dst + (q[r] - U.base) + c * 16) = wv[r];
            st_meta<Q>(U.dst + (sp0[r] - U.base), c, sv[r]);
          }
        }
        float dv[kRowsPerItem];
#pragma unroll
        for (int r = 0; r < kRowsPerItem; ++r) dv[r] = meta_scale<Q>(sv[r]);
#pragma unroll
        for (int m = 0; m < TM; ++m) {
          if (m < mcount) {
            const float* hr = hs + hrow[m] * ldh;
            if (Q == MOE_Q8_0) {
              float hv[16];
              load_chunk16(hr, c, hv);
#pragma unroll
              for (int r = 0; r < kRowsPerItem; ++r) pm[r][m] = fmaf(dv[r], dot_q8(wv[r], hv), pm[r][m]);
            } else if (Q == MOE_Q4_0) {
              float hl[16], hh[16];
              load_chunk16(hr, 2 * c, hl);
              load_chunk16(hr, 2 * c + 1, hh);
#pragma unroll
              for (int r = 0; r < kRowsPerItem; ++r) pm[r][m] = fmaf(dv[r], dot_q4(wv[r], hl, hh), pm[r][m]);
            } else {
              float hl[16], hh[16];
              load_chunk16(hr, 2 * c, hl);
              load_chunk16(hr, 2 * c + 1, hh);
              const float hsum = sum32(hl, hh);
#pragma unroll
              for (int r = 0; r < kRowsPerItem; ++r)
                pm[r][m] = fmaf(dv[r], dot_u4(wv[r], hl, hh), fmaf(meta_bias<Q>(sv[r]), hsum, pm[r][m]));
            }
          }
        }
      }
      // a slot that does not hold the expected generation is refused
      const bool ok = U.miss ? true : (routed ? (U.slot < a.S && gb[b] == U.egen) : a.shared != nullptr);
      float acc[kRowsPerItem][TM];
#pragma unroll
      for (int r = 0; r < kRowsPerItem; ++r)
#pragma unroll
        for (int t = 0; t < TM; ++t) acc[r][t] = 0.f;
      if (ok) {
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
      } else if (lane == 0) {
        atomicOr(a.err, MOE_DEVERR_STALE);
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
          for (int m = 0; m < TM; ++m) part[(u * rpb + rp * kRowsPerItem + r) * TM + m] = acc[r][m];
      }
    }
  }
  __syncthreads();
  // y[t][o] = sum over units in order
  for (int i = tid; i < rpb * T; i += kDownThreads) {
    const int r = i / T, t = i - r * T;
    const int o = o0 + r;
    if (o >= a.H) continue;
    float v = 0.f;
    for (int u = 0; u < units; ++u) v += part[(u * rpb + r) * TM + t];
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
      for (int u = tid; u < units; u += kDownThreads) {
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

// ------------------------------------------------------------ fused kernel
// One persistent launch per layer step, one CTA per SM (a cooperative launch,
// so every CTA is resident and the waits below always end):
//   before the router's results are visible (griddepcontrol.wait): stage the
//     activations and compute the shared expert's gate/up rows into shared
//     memory (they depend on neither the routing nor the cache; nothing
//     global is written before the wait);
//   then each CTA starts asynchronous copies (cp.async) of its down-phase
//     rows of every resident unit into shared memory, which land while
//   phase B runs over every warp of the grid: the routed units' gate/up rows,
//     then the read-through misses' down planes copied from the pinned store
//     into their slots in chunks of at most 8 KiB, tile by tile (a counter
//     per tile: the tile-granular page table of a miss being filled,
//     "Nanite for Experts" §5.4);
//   phase C: once every gate/up row is done (one counter, one release per
//     warp) and the tiles that hold its rows of each miss have landed, each
//     CTA stages h in shared memory and computes its even run of output rows
//     of every unit (as the down kernel), from the prefetched rows;
//   the combine adds the units' partial rows in unit order, so outputs are
//     bitwise those of the two-kernel path; the last CTA publishes the
//     misses' generations and clears the counters.
// Every wait is bounded: past the limit the kernel sets the timeout bit and
// an abort flag that every waiting warp checks, and returns.
template <int TM>
struct FShape {
  static constexpr int kThreads = TM == 1 ? 512 : 256;
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kRowsB = TM == 1 ? 1 : 2;  // gate/up rows per phase-B item
  static constexpr int kBatch = TM == 1 ? 4 : (TM <= 4 ? 4 : 2);  // phase-C items loaded at once
};
constexpr int kCopyChunk = 8192;
constexpr int kSharedEarly = 4;  // shared-expert items a warp computes before the wait
constexpr size_t kFusedSmemMax = 220 * 1024;

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Every lane of the warp calls it: true once *p >= need (each lane has made
// its own acquire load that saw it), false on abort or timeout.
__device__ __noinline__ bool warp_wait_count(const unsigned int* p, unsigned int need, unsigned int* abort_flag,
                                             uint32_t* err, long long limit) {
  const int lane = threadIdx.x & 31;
  const long long t0 = clock64();
  for (unsigned int it = 0;; ++it) {
    const unsigned int v = ld_acquire_u32(p);
    if (__all_sync(0xffffffffu, v >= need)) return true;
    int stop = 0;
    if (lane == 0 && (it & 7u) == 7u) {
      if (ld_relaxed_u32(abort_flag)) {
        stop = 1;
      } else if (clock64() - t0 > limit) {
        atomicOr(err, MOE_DEVERR_TIMEOUT);
        atomicExch(abort_flag, 1u);
        stop = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    __nanosleep(32);
  }
}

// Loads of data written earlier in this launch (h rows, a miss's down plane):
// at L2, never a stale L1 line.
__device__ __forceinline__ uint4 ld_cg16(const void* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }
template <int Q>
__device__ __forceinline__ uint32_t ld_meta_cg(const uint8_t* row, int c) {
  const uint8_t* p = row + meta_off<Q>(c);
  return Q == MOE_I4_G64 ? __ldcg(reinterpret_cast<const unsigned int*>(p))
                         : static_cast<uint32_t>(__ldcg(reinterpret_cast<const unsigned short*>(p)));
}
template <int Q>
__device__ __forceinline__ uint32_t ld_meta_smem(const uint8_t* row, int c) {
  const uint8_t* p = row + meta_off<Q>(c);
  return Q == MOE_I4_G64 ? *reinterpret_cast<const unsigned int*>(p)
                         : static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p));
}
// One bulk copy (the TMA engine) of bytes (a multiple of 16; both addresses
// 16-byte aligned) from global into shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(d),
               "l"(gsrc), "r"(bytes), "r"(b)
               : "memory");
}
// Bounded wait on phase 0 of an mbarrier (every waiting thread observes the
// completion itself); false past the limit, which raises the abort flag.
__device__ __noinline__ bool mbar_wait0(uint64_t* bar, unsigned int* abort_flag, uint32_t* err, long long limit) {
  const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(b)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > limit) {
      atomicOr(err, MOE_DEVERR_TIMEOUT);
      atomicExch(abort_flag, 1u);
      return false;
    }
  }
}

struct FusedArgs {
  unsigned int* sync;  // [0] end ticket, [1] abort, [2] gate/up items done,
                       // [3 + u * max_tiles + t] chunks landed in tile t of unit u's down plane
  int max_tiles;
  int64_t tile_bytes;  // tile of the down-plane copies (the staging tile)
  int rpb;             // output rows per CTA in phase C (even)
  int pf_bytes;        // shared memory for the prefetched down rows
  long long wait_cycles;
};

// Gate/up rows [r0, r0 + ROWS) of unit U (weights at base with the offsets
// of its geometry) for every token routed to it: h = silu(gate . x) *
// (up . x) into h rows (expert-major assignment p0 + m, or token m for the
// shared expert at p0 < 0), or, with hout, into hout[m * ROWS + r] (lane 0;
// the unit's tokens fit one group of TM). A read-through miss (dst set) is
// read from the store and its gate and up rows are written into its slot.
// tok_of: the tokens of the expert-major assignments (shared memory).
template <int Q, int TM, int ROWS>
__device__ __noinline__ void gateup_rows(const FfnArgs& a, const float* xs, const uint8_t* base, uint8_t* dst,
                                            const int64_t* qoff, const int64_t* soff, int M, int p0, int r0,
                                            const int* tok_of, int lane, float* hout) {
  const int H = a.H;
  const int rowbytes = Q == MOE_Q8_0 ? H : H / 2;
  const int nch = rowbytes / 16;
  const int sc_row = (H / 32) * 2;
  const bool miss = dst != nullptr;
  const uint8_t* q[2 * ROWS];
  const uint8_t* sr[2 * ROWS];
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      q[m * ROWS + r] = base + qoff[m] + static_cast<int64_t>(r0 + r) * rowbytes;
      sr[m * ROWS + r] = base + soff[m] + static_cast<int64_t>(r0 + r) * sc_row;
    }
  }
  for (int m0 = 0; m0 < M; m0 += TM) {
    const int mcount = min(TM, M - m0);
    int tok[TM];
#pragma unroll
    for (int m = 0; m < TM; ++m) tok[m] = (m < mcount) ? (p0 >= 0 ? tok_of[p0 + m0 + m] : m0 + m) : 0;
    float acc[2 * ROWS][TM];
#pragma unroll
    for (int r = 0; r < 2 * ROWS; ++r)
#pragma unroll
      for (int m = 0; m < TM; ++m) acc[r][m] = 0.f;
#pragma unroll(ROWS == 1 ? 4 : 2)
    for (int c = lane; c < nch; c += 32) {
      uint4 w[2 * ROWS];
      uint32_t mb[2 * ROWS];
      if (miss) {
#pragma unroll
        for (int r = 0; r < 2 * ROWS; ++r) {
          w[r] = ld_host(q[r] + c * 16);
          mb[r] = ld_meta_host<Q>(sr[r], c);
        }
        if (m0 == 0) {
#pragma unroll
          for (int r = 0; r < 2 * ROWS; ++r) {
            *reinterpret_cast<uint4*>(dst + (q[r] - base) + c * 16) = w[r];
            st_meta<Q>(dst + (sr[r] - base), c, mb[r]);
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < 2 * ROWS; ++r) {
          w[r] = ldg_stream(q[r] + c * 16);
          mb[r] = ld_meta<Q>(sr[r], c);
        }
      }
      float d[2 * ROWS];
#pragma unroll
      for (int r = 0; r < 2 * ROWS; ++r) d[r] = meta_scale<Q>(mb[r]);
#pragma unroll
      for (int m = 0; m < TM; ++m) {
        if (m < mcount) {
          const float* xr = xs + tok[m] * H;
          if (Q == MOE_Q8_0) {
            float xv[16];
            load_chunk16(xr, c, xv);
#pragma unroll
            for (int r = 0; r < 2 * ROWS; ++r) acc[r][m] = fmaf(d[r], dot_q8(w[r], xv), acc[r][m]);
          } else if (Q == MOE_Q4_0) {
            float xl[16], xh[16];
            load_chunk16(xr, 2 * c, xl);
            load_chunk16(xr, 2 * c + 1, xh);
#pragma unroll
            for (int r = 0; r < 2 * ROWS; ++r) acc[r][m] = fmaf(d[r], dot_q4(w[r], xl, xh), acc[r][m]);
          } else {
            float xl[16], xh[16];
            load_chunk16(xr, 2 * c, xl);
            load_chunk16(xr, 2 * c + 1, xh);
            const float xsum = sum32(xl, xh);
#pragma unroll
            for (int r = 0; r < 2 * ROWS; ++r)
              acc[r][m] = fmaf(d[r], dot_u4(w[r], xl, xh), fmaf(meta_bias<Q>(mb[r]), xsum, acc[r][m]));
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 2 * ROWS; ++r)
#pragma unroll
      for (int m = 0; m < TM; ++m)
#pragma unroll
        for (int off = 16; off; off >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < TM; ++m) {
        if (m < mcount) {
#pragma unroll
          for (int r = 0; r < ROWS; ++r) {
            const float hv = silu(acc[r][m]) * acc[ROWS + r][m];
            if (hout)
              hout[(m0 + m) * ROWS + r] = hv;
            else
              a.h[static_cast<int64_t>(p0 >= 0 ? p0 + m0 + m : a.T * a.k + m0 + m) * a.ldh + r0 + r] = hv;
          }
        }
      }
    }
  }
}

// Shared-memory layout of the fused kernel.
struct FusedSmem {
  size_t part, units, perm, order, hsh, pf, total;
};
__host__ __device__ inline FusedSmem fused_smem(int T, int H, int cap, int rpb, int TM, int A, int nrows, int ldh,
                                                int warps, int pf_bytes) {
  FusedSmem L{};
  // region 0: the activations [T][H], later h [nrows][ldh]
  const size_t r0 = static_cast<size_t>(T) * H > static_cast<size_t>(nrows) * ldh ? static_cast<size_t>(T) * H
                                                                                   : static_cast<size_t>(nrows) * ldh;
  L.part = (r0 * sizeof(float) + 15) & ~size_t(15);
  // every region starts on a 16-byte boundary (the prefetched rows are
  // written by 16-byte asynchronous copies and read as 16-byte vectors)
  L.units = L.part + ((static_cast<size_t>(cap) * rpb * TM * sizeof(float) + 15) & ~size_t(15));
  L.perm = L.units + ((sizeof(DUnit) * static_cast<size_t>(cap) + 15) & ~size_t(15));
  L.order = L.perm + ((static_cast<size_t>(A) * 8 + 15) & ~size_t(15));
  L.hsh = L.order + ((sizeof(int) * static_cast<size_t>(2 * cap + 4) + 15) & ~size_t(15));
  L.pf = L.hsh + ((sizeof(float) * static_cast<size_t>(warps) * kSharedEarly * 8 * 2 + 15) & ~size_t(15));
  L.total = L.pf + static_cast<size_t>(pf_bytes);
  return L;
}

// Output rows o0 + 2 rp, +1 of unit U for its tokens, weighted by their
// combine weights and accumulated per token into part[u][row][t]: the rows
// come from pf (this CTA's prefetched down rows of the unit, quants then
// scales) when given, else from the slot (a miss just written in this
// launch: at L2) or the payload. A slot whose generation differs from the
// unit's is refused (nothing accumulated, the stale bit set).
template <int Q, int TM>
__device__ __noinline__ void down_item(const FfnArgs& a, const DUnit& U, int u, int rp, int o0, int rows_cta, int rpb,
                                       const unsigned char* pf, const float* hs, const int* ptok, const float* pw,
                                       float* part, int lane) {
  const int H = a.H, A = a.T * a.k;
  const bool routed = U.p0 >= 0;
  const int K = routed ? a.I : a.Is;
  const int rowbytes = Q == MOE_Q8_0 ? K : K / 2;
  const int nch = rowbytes / 16;
  const int sc_row = (K / 32) * 2;
  const int64_t qo = routed ? a.g.qoff[2] : a.gs.qoff[2];
  const int64_t so = routed ? a.g.soff[2] : a.gs.soff[2];
  const uint8_t* wb = U.miss ? U.dst : U.base;
  const uint32_t gen = (!U.miss && routed && U.slot < a.S) ? __ldg(a.gen + U.slot) : 0u;
  const int mcount = U.M;  // <= T <= TM
  float pm[kRowsPerItem][TM];
#pragma unroll
  for (int r = 0; r < kRowsPerItem; ++r)
#pragma unroll
    for (int m = 0; m < TM; ++m) pm[r][m] = 0.f;
  for (int c = lane; c < nch; c += 32) {
    uint4 wv[kRowsPerItem];
    uint32_t sv[kRowsPerItem];
#pragma unroll
    for (int r = 0; r < kRowsPerItem; ++r) {
      const int lr = rp * kRowsPerItem + r;  // row within the CTA's run
      if (lr >= rows_cta) {
        wv[r] = make_uint4(0, 0, 0, 0);
        sv[r] = 0u;
      } else if (pf) {
        wv[r] = *reinterpret_cast<const uint4*>(pf + lr * rowbytes + c * 16);
        sv[r] = ld_meta_smem<Q>(pf + rows_cta * rowbytes + lr * sc_row, c);
      } else {
        const uint8_t* qp = wb + qo + static_cast<int64_t>(o0 + lr) * rowbytes + c * 16;
        const uint8_t* srow = wb + so + static_cast<int64_t>(o0 + lr) * sc_row;
        wv[r] = U.miss ? ld_cg16(qp) : ldg_stream(qp);
        sv[r] = U.miss ? ld_meta_cg<Q>(srow, c) : ld_meta<Q>(srow, c);
      }
    }
    float dv[kRowsPerItem];
#pragma unroll
    for (int r = 0; r < kRowsPerItem; ++r) dv[r] = meta_scale<Q>(sv[r]);
    for (int m = 0; m < mcount; ++m) {
      const float* hr = hs + (routed ? U.p0 + m : A + m) * a.ldh;
      if (Q == MOE_Q8_0) {
        float hv[16];
        load_chunk16(hr, c, hv);
#pragma unroll
        for (int r = 0; r < kRowsPerItem; ++r) pm[r][m] = fmaf(dv[r], dot_q8(wv[r], hv), pm[r][m]);
      } else if (Q == MOE_Q4_0) {
        float hl[16], hh[16];
        load_chunk16(hr, 2 * c, hl);
        load_chunk16(hr, 2 * c + 1, hh);
#pragma unroll
        for (int r = 0; r < kRowsPerItem; ++r) pm[r][m] = fmaf(dv[r], dot_q4(wv[r], hl, hh), pm[r][m]);
      } else {
        float hl[16], hh[16];
        load_chunk16(hr, 2 * c, hl);
        load_chunk16(hr, 2 * c + 1, hh);
        const float hsum = sum32(hl, hh);
#pragma unroll
        for (int r = 0; r < kRowsPerItem; ++r)
          pm[r][m] = fmaf(dv[r], dot_u4(wv[r], hl, hh), fmaf(meta_bias<Q>(sv[r]), hsum, pm[r][m]));
      }
    }
  }
  const bool ok = U.miss ? true : (routed ? (U.slot < a.S && gen == U.egen) : a.shared != nullptr);
  float acc[kRowsPerItem][TM];
#pragma unroll
  for (int r = 0; r < kRowsPerItem; ++r)
#pragma unroll
    for (int t = 0; t < TM; ++t) acc[r][t] = 0.f;
  if (ok) {
    // weight by the combine weight, accumulate per token (T <= TM)
    for (int m = 0; m < mcount; ++m) {
      const int hrow = routed ? U.p0 + m : A + m;
      const int tok = routed ? ptok[hrow] : m;
      const float wt = routed ? pw[hrow] : 1.0f;
#pragma unroll
      for (int t = 0; t < TM; ++t)
        if (t == tok)
#pragma unroll
          for (int r = 0; r < kRowsPerItem; ++r) acc[r][t] = fmaf(wt, pm[r][m], acc[r][t]);
    }
  } else if (lane == 0) {
    atomicOr(a.err, MOE_DEVERR_STALE);
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
      for (int m = 0; m < TM; ++m) part[(u * rpb + rp * kRowsPerItem + r) * TM + m] = acc[r][m];
  }
}

template <int Q, int TM, int XT>
__global__ void __launch_bounds__(FShape<TM>::kThreads, 1) ffn_fused_kernel(FfnArgs a, FusedArgs f) {
  using FS = FShape<TM>;
  constexpr int kThr = FS::kThreads, kW = FS::kWarps, RB = FS::kRowsB;
  extern __shared__ __align__(16) float fsm[];
  __shared__ __align__(8) uint64_t s_pf_bar;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, T = a.T, A = a.T * a.k;
  const int cap = min(a.E, A) + 1;
  const int rpb = f.rpb;
  const FusedSmem L =
      fused_smem(T, H, cap, rpb, TM, A, A + (a.shared ? T : 0), a.ldh, kW, f.pf_bytes);
  unsigned char* base = reinterpret_cast<unsigned char*>(fsm);
  float* xs = fsm;                                        // [T][H] swizzled
  float* part = reinterpret_cast<float*>(base + L.part);  // [units][rpb][TM]
  DUnit* su = reinterpret_cast<DUnit*>(base + L.units);
  int* ptok = reinterpret_cast<int*>(base + L.perm);
  float* pw = reinterpret_cast<float*>(ptok + A);
  int* pf_off = reinterpret_cast<int*>(base + L.order);   // [cap] prefetched rows of unit u (offset) or -1
  int* miss_of = pf_off + cap;                            // [cap] index among the misses, or -1
  int* s_misc = pf_off + 2 * cap;                         // [0] misses
  float* hsh = reinterpret_cast<float*>(base + L.hsh) + warp * kSharedEarly * 8 * RB;
  unsigned char* pf = base + L.pf;
  unsigned int* abort_flag = f.sync + 1;
  unsigned int* gu_done = f.sync + 2;
  unsigned int* tile_done = f.sync + 3;
  const int gw = blockIdx.x * kW + warp, W = gridDim.x * kW;

  // ---- before the routing is visible: activations and the shared expert.
  // Nothing global is written until the wait: the previous kernel on the
  // stream may still read h and the counters.
  for (int i = tid; i < T * H; i += kThr) {
    const int t = i / H, kk = i - t * H;
    xs[t * H + swz(kk)] = load_act<XT>(a.x, i);
  }
  __syncthreads();
  const int n_sh = a.shared ? a.Is / RB : 0;
  int n_early = 0;
  for (int it = gw; it < n_sh && n_early < kSharedEarly; it += W, ++n_early)
    gateup_rows<Q, TM, RB>(a, xs, a.shared, nullptr, a.gs.qoff, a.gs.soff, T, -1, it * RB, nullptr, lane,
                           hsh + n_early * 8 * RB);
  pdl_wait();
  pdl_trigger();
  unsigned int my_gu = 0;  // gate/up items this warp finished
  {
    int e = 0;
    for (int it = gw; it < n_sh; it += W, ++e, ++my_gu) {
      if (e < n_early) {
        if (lane == 0)
          for (int m = 0; m < T; ++m)
            for (int r = 0; r < RB; ++r)
              a.h[static_cast<int64_t>(A + m) * a.ldh + it * RB + r] = hsh[e * 8 * RB + m * RB + r];
      } else {
        gateup_rows<Q, TM, RB>(a, xs, a.shared, nullptr, a.gs.qoff, a.gs.soff, T, -1, it * RB, nullptr, lane,
                               nullptr);
      }
    }
  }
  // ---- the step's unit table and permutation
  const int n_units = min(__ldg(a.units), cap);
  const int nu = n_units - (a.shared ? 1 : 0);
  for (int u = tid; u < n_units; u += kThr) {
    const UnitRef U = resolve_unit(a, u);
    DUnit r;
    r.base = U.base;
    r.dst = U.miss ? U.dst : nullptr;
    r.M = U.M;
    r.p0 = U.p0;
    r.slot = U.slot;
    r.egen = U.egen;
    r.miss = U.miss ? 1 : 0;
    r.pad = 0;
    su[u] = r;
  }
  for (int i = tid; i < A; i += kThr) {
    ptok[i] = __ldg(a.plan.perm_tok + i);
    pw[i] = __ldg(a.plan.perm_w + i);
  }
  __syncthreads();
  const int o0 = blockIdx.x * rpb;
  const int rows_cta = max(0, min(rpb, H - o0));
  if (tid == 0) {
    // which units' down rows of this CTA are prefetched (resident units,
    // 16-byte aligned rows, as many as fit)
    int nm = 0, at = 0;
    for (int u = 0; u < n_units; ++u) {
      miss_of[u] = su[u].miss ? nm++ : -1;
      const int K = su[u].p0 >= 0 ? a.I : a.Is;
      const int rowbytes = Q == MOE_Q8_0 ? K : K / 2;
      const int qb = rows_cta * rowbytes, sb = rows_cta * (K / 16);
      const bool ok = !su[u].miss && rows_cta > 0 && (K % 256) == 0 && at + qb + sb <= f.pf_bytes;
      pf_off[u] = ok ? at : -1;
      if (ok) at += qb + sb;
    }
    s_misc[0] = nm;
    // the prefetch's barrier, initialised before any thread can wait on it
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&s_pf_bar));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int n_miss = s_misc[0];
  // the prefetch: this CTA's down rows of the resident units, quants then
  // scales, two bulk copies per unit issued by one thread
  if (tid == 0) {
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&s_pf_bar));
    uint32_t total = 0;
    for (int u = 0; u < n_units; ++u) {
      if (pf_off[u] < 0) continue;
      const int K = su[u].p0 >= 0 ? a.I : a.Is;
      total += static_cast<uint32_t>(rows_cta * ((Q == MOE_Q8_0 ? K : K / 2) + K / 16));
    }
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(total) : "memory");
    for (int u = 0; u < n_units; ++u) {
      if (pf_off[u] < 0) continue;
      const bool routed = su[u].p0 >= 0;
      const int K = routed ? a.I : a.Is;
      const int rowbytes = Q == MOE_Q8_0 ? K : K / 2;
      const int qb = rows_cta * rowbytes, sb = rows_cta * (K / 16);
      const uint8_t* qsrc = su[u].base + (routed ? a.g.qoff[2] : a.gs.qoff[2]) + static_cast<int64_t>(o0) * rowbytes;
      const uint8_t* ssrc = su[u].base + (routed ? a.g.soff[2] : a.gs.soff[2]) + static_cast<int64_t>(o0) * (K / 16);
      bulk_g2s(pf + pf_off[u], qsrc, static_cast<uint32_t>(qb), &s_pf_bar);
      bulk_g2s(pf + pf_off[u] + qb, ssrc, static_cast<uint32_t>(sb), &s_pf_bar);
    }
  }

  // the down plane of a miss: quant plane then scale plane, contiguous
  const int64_t dn_off = a.g.qoff[2];
  const int64_t dn_bytes = a.g.qbytes[2] + a.g.sbytes[2];
  const int n_tiles = static_cast<int>((dn_bytes + f.tile_bytes - 1) / f.tile_bytes);
  const int sub = static_cast<int>((f.tile_bytes + kCopyChunk - 1) / kCopyChunk);  // chunks per full tile
  const int64_t chunk = ((f.tile_bytes + sub - 1) / sub + 15) & ~int64_t(15);      // bytes per chunk
  const int copies_per_miss = n_tiles * sub;

  // ---- phase B: routed gate/up rows, then the misses' down-plane chunks
  const int per_routed = a.I / RB;
  const int n_gu = max(0, nu) * per_routed;
  const int n_b = n_gu + n_miss * copies_per_miss;
  for (int it = gw; it < n_b; it += W) {
    if (ld_relaxed_u32(abort_flag)) break;
    if (it < n_gu) {
      const int u = it / per_routed;
      const int r0 = (it - u * per_routed) * RB;
      const DUnit U = su[u];
      const bool ok = U.miss || (U.slot < a.S && __ldg(a.gen + U.slot) == U.egen);
      if (ok)
        gateup_rows<Q, TM, RB>(a, xs, U.base, U.dst, a.g.qoff, a.g.soff, U.M, U.p0, r0, ptok, lane, nullptr);
      else if (lane == 0)
        atomicOr(a.err, MOE_DEVERR_STALE);
      ++my_gu;
    } else {
      const int c = it - n_gu;
      const int mi = c / copies_per_miss, j = c - mi * copies_per_miss;
      const int t = j / sub, sj = j - t * sub;
      int u = 0;
      for (int v = 0; v < n_units; ++v)
        if (miss_of[v] == mi) u = v;
      const int64_t lo = static_cast<int64_t>(t) * f.tile_bytes + sj * chunk;
      const int64_t hi = min(min(static_cast<int64_t>(t + 1) * f.tile_bytes, lo + chunk), dn_bytes);
      const uint8_t* src = su[u].base + dn_off;
      uint8_t* dst = su[u].dst + dn_off;
      for (int64_t o = lo + lane * 16; o < hi; o += 32 * 16)
        *reinterpret_cast<uint4*>(dst + o) = ld_host(src + o);
      if (lo < hi) {  // release: every lane's stores, then the count
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(tile_done + static_cast<int64_t>(u) * f.max_tiles + t, 1u);
      }
    }
  }
  // release of this warp's gate/up rows (lane 0 wrote every h value)
  if (lane == 0 && my_gu) {
    __threadfence();
    atomicAdd(gu_done, my_gu);
  }

  // ---- phase C: output rows [o0, o0 + rpb) of every unit, once every
  // gate/up row is done and, for a miss, the tiles that hold these rows of
  // its down plane have landed; h staged in shared memory (over the
  // activations, no longer needed)
  bool go = true;
  if (warp == 0)
    go = warp_wait_count(gu_done, static_cast<unsigned int>(n_gu + n_sh), abort_flag, a.err, f.wait_cycles);
  for (int u = warp; u < n_units && go; u += kW) {
    if (!su[u].miss || rows_cta == 0) continue;
    const int rowbytes = Q == MOE_Q8_0 ? a.I : a.I / 2;
    const int sc_row = (a.I / 32) * 2;
    const int64_t rng[4] = {static_cast<int64_t>(o0) * rowbytes, static_cast<int64_t>(o0 + rows_cta) * rowbytes - 1,
                            a.g.qbytes[2] + static_cast<int64_t>(o0) * sc_row,
                            a.g.qbytes[2] + static_cast<int64_t>(o0 + rows_cta) * sc_row - 1};
    for (int pr = 0; pr < 4 && go; pr += 2) {
      for (int t = static_cast<int>(rng[pr] / f.tile_bytes); t <= static_cast<int>(rng[pr + 1] / f.tile_bytes) && go;
           ++t) {
        const int64_t tb = min(f.tile_bytes, dn_bytes - static_cast<int64_t>(t) * f.tile_bytes);
        const unsigned int need_t = static_cast<unsigned int>((tb + chunk - 1) / chunk);
        go = warp_wait_count(tile_done + static_cast<int64_t>(u) * f.max_tiles + t, need_t, abort_flag, a.err,
                             f.wait_cycles);
      }
    }
  }
  // every thread observes the prefetch's completion itself (it also drains
  // the copies before any exit)
  go = mbar_wait0(&s_pf_bar, abort_flag, a.err, f.wait_cycles) && go;
  const bool all_go = __syncthreads_and(go) != 0;
  const int nrows = A + (a.shared ? T : 0);
  const int ldh = a.ldh;
  float* hs = fsm;  // [nrows][ldh] swizzled
  if (all_go) {
    constexpr int kU = 4;
    const int n = nrows * ldh;
    for (int i0 = tid * 4; i0 < n; i0 += kThr * 4 * kU) {
      float4 v[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int i = i0 + j * kThr * 4;
        if (i < n) v[j] = __ldcg(reinterpret_cast<const float4*>(a.h + i));
      }
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int i = i0 + j * kThr * 4;
        if (i < n) {
          const int pr = i / ldh, kk = i - pr * ldh;
          *reinterpret_cast<float4*>(hs + pr * ldh + swz(kk)) = v[j];
        }
      }
    }
  }
  __syncthreads();
  const int pairs = rpb / kRowsPerItem;
  const int items = all_go ? n_units * pairs : 0;
  for (int it = warp; it < items; it += kW) {
    const int u = it / pairs, rp = it - u * pairs;
    down_item<Q, TM>(a, su[u], u, rp, o0, rows_cta, rpb, pf_off[u] >= 0 ? pf + pf_off[u] : nullptr, hs, ptok, pw,
                     part, lane);
  }
  __syncthreads();
  // y[t][o] = sum over units in unit order
  for (int i = tid; i < rpb * T; i += kThr) {
    const int r = i / T, t = i - r * T;
    const int o = o0 + r;
    if (o >= H) continue;
    float v = 0.f;
    if (all_go)
      for (int u = 0; u < n_units; ++u) v += part[(u * rpb + r) * TM + t];
    a.y[static_cast<int64_t>(t) * H + o] = v;
  }
  // ---- the last CTA: publish the misses' generations, clear the counters
  __shared__ unsigned int s_ticket;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_ticket = atomicAdd(f.sync, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  __threadfence();
  const bool aborted = ld_relaxed_u32(abort_flag) != 0;
  if (a.store && !aborted) {
    int nmiss = 0;
    for (int u = tid; u < n_units; u += kThr) {
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
  }
  for (int u = 0; u < n_units; ++u)
    if (su[u].miss)
      for (int t = tid; t < n_tiles; t += kThr) tile_done[static_cast<int64_t>(u) * f.max_tiles + t] = 0u;
  __syncthreads();
  if (tid == 0) {
    f.sync[2] = 0u;
    f.sync[1] = 0u;
    f.sync[0] = 0u;
  }
}

template <int Q, int TM>
cudaError_t launch_fused_tm(const FfnArgs& a, const FusedLaunch& fl, cudaStream_t st) {
  using FS = FShape<TM>;
  const int A = a.T * a.k;
  const int cap = std::min(a.E, A) + 1;
  const int nrows = A + (a.shared ? a.T : 0);
  FusedArgs f{};
  f.sync = fl.sync;
  f.max_tiles = fl.max_tiles;
  f.tile_bytes = fl.tile_bytes;
  f.wait_cycles = fl.wait_cycles;
  f.rpb = std::max(2, ((a.H + fl.grid - 1) / fl.grid + 1) & ~1);
  // shared memory for the prefetched down rows: every unit's if it fits
  const int kmax = std::max(a.I, a.Is);
  const size_t want = static_cast<size_t>(cap) * f.rpb * ((Q == MOE_Q8_0 ? kmax : kmax / 2) + kmax / 16);
  const size_t fixed = fused_smem(a.T, a.H, cap, f.rpb, TM, A, nrows, a.ldh, FS::kWarps, 0).total;
  if (fixed > kFusedSmemMax) return cudaErrorInvalidValue;
  f.pf_bytes = static_cast<int>(std::min(want, kFusedSmemMax - fixed) & ~size_t(15));
  const size_t smem = fixed + f.pf_bytes;
  void (*kern)(FfnArgs, FusedArgs) =
      a.xt == MOE_BF16 ? ffn_fused_kernel<Q, TM, MOE_BF16> : ffn_fused_kernel<Q, TM, MOE_F32>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(fl.grid);
  cfg.blockDim = dim3(FS::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = fl.pdl ? 2 : 1;
  if (a.ev[0]) cudaEventRecord(a.ev[0], st);
  err = cudaLaunchKernelEx(&cfg, kern, a, f);
  if (a.ev[1]) cudaEventRecord(a.ev[1], st);
  return err != cudaSuccess ? err : cudaGetLastError();
}

template <int Q>
cudaError_t launch_fused_q(const FfnArgs& a, const FusedLaunch& fl, cudaStream_t st) {
  if (a.T <= 1) return launch_fused_tm<Q, 1>(a, fl, st);
  if (a.T <= 4) return launch_fused_tm<Q, 4>(a, fl, st);
  return launch_fused_tm<Q, 8>(a, fl, st);
}

// Blocks of the gate/up kernel resident on one SM at a dynamic shared memory
// size (the last size asked for is cached per instantiation).
template <int Q, int TM, int XT>
int gateup_blocks_per_sm(size_t smem) {
  static std::mutex mu;
  static size_t last_smem = 0;
  static int last_n = 0;
  std::lock_guard<std::mutex> lock(mu);
  if (last_n == 0 || last_smem != smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gateup_kernel<Q, TM, XT>, kThreads, smem) != cudaSuccess ||
        n < 1)
      n = GateupRows<Q, TM>::kMinBlocks;
    last_smem = smem;
    last_n = n;
  }
  return last_n;
}

template <int Q, int TM>
cudaError_t launch_tm(const FfnArgs& a, int num_sms, cudaStream_t st) {
  const size_t smem1 = sizeof(float) * static_cast<size_t>(a.T) * a.H;
  const int A = a.T * a.k;
  const int nrows = A + (a.shared ? a.T : 0);
  const int max_units = std::min(a.E, A) + (a.shared ? 1 : 0);
  // down: one block per SM, an even number of output rows each
  const int rpb = std::max(2, ((a.H + num_sms - 1) / num_sms + 1) & ~1);
  const int grid2 = (a.H + rpb - 1) / rpb;
  const size_t smem2 = down_smem(nrows, a.ldh, max_units, rpb, TM, A).total;
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
  const int items1 = max_units * (std::max(a.I, a.Is) / GateupRows<Q, TM>::R);
  // one wave: the items are walked grid-stride by the blocks that fit at
  // once (each block stages the step's activations once)
  const int resident = a.xt == MOE_BF16 ? gateup_blocks_per_sm<Q, TM, MOE_BF16>(smem1)
                                        : gateup_blocks_per_sm<Q, TM, MOE_F32>(smem1);
  const int grid1 = std::max(1, std::min((items1 + kWarps - 1) / kWarps, num_sms * resident));
  if (a.ev[0]) cudaEventRecord(a.ev[0], st);
  err = a.xt == MOE_BF16 ? pdl_launch(gateup_kernel<Q, TM, MOE_BF16>, dim3(grid1), dim3(kThreads), smem1, st, a)
                         : pdl_launch(gateup_kernel<Q, TM, MOE_F32>, dim3(grid1), dim3(kThreads), smem1, st, a);
  if (err == cudaSuccess) err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (a.ev[1]) cudaEventRecord(a.ev[1], st);
  if (a.ev[2]) cudaEventRecord(a.ev[2], st);
  err = pdl_launch(down_kernel<Q, TM>, dim3(grid2), dim3(kDownThreads), smem2, st, a, rpb);
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

cudaError_t launch_ffn_decode_fused(const FfnArgs& a, const FusedLaunch& fl, cudaStream_t st) {
  if (a.T < 1 || a.T > 8) return cudaErrorInvalidValue;
  if (a.quant == MOE_Q8_0) return launch_fused_q<MOE_Q8_0>(a, fl, st);
  if (a.quant == MOE_I4_G64) return launch_fused_q<MOE_I4_G64>(a, fl, st);
  return launch_fused_q<MOE_Q4_0>(a, fl, st);
}

cudaError_t launch_ffn_decode(const FfnArgs& a, int num_sms, cudaStream_t st) {
  if (a.T < 1 || a.T > 8) return cudaErrorInvalidValue;
  if (a.quant == MOE_Q8_0) return launch_q<MOE_Q8_0>(a, num_sms, st);
  if (a.quant == MOE_I4_G64) return launch_q<MOE_I4_G64>(a, num_sms, st);
  return launch_q<MOE_Q4_0>(a, num_sms, st);
}

}  // namespace moe
