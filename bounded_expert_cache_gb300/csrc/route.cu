// Router logits, certified top-k, combine weights and the expert-major plan.
//
// "Nanite for Experts" §3.1 and §9: routing is authoritative — the selected
// experts must be the ones the exact router picks, whatever the arithmetic of
// the fast path. The selection is defined on the correctly rounded fp64 value
// of the exact sum sum_i x_i*w_i (+ b); ties go to the lower expert id; the
// selection is ordered by descending logit, then id; combine weights are the
// softmax over the k selected logits ("Paging the Experts" §3.1: top-eight).
//
// Fast path (one launch, one block per expert): each logit is a compensated
// dot product (error-free products by FMA, error-free sums, fp32 error
// accumulator; Ogita, Rump and Oishi, "Accurate sum and dot product", 2005)
// kept as an fp64 value with a rigorous error bound. The last block to finish
// selects the top-k of every token and certifies that the bound intervals of
// consecutive selections (and of the k-th against every other expert) are
// disjoint, so the order of the exact values — and of their correctly rounded
// fp64 images — is the fast order. A token that fails is recomputed exactly:
// every product of a float activation and an fp32 weight is an integer times
// a power of two, so an integer super-accumulator (Kulisch) holds the exact
// sum, which is then rounded to nearest-even fp64 once.
//
// Expert-major plan ("Nanite for Experts" §5.3 union, §5.5 merge into the
// original positions): counts, exclusive offsets, ascending union, and a
// stable (token-ascending) scatter of the assignments.
#include <algorithm>
#include <cfloat>
#include <climits>
#include <mutex>
#include <string>

#include <cuda_bf16.h>

#include "internal.h"
#include "pdl.cuh"
#include "prefill.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteTB = 8;   // tokens per pass of the logits loop
constexpr int kRouteMaxT = 64; // tokens per launch of the small-T router
constexpr int kLimbs = 19;    // 32-bit limbs of the exact accumulator (608 bits)
constexpr int kLsbBias = 298; // -(smallest product LSB exponent): 2^-149 * 2^-149

template <int XT>
__device__ __forceinline__ float load_x(const void* x, size_t i) {
  if (XT == MOE_BF16) {
    uint16_t b = static_cast<const uint16_t*>(x)[i];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  } else {
    return static_cast<const float*>(x)[i];
  }
}

// Four consecutive activations (i a multiple of 4; rows 16-byte aligned).
template <int XT>
__device__ __forceinline__ void load_x4(const void* x, size_t i, float* v) {
  if (XT == MOE_BF16) {
    const uint2 b = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) + i));
    v[0] = __uint_as_float(b.x << 16);
    v[1] = __uint_as_float(b.x & 0xFFFF0000u);
    v[2] = __uint_as_float(b.y << 16);
    v[3] = __uint_as_float(b.y & 0xFFFF0000u);
  } else {
    const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + i));
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  }
}

// Error-free sum: a + b == s + e exactly (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bp = __fsub_rn(s, a);
  float ap = __fsub_rn(s, bp);
  e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

// ------------------------------------------------------------ exact logits
// Integer significand and LSB exponent of a finite float: v = m * 2^e.
__device__ __forceinline__ bool float_parts(float v, uint32_t& m, int& e, bool& neg) {
  uint32_t b = __float_as_uint(v);
  neg = (b >> 31) != 0;
  uint32_t ex = (b >> 23) & 0xFF;
  uint32_t man = b & 0x7FFFFF;
  if (ex == 0xFF) return false;
  if (ex == 0) {
    m = man;
    e = -149;
  } else {
    m = man | 0x800000u;
    e = static_cast<int>(ex) - 150;
  }
  return true;
}

// acc += (neg ? -1 : 1) * mp * 2^(lsb), with lsb >= -298. Limb j holds bits
// [32j, 32j+32) of the sum scaled by 2^298, as a signed carry-save int64.
__device__ __forceinline__ void acc_add(long long* acc, unsigned long long mp, int lsb, bool neg) {
  if (mp == 0) return;
  int s = lsb + kLsbBias;
  int j = s >> 5, b = s & 31;
  unsigned long long lo = mp << b;
  unsigned long long hi = b ? (mp >> (64 - b)) : 0ull;
  long long p0 = static_cast<long long>(lo & 0xFFFFFFFFull);
  long long p1 = static_cast<long long>(lo >> 32);
  long long p2 = static_cast<long long>(hi);
  if (neg) {
    acc[j] -= p0;
    acc[j + 1] -= p1;
    acc[j + 2] -= p2;
  } else {
    acc[j] += p0;
    acc[j + 1] += p1;
    acc[j + 2] += p2;
  }
}

// Bits [lo, lo+64) of a canonical (non-negative, 32-bit limbs) accumulator.
__device__ __forceinline__ unsigned long long acc_bits64(const long long* acc, int lo) {
  unsigned long long r = 0;
  for (int i = 0; i < 64; i += 32) {
    int bit = lo + i;
    // 32 bits starting at `bit` (bit may be negative or unaligned)
    unsigned long long w = 0;
    int j = bit >> 5;  // floor division for negatives too (arithmetic shift)
    int o = bit & 31;
    unsigned long long a0 = (j >= 0 && j < kLimbs) ? static_cast<unsigned long long>(acc[j]) : 0ull;
    unsigned long long a1 = (j + 1 >= 0 && j + 1 < kLimbs) ? static_cast<unsigned long long>(acc[j + 1]) : 0ull;
    w = ((a0 | (a1 << 32)) >> o) & 0xFFFFFFFFull;
    r |= w << i;
  }
  return r;
}

__device__ __forceinline__ bool acc_any_below(const long long* acc, int bit) {
  if (bit <= 0) return false;
  int j = bit >> 5, o = bit & 31;
  for (int i = 0; i < j && i < kLimbs; ++i)
    if (acc[i] != 0) return true;
  if (o && j < kLimbs && (static_cast<unsigned long long>(acc[j]) & ((1ull << o) - 1))) return true;
  return false;
}

// Round the exact accumulated sum to the nearest fp64 (ties to even).
__device__ double acc_round(long long* acc) {
  for (int j = 0; j < kLimbs - 1; ++j) {
    long long carry = acc[j] >> 32;  // arithmetic
    acc[j] -= carry * 4294967296ll;
    acc[j + 1] += carry;
  }
  bool neg = acc[kLimbs - 1] < 0;
  if (neg) {
    for (int j = 0; j < kLimbs; ++j) acc[j] = -acc[j];
    for (int j = 0; j < kLimbs - 1; ++j) {
      long long carry = acc[j] >> 32;
      acc[j] -= carry * 4294967296ll;
      acc[j + 1] += carry;
    }
  }
  int J = kLimbs - 1;
  while (J >= 0 && acc[J] == 0) --J;
  if (J < 0) return 0.0;
  int nb = 64 - __clzll(static_cast<unsigned long long>(acc[J]));
  int P = 32 * J + nb - 1;                       // index of the leading 1
  unsigned long long top = acc_bits64(acc, P - 63);  // leading 1 at bit 63
  unsigned long long mant = top >> 11;           // 53 bits
  bool round = (top >> 10) & 1ull;
  bool sticky = (top & 0x3FFull) != 0 || acc_any_below(acc, P - 63);
  if (round && (sticky || (mant & 1ull))) {
    ++mant;
    if (mant == (1ull << 53)) {
      mant >>= 1;
      ++P;
    }
  }
  double r = ldexp(static_cast<double>(mant), P - 52 - kLsbBias);
  return neg ? -r : r;
}

// Exact correctly rounded logit of one (token, expert), computed by a warp.
// Returns false if an input is not finite.
template <int XT>
__device__ bool warp_exact_logit(const void* x, size_t xoff, const float* wrow, int H,
                                 const float* bias, int e, double& out) {
  const int lane = threadIdx.x & 31;
  long long acc[kLimbs];
#pragma unroll
  for (int j = 0; j < kLimbs; ++j) acc[j] = 0;
  bool ok = true;
  for (int kk = lane; kk < H; kk += 32) {
    uint32_t mx, mw;
    int ex, ew;
    bool nx, nw;
    ok &= float_parts(load_x<XT>(x, xoff + kk), mx, ex, nx);
    ok &= float_parts(wrow[kk], mw, ew, nw);
    if (ok) acc_add(acc, static_cast<unsigned long long>(mx) * mw, ex + ew, nx != nw);
  }
  if (lane == 0 && bias) {
    uint32_t mb;
    int eb;
    bool nb;
    ok &= float_parts(bias[e], mb, eb, nb);
    if (ok) acc_add(acc, mb, eb, nb);
  }
#pragma unroll
  for (int j = 0; j < kLimbs; ++j) {
    long long v = acc[j];
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    acc[j] = v;
  }
  ok = __all_sync(0xffffffffu, ok);
  out = acc_round(acc);
  return ok;
}

// ------------------------------------------------------------ selection
// Selection and certification compare order-preserving integer keys of the
// fp64 logits and of their bound intervals (FP64 compares are slow on this
// GPU; integer ones are not). okey is strictly monotone on non-NaN doubles,
// maps -0 and +0 to the same key and NaN below everything.
__device__ __forceinline__ unsigned long long okey(double x) {
  if (isnan(x)) return 0ull;
  x = x + 0.0;  // -0 -> +0
  const long long b = __double_as_longlong(x);
  return b >= 0 ? (static_cast<unsigned long long>(b) | 0x8000000000000000ull)
                : ~static_cast<unsigned long long>(b);
}
__device__ __forceinline__ double okey_value(unsigned long long k) {
  const unsigned long long b = (k & 0x8000000000000000ull) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k;
  return __longlong_as_double(static_cast<long long>(b));
}

struct TokenKeys {
  const unsigned long long* l;   // [E] logit keys
  const unsigned long long* lo;  // [E] lower-bound keys (rounded down)
  const unsigned long long* hi;  // [E] upper-bound keys (rounded up)
};

__device__ __forceinline__ bool kbetter(unsigned long long v, int e, unsigned long long bv, int be) {
  return v > bv || (v == bv && e < be);
}

// Top-k of one token by a warp: lane owns experts lane, lane+32, ...
// (E <= 32*NPL). Returns the selection in sel and its keys in selk (all lanes;
// descending logit, ties to the lower id) and, if certify, whether the bound
// intervals of consecutive selections and of the k-th against every other
// expert are disjoint.
template <int NPL>
__device__ bool warp_select_keys(const TokenKeys& K, int E, int k, int* sel,
                                 unsigned long long* selk, bool certify) {
  const int lane = threadIdx.x & 31;
  unsigned long long v[NPL];
  uint32_t live = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = i * 32 + lane;
    v[i] = e < E ? __ldcg(K.l + e) : 0ull;
    if (e < E) live |= 1u << i;
  }
  for (int r = 0; r < k; ++r) {
    unsigned long long bv = 0ull;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      if (((live >> i) & 1u) && (be == INT_MAX || kbetter(v[i], i * 32 + lane, bv, be))) {
        bv = v[i];
        be = i * 32 + lane;
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const unsigned long long ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (oe != INT_MAX && (be == INT_MAX || kbetter(ov, oe, bv, be))) {
        bv = ov;
        be = oe;
      }
    }
    sel[r] = be;
    selk[r] = bv;
    if ((be & 31) == lane) live &= ~(1u << (be >> 5));
  }
  if (!certify) return true;
  // bounds of the selection (lane j < k holds selection j's), and the
  // largest upper bound outside it
  unsigned long long my_lo = 0ull, my_hi = 0ull;
  if (lane < k) {
    int sj = 0;
    for (int j = 0; j < k; ++j)
      if (j == lane) sj = sel[j];
    my_lo = __ldcg(K.lo + sj);
    my_hi = __ldcg(K.hi + sj);
  }
  unsigned long long rest = 0ull;
  bool any = false;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    if ((live >> i) & 1u) {
      const unsigned long long h = __ldcg(K.hi + i * 32 + lane);
      rest = (!any || h > rest) ? h : rest;
      any = true;
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, rest, off);
    const int oa = __shfl_xor_sync(0xffffffffu, any ? 1 : 0, off);
    if (oa) {
      rest = (!any || o > rest) ? o : rest;
      any = true;
    }
  }
  // lane j < k-1 checks lower(sel j) > upper(sel j+1); lane k-1 checks the rest
  const unsigned long long next_hi = __shfl_down_sync(0xffffffffu, my_hi, 1);
  bool ok = true;
  if (lane + 1 < k) ok = my_lo > next_hi;
  if (lane == k - 1 && any) ok = my_lo > rest;
  return __all_sync(0xffffffffu, ok);
}

__device__ bool warp_select(const TokenKeys& K, int E, int k, int* sel, unsigned long long* selk,
                            bool certify) {
  if (E <= 32) return warp_select_keys<1>(K, E, k, sel, selk, certify);
  if (E <= 64) return warp_select_keys<2>(K, E, k, sel, selk, certify);
  if (E <= 128) return warp_select_keys<4>(K, E, k, sel, selk, certify);
  if (E <= 256) return warp_select_keys<8>(K, E, k, sel, selk, certify);
  if (E <= 512) return warp_select_keys<16>(K, E, k, sel, selk, certify);
  return warp_select_keys<32>(K, E, k, sel, selk, certify);
}

// ---- decode selection from keys staged in shared memory (l, lo, hi [E])
// One warp round: the warp's best head by the high key word, then the low
// word, then the lowest id (32-bit warp reductions; keys descending, ties
// to the lower expert id). Returns the winning id (or -1) and its key.
__device__ __forceinline__ int warp_round(bool has, unsigned long long v, int id, unsigned long long& key) {
  const uint32_t h32 = has ? static_cast<uint32_t>(v >> 32) : 0u;
  const uint32_t m1 = __reduce_max_sync(0xffffffffu, h32);
  const bool c1 = has && h32 == m1;
  const uint32_t m2 = __reduce_max_sync(0xffffffffu, c1 ? static_cast<uint32_t>(v) : 0u);
  const bool c2 = c1 && static_cast<uint32_t>(v) == m2;
  key = (static_cast<unsigned long long>(m1) << 32) | m2;
  return static_cast<int>(__reduce_min_sync(0xffffffffu, c2 ? static_cast<unsigned>(id) : 0xffffffffu));
}

// Certification of a selection s_idx[k] (the same test as warp_select_keys):
// the bound intervals of consecutive selections and of the k-th against
// every other expert are disjoint. taken[e] marks the selected experts.
__device__ bool warp_certify(const unsigned long long* slo, const unsigned long long* shi,
                             const unsigned char* taken, const int* s_idx, int E, int k) {
  const int lane = threadIdx.x & 31;
  unsigned long long rest = 0ull;
  bool any = false;
#pragma unroll 1
  for (int e = lane; e < E; e += 32) {
    if (taken[e]) continue;
    const unsigned long long h = shi[e];
    rest = (!any || h > rest) ? h : rest;
    any = true;
  }
  const uint32_t rh = __reduce_max_sync(0xffffffffu, any ? static_cast<uint32_t>(rest >> 32) : 0u);
  const uint32_t rl =
      __reduce_max_sync(0xffffffffu, any && static_cast<uint32_t>(rest >> 32) == rh ? static_cast<uint32_t>(rest) : 0u);
  const bool any_rest = __any_sync(0xffffffffu, any);
  const unsigned long long restmax = (static_cast<unsigned long long>(rh) << 32) | rl;
  bool ok = true;
  if (lane + 1 < k) ok = slo[s_idx[lane]] > shi[s_idx[lane + 1]];
  if (lane == k - 1 && any_rest) ok = slo[s_idx[lane]] > restmax;
  return __all_sync(0xffffffffu, ok);
}

// Top-k of one token by one warp (E <= 256): every lane sorts its 8 keys in
// registers once (odd-even transposition), then each round takes the best
// head over the warp and the winning lane pops it. Writes s_idx/s_key and
// marks taken[].
__device__ void warp_select_heads(const unsigned long long* sl, int E, int k, int* s_idx,
                                  unsigned long long* s_key, unsigned char* taken) {
  const int lane = threadIdx.x & 31;
  unsigned long long sv[8];
  int sid[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = i * 32 + lane;
    sv[i] = e < E ? sl[e] : 0ull;
    sid[i] = e < E ? e : -1;
  }
#pragma unroll
  for (int p = 0; p < 8; ++p) {
#pragma unroll
    for (int i = p & 1; i + 1 < 8; i += 2) {
      const bool swap =
          sid[i + 1] >= 0 && (sid[i] < 0 || sv[i + 1] > sv[i] || (sv[i + 1] == sv[i] && sid[i + 1] < sid[i]));
      const unsigned long long x = sv[i], y = sv[i + 1];
      const int ix = sid[i], iy = sid[i + 1];
      sv[i] = swap ? y : x;
      sv[i + 1] = swap ? x : y;
      sid[i] = swap ? iy : ix;
      sid[i + 1] = swap ? ix : iy;
    }
  }
#pragma unroll 1
  for (int r = 0; r < k; ++r) {
    unsigned long long key;
    const int mi = warp_round(sid[0] >= 0, sv[0], sid[0], key);
    if (lane == 0) {
      s_idx[r] = mi;
      s_key[r] = key;
      taken[mi] = 1;
    }
    const bool pop = sid[0] == mi;
#pragma unroll
    for (int i = 0; i < 7; ++i) {
      sv[i] = pop ? sv[i + 1] : sv[i];
      sid[i] = pop ? sid[i + 1] : sid[i];
    }
    sv[7] = pop ? 0ull : sv[7];
    sid[7] = pop ? -1 : sid[7];
  }
  __syncwarp();
}

// Top-k (k <= 8) of one token by the whole block (E <= 256): warp w selects
// the top k of experts 32w .. 32w+31 (one key per lane), then warp 0 merges
// the 8k candidates (two per lane). Called by every thread of the block;
// s_idx/s_key/taken are written by warp 0.
__device__ void block_select_tournament(const unsigned long long* sl, int E, int k, int* cand_idx,
                                        unsigned long long* cand_key, int* s_idx, unsigned long long* s_key,
                                        unsigned char* taken) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {
    const int e = warp * 32 + lane;
    const unsigned long long v = e < E ? sl[e] : 0ull;
    bool has = e < E;
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
      unsigned long long key;
      const int mi = warp_round(has, v, e, key);
      if (lane == 0) {
        cand_idx[warp * 8 + r] = mi;
        cand_key[warp * 8 + r] = key;
      }
      if (e == mi) has = false;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // candidates lane and lane + 32 (each warp's list is in order)
    unsigned long long a = cand_key[lane], b = cand_key[lane + 32];
    const int ia = (lane % 8) < k ? cand_idx[lane] : -1, ib = (lane % 8) < k ? cand_idx[lane + 32] : -1;
    bool ha = ia >= 0, hb = ib >= 0;
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
      const bool useb = hb && (!ha || b > a || (b == a && ib < ia));
      unsigned long long key;
      const int mi = warp_round(ha || hb, useb ? b : a, useb ? ib : ia, key);
      if (lane == 0) {
        s_idx[r] = mi;
        s_key[r] = key;
        taken[mi] = 1;
      }
      if ((useb ? ib : ia) == mi && (ha || hb)) {
        if (useb)
          hb = false;
        else
          ha = false;
      }
    }
    __syncwarp();
  }
}

// Combine weights of a selection held in shared memory (same arithmetic and
// order as warp_write_selection); also keeps the weights in shared memory.
__device__ void fast_write_selection(const int* s_idx, const unsigned long long* s_key, int k, int32_t* idx,
                                     float* w, float* s_w) {
  const int lane = threadIdx.x & 31;
  float z = 0.f;
  if (lane < k) z = expf(static_cast<float>(okey_value(s_key[lane]) - okey_value(s_key[0])));
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, z, j);  // fixed order
  if (lane < k) {
    const float wl = z / sum;
    idx[lane] = s_idx[lane];
    w[lane] = wl;
    s_w[lane] = wl;
  }
}

// Combine weights of a selection: softmax over the k selected logits, the
// differences taken in fp64 and exponentiated in fp32.
__device__ void warp_write_selection(const int* sel, const unsigned long long* selk, int k,
                                     int32_t* idx, float* w) {
  const int lane = threadIdx.x & 31;
  float z = 0.f;
  int sj = 0;
  unsigned long long kj = selk[0];
  for (int j = 0; j < k; ++j)
    if (j == lane) {
      sj = sel[j];
      kj = selk[j];
    }
  if (lane < k) z = expf(static_cast<float>(okey_value(kj) - okey_value(selk[0])));
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, z, j);  // fixed order
  if (lane < k) {
    idx[lane] = sj;
    w[lane] = z / sum;
  }
}

// ------------------------------------------------------------ block scan
// In-place exclusive scan of n ints in shared memory by the whole block.
template <int NT>
__device__ int block_exclusive_scan(int* data, int n, int* scratch) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + NT - 1) / NT;
  const int b0 = tid * per;
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (b0 + i < n) local += data[b0 + i];
  int incl = local;
  for (int off = 1; off < 32; off <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = lane < NW ? scratch[lane] : 0;
    int vi = v;
    for (int off = 1; off < 32; off <<= 1) {
      int o = __shfl_up_sync(0xffffffffu, vi, off);
      if (lane >= off) vi += o;
    }
    if (lane < NW) scratch[lane] = vi - v;  // exclusive warp offsets
    if (lane == NW - 1) scratch[NW] = vi;   // total
  }
  __syncthreads();
  int run = scratch[warp] + incl - local;
  for (int i = 0; i < per; ++i) {
    if (b0 + i < n) {
      int v = data[b0 + i];
      data[b0 + i] = run;
      run += v;
    }
  }
  int total = scratch[NW];
  __syncthreads();
  return total;
}


// Expert-major plan of A = T*k assignments (a = t*k + j) by one block of NT
// threads. smem: counts[E] cursor[E] wcount[NW*E] scratch[NW+1].
template <int NT>
__device__ void plan_block(const int32_t* idx, const float* w, int A, int k, int E,
                           const moe_plan_t& P, int* smem, uint32_t* err) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* counts = smem;
  int* cursor = counts + E;
  int* wcount = cursor + E;
  int* scratch = wcount + NW * E;
  for (int e = tid; e < E; e += NT) counts[e] = 0;
  __syncthreads();
  for (int a = tid; a < A; a += NT) {
    int e = __ldcg(idx + a);
    if (e >= 0 && e < E)
      atomicAdd(&counts[e], 1);
    else
      atomicOr(err, MOE_DEVERR_BADIDX);
  }
  __syncthreads();
  // ascending union
  for (int e = tid; e < E; e += NT) {
    P.counts[e] = counts[e];
    cursor[e] = counts[e] > 0 ? 1 : 0;
  }
  __syncthreads();
  const int nu = block_exclusive_scan<NT>(cursor, E, scratch);
  for (int e = tid; e < E; e += NT)
    if (counts[e] > 0) P.uniq[cursor[e]] = e;
  if (tid == 0) *P.n_uniq = nu;
  __syncthreads();
  // offsets
  for (int e = tid; e < E; e += NT) cursor[e] = counts[e];
  __syncthreads();
  const int total = block_exclusive_scan<NT>(cursor, E, scratch);
  for (int e = tid; e < E; e += NT) P.offsets[e] = cursor[e];
  if (tid == 0) P.offsets[E] = total;
  __syncthreads();
  // stable scatter, NT assignments at a time in assignment order; a token
  // holds an expert at most once, so assignment order within an expert is
  // token order
  for (int base = 0; base < A; base += NT) {
    for (int i = tid; i < NW * E; i += NT) wcount[i] = 0;
    __syncthreads();
    const int a = base + tid;
    int e = (a < A) ? __ldcg(idx + a) : -1;
    const bool valid = e >= 0 && e < E;
    const int key = valid ? e : -1 - lane;  // invalid lanes never share a group
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const bool leader = (__ffs(peers) - 1) == lane;
    if (valid && leader) wcount[warp * E + e] = __popc(peers);
    __syncthreads();
    if (valid) {
      int pos = cursor[e] + rank;
      for (int w2 = 0; w2 < warp; ++w2) pos += wcount[w2 * E + e];
      P.perm_tok[pos] = a / k;
      P.perm_rank[pos] = a % k;
      P.perm_w[pos] = __ldcg(w + a);
      P.inv[a] = pos;
    }
    __syncthreads();
    for (int e2 = tid; e2 < E; e2 += NT) {
      int add = 0;
      for (int w2 = 0; w2 < NW; ++w2) add += wcount[w2 * E + e2];
      cursor[e2] += add;
    }
    __syncthreads();
  }
}


// ------------------------------------------------------------ on-device admission
__device__ __forceinline__ unsigned long long splitmix64_next(unsigned long long& st) {
  unsigned long long z = (st += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Cache resolve of one step by one warp, the same policy as the host slot
// manager ("MawForge" §IV-C materialise into an available slot and update the
// route-to-slot map; "Paging the Experts" §3.2 entries pinned per layer,
// §4.1 LRU and seeded random eviction): resident experts of the union are
// touched in ascending id, then missing experts are admitted in ascending id,
// one tick per access; a miss takes the lowest free slot, else the LRU victim
// (oldest tick) or cand[next() mod n] over resident experts outside the
// union listed by slot. The layer's slot state and the union's page-table
// entries are read once into shared memory, decided there, and written back;
// the warp then writes the fill list, the FFN's unit table, and resets the
// staging counters.
__host__ __device__ constexpr size_t admit_smem_bytes(int E, int S, int max_units) {
  return 8 * static_cast<size_t>(S)                    // last
         + 4 * static_cast<size_t>(S) * 2              // owner, sgen
         + 4 * static_cast<size_t>((E + 31) / 32)      // union bitmap
         + 4 * static_cast<size_t>(max_units) * 2 + 16;  // union ids, their slots
}

// Inputs another warp of the block may have staged in shared memory before
// the admission runs (the decode router's last block does so while it
// selects): the slot state, the layer's page table, and the plan's union,
// counts and offsets. Null pointers / false mean "read from global memory".
struct AdmitStaged {
  bool slots = false;        // last/owner/sgen already in the admission's smem
  const int* pt = nullptr;   // [E] page table
  int nu = 0;
  const int* uniq = nullptr;  // [nu] union, ascending
  const int* cnt = nullptr;   // [E] assignments per expert
  const int* off = nullptr;   // [E] first expert-major assignment per expert
  unsigned long long tick = 0, rng = 0;
  bool have_tick = false;
};

// Asynchronous copies global -> shared (4 or 8 bytes, naturally aligned).
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<unsigned>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(static_cast<unsigned>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Every block of the decode router copies the layer's cache state (slot
// state, page table, tick and generator state) into the admission area of
// its shared memory when it starts; only the last block uses it, but the
// copies are small and have landed by the time the tail needs them.
__device__ void admit_stage_async(const AdmitArgs& A, unsigned char* smem, int* pt_s, unsigned long long* tick_rng) {
  const int S = A.S;
  const DevCacheLayer c = A.c;
  unsigned long long* s_last = reinterpret_cast<unsigned long long*>(smem);
  int* s_owner = reinterpret_cast<int*>(s_last + S);
  uint32_t* s_sgen = reinterpret_cast<uint32_t*>(s_owner + S);
  for (int i = threadIdx.x; i < S; i += blockDim.x) {
    cp_async8(s_last + i, c.last + i);
    cp_async4(s_owner + i, c.owner + i);
    cp_async4(s_sgen + i, c.sgen + i);
  }
  for (int e = threadIdx.x; e < A.E; e += blockDim.x) cp_async4(pt_s + e, c.pt + e);
  if (threadIdx.x == 0) {
    cp_async8(tick_rng, c.tick);
    cp_async8(tick_rng + 1, c.rng);
  }
  cp_async_commit();
}

__device__ void admit_warp(const AdmitArgs& A, const moe_plan_t& P, unsigned char* smem,
                           uint32_t* err, const AdmitStaged& st = AdmitStaged()) {
  const int lane = threadIdx.x & 31;
  const int E = A.E, S = A.S;
  const DevCacheLayer c = A.c;
  const int nu = st.uniq ? st.nu : __ldcg(P.n_uniq);
  unsigned long long* s_last = reinterpret_cast<unsigned long long*>(smem);
  int* s_owner = reinterpret_cast<int*>(s_last + S);
  uint32_t* s_sgen = reinterpret_cast<uint32_t*>(s_owner + S);
  unsigned* bm = reinterpret_cast<unsigned*>(s_sgen + S);
  int* uq = reinterpret_cast<int*>(bm + (E + 31) / 32);
  int* upt = uq + nu;
  const int nwords = (E + 31) / 32;
  for (int w = lane; w < nwords; w += 32) bm[w] = 0u;
  // global state is read in batches of kAdmB entries a lane, every load of a
  // batch issued before the first is used
  constexpr int kAdmB = 8;
  if (!st.slots) {
    for (int s0 = 0; s0 < S; s0 += 32 * kAdmB) {
      unsigned long long vl[kAdmB];
      int vo[kAdmB];
      uint32_t vg[kAdmB];
#pragma unroll
      for (int j = 0; j < kAdmB; ++j) {
        const int s = s0 + 32 * j + lane;
        vl[j] = s < S ? __ldcg(c.last + s) : 0ull;
        vo[j] = s < S ? __ldcg(c.owner + s) : 0;
        vg[j] = s < S ? __ldcg(c.sgen + s) : 0u;
      }
#pragma unroll
      for (int j = 0; j < kAdmB; ++j) {
        const int s = s0 + 32 * j + lane;
        if (s < S) {
          s_last[s] = vl[j];
          s_owner[s] = vo[j];
          s_sgen[s] = vg[j];
        }
      }
    }
  }
  __syncwarp();
  if (st.uniq && st.pt) {
    // staged in shared memory: nothing to overlap
    for (int u = lane; u < nu; u += 32) {
      const int e = st.uniq[u];
      uq[u] = e;
      upt[u] = st.pt[e];
      atomicOr(&bm[e >> 5], 1u << (e & 31));
    }
  } else {
    for (int u0 = 0; u0 < nu; u0 += 32 * kAdmB) {
      int ve[kAdmB], vp[kAdmB];
#pragma unroll
      for (int j = 0; j < kAdmB; ++j) {
        const int u = u0 + 32 * j + lane;
        ve[j] = u < nu ? (st.uniq ? st.uniq[u] : __ldcg(P.uniq + u)) : 0;
      }
#pragma unroll
      for (int j = 0; j < kAdmB; ++j) {
        const int u = u0 + 32 * j + lane;
        vp[j] = u < nu ? (st.pt ? st.pt[ve[j]] : __ldcg(c.pt + ve[j])) : 0;
      }
#pragma unroll
      for (int j = 0; j < kAdmB; ++j) {
        const int u = u0 + 32 * j + lane;
        if (u < nu) {
          uq[u] = ve[j];
          upt[u] = vp[j];
          atomicOr(&bm[ve[j] >> 5], 1u << (ve[j] & 31));
        }
      }
    }
  }
  __syncwarp();
  auto in_u = [&](int o) { return o >= 0 && ((bm[o >> 5] >> (o & 31)) & 1u); };
  // counts before any change, so a refused step leaves the state untouched
  int nmiss = 0, nfree = 0, res_in_u = 0;
  for (int u0 = 0; u0 < nu; u0 += 32) {
    const int u = u0 + lane;
    nmiss += __popc(__ballot_sync(0xffffffffu, u < nu && upt[u] < 0));
  }
  for (int s0 = 0; s0 < S; s0 += 32) {
    const int s = s0 + lane;
    const int o = s < S ? s_owner[s] : -2;
    nfree += __popc(__ballot_sync(0xffffffffu, o == -1));
    res_in_u += __popc(__ballot_sync(0xffffffffu, in_u(o)));
  }
  const int cand0 = (S - nfree) - res_in_u;
  if (nu > S || (A.policy == MOE_RANDOM && nmiss > nfree + cand0)) {
    if (lane == 0) {
      atomicOr(err, MOE_DEVERR_CAPACITY);
      A.units[0] = 0;
      A.fills[0] = 0;
    }
    return;
  }
  unsigned long long tick = st.have_tick ? st.tick : __ldcg(c.tick);
  // hits in ascending id, consecutive ticks
  for (int u0 = 0; u0 < nu; u0 += 32) {
    const int u = u0 + lane;
    const int slot = u < nu ? upt[u] : -1;
    const unsigned hm = __ballot_sync(0xffffffffu, slot >= 0);
    if (slot >= 0) s_last[slot] = tick + 1 + __popc(hm & ((1u << lane) - 1u));
    tick += __popc(hm);
  }
  __syncwarp();
  // misses in ascending id, one at a time
  unsigned long long rng = st.have_tick ? st.rng : __ldcg(c.rng);
  int nfill = 0, nevict = 0;
  for (int u0 = 0; u0 < nu; u0 += 32) {
    // the chunk's misses, in ascending unit order (a miss changes only its own entry)
    unsigned mm = __ballot_sync(0xffffffffu, u0 + lane < nu && upt[u0 + lane] < 0);
    while (mm) {
      const int u = u0 + __ffs(mm) - 1;
      mm &= mm - 1;
      const int e = uq[u];
      ++tick;
      int slot = -1;
      for (int s0 = 0; s0 < S && slot < 0; s0 += 32) {
        const int s = s0 + lane;
        const unsigned fm = __ballot_sync(0xffffffffu, s < S && s_owner[s] < 0);
        if (fm) slot = s0 + __ffs(fm) - 1;
      }
      if (slot < 0) {
        if (A.policy == MOE_LRU) {
          unsigned long long best = ~0ull;
          int bs = INT_MAX;
          for (int s = lane; s < S; s += 32) {
            const unsigned long long v = s_last[s];
            if (v < best || (v == best && s < bs)) {
              best = v;
              bs = s;
            }
          }
          for (int off = 16; off; off >>= 1) {
            const unsigned long long ov = __shfl_xor_sync(0xffffffffu, best, off);
            const int os = __shfl_xor_sync(0xffffffffu, bs, off);
            if (ov < best || (ov == best && os < bs)) {
              best = ov;
              bs = os;
            }
          }
          slot = bs;
        } else {
          int n = 0;
          for (int s0 = 0; s0 < S; s0 += 32) {
            const int s = s0 + lane;
            const int o = s < S ? s_owner[s] : -1;
            n += __popc(__ballot_sync(0xffffffffu, o >= 0 && !in_u(o)));
          }
          const unsigned long long r = splitmix64_next(rng);
          int target = static_cast<int>(r % static_cast<unsigned long long>(n));
          for (int s0 = 0; s0 < S && slot < 0; s0 += 32) {
            const int s = s0 + lane;
            const int o = s < S ? s_owner[s] : -1;
            unsigned cm = __ballot_sync(0xffffffffu, o >= 0 && !in_u(o));
            const int pc = __popc(cm);
            if (target < pc) {
              for (int i = 0; i < target; ++i) cm &= cm - 1;
              slot = s0 + __ffs(cm) - 1;
            } else {
              target -= pc;
            }
          }
        }
        if (lane == 0) c.pt[s_owner[slot]] = -1;  // victims are never in the union
        ++nevict;
      }
      if (lane == 0) {
        s_owner[slot] = e;
        s_sgen[slot] += 1u;
        s_last[slot] = tick;
        upt[u] = -2 - slot;  // filled this step
        A.fills[1 + 2 * nfill] = e;
        A.fills[2 + 2 * nfill] = slot;
        A.done[nfill] = 0u;
      }
      ++nfill;
      __syncwarp();
    }
  }
  // write back the slot state and the union's page-table entries
  for (int s = lane; s < S; s += 32) {
    c.last[s] = s_last[s];
    c.owner[s] = s_owner[s];
    c.sgen[s] = s_sgen[s];
  }
  long long assignments = 0;
  // unit table: routed units in union order, then the shared expert
  auto unit_entry = [&](int u, int cnt, int off) {
    const int e = uq[u];
    const bool was_miss = upt[u] <= -2;
    const int slot = was_miss ? -2 - upt[u] : upt[u];
    assignments += cnt;
    c.pt[e] = slot;
    c.ptgen[e] = s_sgen[slot];
    int* U = A.units + kUnitHeader + kUnitInts * u;
    const bool filled = A.read_through && was_miss;
    U[0] = filled ? -2 - slot : slot;
    U[1] = off;
    U[2] = cnt;
    U[3] = filled ? e : static_cast<int>(s_sgen[slot]);
  };
  if (st.cnt && st.off) {
    for (int u = lane; u < nu; u += 32) unit_entry(u, st.cnt[uq[u]], st.off[uq[u]]);
  } else {
    for (int u0 = 0; u0 < nu; u0 += 32 * kAdmB) {
      int vc[kAdmB], vo[kAdmB];
#pragma unroll
      for (int j = 0; j < kAdmB; ++j) {
        const int u = u0 + 32 * j + lane;
        const int e = u < nu ? uq[u] : 0;
        vc[j] = u < nu ? (st.cnt ? st.cnt[e] : __ldcg(P.counts + e)) : 0;
        vo[j] = u < nu ? (st.off ? st.off[e] : __ldcg(P.offsets + e)) : 0;
      }
#pragma unroll
      for (int j = 0; j < kAdmB; ++j) {
        const int u = u0 + 32 * j + lane;
        if (u < nu) unit_entry(u, vc[j], vo[j]);
      }
    }
  }
  for (int off = 16; off; off >>= 1) assignments += __shfl_xor_sync(0xffffffffu, assignments, off);
  if (lane == 0) {
    if (A.has_shared) {
      int* U = A.units + kUnitHeader + kUnitInts * nu;
      U[0] = -1;
      U[1] = -1;
      U[2] = A.T;
      U[3] = 0;
    }
    A.units[0] = nu + (A.has_shared ? 1 : 0);
    A.fills[0] = nfill;
    c.tick[0] = tick;
    c.rng[0] = rng;
    c.stats[kStatSteps] += 1;
    c.stats[kStatHits] += assignments - nfill;
    c.stats[kStatMisses] += nfill;
    c.stats[kStatEvictions] += nevict;
    c.stats[kStatMaterialized] += static_cast<long long>(nfill) * A.payload;
  }
}

// Expert-major plan of A <= 32 assignments by one warp (every decode step):
// same outputs as plan_block. smem: counts[E], offsets[E].
__device__ void plan_warp(const int32_t* idx, const float* w, int A, int k, int E,
                          const moe_plan_t& P, int* smem, uint32_t* err, int* uniq_s = nullptr,
                          int* nu_s = nullptr) {
  const int lane = threadIdx.x & 31;
  int* cnt = smem;
  int* off = smem + E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const bool live = lane < A;
  int e = live ? idx[lane] : -1;  // global (written before) or shared memory
  const bool valid = live && e >= 0 && e < E;
  if (live && !valid) atomicOr(err, MOE_DEVERR_BADIDX);
  const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1 - lane);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid && (__ffs(peers) - 1) == lane) cnt[e] = __popc(peers);
  __syncwarp();
  // exclusive scans of counts and of (count > 0) over the experts; lane owns
  // a contiguous range of experts
  const int per = (E + 31) / 32, b0 = lane * per;
  int sc = 0, sn = 0;
  for (int i = 0; i < per; ++i)
    if (b0 + i < E) {
      sc += cnt[b0 + i];
      sn += cnt[b0 + i] > 0;
    }
  int ic = sc, in = sn;
  for (int d = 1; d < 32; d <<= 1) {
    const int oc = __shfl_up_sync(0xffffffffu, ic, d);
    const int on = __shfl_up_sync(0xffffffffu, in, d);
    if (lane >= d) {
      ic += oc;
      in += on;
    }
  }
  int rc = ic - sc, rn = in - sn;
  for (int i = 0; i < per; ++i) {
    const int ee = b0 + i;
    if (ee < E) {
      const int c = cnt[ee];
      off[ee] = rc;
      P.counts[ee] = c;
      P.offsets[ee] = rc;
      if (c > 0) {
        if (uniq_s) uniq_s[rn] = ee;
        P.uniq[rn++] = ee;
      }
      rc += c;
    }
  }
  if (lane == 31) {
    P.offsets[E] = ic;
    *P.n_uniq = in;
    if (nu_s) *nu_s = in;
  }
  __syncwarp();
  if (valid) {
    const int pos = off[e] + rank;  // lanes are assignments in token order
    P.perm_tok[pos] = lane / k;
    P.perm_rank[pos] = lane % k;
    P.perm_w[pos] = w[lane];
    P.inv[lane] = pos;
  }
}

constexpr int kPlanThreads = 256;

size_t plan_smem_bytes(int E) {
  return sizeof(int) * (2 * E + (kPlanThreads / 32) * E + kPlanThreads / 32 + 1);
}

// ------------------------------------------------------------ decode tail
// Shared-memory layout of the router's last block on the decode fast path
// (T*k <= 32 assignments, E <= 256): admission scratch, the plan's counts and
// offsets, the layer's page table, and the selection.
struct FastTailLayout {
  size_t admit, plan, pt, key, idx, w, uniq, tick, nu, cand, keys, taken, one, total;
};
__host__ __device__ constexpr size_t r16(size_t v) { return (v + 15) & ~size_t(15); }

// Scratch of the one-token tail: candidate keys [E] and ids [E], per-warp
// maxima and reductions, counters, the slots hit by the step [S] and the
// slot of each miss.
struct OneTokenScratch {
  unsigned long long* ckey;   // [E]
  int* cid;                   // [E]
  unsigned long long* wrest;  // [kRouteWarps] largest upper bound outside the selection
  uint32_t* wmax;             // [kRouteWarps]
  int* cnt;                   // [8]: 0 candidates, 1 certified, 2 free slots
  unsigned char* hit;         // [S]
  int* mslot;                 // [32] slot of the r-th miss
};
__host__ __device__ constexpr size_t one_token_scratch_bytes(int E, int S) {
  return 8 * static_cast<size_t>(E) + r16(4 * static_cast<size_t>(E)) + 8 * kRouteWarps + 4 * kRouteWarps +
         32 + r16(static_cast<size_t>(S)) + 4 * 32;
}
__device__ inline OneTokenScratch one_token_scratch(unsigned char* p, int E, int S) {
  OneTokenScratch o;
  o.ckey = reinterpret_cast<unsigned long long*>(p);
  p += 8 * static_cast<size_t>(E);
  o.cid = reinterpret_cast<int*>(p);
  p += r16(4 * static_cast<size_t>(E));
  o.wrest = reinterpret_cast<unsigned long long*>(p);
  p += 8 * kRouteWarps;
  o.wmax = reinterpret_cast<uint32_t*>(p);
  p += 4 * kRouteWarps;
  o.cnt = reinterpret_cast<int*>(p);
  p += 32;
  o.hit = p;
  p += r16(static_cast<size_t>(S));
  o.mslot = reinterpret_cast<int*>(p);
  return o;
}
__host__ __device__ inline FastTailLayout fast_tail_layout(int T, int E, int S, int max_units, bool admit) {
  FastTailLayout L{};
  L.admit = 0;
  L.plan = admit ? r16(admit_smem_bytes(E, S, max_units)) : 0;
  L.pt = L.plan + r16(8 * static_cast<size_t>(E));
  L.key = L.pt + r16(4 * static_cast<size_t>(E));
  L.idx = L.key + 8 * 32;
  L.w = L.idx + 4 * 32;
  L.uniq = L.w + 4 * 32;
  L.tick = L.uniq + 4 * 32;
  L.nu = L.tick + 16;
  L.cand = L.nu + 16;                                             // tournament: 64 ids, 64 keys
  L.keys = L.cand + 4 * 64 + 8 * 64;                              // [3][T][E] u64
  L.taken = L.keys + 24 * static_cast<size_t>(T) * E;             // [T][E] bytes
  L.one = L.taken + r16(static_cast<size_t>(T) * E);                // one-token tail scratch
  L.total = L.one + (T == 1 ? one_token_scratch_bytes(E, S) : 0);
  return L;
}
__host__ __device__ constexpr bool fast_tail_ok(int T, int k, int E) {
  return T * k <= 32 && E <= 256 && T * E <= 2048;
}

// LRU admission of one token's selection by one warp (the shared-memory
// cache state copied when the router started): the r-th miss in ascending id
// takes the r-th free slot by index, then the untouched occupied slots in
// ascending (last access, slot) order. Sets o.cnt[4] if nothing was admitted
// (the union does not fit); the slot state is written back by the caller.
__device__ void one_token_admit_lru(const RouteArgs& a, unsigned char* sm, const FastTailLayout& L,
                                    const OneTokenScratch& o) {
  const int lane = threadIdx.x & 31;
  const int k = a.k, S = a.admit.S;
  const AdmitArgs& A = a.admit;
  const DevCacheLayer c = A.c;
  const int* s_idx = reinterpret_cast<const int*>(sm + L.idx);
  const int* s_pt = reinterpret_cast<const int*>(sm + L.pt);
  unsigned long long* s_last = reinterpret_cast<unsigned long long*>(sm + L.admit);
  int* s_owner = reinterpret_cast<int*>(s_last + S);
  uint32_t* s_sgen = reinterpret_cast<uint32_t*>(s_owner + S);
  const unsigned long long tick0 = reinterpret_cast<const unsigned long long*>(sm + L.tick)[0];
  if (k > S) {
    if (lane == 0) {
      atomicOr(a.err, MOE_DEVERR_CAPACITY);
      A.units[0] = 0;
      A.fills[0] = 0;
      o.cnt[4] = 1;
    }
    return;
  }
  for (int i = lane; i < S; i += 32) o.hit[i] = 0;
  o.mslot[lane] = -1;
  __syncwarp();
  // selection j (lane j): its slot before the step
  int e_j = -1, slot_j = -1, hr = 0, mr = 0;
  if (lane < k) {
    e_j = s_idx[lane];
    slot_j = s_pt[e_j];
  }
  const bool hit = lane < k && slot_j >= 0;
  const unsigned hm = __ballot_sync(0xffffffffu, hit), mm = __ballot_sync(0xffffffffu, lane < k && !hit);
  const int nh = __popc(hm), nm = k - nh;
  for (int i = 0; i < k; ++i) {
    const int ei = __shfl_sync(0xffffffffu, e_j, i);
    if (ei < e_j) {
      hr += (hm >> i) & 1u;
      mr += (mm >> i) & 1u;
    }
  }
  if (hit) o.hit[slot_j] = 1;
  __syncwarp();
  // the misses take the free slots in index order
  int nfree = 0;
  for (int s0 = 0; s0 < S; s0 += 32) {
    const int s2 = s0 + lane;
    const bool fr = s2 < S && s_owner[s2] < 0;
    const unsigned fb = __ballot_sync(0xffffffffu, fr);
    const int r = nfree + __popc(fb & ((1u << lane) - 1u));
    if (fr && r < nm) o.mslot[r] = s2;
    nfree += __popc(fb);
  }
  // then the untouched occupied slots, oldest access first (ties: lower slot)
  unsigned chosen = 0u;  // bit j: slot lane + 32 j taken by an earlier round
  for (int r = nfree; r < nm; ++r) {
    unsigned long long best = ~0ull;
    int bs = INT_MAX;
    for (int j = 0; j * 32 < S; ++j) {
      const int s2 = j * 32 + lane;
      if (s2 < S && s_owner[s2] >= 0 && !o.hit[s2] && !((chosen >> j) & 1u)) {
        const unsigned long long v = s_last[s2];
        if (v < best) {
          best = v;
          bs = s2;
        }
      }
    }
    const uint32_t mh = __reduce_min_sync(0xffffffffu, static_cast<uint32_t>(best >> 32));
    const bool c1 = static_cast<uint32_t>(best >> 32) == mh;
    const uint32_t ml = __reduce_min_sync(0xffffffffu, c1 ? static_cast<uint32_t>(best) : 0xffffffffu);
    const bool c2 = c1 && static_cast<uint32_t>(best) == ml;
    const int win = static_cast<int>(__reduce_min_sync(0xffffffffu, c2 ? static_cast<unsigned>(bs) : 0xffffffffu));
    if (lane == 0) o.mslot[r] = win < S ? win : -1;
    if (win < S && (win & 31) == lane) chosen |= 1u << (win >> 5);
  }
  __syncwarp();
  // every miss has a slot (guaranteed while the union fits the slots)
  const bool bad = __any_sync(0xffffffffu, lane < k && !hit && o.mslot[mr] < 0);
  if (bad) {
    if (lane == 0) {
      atomicOr(a.err, MOE_DEVERR_CAPACITY);
      A.units[0] = 0;
      A.fills[0] = 0;
      o.cnt[4] = 1;
    }
    return;
  }
  int nevict = 0;
  if (lane < k) {
    int slot = slot_j;
    if (!hit) {
      slot = o.mslot[mr];
      const int victim = s_owner[slot];
      if (victim >= 0) {
        c.pt[victim] = -1;  // victims are never in the union
        nevict = 1;
      }
      s_owner[slot] = e_j;
      s_sgen[slot] += 1u;
      s_last[slot] = tick0 + nh + 1 + mr;
      A.fills[1 + 2 * mr] = e_j;
      A.fills[2 + 2 * mr] = slot;
      A.done[mr] = 0u;
    } else {
      s_last[slot] = tick0 + 1 + hr;
    }
    const uint32_t g = s_sgen[slot];
    c.pt[e_j] = slot;
    c.ptgen[e_j] = g;
    int pos = 0;
    for (int i = 0; i < k; ++i) pos += s_idx[i] < e_j ? 1 : 0;
    int* U = A.units + kUnitHeader + kUnitInts * pos;
    const bool filled = A.read_through && !hit;
    U[0] = filled ? -2 - slot : slot;
    U[1] = pos;
    U[2] = 1;
    U[3] = filled ? e_j : static_cast<int>(g);
  }
  nevict = __reduce_add_sync(0xffffffffu, nevict);
  if (lane == 0) {
    if (A.has_shared) {
      int* U = A.units + kUnitHeader + kUnitInts * k;
      U[0] = -1;
      U[1] = -1;
      U[2] = 1;
      U[3] = 0;
    }
    A.units[0] = k + (A.has_shared ? 1 : 0);
    A.fills[0] = nm;
    c.tick[0] = tick0 + k;
    atomicAdd(reinterpret_cast<unsigned long long*>(c.stats + kStatSteps), 1ull);
    atomicAdd(reinterpret_cast<unsigned long long*>(c.stats + kStatHits), static_cast<unsigned long long>(k - nm));
    atomicAdd(reinterpret_cast<unsigned long long*>(c.stats + kStatMisses), static_cast<unsigned long long>(nm));
    atomicAdd(reinterpret_cast<unsigned long long*>(c.stats + kStatEvictions), static_cast<unsigned long long>(nevict));
    atomicAdd(reinterpret_cast<unsigned long long*>(c.stats + kStatMaterialized),
              static_cast<unsigned long long>(nm) * static_cast<unsigned long long>(A.payload));
  }
}

// One token (T == 1) on the whole block. Selection: experts whose high key
// word reaches the smallest of the per-warp maxima (when at least k warps
// hold experts, at least k experts do, so the top k are among them) are
// ranked among themselves by (key descending, id ascending). If the
// selection is certified, the weights, the plan and, for LRU, the
// admission are computed in parallel: for one token the sequential rule
// "a miss takes the lowest free slot, else the slot of oldest access" gives
// the r-th miss (ascending id) the r-th free slot by index, and past the
// free slots the untouched occupied slots in ascending (last access, slot)
// order, since every slot the step touches gets a newer tick than any
// earlier access. Returns false, having written nothing global, when the
// selection is not certified.
__device__ bool one_token_tail(const RouteArgs& a, unsigned char* sm, const FastTailLayout& L) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k;
  const bool adm = a.admit.enabled != 0;
  const int S = a.admit.S;
  const unsigned long long* sl = reinterpret_cast<const unsigned long long*>(sm + L.keys);
  const unsigned long long* slo = sl + E;
  const unsigned long long* shi = sl + 2 * E;
  unsigned char* taken = sm + L.taken;
  int* s_idx = reinterpret_cast<int*>(sm + L.idx);
  unsigned long long* s_key = reinterpret_cast<unsigned long long*>(sm + L.key);
  float* s_w = reinterpret_cast<float*>(sm + L.w);
  int* s_plan = reinterpret_cast<int*>(sm + L.plan);
  int* s_uniq = reinterpret_cast<int*>(sm + L.uniq);
  int* s_nu = reinterpret_cast<int*>(sm + L.nu);
  const OneTokenScratch o = one_token_scratch(sm + L.one, E, S);
  // ---- candidates
  const bool live = tid < E;
  const unsigned long long ke = live ? sl[tid] : 0ull;
  const uint32_t he = static_cast<uint32_t>(ke >> 32);
  const uint32_t wm = __reduce_max_sync(0xffffffffu, live ? he : 0u);
  const int nwarps = (E + 31) / 32;
  if (lane == 0) o.wmax[warp] = warp < nwarps ? wm : 0xffffffffu;
  if (tid < 8) o.cnt[tid] = 0;
  __syncthreads();
  uint32_t t = 0u;
  if (nwarps >= k) {
    t = 0xffffffffu;
    for (int w = 0; w < kRouteWarps; ++w) t = min(t, o.wmax[w]);
  }
  if (live && he >= t) {
    const int c = atomicAdd(&o.cnt[0], 1);
    o.ckey[c] = ke;
    o.cid[c] = tid;
  }
  __syncthreads();
  const int nc = o.cnt[0];
  if (nc <= kRouteThreads / 2) {
    // g threads per candidate (8, 4 or 2), each comparing against every g-th
    const int lg = nc <= kRouteThreads / 8 ? 3 : (nc <= kRouteThreads / 4 ? 2 : 1);
    const int g = 1 << lg;
    const int i = tid >> lg, part = tid & (g - 1);
    const bool ci = i < nc;
    const unsigned long long ki = ci ? o.ckey[i] : 0ull;
    const int ei = ci ? o.cid[i] : 0;
    int r = 0;
    if (ci) {
      for (int j = part; j < nc; j += g) {
        const unsigned long long kj = o.ckey[j];
        const int ej = o.cid[j];
        r += (kj > ki || (kj == ki && ej < ei)) ? 1 : 0;
      }
    }
    for (int d = 1; d < g; d <<= 1) r += __shfl_xor_sync(0xffffffffu, r, d);
    if (ci && part == 0 && r < k) {
      s_idx[r] = ei;
      s_key[r] = ki;
      taken[ei] = 1;
    }
  } else {
    for (int i = tid; i < nc; i += kRouteThreads) {
      const unsigned long long ki = o.ckey[i];
      const int ei = o.cid[i];
      int r = 0;
      for (int j = 0; j < nc; ++j) {
        const unsigned long long kj = o.ckey[j];
        const int ej = o.cid[j];
        r += (kj > ki || (kj == ki && ej < ei)) ? 1 : 0;
      }
      if (r < k) {
        s_idx[r] = ei;
        s_key[r] = ki;
        taken[ei] = 1;
      }
    }
  }
  __syncthreads();
  // ---- certification: consecutive selections, and the k-th against the
  // largest upper bound outside the selection
  {
    const bool out = live && !taken[tid];
    const unsigned long long h = out ? shi[tid] : 0ull;
    const uint32_t rh = __reduce_max_sync(0xffffffffu, out ? static_cast<uint32_t>(h >> 32) : 0u);
    const uint32_t rl =
        __reduce_max_sync(0xffffffffu, out && static_cast<uint32_t>(h >> 32) == rh ? static_cast<uint32_t>(h) : 0u);
    const bool any = __any_sync(0xffffffffu, out);
    if (lane == 0) o.wrest[warp] = any ? ((static_cast<unsigned long long>(rh) << 32) | rl) : 0ull;
    if (lane == 0 && any) atomicOr(&o.cnt[3], 1);
  }
  __syncthreads();
  if (warp == 0) {
    unsigned long long rest = 0ull;
    for (int w = 0; w < kRouteWarps; ++w) rest = o.wrest[w] > rest ? o.wrest[w] : rest;
    const bool any_rest = o.cnt[3] != 0;
    bool ok = true;
    if (lane + 1 < k) ok = slo[s_idx[lane]] > shi[s_idx[lane + 1]];
    if (lane == k - 1 && any_rest) ok = slo[s_idx[lane]] > rest;
    ok = __all_sync(0xffffffffu, ok);
    if (lane == 0) o.cnt[1] = ok ? 1 : 0;
  }
  __syncthreads();
  if (!o.cnt[1]) return false;
  const moe_plan_t& P = a.plan;
  const bool lru = adm && a.admit.policy == MOE_LRU;
  // LRU admission needs only the selection and the page table before the
  // step: warp 1 admits while warp 0 writes the weights and permutation and
  // the other warps the plan's per-expert arrays
  if (warp == 0) {
    float z = 0.f;
    int pos = 0;
    if (lane < k) {
      z = expf(static_cast<float>(okey_value(s_key[lane]) - okey_value(s_key[0])));
      const int e = s_idx[lane];
      for (int i = 0; i < k; ++i) pos += s_idx[i] < e ? 1 : 0;
    }
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, z, j);  // fixed order
    if (lane < k) {
      const float wl = z / sum;
      const int e = s_idx[lane];
      a.topk_idx[lane] = e;
      a.topk_w[lane] = wl;
      s_w[lane] = wl;
      s_uniq[pos] = e;
      P.uniq[pos] = e;
      P.perm_tok[pos] = 0;
      P.perm_rank[pos] = lane;
      P.perm_w[pos] = wl;
      P.inv[lane] = pos;
    }
    if (lane == 0) {
      P.offsets[E] = k;
      *P.n_uniq = k;
      *s_nu = k;
    }
  } else if (warp == 1 && lru) {
    one_token_admit_lru(a, sm, L, o);
  }
  {
    const int busy = lru ? 64 : 32;  // threads of warp 0 (and 1)
    for (int e = tid - busy; e >= 0 && e < E; e += kRouteThreads - busy) {
      int off = 0;
      for (int i = 0; i < k; ++i) off += s_idx[i] < e ? 1 : 0;
      const int c = taken[e];
      P.counts[e] = c;
      P.offsets[e] = off;
      s_plan[e] = c;
      s_plan[E + e] = off;
    }
  }
  __syncthreads();  // the caller's admission (random policy) reads the plan from shared memory
  if (!lru || o.cnt[4]) return true;
  // write back the layer's slot state
  const DevCacheLayer c = a.admit.c;
  const unsigned long long* s_last = reinterpret_cast<const unsigned long long*>(sm + L.admit);
  const int* s_owner = reinterpret_cast<const int*>(s_last + S);
  const uint32_t* s_sgen = reinterpret_cast<const uint32_t*>(s_owner + S);
  for (int s2 = tid; s2 < S; s2 += kRouteThreads) {
    c.last[s2] = s_last[s2];
    c.owner[s2] = s_owner[s2];
    c.sgen[s2] = s_sgen[s2];
  }
  return true;
}

// The decode fast path of the router's last block: warps 0..T-1 select the
// tokens' experts (fast_select) while the last warp stages the layer's cache
// state; uncertified tokens are repaired exactly (rare); then warp 0 plans
// and admits from shared memory, so the tail costs one round of loads.
template <int XT>
__device__ void fast_tail(const RouteArgs& a, unsigned char* sm, int* s_flagged, int* s_nflag) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, E = a.E, H = a.H, k = a.k;
  const bool adm = a.admit.enabled != 0;
  const FastTailLayout L = fast_tail_layout(T, E, a.admit.S, min(E, T * k), adm);
  unsigned char* s_admit = sm + L.admit;
  int* s_plan = reinterpret_cast<int*>(sm + L.plan);
  int* s_pt = reinterpret_cast<int*>(sm + L.pt);
  unsigned long long* s_key = reinterpret_cast<unsigned long long*>(sm + L.key);
  unsigned long long* s_keys = reinterpret_cast<unsigned long long*>(sm + L.keys);
  unsigned char* s_taken = sm + L.taken;
  int* s_idx = reinterpret_cast<int*>(sm + L.idx);
  float* s_w = reinterpret_cast<float*>(sm + L.w);
  int* s_uniq = reinterpret_cast<int*>(sm + L.uniq);
  unsigned long long* s_tick = reinterpret_cast<unsigned long long*>(sm + L.tick);
  int* s_nu = reinterpret_cast<int*>(sm + L.nu);
  const size_t te = static_cast<size_t>(T) * E;
  // the block stages every token's keys (one round of loads); the last warp
  // stages the layer's cache state meanwhile
  if (adm) cp_async_wait_all();  // the cache state copied when the kernel started
  for (int i = tid; i < static_cast<int>(te); i += kRouteThreads) {
    s_keys[i] = __ldcg(a.keys + i);
    s_keys[te + i] = __ldcg(a.keys + te + i);
    s_keys[2 * te + i] = __ldcg(a.keys + 2 * te + i);
    s_taken[i] = 0;
  }
  __syncthreads();
  if (T == 1 && one_token_tail(a, sm, L)) {
    if (adm && a.admit.policy != MOE_LRU && warp == 0) {
      AdmitStaged st;
      st.slots = true;
      st.pt = s_pt;
      st.nu = *s_nu;
      st.uniq = s_uniq;
      st.cnt = s_plan;
      st.off = s_plan + E;
      st.tick = s_tick[0];
      st.rng = s_tick[1];
      st.have_tick = true;
      __syncwarp();
      admit_warp(a.admit, a.plan, s_admit, a.err, st);
    }
    return;
  }
  if (T == 1 && k <= 8) {
    // one token: tournament over the whole block
    int* cand_idx = reinterpret_cast<int*>(sm + L.cand);
    unsigned long long* cand_key = reinterpret_cast<unsigned long long*>(sm + L.cand + 4 * 64);
    block_select_tournament(s_keys, E, k, cand_idx, cand_key, s_idx, s_key, s_taken);
    if (warp == 0) {
      const bool ok = warp_certify(s_keys + te, s_keys + 2 * te, s_taken, s_idx, E, k);
      if (ok)
        fast_write_selection(s_idx, s_key, k, a.topk_idx, a.topk_w, s_w);
      else if (lane == 0)
        s_flagged[atomicAdd(s_nflag, 1)] = 0;
    }
  } else {
    for (int t = warp; t < T; t += kRouteWarps) {
      const size_t o = static_cast<size_t>(t) * E;
      warp_select_heads(s_keys + o, E, k, s_idx + t * k, s_key + t * k, s_taken + o);
      const bool ok = warp_certify(s_keys + te + o, s_keys + 2 * te + o, s_taken + o, s_idx + t * k, E, k);
      if (ok)
        fast_write_selection(s_idx + t * k, s_key + t * k, k, a.topk_idx + t * k, a.topk_w + t * k, s_w + t * k);
      else if (lane == 0)
        s_flagged[atomicAdd(s_nflag, 1)] = t;
    }
  }
  __syncthreads();
  const int nflag = *s_nflag;
  if (nflag) {
    // exact logits of every expert of the uncertified tokens, then selection
    // by the exact keys
    for (int fi = 0; fi < nflag; ++fi) {
      const int t = s_flagged[fi];
      for (int ee = warp; ee < E; ee += kRouteWarps) {
        double v;
        const bool fin = warp_exact_logit<XT>(a.x, static_cast<size_t>(t) * H, a.w + static_cast<size_t>(ee) * H,
                                              H, a.bias, ee, v);
        if (lane == 0) {
          if (!fin) atomicOr(a.err, MOE_DEVERR_NONFINITE);
          const size_t o = static_cast<size_t>(t) * E + ee;
          a.keys[o] = a.keys[te + o] = a.keys[2 * te + o] = okey(v);
        }
      }
    }
    __syncthreads();
    for (int fi = warp; fi < nflag; fi += kRouteWarps) {
      const int t = s_flagged[fi];
      const size_t o = static_cast<size_t>(t) * E;
      for (int e = lane; e < E; e += 32) {
        s_keys[o + e] = __ldcg(a.keys + o + e);
        s_taken[o + e] = 0;
      }
      __syncwarp();
      warp_select_heads(s_keys + o, E, k, s_idx + t * k, s_key + t * k, s_taken + o);
      fast_write_selection(s_idx + t * k, s_key + t * k, k, a.topk_idx + t * k, a.topk_w + t * k, s_w + t * k);
      if (lane == 0) atomicAdd(a.repairs, 1ull);
    }
    __syncthreads();
  }
  if (warp == 0) {
    plan_warp(s_idx, s_w, T * k, k, E, a.plan, s_plan, a.err, s_uniq, s_nu);
    if (adm) {
      __syncwarp();
      AdmitStaged st;
      st.slots = true;
      st.pt = s_pt;
      st.nu = *s_nu;
      st.uniq = s_uniq;
      st.cnt = s_plan;
      st.off = s_plan + E;
      st.tick = s_tick[0];
      st.rng = s_tick[1];
      st.have_tick = true;
      admit_warp(a.admit, a.plan, s_admit, a.err, st);
    }
  }
}

// ------------------------------------------------------------ kernels
template <int XT>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteArgs a) {
  extern __shared__ int dyn_smem[];
  __shared__ float red[kRouteWarps][kRouteTB][3];
  __shared__ unsigned int s_ticket;
  __shared__ int s_nflag;
  __shared__ int s_flagged[kRouteMaxT];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e = blockIdx.x;
  const int H = a.H, E = a.E, T = a.T;
  const float* wrow = a.w + static_cast<size_t>(e) * H;
  const int nterm = 4 * ((H / 4 + kRouteThreads - 1) / kRouteThreads);  // terms per thread
  // the router weights are constant: start this block's row before waiting
  // for the kernels that produce x and reuse the scratch
  for (int v = tid; v < (H >> 2); v += kRouteThreads)
    asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<const float4*>(wrow) + v));
  // the decode tail's cache state (not written by the kernels this launch may
  // overlap): start copying it into shared memory now
  const bool early_admit = a.admit.enabled && a.plan.counts != nullptr && fast_tail_ok(T, a.k, E);
  if (early_admit) {
    const FastTailLayout L = fast_tail_layout(T, E, a.admit.S, min(E, T * a.k), true);
    unsigned char* sm = reinterpret_cast<unsigned char*>(dyn_smem);
    admit_stage_async(a.admit, sm + L.admit, reinterpret_cast<int*>(sm + L.pt),
                      reinterpret_cast<unsigned long long*>(sm + L.tick));
  }
  pdl_wait();
  pdl_trigger();

  for (int t0 = 0; t0 < T; t0 += kRouteTB) {
    float s[kRouteTB], c[kRouteTB], ab[kRouteTB];
#pragma unroll
    for (int i = 0; i < kRouteTB; ++i) s[i] = c[i] = ab[i] = 0.f;
    // four consecutive weights per load; the unrolled loop issues every
    // load of the row before the first product
    const int nvec = H >> 2;
#pragma unroll 4
    for (int v = tid; v < nvec; v += kRouteThreads) {
      const float4 w4 = __ldg(reinterpret_cast<const float4*>(wrow) + v);
      const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int i = 0; i < kRouteTB; ++i) {
        if (t0 + i < T) {
          float xv[4];
          load_x4<XT>(a.x, static_cast<size_t>(t0 + i) * H + 4 * v, xv);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float p = __fmul_rn(xv[j], wv[j]);
            const float ep = fmaf(xv[j], wv[j], -p);  // exact low part of the product
            float ns, es;
            two_sum(s[i], p, ns, es);
            s[i] = ns;
            c[i] = __fadd_rn(c[i], __fadd_rn(ep, es));
            ab[i] = fmaf(fabsf(xv[j]), fabsf(wv[j]), ab[i]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kRouteTB; ++i) {
      if (t0 + i >= T) continue;  // uniform across the block
      for (int off = 16; off; off >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s[i], off);
        const float c2 = __shfl_xor_sync(0xffffffffu, c[i], off);
        const float a2 = __shfl_xor_sync(0xffffffffu, ab[i], off);
        float ns, es;
        two_sum(s[i], s2, ns, es);
        s[i] = ns;
        c[i] = __fadd_rn(__fadd_rn(c[i], c2), es);
        ab[i] = __fadd_rn(ab[i], a2);
      }
      if (lane == 0) {
        red[warp][i][0] = s[i];
        red[warp][i][1] = c[i];
        red[warp][i][2] = ab[i];
      }
    }
    __syncthreads();
    if (tid < kRouteTB && t0 + tid < T) {
      float S = red[0][tid][0], C = red[0][tid][1], AB = red[0][tid][2];
      for (int w2 = 1; w2 < kRouteWarps; ++w2) {
        float ns, es;
        two_sum(S, red[w2][tid][0], ns, es);
        S = ns;
        C = __fadd_rn(__fadd_rn(C, red[w2][tid][1]), es);
        AB = __fadd_rn(AB, red[w2][tid][2]);
      }
      const double b = a.bias ? static_cast<double>(a.bias[e]) : 0.0;
      const double l = (static_cast<double>(S) + static_cast<double>(C)) + b;
      // |exact - (S + C)| <= (D u)^2 (1 + 2 D u) sum|x w| with D = terms per
      // thread + reduction depth + 2; the fp64 sums add <= 2^-51 |l|;
      // products below the fp32 normal range add <= 2^-140 each.
      const double Du = static_cast<double>(nterm + 5 + 3 + 2) * 0x1p-24;
      const double bnd = Du * Du * (1.0 + 2.0 * Du) * 1.01 * static_cast<double>(AB) +
                         fabs(l) * 0x1p-51 + static_cast<double>(H + 1) * 0x1p-140;
      // interval keys, rounded outward; widened by 2^-50 |l| so that
      // disjoint intervals also separate the correctly rounded fp64 images
      const double wid = __dadd_ru(bnd, __dmul_ru(fabs(l), 0x1p-50));
      const double lower = __dsub_rd(l, wid), upper = __dadd_ru(l, wid);
      const size_t o = static_cast<size_t>(t0 + tid) * E + e;
      const size_t te = static_cast<size_t>(T) * E;
      const bool fin = isfinite(l) && isfinite(wid);
      a.keys[o] = okey(l);
      a.keys[te + o] = fin ? okey(lower) : 0ull;
      a.keys[2 * te + o] = fin ? okey(upper) : ~0ull;
    }
    __syncthreads();
  }

  // ---- the last block to finish selects for every token
  __threadfence();
  if (tid == 0) s_ticket = atomicAdd(a.ticket, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) {
    if (early_admit) cp_async_wait_all();
    return;
  }
  __threadfence();
  if (tid == 0) s_nflag = 0;
  __syncthreads();
  if (a.plan.counts != nullptr && fast_tail_ok(T, a.k, E)) {
    fast_tail<XT>(a, reinterpret_cast<unsigned char*>(dyn_smem), s_flagged, &s_nflag);
    if (tid == 0) *a.ticket = 0u;
    return;
  }
  int sel[16];
  unsigned long long selk[16];
  const size_t te = static_cast<size_t>(T) * E;
  for (int t = warp; t < T; t += kRouteWarps) {
    const size_t o = static_cast<size_t>(t) * E;
    const TokenKeys K{a.keys + o, a.keys + te + o, a.keys + 2 * te + o};
    const bool ok = warp_select(K, E, a.k, sel, selk, true);
    if (ok) {
      warp_write_selection(sel, selk, a.k, a.topk_idx + static_cast<size_t>(t) * a.k,
                           a.topk_w + static_cast<size_t>(t) * a.k);
    } else if (lane == 0) {
      s_flagged[atomicAdd(&s_nflag, 1)] = t;
    }
  }
  __syncthreads();
  // exact repair of uncertified tokens (T <= kRouteMaxT, so all fit the list)
  const int nflag = s_nflag;
  for (int fi = 0; fi < nflag; ++fi) {
    const int t = s_flagged[fi];
    for (int ee = warp; ee < E; ee += kRouteWarps) {
      double v;
      const bool fin = warp_exact_logit<XT>(a.x, static_cast<size_t>(t) * H,
                                            a.w + static_cast<size_t>(ee) * H, H, a.bias, ee, v);
      if (lane == 0) {
        if (!fin) atomicOr(a.err, MOE_DEVERR_NONFINITE);
        const size_t o = static_cast<size_t>(t) * E + ee;
        a.keys[o] = a.keys[te + o] = a.keys[2 * te + o] = okey(v);
      }
    }
  }
  __syncthreads();
  for (int fi = warp; fi < nflag; fi += kRouteWarps) {
    const int t = s_flagged[fi];
    const size_t o = static_cast<size_t>(t) * E;
    const TokenKeys K{a.keys + o, a.keys + te + o, a.keys + 2 * te + o};
    warp_select(K, E, a.k, sel, selk, false);
    warp_write_selection(sel, selk, a.k, a.topk_idx + static_cast<size_t>(t) * a.k,
                         a.topk_w + static_cast<size_t>(t) * a.k);
    if (lane == 0) atomicAdd(a.repairs, 1ull);
  }
  if (a.plan.counts != nullptr) {
    __syncthreads();
    if (T * a.k <= 32) {
      if (warp == 0) plan_warp(a.topk_idx, a.topk_w, T * a.k, a.k, E, a.plan, dyn_smem, a.err);
    } else {
      plan_block<kRouteThreads>(a.topk_idx, a.topk_w, T * a.k, a.k, E, a.plan, dyn_smem, a.err);
    }
    if (a.admit.enabled) {
      __syncthreads();
      if (warp == 0) admit_warp(a.admit, a.plan, reinterpret_cast<unsigned char*>(dyn_smem), a.err);
    }
  }
  if (tid == 0) *a.ticket = 0u;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  extern __shared__ int dyn_smem[];
  if (a.T * a.k <= 32) {
    if (threadIdx.x < 32) plan_warp(a.idx, a.w, a.T * a.k, a.k, a.E, a.plan, dyn_smem, a.err);
  } else {
    plan_block<kPlanThreads>(a.idx, a.w, a.T * a.k, a.k, a.E, a.plan, dyn_smem, a.err);
  }
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t st) {
  (void)num_sms;
  if (a.T < 1 || a.T > kRouteMaxT || a.k > 16 || a.E > 1024) return cudaErrorInvalidValue;
  size_t smem = a.plan.counts ? plan_smem_bytes(a.E) : 0;
  if (a.admit.enabled)
    smem = std::max(smem, admit_smem_bytes(a.E, a.admit.S, std::min(a.E, a.T * a.k)));
  if (a.plan.counts && fast_tail_ok(a.T, a.k, a.E))
    smem = std::max(smem, fast_tail_layout(a.T, a.E, a.admit.S, std::min(a.E, a.T * a.k), a.admit.enabled != 0).total);
  if (smem > 48 * 1024) {
    cudaError_t e = a.xt == MOE_BF16
        ? cudaFuncSetAttribute(route_kernel<MOE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem))
        : cudaFuncSetAttribute(route_kernel<MOE_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const cudaError_t e = a.xt == MOE_BF16
      ? pdl_launch(route_kernel<MOE_BF16>, dim3(a.E), dim3(kRouteThreads), smem, st, a)
      : pdl_launch(route_kernel<MOE_F32>, dim3(a.E), dim3(kRouteThreads), smem, st, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t st) {
  plan_kernel<<<1, kPlanThreads, plan_smem_bytes(a.E), st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

// ------------------------------------------------------------ no-allocation router
// A standalone router entry point for callers that cannot allocate device
// memory: code running inside another framework's memory pool or arena, hosts
// that forbid cudaMalloc after start-up, or pipelines being captured into a
// CUDA graph where an allocation would break the capture. Its scratch (fast
// logits, their bounds, the last-block counter, the repair counter and an
// error word) lives in one file-scope device array below, sized for at most
// kNoAllocMaxTE = 8192 (token, expert) logits (192 KiB of logit and bound keys);
// every GPU that loads this library holds that array until the process exits.
namespace moe {
namespace {

constexpr int kNoAllocMaxTE = 8192;
constexpr int kNoAllocMaxDevices = 64;

// [0, 3 TE) logit, lower-bound and upper-bound keys, then a 32-byte header:
// ticket (u32), error word (u32), repaired-token counter (u64).
static __device__ __align__(256) unsigned long long g_route_scratch[3 * kNoAllocMaxTE + 4];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_noalloc(const void* x, int32_t xt, int32_t T, int32_t H,
                                          int32_t E, int32_t k, const float* w_router,
                                          const float* bias, int32_t* topk_idx, float* topk_w,
                                          moe_stream_t stream) {
  using namespace moe;
  if (!x || !w_router || !topk_idx || !topk_w) {
    set_thread_error("moe_route_noalloc: null pointer");
    return MOE_ERR_ARG;
  }
  if (xt != MOE_F32 && xt != MOE_BF16) {
    set_thread_error("moe_route_noalloc: activation dtype must be MOE_F32 or MOE_BF16");
    return MOE_ERR_ARG;
  }
  if (T < 1 || T > kRouteMaxT || H < 4 || H % 4 || E < 1 || E > 1024 || k < 1 || k > 16 || k > E) {
    set_thread_error("moe_route_noalloc: need 1 <= T <= 64, H a positive multiple of 4, "
                     "1 <= E <= 1024, 1 <= k <= min(16, E)");
    return MOE_ERR_ARG;
  }
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(w_router) % 16) {
    set_thread_error("moe_route_noalloc: x and w_router must be 16-byte aligned");
    return MOE_ERR_ARG;
  }
  if (static_cast<int64_t>(T) * E > kNoAllocMaxTE) {
    set_thread_error("moe_route_noalloc: T*E = " + std::to_string(static_cast<int64_t>(T) * E) +
                     " exceeds the static scratch limit of " + std::to_string(kNoAllocMaxTE) +
                     " logits");
    return MOE_ERR_ARG;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
    set_thread_error(std::string("moe_route_noalloc: cudaGetDevice: ") + cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  void* base = nullptr;
  {
    // once per device, with that device current: the host-side name of a
    // __device__ array is not a device address; ask the runtime for it
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      e = cudaGetSymbolAddress(&g_noalloc_ptr[dev], g_route_scratch);
      if (e != cudaSuccess) {
        g_noalloc_ptr[dev] = nullptr;
        set_thread_error(std::string("moe_route_noalloc: cudaGetSymbolAddress: ") +
                         cudaGetErrorString(e));
        return MOE_ERR_CUDA;
      }
    }
    base = g_noalloc_ptr[dev];
  }
  unsigned long long* scratch = static_cast<unsigned long long*>(base);
  unsigned char* header = reinterpret_cast<unsigned char*>(scratch + 3 * kNoAllocMaxTE);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the counter and flags must start at zero; the array keeps the last call's contents
  e = cudaMemsetAsync(header, 0, 32, st);
  if (e != cudaSuccess) {
    set_thread_error(std::string("moe_route_noalloc: cudaMemsetAsync: ") + cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  RouteArgs a{};
  a.x = x;
  a.xt = xt;
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = k;
  a.w = w_router;
  a.bias = bias;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.keys = scratch;
  a.ticket = reinterpret_cast<unsigned int*>(header);
  a.err = reinterpret_cast<uint32_t*>(header + 4);
  a.repairs = reinterpret_cast<unsigned long long*>(header + 8);
  e = launch_route(a, 0, st);
  if (e != cudaSuccess) {
    set_thread_error(std::string("moe_route_noalloc: launch: ") + cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// ------------------------------------------------------------ many-token routing
// Prefill chunks route thousands of tokens at once. Logits come from a tiled
// fp32 GEMM (split along K) that sums each 32-term chunk with plain FMAs and
// folds the chunk sums into an error-free (hi, lo) pair; the chunk error is at most
// gamma_32 * sum|x w| <= gamma_32 * ||x|| * ||w|| (Cauchy-Schwarz), so the
// same integer-key certification applies, and uncertified tokens are
// recomputed exactly as in the few-token router.
namespace moe {
namespace {

constexpr int kLT = 64;   // tokens per logits tile
constexpr int kLE = 64;   // experts per logits tile
constexpr int kLK = 32;   // K chunk

template <int XT>
__global__ void __launch_bounds__(256) row_norms_kernel(const void* x, int T, const float* w, int E, int H,
                                                        float* xn, float* wn) {
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (gw >= T + E) return;
  float s = 0.f;
  if (gw < T) {
    for (int k = lane; k < H; k += 32) {
      const float v = load_x<XT>(x, static_cast<size_t>(gw) * H + k);
      s = fmaf(v, v, s);
    }
  } else {
    const float* r = w + static_cast<size_t>(gw - T) * H;
    for (int k = lane; k < H; k += 32) s = fmaf(r[k], r[k], s);
  }
  for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  // the fp32 sum of squares is within a relative 1e-3 of the exact one
  const float nrm = sqrtf(s) * 1.001f;
  if (lane == 0) {
    if (gw < T)
      xn[gw] = isfinite(nrm) ? nrm : INFINITY;
    else
      wn[gw - T] = isfinite(nrm) ? nrm : INFINITY;
  }
}

// Split-K logits: one 64-token x 64-expert tile and one of up to four
// slices of K per 128-thread block. A thread owns 8 tokens x 4 experts; a
// warp spans 8 token groups x 4 expert groups, so each of its shared loads
// touches at most 128 bytes. K advances in chunks of 32 through a
// double-buffered, transposed shared-memory stage (the next chunk's global
// loads are issued before the current chunk's FMAs). Each chunk sum is
// folded into an error-free (hi, lo) pair; the slice's pair goes to a
// partial buffer and logits_keys_kernel folds the slices in slice order, so
// the result does not depend on scheduling.
constexpr int kLThreads = 128;
constexpr int kLPad = kLT + 4;

template <int XT>
__device__ __forceinline__ void logits_fetch(const RouteArgs& a, int t0, int e0, int kc, float (&xv)[2][8],
                                             float4 (&wv)[4]) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int rep = 0; rep < 2; ++rep) {
    const int idx = tid + kLThreads * rep, r = idx & 63, part = idx >> 6;  // k = part*8 .. +7
    const int t = t0 + r;
    const size_t off = static_cast<size_t>(t) * a.H + kc + part * 8;
    if (t >= a.T) {
#pragma unroll
      for (int j = 0; j < 8; ++j) xv[rep][j] = 0.f;
    } else if (XT == MOE_BF16) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + off));
      const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xv[rep][2 * j] = __uint_as_float(wds[j] << 16);
        xv[rep][2 * j + 1] = __uint_as_float(wds[j] & 0xFFFF0000u);
      }
    } else {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + off);
      const float4 p = __ldg(src), q = __ldg(src + 1);
      xv[rep][0] = p.x, xv[rep][1] = p.y, xv[rep][2] = p.z, xv[rep][3] = p.w;
      xv[rep][4] = q.x, xv[rep][5] = q.y, xv[rep][6] = q.z, xv[rep][7] = q.w;
    }
  }
#pragma unroll
  for (int rep = 0; rep < 4; ++rep) {
    const int idx = tid + kLThreads * rep, r = idx & 63, q = idx >> 6;  // k = q*4 .. +3
    const int e = e0 + r;
    wv[rep] = e < a.E ? __ldg(reinterpret_cast<const float4*>(a.w + static_cast<size_t>(e) * a.H + kc + q * 4))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__device__ __forceinline__ void logits_stash(float (*xs)[kLPad], float (*ws)[kLPad], const float (&xv)[2][8],
                                             const float4 (&wv)[4]) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int rep = 0; rep < 2; ++rep) {
    const int idx = tid + kLThreads * rep, r = idx & 63, part = idx >> 6;
#pragma unroll
    for (int j = 0; j < 8; ++j) xs[part * 8 + j][r] = xv[rep][j];
  }
#pragma unroll
  for (int rep = 0; rep < 4; ++rep) {
    const int idx = tid + kLThreads * rep, r = idx & 63, q = idx >> 6;
    ws[q * 4 + 0][r] = wv[rep].x;
    ws[q * 4 + 1][r] = wv[rep].y;
    ws[q * 4 + 2][r] = wv[rep].z;
    ws[q * 4 + 3][r] = wv[rep].w;
  }
}

// part: [slices][T][E] (hi, lo) pairs of the K slices
template <int XT>
__global__ void __launch_bounds__(kLThreads, 4) logits_tiled_kernel(RouteArgs a, float2* part) {
  __shared__ __align__(16) float xs[2][kLK][kLPad];
  __shared__ __align__(16) float ws[2][kLK][kLPad];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ty = lane & 7, tx = warp * 4 + (lane >> 3);  // tokens ty*8.., experts tx*4..
  const int t0 = blockIdx.y * kLT, e0 = blockIdx.x * kLE;
  const int T = a.T, E = a.E;
  const int klen = a.H / gridDim.z, kbeg = blockIdx.z * klen;
  float hi[8][4], lo[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) hi[i][j] = lo[i][j] = 0.f;
  float xv[2][8];
  float4 wv[4];
  logits_fetch<XT>(a, t0, e0, kbeg, xv, wv);
  logits_stash(xs[0], ws[0], xv, wv);
  __syncthreads();
  const int nch = klen / kLK;
  for (int c = 0; c < nch; ++c) {
    const int buf = c & 1;
    if (c + 1 < nch) logits_fetch<XT>(a, t0, e0, kbeg + (c + 1) * kLK, xv, wv);
    float p[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) p[i][j] = 0.f;
#pragma unroll 4
    for (int k = 0; k < kLK; ++k) {
      const float4 x0 = *reinterpret_cast<const float4*>(&xs[buf][k][ty * 8]);
      const float4 x1 = *reinterpret_cast<const float4*>(&xs[buf][k][ty * 8 + 4]);
      const float4 w4 = *reinterpret_cast<const float4*>(&ws[buf][k][tx * 4]);
      const float xa[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const float wa[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) p[i][j] = fmaf(xa[i], wa[j], p[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float ns, es;
        two_sum(hi[i][j], p[i][j], ns, es);
        hi[i][j] = ns;
        lo[i][j] = __fadd_rn(lo[i][j], es);
      }
    if (c + 1 < nch) logits_stash(xs[buf ^ 1], ws[buf ^ 1], xv, wv);
    __syncthreads();
  }
  float2* dst = part + static_cast<size_t>(blockIdx.z) * T * E;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + ty * 8 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) dst[static_cast<size_t>(t) * E + e] = make_float2(hi[i][j], lo[i][j]);
    }
  }
}

// Keys of a logit summed in chunks of at most 32 plain-FMA products whose
// chunk sums were folded error-free into (hi, lo): the logit
// l = hi + lo + b in fp64 and its outward-rounded bound interval. The bound
// is formed in fp32 with every operation rounded up (an upper bound of the
// fp64 expression gamma_32 * 1.01 * ||x|| ||w|| + |l| (2^-51 + 2^-50) +
// (H+1) 2^-126; ||x|| ||w|| bounds sum |x w| by Cauchy-Schwarz), so only the
// logit and the two interval ends use fp64. A non-finite logit or bound
// gives the widest interval.
__device__ __forceinline__ void chunked_keys(float hi, float lo, float bf, float xn, float wn, int H,
                                             unsigned long long& kl, unsigned long long& klo,
                                             unsigned long long& khi) {
  const double l = (static_cast<double>(hi) + static_cast<double>(lo)) + static_cast<double>(bf);
  // 1.01 * gamma_32 rounded up; gamma_32 = 32u / (1 - 32u), u = 2^-24
  const float c1 = 1.9314e-6f;
  const float A = __fmul_ru(xn, wn);
  const float absl = __fadd_ru(__fadd_ru(fabsf(hi), fabsf(lo)), fabsf(bf));
  const float wid =
      __fadd_ru(__fadd_ru(__fmul_ru(c1, A), __fmul_ru(absl, 0x1.8p-50f)), static_cast<float>(H + 1) * 0x1p-126f);
  const bool fin = isfinite(l) && isfinite(wid);
  kl = okey(l);
  klo = fin ? okey(__dsub_rd(l, static_cast<double>(wid))) : 0ull;
  khi = fin ? okey(__dadd_ru(l, static_cast<double>(wid))) : ~0ull;
}

// Folds the slices' (hi, lo) pairs in slice order and writes the logit keys
// and the outward-rounded bound keys (one thread per token and expert).
__global__ void __launch_bounds__(256) logits_keys_kernel(RouteArgs a, const float2* part, int slices,
                                                          const float* xn, const float* wn) {
  const size_t te = static_cast<size_t>(a.T) * a.E;
  const int t = blockIdx.y, e = blockIdx.x * 256 + threadIdx.x;  // grid (ceil(E/256), T)
  if (e >= a.E) return;
  const size_t o = static_cast<size_t>(t) * a.E + e;
  float2 v = __ldcs(part + o);
  float hi = v.x, lo = v.y;
  for (int z = 1; z < slices; ++z) {
    v = __ldcs(part + z * te + o);
    float ns, es;
    two_sum(hi, v.x, ns, es);
    hi = ns;
    lo = __fadd_rn(__fadd_rn(lo, v.y), es);
  }
  const float bf = a.bias ? a.bias[e] : 0.f;
  unsigned long long kl, klo, khi;
  chunked_keys(hi, lo, bf, __ldg(xn + t), __ldg(wn + e), a.H, kl, klo, khi);
  a.keys[o] = kl;
  a.keys[te + o] = klo;
  a.keys[2 * te + o] = khi;
}

// Per-token selection and certification from the keys (one warp per
// token). gated: only the tokens the refining kernel left with flag 2.
__global__ void __launch_bounds__(256) select_kernel(RouteArgs a, int* flags, int gated) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= a.T) return;
  if (gated && flags[t] != 2) return;
  const size_t te = static_cast<size_t>(a.T) * a.E, o = static_cast<size_t>(t) * a.E;
  const TokenKeys K{a.keys + o, a.keys + te + o, a.keys + 2 * te + o};
  int sel[16];
  unsigned long long selk[16];
  const bool ok = warp_select(K, a.E, a.k, sel, selk, true);
  if (ok)
    warp_write_selection(sel, selk, a.k, a.topk_idx + static_cast<size_t>(t) * a.k,
                         a.topk_w + static_cast<size_t>(t) * a.k);
  if (lane == 0) flags[t] = ok ? 0 : 1;
}

// Exact repair of an uncertified token. Only the experts whose rank the bound
// intervals leave open are recomputed: the candidates are the experts that
// fewer than k others beat for certain (lower bound above their upper
// bound); a candidate whose interval meets another candidate's is
// recomputed exactly (its three keys collapse to the exact logit's). Every
// other expert is either certainly outside the top k or certainly ordered
// against each candidate, so selecting by the logit keys afterwards yields
// the ranking of the exact logits, ties to the lower expert id. Each block
// reads the flags of 32 tokens at once and repairs the flagged ones.
constexpr int kRepairGrid = 512;  // blocks at most (32 tokens each per pass)
template <int XT>
__global__ void __launch_bounds__(kRouteThreads) repair_kernel(RouteArgs a, const int* flags) {
  __shared__ unsigned long long s_lo[1024], s_hi[1024];
  __shared__ unsigned char s_cand[1024];
  __shared__ int s_amb[1024];
  __shared__ int s_namb;
  __shared__ unsigned s_mask;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, H = a.H, k = a.k;
  for (int base = blockIdx.x * 32; base < a.T; base += gridDim.x * 32) {
    if (warp == 0) {
      const unsigned m = __ballot_sync(0xffffffffu, base + lane < a.T && flags[base + lane] != 0);
      if (lane == 0) s_mask = m;
    }
    __syncthreads();
    unsigned mask = s_mask;
    __syncthreads();
    while (mask) {
      const int t = base + __ffs(mask) - 1;
      mask &= mask - 1;
      const size_t te = static_cast<size_t>(a.T) * E, o = static_cast<size_t>(t) * E;
      for (int e = tid; e < E; e += kRouteThreads) {
        s_lo[e] = __ldcg(a.keys + te + o + e);
        s_hi[e] = __ldcg(a.keys + 2 * te + o + e);
      }
      if (tid == 0) s_namb = 0;
      __syncthreads();
      for (int e = tid; e < E; e += kRouteThreads) {
        const unsigned long long h = s_hi[e];
        int above = 0;
        for (int j = 0; j < E; ++j) above += s_lo[j] > h ? 1 : 0;
        s_cand[e] = above < k ? 1 : 0;
      }
      __syncthreads();
      for (int e = tid; e < E; e += kRouteThreads) {
        if (!s_cand[e]) continue;
        const unsigned long long l = s_lo[e], h = s_hi[e];
        bool meets = false;
        for (int j = 0; j < E && !meets; ++j)
          meets = j != e && s_cand[j] && !(l > s_hi[j] || s_lo[j] > h);
        if (meets) s_amb[atomicAdd(&s_namb, 1)] = e;
      }
      __syncthreads();
      const int namb = s_namb;
      for (int i = warp; i < namb; i += kRouteWarps) {
        const int ee = s_amb[i];
        double v;
        const bool fin = warp_exact_logit<XT>(a.x, static_cast<size_t>(t) * H, a.w + static_cast<size_t>(ee) * H,
                                              H, a.bias, ee, v);
        if (lane == 0) {
          if (!fin) atomicOr(a.err, MOE_DEVERR_NONFINITE);
          a.keys[o + ee] = a.keys[te + o + ee] = a.keys[2 * te + o + ee] = okey(v);
        }
      }
      __syncthreads();
      if (warp == 0) {
        const TokenKeys K{a.keys + o, a.keys + te + o, a.keys + 2 * te + o};
        int sel[16];
        unsigned long long selk[16];
        warp_select(K, E, k, sel, selk, false);
        warp_write_selection(sel, selk, k, a.topk_idx + static_cast<size_t>(t) * k,
                             a.topk_w + static_cast<size_t>(t) * k);
        if (lane == 0) atomicAdd(a.repairs, 1ull);
      }
      __syncthreads();
    }
  }
}

// ---- many-token logits on the tensor cores, as a filter
// The router weights are split into two bf16 parts, w = hi + mid + r with
// hi = bf16(w) and mid = bf16(w - hi), both rounded to nearest (w - hi is
// exact in fp32, |r| <= 2^-16 |w|). One tcgen05 GEMM per 128-token x
// 64-expert tile computes G = x hi^T and M = x mid^T (bf16 operands, so every
// product is exact; fp32 accumulators in TMEM) and writes L = G + M. The
// tensor cores' accumulation order and rounding are not specified, so L only
// excludes experts, under a deliberately loose error model:
//   |L - x.w| <= 2^-9 ||x|| ||w|| + 2^-22 |L| + 2^-124 sqrt(H) ||w|| + (2H+2) 2^-126,
// i.e. an accumulation error of at most 2^-10 of the summed magnitudes (64
// times the error of an fp32 accumulation that truncates after every
// 16-product step at H = 2048), the split residual 2^-16, the fp32 sum
// G + M, and flushed subnormal operands and products. An expert whose upper
// bound lies below the k-th largest lower bound cannot be among the top k
// (at least k experts are certainly above it, ties included). The others,
// the candidates (about ten of 256 on the prefill workload), get certified
// logits on the CUDA cores: first summed in chunks of 32 products (the same
// keys as the CUDA-core path); for a token they leave uncertified, the
// candidates whose rank stays open are recomputed as compensated dot
// products (error-free products and sums; Ogita, Rump and Oishi 2005),
// whose bound is some five orders of magnitude tighter. Each candidate's certified logit is also checked against its
// filter interval; a token whose check fails, or whose filter is not
// finite, takes every expert as a candidate. A token still uncertified gets
// full keys (non-candidates a key below every logit) and goes through the
// per-token selection and the exact repair.
constexpr int kTcTok = 128;  // tokens per CTA (MMA M)
constexpr int kTcExp = 64;   // experts per CTA; MMA N = 128: their hi rows, then their mid rows
constexpr int kTcBK = 64;    // K per stage: 128 bytes of bf16 per row
constexpr int kTcStages = 6;
constexpr uint32_t kTcABytes = kTcTok * kTcBK * 2;      // 16 KiB of tokens
constexpr uint32_t kTcBBytes = 2 * kTcExp * kTcBK * 2;  // 16 KiB of weight parts
constexpr uint32_t kTcStage = kTcABytes + kTcBBytes;
constexpr size_t kTcSmem = static_cast<size_t>(kTcStages) * kTcStage + 1024;
constexpr long long kTcWaitCycles = 4000000000ll;  // about 2 s at the SM clock
static_assert(kTcABytes % 1024 == 0 && kTcStage % 1024 == 0, "stage alignment");

// ws: bf16 [ceil(E/64)][2][64][H]: block b holds the hi rows of experts
// 64b .. 64b+63, then their mid rows; rows of experts >= E are zero. One
// 128-thread block per row (each warp a quarter of it); it also writes the
// row's norm bound wn[e] = 1.001 * sqrt(sum w^2) in fp32 (the fp32 sum of
// squares, its four quarters added in order, is within a relative 1e-3 of
// the exact one), infinite if not finite.
__global__ void __launch_bounds__(128) router_split_kernel(const float* w, int E, int H, uint16_t* ws, float* wn) {
  __shared__ float s_part[4];
  const int e = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = e / kTcExp, r = e % kTcExp;
  uint16_t* hrow = ws + (static_cast<int64_t>(2 * b) * kTcExp + r) * H;
  uint16_t* mrow = ws + (static_cast<int64_t>(2 * b + 1) * kTcExp + r) * H;
  const int q = H / 4, c0 = warp * q;  // the warp's quarter (H % 64 == 0)
  float s = 0.f;
#pragma unroll 4
  for (int c = c0 + lane * 4; c < c0 + q; c += 128) {
    const float4 v = e < E ? __ldg(reinterpret_cast<const float4*>(w + static_cast<int64_t>(e) * H + c))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    const float f[4] = {v.x, v.y, v.z, v.w};
    uint32_t hb[2], mb[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(f[2 * j]), h1 = __float2bfloat16_rn(f[2 * j + 1]);
      const __nv_bfloat16 m0 = __float2bfloat16_rn(f[2 * j] - __bfloat162float(h0));
      const __nv_bfloat16 m1 = __float2bfloat16_rn(f[2 * j + 1] - __bfloat162float(h1));
      hb[j] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
      mb[j] = static_cast<uint32_t>(__bfloat16_as_ushort(m0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(m1)) << 16);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) s = fmaf(f[j], f[j], s);
    *reinterpret_cast<uint2*>(hrow + c) = make_uint2(hb[0], hb[1]);
    *reinterpret_cast<uint2*>(mrow + c) = make_uint2(mb[0], mb[1]);
  }
  for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) s_part[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0 && e < E) {
    const float nrm = sqrtf(((s_part[0] + s_part[1]) + s_part[2]) + s_part[3]) * 1.001f;
    wn[e] = isfinite(nrm) ? nrm : INFINITY;
  }
}

struct TcArgs {
  int T, E, H;
  float* out;  // [T][E] approximate logits
  uint32_t* err;
  long long wait_cycles;
};

// D (TMEM) += A (shared-memory descriptor) * B (shared-memory descriptor)
__device__ __forceinline__ void umma_ss(uint32_t dt, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(dt),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// One 128-token x 64-expert tile per CTA of 4 warps: lane 0 of warp 0 issues
// the TMA copies (token rows and the hi + mid rows, 64 K per stage, 128-byte
// swizzle), lane 0 of warp 1 the MMAs (M 128, N 128, K 16; A and B from
// shared memory); then every warp reads its 32 TMEM lanes (tokens) and
// writes G + M. Every wait is bounded: past the limit the CTA's abort flag
// and the timeout bit are set, copies and MMAs in flight are drained, and no
// logit is written.
__global__ void __launch_bounds__(128, 1) logits_tc_kernel(const __grid_constant__ CUtensorMap map_x,
                                                           const __grid_constant__ CUtensorMap map_w, TcArgs a) {
  using namespace tc;
  extern __shared__ unsigned char smraw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_full[kTcStages], bar_free[kTcStages], bar_acc, bar_drain;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_abort;
  volatile int* abort_flag = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = su32(sm);
  const int t0 = blockIdx.x * kTcTok, eb = blockIdx.y;
  const int nkb = a.H / kTcBK;
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(su32(&bar_full[s]), 1);
      mbar_init(su32(&bar_free[s]), 1);
    }
    mbar_init(su32(&bar_acc), 1);
    mbar_init(su32(&bar_drain), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_holder)),
                 "r"(2 * kTcExp));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = tmem_holder;

  if (warp == 0 && lane == 0) {
    uint32_t ring = 0;
    RingPos rp;
    for (int kb = 0; kb < nkb; ++kb, ++ring, rp.next(kTcStages)) {
      if (ring >= static_cast<uint32_t>(kTcStages) &&
          !mbar_wait(su32(&bar_free[rp.s]), rp.ph ^ 1u, abort_flag, a.err, a.wait_cycles))
        break;
      const uint32_t st = sbase + static_cast<uint32_t>(rp.s) * kTcStage, fb = su32(&bar_full[rp.s]);
      mbar_expect_tx(fb, kTcStage);
      tma2d(st, &map_x, fb, kb * kTcBK, t0);
      tma2d(st + kTcABytes, &map_w, fb, kb * kTcBK, eb * 2 * kTcExp);
    }
    // drain: the last copies into each stage complete before exit
    const uint32_t n = ring < static_cast<uint32_t>(kTcStages) ? ring : static_cast<uint32_t>(kTcStages);
    for (uint32_t j = 0; j < n; ++j) {
      const uint32_t r = ring - 1 - j;
      mbar_drain(su32(&bar_full[r % kTcStages]), (r / kTcStages) & 1u, a.err, a.wait_cycles);
    }
  } else if (warp == 1 && lane == 0) {
    // kind::f16, bf16 A and B (K-major), fp32 D, N = 128, M = 128
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((static_cast<uint32_t>(2 * kTcExp) >> 3) << 17) |
                           ((static_cast<uint32_t>(kTcTok) >> 4) << 24);
    RingPos rp;
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb, rp.next(kTcStages)) {
      if (!(ok = mbar_wait(su32(&bar_full[rp.s]), rp.ph, abort_flag, a.err, a.wait_cycles))) break;
      asm volatile("tcgen05.fence::after_thread_sync;");
      const uint32_t st = sbase + static_cast<uint32_t>(rp.s) * kTcStage;
      const uint64_t ad = sdesc(st), bd = sdesc(st + kTcABytes);
#pragma unroll
      for (int k = 0; k < kTcBK / 16; ++k)
        umma_ss(tmem, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      umma_commit(su32(&bar_free[rp.s]));
    }
    if (ok) umma_commit(su32(&bar_acc));
    // drain: every MMA issued here has completed before TMEM is released
    umma_commit(su32(&bar_drain));
    mbar_drain(su32(&bar_drain), 0, a.err, a.wait_cycles);
  }
  __syncwarp();
  // epilogue: warp w holds TMEM lanes 32w .. 32w+31, the tile's tokens
  // t0 + 32w + lane; columns 0..63 G, 64..127 M
  const bool ready = __all_sync(0xffffffffu, mbar_wait(su32(&bar_acc), 0, abort_flag, a.err, a.wait_cycles));
  if (ready) {
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int t = t0 + warp * 32 + lane;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      uint32_t g[32], m[32];
      tmem_ld32(tmem + lane_base + half * 32, g);
      tmem_ld32(tmem + lane_base + kTcExp + half * 32, m);
      const int e0 = eb * kTcExp + half * 32;
      if (t < a.T && e0 < a.E) {
        float* dst = a.out + static_cast<int64_t>(t) * a.E + e0;
        if (e0 + 32 <= a.E && (a.E & 3) == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4*>(dst)[j] = make_float4(
                __uint_as_float(g[4 * j]) + __uint_as_float(m[4 * j]),
                __uint_as_float(g[4 * j + 1]) + __uint_as_float(m[4 * j + 1]),
                __uint_as_float(g[4 * j + 2]) + __uint_as_float(m[4 * j + 2]),
                __uint_as_float(g[4 * j + 3]) + __uint_as_float(m[4 * j + 3]));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (e0 + j < a.E) dst[j] = __uint_as_float(g[j]) + __uint_as_float(m[j]);
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kTcExp));
}

// Order-preserving key of a non-NaN float (-0 first made +0 by the caller).
__device__ __forceinline__ uint32_t fkey(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Logit of token row xr (bf16) and weight row wr by the warp, summed in
// chunks of at most 32 plain-FMA products per lane, each chunk sum folded
// error-free into (hi, lo), the lanes combined by error-free sums (every
// lane returns the same pair). The keys come from chunked_keys.
__device__ void warp_dot_chunked(const uint16_t* xr, const float* wr, int H, float& hi, float& lo) {
  const int lane = threadIdx.x & 31;
  hi = 0.f;
  lo = 0.f;
  float p = 0.f;
  int n = 0;
  for (int g = lane; g < (H >> 2); g += 32) {
    const float4 w4 = __ldg(reinterpret_cast<const float4*>(wr) + g);
    const uint2 xb = __ldg(reinterpret_cast<const uint2*>(xr) + g);
    p = fmaf(__uint_as_float(xb.x << 16), w4.x, p);
    p = fmaf(__uint_as_float(xb.x & 0xFFFF0000u), w4.y, p);
    p = fmaf(__uint_as_float(xb.y << 16), w4.z, p);
    p = fmaf(__uint_as_float(xb.y & 0xFFFF0000u), w4.w, p);
    if (++n == 8) {  // 32 products
      float ns, es;
      two_sum(hi, p, ns, es);
      hi = ns;
      lo = __fadd_rn(lo, es);
      p = 0.f;
      n = 0;
    }
  }
  {
    float ns, es;
    two_sum(hi, p, ns, es);
    hi = ns;
    lo = __fadd_rn(lo, es);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, lo, off);
    float ns, es;
    two_sum(hi, h2, ns, es);
    hi = ns;
    lo = __fadd_rn(__fadd_rn(lo, l2), es);
  }
}

// Top-k of the candidates held one per lane (lane j < C: expert my_e, keys
// my_l, my_lo, my_hi) by descending logit key, ties to the lower id. Lane
// r < k ends with selection r (sel_e, sel_k). Returns whether the bound
// intervals of consecutive selections, and of the k-th against every other
// candidate, are disjoint (the other experts are excluded by the filter).
__device__ bool cand_select(int C, int k, int my_e, unsigned long long my_l, unsigned long long my_lo,
                            unsigned long long my_hi, int& sel_e, unsigned long long& sel_k) {
  const int lane = threadIdx.x & 31;
  const bool has = lane < C;
  bool taken = false;
  unsigned long long r_lo = 0ull, r_hi = 0ull;
  for (int r = 0; r < k; ++r) {
    unsigned long long key;
    const int mi = warp_round(has && !taken, my_l, my_e, key);
    const unsigned ow = __ballot_sync(0xffffffffu, has && !taken && my_e == mi);
    const int owner = __ffs(ow) - 1;
    const unsigned long long lo_o = __shfl_sync(0xffffffffu, my_lo, owner & 31);
    const unsigned long long hi_o = __shfl_sync(0xffffffffu, my_hi, owner & 31);
    if (lane == owner) taken = true;
    if (lane == r) {
      sel_e = mi;
      sel_k = key;
      r_lo = lo_o;
      r_hi = hi_o;
    }
  }
  const bool rest = has && !taken;
  const uint32_t rh = __reduce_max_sync(0xffffffffu, rest ? static_cast<uint32_t>(my_hi >> 32) : 0u);
  const uint32_t rl = __reduce_max_sync(
      0xffffffffu, rest && static_cast<uint32_t>(my_hi >> 32) == rh ? static_cast<uint32_t>(my_hi) : 0u);
  const bool any_rest = __any_sync(0xffffffffu, rest);
  const unsigned long long restmax = (static_cast<unsigned long long>(rh) << 32) | rl;
  const unsigned long long next_hi = __shfl_down_sync(0xffffffffu, r_hi, 1);
  bool ok = true;
  if (lane + 1 < k) ok = r_lo > next_hi;
  if (lane == k - 1 && any_rest) ok = r_lo > restmax;
  return __all_sync(0xffffffffu, ok);
}

constexpr int kRfWarps = 8;

// Filter interval of expert e for token t: the approximate logit v plus the
// bias, widened by the error model above, rounded outward (-0 made +0).
__device__ __forceinline__ void filter_bounds(float v, float b, float xnt, float wne, float rs, float c0,
                                              float& lv, float& uv) {
  const float d = __fadd_ru(__fadd_ru(__fmul_ru(0x1p-9f, __fmul_ru(xnt, wne)), __fmul_ru(0x1p-22f, fabsf(v))),
                            __fmaf_ru(rs, wne, c0));
  lv = __fadd_rn(__fsub_rd(__fadd_rd(v, b), d), 0.f);
  uv = __fadd_rn(__fadd_ru(__fadd_ru(v, b), d), 0.f);
}

// One chunk of a lane's share of a logit: the weights of groups g0 + 32 m
// (m < 8) of four products each, 32 products; groups past the row are zero.
struct RfChunk {
  float4 w[8];
};
__device__ __forceinline__ void rf_load(RfChunk& c, const float* wr, int g0, int ng) {
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int g = g0 + 32 * m;
    c.w[m] = g < ng ? __ldg(reinterpret_cast<const float4*>(wr) + g) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}
// The chunk's 32 products (activations xs: the token row in fp32, zero past
// the row) as four independent sums of eight (one per component of the
// groups), combined error-free: chunk sum s plus the error e of the
// combination.
__device__ __forceinline__ void rf_dot(const RfChunk& c, const float* xs, int g0, float& s, float& e) {
  float2 p01 = make_float2(0.f, 0.f), p23 = make_float2(0.f, 0.f);  // paired FMAs, each lane of a pair rounded alone
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float4 x4 = reinterpret_cast<const float4*>(xs)[g0 + 32 * m];
    p01 = __ffma2_rn(make_float2(x4.x, x4.y), make_float2(c.w[m].x, c.w[m].y), p01);
    p23 = __ffma2_rn(make_float2(x4.z, x4.w), make_float2(c.w[m].z, c.w[m].w), p23);
  }
  float s01, e01, s23, e23, e2;
  two_sum(p01.x, p01.y, s01, e01);
  two_sum(p23.x, p23.y, s23, e23);
  two_sum(s01, s23, s, e2);
  e = __fadd_rn(__fadd_rn(e01, e23), e2);
}

// Chunked logits of the warp's C <= 32 candidates cand[0..C) against the
// token row xs (fp32, shared memory), as one stream of (candidate, chunk)
// steps with the weight loads of two steps in flight. Each lane's chunk of 32 products is four plain-FMA sums
// of eight; their combination and the fold of every chunk into (hi, lo) are
// error-free, and the lanes are combined error-free, so the chunk error
// stays within gamma_8 <= gamma_32 of its magnitudes and chunked_keys
// applies. Lane j ends with candidate j's (hi, lo).
__device__ void rf_candidate_logits(const RouteArgs& a, const float* xs, const int* cand, int C, float& my_hi,
                                    float& my_lo) {
  const int lane = threadIdx.x & 31;
  const int H = a.H, ng = H >> 2;
  const int nch = (((ng + 31) >> 5) + 7) >> 3;  // chunks per logit
  const int S = C * nch;
  RfChunk A, B;
  int lj = 0, lc = 0;  // (candidate, chunk) of the next load
  auto load = [&](RfChunk& c) {
    rf_load(c, a.w + static_cast<size_t>(cand[lj]) * H, lane + 256 * lc, ng);
    if (++lc == nch) {
      lc = 0;
      ++lj;
    }
  };
  float hi = 0.f, lo = 0.f;
  int sj = 0, sc = 0;  // (candidate, chunk) of the next step
  auto step = [&](const RfChunk& c) {
    float cs, ce, ns, es;
    rf_dot(c, xs, lane + 256 * sc, cs, ce);
    two_sum(hi, cs, ns, es);
    hi = ns;
    lo = __fadd_rn(lo, __fadd_rn(ce, es));
    if (++sc == nch) {  // the candidate's last chunk: combine the lanes
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, off);
        const float l2 = __shfl_xor_sync(0xffffffffu, lo, off);
        two_sum(hi, h2, ns, es);
        hi = ns;
        lo = __fadd_rn(__fadd_rn(lo, l2), es);
      }
      if (lane == sj) {
        my_hi = hi;
        my_lo = lo;
      }
      hi = 0.f;
      lo = 0.f;
      sc = 0;
      ++sj;
    }
  };
  if (S > 0) load(A);
  if (S > 1) load(B);
  for (int s = 0; s < S; s += 2) {
    step(A);
    if (s + 2 < S) load(A);
    if (s + 1 < S) {
      step(B);
      if (s + 3 < S) load(B);
    }
  }
}

// Compensated logits (error-free products by FMA, error-free sums, fp32
// error accumulators; Ogita, Rump and Oishi 2005) of the warp's C <= 32
// experts cand[0..C) against the token row xs (fp32, shared memory), streamed as
// rf_candidate_logits streams the chunked ones. Each lane keeps four such
// sums (one per component of the groups), combined error-free per
// candidate, then the lanes. Keys as the few-token router's:
// |exact - (S + C)| <= (D u)^2 (1 + 2 D u) sum |x w| with D = terms per lane
// + 10, above the summation depth. Lane j ends with candidate j's keys.
__device__ void rf_candidate_compensated(const RouteArgs& a, const float* xs, const int* cand, int C,
                                         const float* s_b, unsigned long long& my_l, unsigned long long& my_lo,
                                         unsigned long long& my_hi) {
  const int lane = threadIdx.x & 31;
  const int H = a.H, ng = H >> 2;
  const int nch = (((ng + 31) >> 5) + 7) >> 3;
  const int S = C * nch;
  RfChunk A, B;
  int lj = 0, lc = 0;
  auto load = [&](RfChunk& c) {
    rf_load(c, a.w + static_cast<size_t>(cand[lj]) * H, lane + 256 * lc, ng);
    if (++lc == nch) {
      lc = 0;
      ++lj;
    }
  };
  float s[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f}, ab[4] = {0.f, 0.f, 0.f, 0.f};
  float rs = 0.f, rc = 0.f, rab = 0.f;  // lane j: candidate j's sums
  int sj = 0, sc = 0;
  auto step = [&](const RfChunk& ch) {
    const int g0 = lane + 256 * sc;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float4 x4 = reinterpret_cast<const float4*>(xs)[g0 + 32 * m];
      const float xv[4] = {x4.x, x4.y, x4.z, x4.w};
      const float wv[4] = {ch.w[m].x, ch.w[m].y, ch.w[m].z, ch.w[m].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float pr = __fmul_rn(xv[q], wv[q]);
        const float ep = fmaf(xv[q], wv[q], -pr);  // exact low part of the product
        float ns, es;
        two_sum(s[q], pr, ns, es);
        s[q] = ns;
        c[q] = __fadd_rn(c[q], __fadd_rn(ep, es));
        ab[q] = fmaf(fabsf(xv[q]), fabsf(wv[q]), ab[q]);
      }
    }
    if (++sc == nch) {
      float ss, es, s01, s23, e01, e23;
      two_sum(s[0], s[1], s01, e01);
      two_sum(s[2], s[3], s23, e23);
      two_sum(s01, s23, ss, es);
      float cc = __fadd_rn(__fadd_rn(__fadd_rn(c[0], c[1]), __fadd_rn(c[2], c[3])), __fadd_rn(__fadd_rn(e01, e23), es));
      float aa = __fadd_rn(__fadd_rn(ab[0], ab[1]), __fadd_rn(ab[2], ab[3]));
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, ss, off);
        const float c2 = __shfl_xor_sync(0xffffffffu, cc, off);
        const float a2 = __shfl_xor_sync(0xffffffffu, aa, off);
        float ns, e2;
        two_sum(ss, s2, ns, e2);
        ss = ns;
        cc = __fadd_rn(__fadd_rn(cc, c2), e2);
        aa = __fadd_rn(aa, a2);
      }
      if (lane == sj) {
        rs = ss;
        rc = cc;
        rab = aa;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) s[q] = c[q] = ab[q] = 0.f;
      sc = 0;
      ++sj;
    }
  };
  if (S > 0) load(A);
  if (S > 1) load(B);
  for (int st = 0; st < S; st += 2) {
    step(A);
    if (st + 2 < S) load(A);
    if (st + 1 < S) {
      step(B);
      if (st + 3 < S) load(B);
    }
  }
  if (lane < C) {
    const int nterm = 4 * (((H >> 2) + 31) / 32);
    const double l = (static_cast<double>(rs) + static_cast<double>(rc)) + static_cast<double>(s_b[cand[lane]]);
    const double Du = static_cast<double>(nterm + 5 + 5) * 0x1p-24;
    const double bnd = Du * Du * (1.0 + 2.0 * Du) * 1.01 * static_cast<double>(rab) + fabs(l) * 0x1p-51 +
                       static_cast<double>(H + 1) * 0x1p-140;
    const double wid = __dadd_ru(bnd, __dmul_ru(fabs(l), 0x1p-50));
    const bool fin = isfinite(l) && isfinite(wid);
    my_l = okey(l);
    my_lo = fin ? okey(__dsub_rd(l, wid)) : 0ull;
    my_hi = fin ? okey(__dadd_ru(l, wid)) : ~0ull;
  }
}

// One warp per token: the filter over the approximate logits, certified
// logits of the candidates, selection and combine weights; or, for a token
// left uncertified, full keys and flag 2 for select_kernel and repair_kernel.
template <int NPL>
__device__ void refine_token(const RouteArgs& a, int t, const float* approx, const float (&va)[NPL], float xnt,
                             int* flags, const float* s_wn, const float* s_b, int* cand, int* amb_list, float* xs) {
  const int lane = threadIdx.x & 31;
  const int E = a.E, H = a.H, k = a.k;
  const float rs = __fmul_ru(0x1p-124f, __fsqrt_ru(static_cast<float>(H)));
  const float c0 = static_cast<float>(2 * H + 2) * 0x1p-126f;
  const float* ar = approx + static_cast<size_t>(t) * E;
  const uint16_t* xr = static_cast<const uint16_t*>(a.x) + static_cast<size_t>(t) * H;
  const size_t te = static_cast<size_t>(a.T) * E, o = static_cast<size_t>(t) * E;
  const unsigned lt = (1u << lane) - 1u;
  // the k-th largest lower bound (with multiplicity) and the candidates in
  // expert order: upper bound >= it (every expert if a bound is not finite
  // or, on the second pass, if the filter's model failed)
  uint32_t thr = 0u;
  uint32_t cmask = 0u;  // bit i: expert i * 32 + lane is a candidate
  bool all;
  {
    uint32_t lk[NPL], uk[NPL];
    bool bad = !isfinite(xnt);
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = i * 32 + lane;
      lk[i] = uk[i] = 0u;  // below every finite bound
      if (e < E) {
        float lv, uv;
        filter_bounds(va[i], s_b[e], xnt, s_wn[e], rs, c0, lv, uv);
        bad |= !(isfinite(lv) && isfinite(uv));
        lk[i] = fkey(lv);
        uk[i] = fkey(uv);
      }
    }
    all = __any_sync(0xffffffffu, bad);
    if (!all) {
      // each lane sorts its keys (descending; absent experts are 0, below
      // every bound); each round the lowest lane holding the largest head
      // pops it
      uint32_t sk[NPL];
#pragma unroll
      for (int i = 0; i < NPL; ++i) sk[i] = lk[i];
#pragma unroll
      for (int p = 0; p < NPL; ++p)
#pragma unroll
        for (int i = p & 1; i + 1 < NPL; i += 2) {
          const uint32_t hi2 = max(sk[i], sk[i + 1]), lo2 = min(sk[i], sk[i + 1]);
          sk[i] = hi2;
          sk[i + 1] = lo2;
        }
      for (int r = 0; r < k; ++r) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, sk[0]);
        const unsigned own = __ballot_sync(0xffffffffu, sk[0] == m);
        if (lane == __ffs(own) - 1) {
#pragma unroll
          for (int i = 0; i + 1 < NPL; ++i) sk[i] = sk[i + 1];
          sk[NPL - 1] = 0u;
        }
        thr = m;
      }
    }
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (i * 32 + lane < E && (all || uk[i] >= thr)) cmask |= 1u << i;
  }
  for (int pass = 0; pass < 2; ++pass) {
    int C = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const bool c = (cmask >> i) & 1u;
      const unsigned bal = __ballot_sync(0xffffffffu, c);
      if (c && C + __popc(bal & lt) < 32) cand[C + __popc(bal & lt)] = i * 32 + lane;
      C += __popc(bal);
    }
    __syncwarp();
    if (C <= 32) {
      int my_e = lane < C ? cand[lane] : -1;
      unsigned long long my_l = 0ull, my_lo = 0ull, my_hi = 0ull;
      {
        float ch = 0.f, cl = 0.f;
        rf_candidate_logits(a, xs, cand, C, ch, cl);
        if (lane < C) chunked_keys(ch, cl, s_b[my_e], xnt, s_wn[my_e], H, my_l, my_lo, my_hi);
      }
      // the certified interval must meet the filter interval (the model of
      // the tensor cores' error, checked on every candidate)
      bool consistent = true;
      if (!all && lane < C) {
        float lv, uv;
        filter_bounds(__ldg(ar + my_e), s_b[my_e], xnt, s_wn[my_e], rs, c0, lv, uv);
        consistent = !(okey_value(my_hi) < static_cast<double>(lv) || okey_value(my_lo) > static_cast<double>(uv));
      }
      if (__all_sync(0xffffffffu, consistent)) {
        int sel_e = -1;
        unsigned long long sel_k = 0ull;
        bool ok = cand_select(C, k, my_e, my_l, my_lo, my_hi, sel_e, sel_k);
        if (!ok) {
          // the candidates whose rank the intervals leave open (fewer than k
          // others certainly above them) and whose interval meets another
          // such candidate's get the compensated logits, some five orders of
          // magnitude tighter
          int above = 0;
          for (int i = 0; i < C; ++i) {
            const unsigned long long loi = __shfl_sync(0xffffffffu, my_lo, i);
            above += (i != lane && loi > my_hi) ? 1 : 0;
          }
          const bool open = lane < C && above < k;
          bool meets = false;
          for (int i = 0; i < C; ++i) {
            const unsigned long long loi = __shfl_sync(0xffffffffu, my_lo, i);
            const unsigned long long hii = __shfl_sync(0xffffffffu, my_hi, i);
            const bool oi = __shfl_sync(0xffffffffu, open, i);
            meets |= open && oi && i != lane && !(my_lo > hii || loi > my_hi);
          }
          const unsigned amb = __ballot_sync(0xffffffffu, meets);
          if (meets) amb_list[__popc(amb & lt)] = my_e;
          __syncwarp();
          unsigned long long kl = 0ull, klo = 0ull, khi = 0ull;
          rf_candidate_compensated(a, xs, amb_list, __popc(amb), s_b, kl, klo, khi);
          const int src = __popc(amb & lt) & 31;
          const unsigned long long nl = __shfl_sync(0xffffffffu, kl, src);
          const unsigned long long nlo = __shfl_sync(0xffffffffu, klo, src);
          const unsigned long long nhi = __shfl_sync(0xffffffffu, khi, src);
          if (meets) {
            my_l = nl;
            my_lo = nlo;
            my_hi = nhi;
          }
          ok = cand_select(C, k, my_e, my_l, my_lo, my_hi, sel_e, sel_k);
        }
        if (ok) {
          const unsigned long long k0 = __shfl_sync(0xffffffffu, sel_k, 0);
          float z = 0.f;
          if (lane < k) z = expf(static_cast<float>(okey_value(sel_k) - okey_value(k0)));
          float sum = 0.f;
          for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, z, j);  // fixed order
          if (lane < k) {
            a.topk_idx[static_cast<size_t>(t) * k + lane] = sel_e;
            a.topk_w[static_cast<size_t>(t) * k + lane] = z / sum;
          }
          if (lane == 0) flags[t] = 0;
          return;
        }
        // full keys: the candidates' (lane j holds the j-th), a key below
        // every logit for the others
        int base = 0;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          const int e = i * 32 + lane;
          const bool c = (cmask >> i) & 1u;
          const unsigned bal = __ballot_sync(0xffffffffu, c);
          const int src = (base + __popc(bal & lt)) & 31;
          const unsigned long long vl = __shfl_sync(0xffffffffu, my_l, src);
          const unsigned long long vlo = __shfl_sync(0xffffffffu, my_lo, src);
          const unsigned long long vhi = __shfl_sync(0xffffffffu, my_hi, src);
          if (e < E) {
            a.keys[o + e] = c ? vl : 1ull;
            a.keys[te + o + e] = c ? vlo : 1ull;
            a.keys[2 * te + o + e] = c ? vhi : 1ull;
          }
          base += __popc(bal);
        }
        if (lane == 0) flags[t] = 2;
        return;
      }
      // the filter's model failed for this token: every expert
      if (lane == 0) atomicAdd(a.repairs + 1, 1ull);
      all = true;
      cmask = 0u;
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (i * 32 + lane < E) cmask |= 1u << i;
      __syncwarp();
      continue;
    }
    // more than 32 candidates: every candidate's chunked keys, written by
    // lane 0 in turn, the others a key below every logit
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = i * 32 + lane;
      if (e < E && !((cmask >> i) & 1u)) a.keys[o + e] = a.keys[te + o + e] = a.keys[2 * te + o + e] = 1ull;
    }
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      unsigned bal = __ballot_sync(0xffffffffu, (cmask >> i) & 1u);
      while (bal) {
        const int e = i * 32 + __ffs(bal) - 1;
        bal &= bal - 1;
        float hi, lo;
        warp_dot_chunked(xr, a.w + static_cast<size_t>(e) * H, H, hi, lo);
        if (lane == 0) {
          unsigned long long kl, klo, khi;
          chunked_keys(hi, lo, s_b[e], xnt, s_wn[e], H, kl, klo, khi);
          a.keys[o + e] = kl;
          a.keys[te + o + e] = klo;
          a.keys[2 * te + o + e] = khi;
        }
      }
    }
    if (lane == 0) flags[t] = 2;
    return;
  }
}

// Activations of one warp's token in shared memory: chunks of 256 groups of
// four fp32 values (zero past the row).
__device__ __forceinline__ int rf_chunks(int H) { return (((H >> 2) + 31) / 32 + 7) / 8; }
size_t rf_smem_bytes(int H) { return static_cast<size_t>(kRfWarps) * ((((H >> 2) + 31) / 32 + 7) / 8) * 4096; }

// One warp per token; the token's activations are staged once, in fp32, in
// the warp's part of the shared memory.
template <int NPL>
__global__ void __launch_bounds__(kRfWarps * 32, 2) refine_kernel(RouteArgs a, const float* approx, const float* wn,
                                                                  int* flags) {
  extern __shared__ float4 rf_dyn[];
  __shared__ float s_wn[1024], s_b[1024];
  __shared__ int s_cand[kRfWarps][32], s_amb[kRfWarps][32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < a.E; e += kRfWarps * 32) {
    s_wn[e] = __ldg(wn + e);
    s_b[e] = a.bias ? __ldg(a.bias + e) : 0.f;
  }
  __syncthreads();
  const int t = blockIdx.x * kRfWarps + warp;
  if (t >= a.T) return;
  const int ngp = rf_chunks(a.H) * 256;  // groups of the padded row
  float4* xs = rf_dyn + static_cast<size_t>(warp) * ngp;
  // the token's approximate logits are loaded first, so that their round
  // trip overlaps the staging of the activations
  float va[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = i * 32 + lane;
    va[i] = e < a.E ? __ldcs(approx + static_cast<size_t>(t) * a.E + e) : 0.f;
  }
  const uint2* xr = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.x) + static_cast<size_t>(t) * a.H);
  float ss = 0.f;
  for (int g = lane; g < ngp; g += 32) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (g < (a.H >> 2)) {
      const uint2 b = __ldg(xr + g);
      v = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u), __uint_as_float(b.y << 16),
                      __uint_as_float(b.y & 0xFFFF0000u));
    }
    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
    xs[g] = v;
  }
  for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  // the token's norm bound, as row_norms_kernel's (within a relative 1e-3)
  const float nrm = sqrtf(ss) * 1.001f;
  __syncwarp();
  refine_token<NPL>(a, t, approx, va, isfinite(nrm) ? nrm : INFINITY, flags, s_wn, s_b, s_cand[warp], s_amb[warp],
                    reinterpret_cast<float*>(xs));
}

constexpr int kRfMaxH = 6144;  // the refining kernel's activations fit shared memory

template <int NPL>
cudaError_t launch_refine(int grid, size_t smem, const RouteArgs& a, const float* approx, const float* wn, int* flags,
                          cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(refine_kernel<NPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  refine_kernel<NPL><<<grid, kRfWarps * 32, smem, st>>>(a, approx, wn, flags);
  return cudaGetLastError();
}

// ---- multi-block plan: per-block counts, one scan, per-block stable scatter
constexpr int kPB = 256;  // assignments per block

__global__ void __launch_bounds__(kPB) plan_count_kernel(PlanArgs a, int* local) {
  extern __shared__ int hist[];
  const int E = a.E, A = a.T * a.k, b = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += kPB) hist[e] = 0;
  __syncthreads();
  const int i = b * kPB + threadIdx.x;
  if (i < A) {
    const int e = __ldg(a.idx + i);
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else
      atomicOr(a.err, MOE_DEVERR_BADIDX);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kPB) {
    local[static_cast<size_t>(b) * E + e] = hist[e];
    if (hist[e]) atomicAdd(a.plan.counts + e, hist[e]);
  }
}

__global__ void __launch_bounds__(1024) plan_scan_kernel(PlanArgs a, int* local, int nb) {
  extern __shared__ int sm[];
  const int E = a.E;
  int* cnt = sm;
  int* cur = sm + E;
  int* scratch = sm + 2 * E;
  for (int e = threadIdx.x; e < E; e += 1024) {
    cnt[e] = __ldcg(a.plan.counts + e);
    cur[e] = cnt[e] > 0 ? 1 : 0;
  }
  __syncthreads();
  const int nu = block_exclusive_scan<1024>(cur, E, scratch);
  for (int e = threadIdx.x; e < E; e += 1024)
    if (cnt[e] > 0) a.plan.uniq[cur[e]] = e;
  if (threadIdx.x == 0) *a.plan.n_uniq = nu;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += 1024) cur[e] = cnt[e];
  __syncthreads();
  const int total = block_exclusive_scan<1024>(cur, E, scratch);
  for (int e = threadIdx.x; e < E; e += 1024) a.plan.offsets[e] = cur[e];
  // each expert's per-block counts become per-block offsets: G threads per
  // expert each take a run of blocks (loads batched ahead of the stores)
  constexpr int kB = 8;
  const int G = max(1, 1024 / E);
  const int seg = (nb + G - 1) / G;
  int* segsum = sm + 2 * E + 33;  // [G][E]
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * E; idx += 1024) {
    const int e = idx % E, g = idx / E;
    const int b0 = g * seg, b1 = min(nb, b0 + seg);
    int sum = 0;
    for (int b = b0; b < b1; b += kB) {
      int v[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) v[j] = b + j < b1 ? __ldcg(local + static_cast<size_t>(b + j) * E + e) : 0;
#pragma unroll
      for (int j = 0; j < kB; ++j) sum += v[j];
    }
    segsum[g * E + e] = sum;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * E; idx += 1024) {
    const int e = idx % E, g = idx / E;
    const int b0 = g * seg, b1 = min(nb, b0 + seg);
    int run = cur[e];
    for (int g2 = 0; g2 < g; ++g2) run += segsum[g2 * E + e];
    for (int b = b0; b < b1; b += kB) {
      int v[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) v[j] = b + j < b1 ? __ldcg(local + static_cast<size_t>(b + j) * E + e) : 0;
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        if (b + j < b1) local[static_cast<size_t>(b + j) * E + e] = run;
        run += v[j];
      }
    }
  }
  if (threadIdx.x == 0) a.plan.offsets[E] = total;
}

__global__ void __launch_bounds__(kPB) plan_scatter_kernel(PlanArgs a, const int* local) {
  extern __shared__ int wcount[];  // [8 warps][E]
  const int E = a.E, A = a.T * a.k, b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 8 * E; i += kPB) wcount[i] = 0;
  __syncthreads();
  const int i = b * kPB + tid;
  const int e = i < A ? __ldg(a.idx + i) : -1;
  const bool valid = e >= 0 && e < E;
  const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1 - lane);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid && (__ffs(peers) - 1) == lane) wcount[warp * E + e] = __popc(peers);
  __syncthreads();
  if (valid) {
    int pos = __ldg(local + static_cast<size_t>(b) * E + e) + rank;
    for (int w2 = 0; w2 < warp; ++w2) pos += wcount[w2 * E + e];
    a.plan.perm_tok[pos] = i / a.k;
    a.plan.perm_rank[pos] = i % a.k;
    a.plan.perm_w[pos] = __ldg(a.w + i);
    a.plan.inv[i] = pos;
  }
}

__global__ void admit_kernel(AdmitArgs A, moe_plan_t P, uint32_t* err) {
  extern __shared__ unsigned char asm_smem[];
  if (threadIdx.x < 32) admit_warp(A, P, asm_smem, err);
}

}  // namespace

size_t router_split_bytes(int E, int H) {
  return static_cast<size_t>((E + kTcExp - 1) / kTcExp) * 2 * kTcExp * static_cast<size_t>(H) * 2;
}

cudaError_t launch_route_large(const RouteArgs& a, float* norms, int* flags, float2* part, uint16_t* wsplit,
                               int num_sms, cudaStream_t st) {
  if (a.T < 1 || a.k > 16 || a.E > 1024 || a.H % kLK) return cudaErrorInvalidValue;
  const int slices = a.H % (kLK * 4) == 0 ? 4 : (a.H % (kLK * 2) == 0 ? 2 : 1);
  float* xn = norms;
  float* wn = norms + a.T;
  if (wsplit && a.xt == MOE_BF16 && a.H % kTcBK == 0 && a.H <= kRfMaxH && encoder() == cudaSuccess) {
    // tensor-core filter, certified logits of the candidates, then the
    // per-token selection and exact repair of the tokens it left (the norm
    // bounds come from the split and the refining kernels)
    const int nb = (a.E + kTcExp - 1) / kTcExp;
    router_split_kernel<<<nb * kTcExp, 128, 0, st>>>(a.w, a.E, a.H, wsplit, wn);
    CUtensorMap mx, mw;
    cudaError_t e = map16(&mx, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.T, a.H, kTcTok);
    if (e != cudaSuccess) return e;
    e = map16(&mw, wsplit, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<int64_t>(nb) * 2 * kTcExp, a.H, 2 * kTcExp);
    if (e != cudaSuccess) return e;
    float* approx = reinterpret_cast<float*>(part);
    const TcArgs ta{a.T, a.E, a.H, approx, a.err, kTcWaitCycles};
    e = cudaFuncSetAttribute(logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kTcSmem));
    if (e != cudaSuccess) return e;
    logits_tc_kernel<<<dim3((a.T + kTcTok - 1) / kTcTok, nb), 128, kTcSmem, st>>>(mx, mw, ta);
    const int rg = (a.T + kRfWarps - 1) / kRfWarps;
    const size_t rsm = rf_smem_bytes(a.H);
    (void)num_sms;
    if (a.E <= 32)
      e = launch_refine<1>(rg, rsm, a, approx, wn, flags, st);
    else if (a.E <= 64)
      e = launch_refine<2>(rg, rsm, a, approx, wn, flags, st);
    else if (a.E <= 128)
      e = launch_refine<4>(rg, rsm, a, approx, wn, flags, st);
    else if (a.E <= 256)
      e = launch_refine<8>(rg, rsm, a, approx, wn, flags, st);
    else if (a.E <= 512)
      e = launch_refine<16>(rg, rsm, a, approx, wn, flags, st);
    else
      e = launch_refine<32>(rg, rsm, a, approx, wn, flags, st);
    if (e != cudaSuccess) return e;
    select_kernel<<<(a.T + 7) / 8, 256, 0, st>>>(a, flags, 1);
    repair_kernel<MOE_BF16><<<std::min((a.T + 31) / 32, kRepairGrid), kRouteThreads, 0, st>>>(a, flags);
    return cudaGetLastError();
  }
  const int nrows = a.T + a.E;
  if (a.xt == MOE_BF16)
    row_norms_kernel<MOE_BF16><<<(nrows + 7) / 8, 256, 0, st>>>(a.x, a.T, a.w, a.E, a.H, xn, wn);
  else
    row_norms_kernel<MOE_F32><<<(nrows + 7) / 8, 256, 0, st>>>(a.x, a.T, a.w, a.E, a.H, xn, wn);
  dim3 grid((a.E + kLE - 1) / kLE, (a.T + kLT - 1) / kLT, slices);
  if (a.xt == MOE_BF16)
    logits_tiled_kernel<MOE_BF16><<<grid, kLThreads, 0, st>>>(a, part);
  else
    logits_tiled_kernel<MOE_F32><<<grid, kLThreads, 0, st>>>(a, part);
  logits_keys_kernel<<<dim3((a.E + 255) / 256, a.T), 256, 0, st>>>(a, part, slices, xn, wn);
  select_kernel<<<(a.T + 7) / 8, 256, 0, st>>>(a, flags, 0);
  if (a.xt == MOE_BF16)
    repair_kernel<MOE_BF16><<<std::min((a.T + 31) / 32, kRepairGrid), kRouteThreads, 0, st>>>(a, flags);
  else
    repair_kernel<MOE_F32><<<std::min((a.T + 31) / 32, kRepairGrid), kRouteThreads, 0, st>>>(a, flags);
  return cudaGetLastError();
}

int plan_blocks(int A) { return (A + kPB - 1) / kPB; }

cudaError_t launch_plan_large(const PlanArgs& a, int* local, cudaStream_t st) {
  const int A = a.T * a.k, nb = plan_blocks(A);
  cudaError_t e = cudaMemsetAsync(a.plan.counts, 0, sizeof(int32_t) * a.E, st);
  if (e != cudaSuccess) return e;
  plan_count_kernel<<<nb, kPB, sizeof(int) * a.E, st>>>(a, local);
  plan_scan_kernel<<<1, 1024, sizeof(int) * (2 * a.E + 33 + std::max(a.E, 1024)), st>>>(a, local, nb);
  plan_scatter_kernel<<<nb, kPB, sizeof(int) * 8 * a.E, st>>>(a, local);
  return cudaGetLastError();
}

cudaError_t launch_admit(const AdmitArgs& A, const moe_plan_t& P, int max_units, uint32_t* err,
                         cudaStream_t st) {
  const size_t smem = admit_smem_bytes(A.E, A.S, max_units);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(admit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  admit_kernel<<<1, 32, smem, st>>>(A, P, err);
  return cudaGetLastError();
}

}  // namespace moe
