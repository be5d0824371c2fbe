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
#include <cfloat>
#include <climits>
#include <mutex>
#include <string>

#include "internal.h"

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
struct Cand {
  double v;
  int e;
};
__device__ __forceinline__ bool better(double v, int e, double bv, int be) {
  return v > bv || (v == bv && e < be);
}

// Top-k of one token by a warp. Returns the selection in sel (all lanes) and
// whether the bounds certify it.
__device__ bool warp_select(const double* l, const double* bnd, int E, int k, int* sel,
                            bool certify) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;
  for (int r = 0; r < k; ++r) {
    double bv = -DBL_MAX;
    int be = INT_MAX;
    for (int i = 0; i * 32 + lane < E; ++i) {
      if ((taken >> i) & 1u) continue;
      int e = i * 32 + lane;
      double v = __ldcg(l + e);
      if (be == INT_MAX || better(v, e, bv, be)) {
        bv = v;
        be = e;
      }
    }
    for (int off = 16; off; off >>= 1) {
      double ov = __shfl_xor_sync(0xffffffffu, bv, off);
      int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (oe != INT_MAX && (be == INT_MAX || better(ov, oe, bv, be))) {
        bv = ov;
        be = oe;
      }
    }
    sel[r] = be;
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
  }
  if (!certify) return true;
  // interval [l - b, l + b] widened by 2^-50 |l| so that disjoint intervals
  // also separate the correctly rounded fp64 images
  auto lower = [&](int e) {
    double v = __ldcg(l + e), b = __ldcg(bnd + e);
    return v - b - fabs(v) * 0x1p-50;
  };
  auto upper = [&](int e) {
    double v = __ldcg(l + e), b = __ldcg(bnd + e);
    return v + b + fabs(v) * 0x1p-50;
  };
  bool ok = true;
  for (int j = 0; j + 1 < k; ++j) ok &= lower(sel[j]) > upper(sel[j + 1]);
  double up = -DBL_MAX;
  bool any = false;
  for (int i = 0; i * 32 + lane < E; ++i) {
    if ((taken >> i) & 1u) continue;
    double u = upper(i * 32 + lane);
    if (!any || !(u <= up)) up = u;  // NaN propagates as "uncertified"
    any = true;
  }
  for (int off = 16; off; off >>= 1) {
    double o = __shfl_xor_sync(0xffffffffu, up, off);
    int oa = __shfl_xor_sync(0xffffffffu, any ? 1 : 0, off);
    if (oa) {
      if (!any || !(o <= up)) up = o;
      any = true;
    }
  }
  if (any) ok &= lower(sel[k - 1]) > up;
  return __all_sync(0xffffffffu, ok);
}

__device__ void warp_write_selection(const double* l, const int* sel, int k, int32_t* idx,
                                     float* w) {
  const int lane = threadIdx.x & 31;
  double m = __ldcg(l + sel[0]);
  double z = 0.0;
  if (lane < k) z = exp(__ldcg(l + sel[lane]) - m);
  double sum = 0.0;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, z, j);  // fixed order
  if (lane < k) {
    idx[lane] = sel[lane];
    w[lane] = static_cast<float>(z / sum);
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

constexpr int kPlanThreads = 256;

size_t plan_smem_bytes(int E) {
  return sizeof(int) * (2 * E + (kPlanThreads / 32) * E + kPlanThreads / 32 + 1);
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
  const int nterm = (H + kRouteThreads - 1) / kRouteThreads;

  for (int t0 = 0; t0 < T; t0 += kRouteTB) {
    float s[kRouteTB], c[kRouteTB], ab[kRouteTB];
#pragma unroll
    for (int i = 0; i < kRouteTB; ++i) s[i] = c[i] = ab[i] = 0.f;
    for (int kk = tid; kk < H; kk += kRouteThreads) {
      const float wv = __ldg(wrow + kk);
#pragma unroll
      for (int i = 0; i < kRouteTB; ++i) {
        if (t0 + i < T) {
          const float xv = load_x<XT>(a.x, static_cast<size_t>(t0 + i) * H + kk);
          const float p = __fmul_rn(xv, wv);
          const float ep = fmaf(xv, wv, -p);  // exact low part of the product
          float ns, es;
          two_sum(s[i], p, ns, es);
          s[i] = ns;
          c[i] = __fadd_rn(c[i], __fadd_rn(ep, es));
          ab[i] = fmaf(fabsf(xv), fabsf(wv), ab[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kRouteTB; ++i) {
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
      const size_t o = static_cast<size_t>(t0 + tid) * E + e;
      a.l_est[o] = l;
      a.l_bnd[o] = isfinite(bnd) ? bnd : INFINITY;
    }
    __syncthreads();
  }

  // ---- the last block to finish selects for every token
  __threadfence();
  if (tid == 0) s_ticket = atomicAdd(a.ticket, 1u);
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  __threadfence();
  if (tid == 0) s_nflag = 0;
  __syncthreads();
  int sel[16];
  for (int t = warp; t < T; t += kRouteWarps) {
    const double* l = a.l_est + static_cast<size_t>(t) * E;
    const double* b = a.l_bnd + static_cast<size_t>(t) * E;
    bool ok = warp_select(l, b, E, a.k, sel, true);
    if (ok) {
      warp_write_selection(l, sel, a.k, a.topk_idx + static_cast<size_t>(t) * a.k,
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
        a.l_est[static_cast<size_t>(t) * E + ee] = v;
        a.l_bnd[static_cast<size_t>(t) * E + ee] = 0.0;
      }
    }
  }
  __syncthreads();
  for (int fi = warp; fi < nflag; fi += kRouteWarps) {
    const int t = s_flagged[fi];
    const double* l = a.l_est + static_cast<size_t>(t) * E;
    warp_select(l, nullptr, E, a.k, sel, false);
    warp_write_selection(l, sel, a.k, a.topk_idx + static_cast<size_t>(t) * a.k,
                         a.topk_w + static_cast<size_t>(t) * a.k);
    if (lane == 0) atomicAdd(a.repairs, 1ull);
  }
  if (a.plan.counts != nullptr) {
    __syncthreads();
    plan_block<kRouteThreads>(a.topk_idx, a.topk_w, T * a.k, a.k, E, a.plan, dyn_smem, a.err);
  }
  if (tid == 0) *a.ticket = 0u;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  extern __shared__ int dyn_smem[];
  plan_block<kPlanThreads>(a.idx, a.w, a.T * a.k, a.k, a.E, a.plan, dyn_smem, a.err);
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t st) {
  (void)num_sms;
  if (a.T < 1 || a.T > kRouteMaxT || a.k > 16 || a.E > 1024) return cudaErrorInvalidValue;
  const size_t smem = a.plan.counts ? plan_smem_bytes(a.E) : 0;
  if (a.xt == MOE_BF16)
    route_kernel<MOE_BF16><<<a.E, kRouteThreads, smem, st>>>(a);
  else
    route_kernel<MOE_F32><<<a.E, kRouteThreads, smem, st>>>(a);
  return cudaGetLastError();
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
// kNoAllocMaxTE = 16384 (token, expert) logits (256 KiB of logits and bounds);
// every GPU that loads this library holds that array until the process exits.
namespace moe {
namespace {

constexpr int kNoAllocMaxTE = 16384;
constexpr int kNoAllocMaxDevices = 64;

// [0, TE) fast logits, [TE, 2 TE) bounds, then a 32-byte header:
// ticket (u32), error word (u32), repaired-token counter (u64).
static __device__ __align__(256) double g_route_scratch[2 * kNoAllocMaxTE + 4];

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
  if (T < 1 || T > kRouteMaxT || H < 1 || E < 1 || E > 1024 || k < 1 || k > 16 || k > E) {
    set_thread_error("moe_route_noalloc: need 1 <= T <= 64, H >= 1, 1 <= E <= 1024, "
                     "1 <= k <= min(16, E)");
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
  double* scratch = static_cast<double*>(base);
  const size_t te = static_cast<size_t>(T) * E;
  unsigned char* header = reinterpret_cast<unsigned char*>(scratch + 2 * kNoAllocMaxTE);
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
  a.l_est = scratch;
  a.l_bnd = scratch + te;
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
