// Prefill expert FFN driver: gather -> grouped gate/up GEMM -> grouped down
// GEMM -> combine.
//
// "Nanite for Experts" §5.3: each unique expert is scheduled once over all its
// tokens (expert-major rows); §5.5: per-expert results merge back into the
// tokens' original positions. The combine adds, per token, the shared
// expert's row and then its k routed rows in selection order, so the output
// is independent of scheduling and of the cache state.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "prefill.h"

namespace moe {
namespace {

// fp16 copy of the activations in expert-major order: row p < T*k is token
// perm_tok[p]; rows T*k .. T*k+T-1 are tokens 0..T-1 (the shared expert's).
// One warp per row; each lane keeps four 8-element loads in flight.
template <int XT>
__global__ void __launch_bounds__(256) gather_kernel(const void* x, int T, int k, int H,
                                                     const int32_t* perm_tok, __half* out, int rows) {
  const int p = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (p >= rows) return;
  const int A = T * k;
  const int t = p < A ? __ldg(perm_tok + p) : p - A;
  __half* dst = out + static_cast<int64_t>(p) * H;
  for (int i0 = lane * 8; i0 < H; i0 += 4 * 256) {
    float v[4][8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int i = i0 + g * 256;
      if (i >= H) continue;
      if (XT == MOE_BF16) {
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) +
                                                            static_cast<int64_t>(t) * H + i));
        const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[g][2 * j] = __uint_as_float(w[j] << 16);
          v[g][2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      } else {
        const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(x) +
                                                          static_cast<int64_t>(t) * H + i);
        const float4 c = __ldg(s), d = __ldg(s + 1);
        v[g][0] = c.x, v[g][1] = c.y, v[g][2] = c.z, v[g][3] = c.w;
        v[g][4] = d.x, v[g][5] = d.y, v[g][6] = d.z, v[g][7] = d.w;
      }
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int i = i0 + g * 256;
      if (i >= H) continue;
      __half2 h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = __floats2half2_rn(v[g][2 * j], v[g][2 * j + 1]);
      *reinterpret_cast<uint4*>(dst + i) = *reinterpret_cast<uint4*>(h);
    }
  }
}

// Work items of both GEMMs from the unit table: per unit, 192-token tiles
// times weight tiles (128 gate rows with the same 128 up rows, or 128 down
// rows); the weight tile varies fastest so that consecutive CTAs share a
// token tile. Unit-major order; the items are written by the whole block
// (each finds its unit by a binary search over the units' first items).
__global__ void __launch_bounds__(1024) items_kernel(const int32_t* units, int I, int Is, int H,
                                                     int32_t* items0, int32_t* n0, int32_t* items1,
                                                     int32_t* n1) {
  __shared__ int c0[1025], c1[1025], s_nt0[1024];
  const int nu = min(__ldg(units), 1024);
  const int u = threadIdx.x;
  const int nt1 = H / 128;
  int a = 0, b = 0;
  if (u < nu) {
    const int4 U = __ldg(reinterpret_cast<const int4*>(units + kUnitHeader) + u);
    const int mt = (U.z + kPrefillTok - 1) / kPrefillTok;
    const int nt0 = ((U.x == -1 ? Is : I) + 127) / 128;
    a = mt * nt0;
    b = mt * nt1;
    s_nt0[u] = nt0;
  }
  c0[u] = a;
  c1[u] = b;
  __syncthreads();
  if (u == 0) {
    int s0 = 0, s1 = 0;
    for (int i = 0; i < nu; ++i) {
      const int x0 = c0[i], x1 = c1[i];
      c0[i] = s0;
      c1[i] = s1;
      s0 += x0;
      s1 += x1;
    }
    c0[nu] = s0;
    c1[nu] = s1;
    *n0 = s0;
    *n1 = s1;
  }
  __syncthreads();
  const int tot0 = c0[nu], tot1 = c1[nu];
  for (int i = threadIdx.x; i < tot0; i += blockDim.x) {
    int lo = 0, hi = nu - 1;  // the last unit whose first item is <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (c0[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int j = i - c0[lo], nt = s_nt0[lo];
    reinterpret_cast<int4*>(items0)[i] = make_int4(lo, (j / nt) * kPrefillTok, (j % nt) * 128, 0);
  }
  for (int i = threadIdx.x; i < tot1; i += blockDim.x) {
    int lo = 0, hi = nu - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (c1[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int j = i - c1[lo];
    reinterpret_cast<int4*>(items1)[i] = make_int4(lo, (j / nt1) * kPrefillTok, (j % nt1) * 128, 0);
  }
}

// Publishes the new generations of one wave's fills once their copies are
// complete (stream order): list = [n, (slot, generation) x n]. Hits are not
// republished, so a slot whose earlier staging failed stays refused.
__global__ void __launch_bounds__(256) publish_kernel(const int32_t* list, uint32_t* gen) {
  const int n = __ldg(list);
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    gen[__ldg(list + 1 + 2 * i)] = static_cast<uint32_t>(__ldg(list + 2 + 2 * i));
}

// y[t] = shared row + sum over j in selection order of w[t,j] * row inv[t,j]
// (the weight of expert-major row p is perm_w[p]).
__global__ void __launch_bounds__(256) combine_kernel(const float* yp, const int32_t* inv, const float* w, int T,
                                                      int k, int H, int has_shared, float* y) {
  const int t = blockIdx.x;
  const int A = T * k;
  for (int i = threadIdx.x * 4; i < H; i += 256 * 4) {
    float4 acc = has_shared ? __ldg(reinterpret_cast<const float4*>(yp + static_cast<int64_t>(A + t) * H + i))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int p = __ldg(inv + t * k + j);
      const float wj = __ldg(w + p);
      const float4 v = __ldg(reinterpret_cast<const float4*>(yp + static_cast<int64_t>(p) * H + i));
      acc.x += wj * v.x;
      acc.y += wj * v.y;
      acc.z += wj * v.z;
      acc.w += wj * v.w;
    }
    *reinterpret_cast<float4*>(y + static_cast<int64_t>(t) * H + i) = acc;
  }
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t encoder() {
  if (g_encode) return cudaSuccess;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&g_encode),
                                                   12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !g_encode) return cudaErrorNotSupported;
  return cudaSuccess;
}

// 16-bit [rows][cols] token operand, 64 x box_rows boxes, 128-byte swizzle.
cudaError_t map16(CUtensorMap* m, const void* base, CUtensorMapDataType t, int64_t rows, int64_t cols,
                  int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, t, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

// Q8_0 quant planes in every slot: bytes x rows x matrix x slot. The box is
// 64 bytes x box_rows x n_mat: the gate/up GEMM reads the same rows of the
// gate plane and of the up plane (mat_stride bytes further) in one copy.
// The 64-byte swizzle lets the dequantising threads read one row each
// without bank conflicts.
cudaError_t mapq(CUtensorMap* m, const void* base, int64_t kbytes, int64_t rows, int64_t mat_stride, int n_mat,
                 int64_t slots, int64_t slot_stride, int box_rows) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(kbytes), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(n_mat), static_cast<cuuint64_t>(slots)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(kbytes), static_cast<cuuint64_t>(mat_stride),
                           static_cast<cuuint64_t>(slot_stride)};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(n_mat), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

// Work items, tensor maps and both GEMMs over the unit table p.units.
static cudaError_t prefill_gemms(const PrefillArgs& p, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  const int A = p.T * p.k, rows = A + p.T;
  const ExpertGeom& g = p.g;
  const ExpertGeom& gs = p.gs;
  if (p.publish_gen) publish_kernel<<<1, 256, 0, st>>>(p.publish_list, p.publish_gen);
  // 2. work items
  items_kernel<<<1, 1024, 0, st>>>(p.units, p.I, p.Is, p.H, p.items0, p.n_items0, p.items1, p.n_items1);
  // 3. tensor maps (pointers are fixed per context and layer)
  GemmMaps m0{}, m1{};
  const int64_t S = p.S;
  const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16, BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if ((e = map16(&m0.b32, p.x16, F16, rows, p.H, 32)) != cudaSuccess) return e;
  if ((e = map16(&m0.btile, p.x16, F16, rows, p.H, kPrefillTok)) != cudaSuccess) return e;
  if ((e = map16(&m1.b32, p.h, BF16, rows, p.ldh, 32)) != cudaSuccess) return e;
  if ((e = map16(&m1.btile, p.h, BF16, rows, p.ldh, kPrefillTok)) != cudaSuccess) return e;
  if ((e = mapq(&m0.q, p.pool + g.qoff[0], p.H, p.I, g.qoff[1] - g.qoff[0], 2, S, p.slot_stride, 128)) != cudaSuccess)
    return e;
  if ((e = mapq(&m1.q, p.pool + g.qoff[2], p.I, p.H, g.qbytes[2], 1, S, p.slot_stride, 128)) != cudaSuccess) return e;
  if (p.shared) {
    if ((e = mapq(&m0.sq, p.shared + gs.qoff[0], p.H, p.Is, gs.qoff[1] - gs.qoff[0], 2, 1, gs.bytes, 128)) !=
        cudaSuccess)
      return e;
    if ((e = mapq(&m1.sq, p.shared + gs.qoff[2], p.Is, p.H, gs.qbytes[2], 1, 1, gs.bytes, 128)) != cudaSuccess)
      return e;
  } else {
    m0.sq = m0.q;
    m1.sq = m1.q;
  }
  GemmArgs a{};
  a.units = p.units;
  a.pool = p.pool;
  a.slot_stride = p.slot_stride;
  a.shared = p.shared;
  for (int i = 0; i < 3; ++i) {
    a.r_soff[i] = g.soff[i];
    a.s_soff[i] = gs.soff[i];
  }
  a.H = p.H;
  a.I = p.I;
  a.Is = p.Is;
  a.rows_routed = A;
  a.h = p.h;
  a.ldh = p.ldh;
  a.yp = p.yp;
  a.err = p.err;
  a.gen = p.gen;
  a.S = p.S;
  // 4. gate/up + SwiGLU
  a.items = p.items0;
  a.n_items = p.n_items0;
  a.wait_cycles = p.wait_cycles > 0 ? p.wait_cycles : kPrefillWaitCycles;
  a.skip_ring = p.skip_ring;
  a.stages = gemm_stages(0);
  if (a.stages == 0) return cudaErrorInvalidValue;
  if (p.ev[0]) cudaEventRecord(p.ev[0], st);
  if ((e = launch_gemm(0, m0, a, std::min(p.max_items0, p.n_sm), st)) != cudaSuccess) return e;
  if (p.ev[1]) cudaEventRecord(p.ev[1], st);
  // 5. down (the combine applies the weights)
  a.items = p.items1;
  a.n_items = p.n_items1;
  a.wait_cycles = kPrefillWaitCycles;
  a.skip_ring = -1;
  a.stages = gemm_stages(1);
  if (a.stages == 0) return cudaErrorInvalidValue;
  if (p.ev[2]) cudaEventRecord(p.ev[2], st);
  if ((e = launch_gemm(1, m1, a, std::min(p.max_items1, p.n_sm), st)) != cudaSuccess) return e;
  if (p.ev[3]) cudaEventRecord(p.ev[3], st);
  return cudaGetLastError();
}

cudaError_t prefill_ffn(const PrefillArgs& p, cudaStream_t st) {
  cudaError_t e = encoder();
  if (e != cudaSuccess) return e;
  const int rows = p.T * p.k + p.T;
  // 1. activations in expert-major order, fp16
  if (p.parts & kPartGather) {
    if (p.xt == MOE_BF16)
      gather_kernel<MOE_BF16><<<(rows + 7) / 8, 256, 0, st>>>(p.x, p.T, p.k, p.H, p.plan.perm_tok, p.x16, rows);
    else
      gather_kernel<MOE_F32><<<(rows + 7) / 8, 256, 0, st>>>(p.x, p.T, p.k, p.H, p.plan.perm_tok, p.x16, rows);
  }
  if (p.parts & kPartGemm) {
    if ((e = prefill_gemms(p, st)) != cudaSuccess) return e;
  }
  // 6. combine into the tokens' positions
  if (p.parts & kPartCombine)
    combine_kernel<<<p.T, 256, 0, st>>>(p.yp, p.plan.inv, p.plan.perm_w, p.T, p.k, p.H, p.shared ? 1 : 0, p.y);
  return cudaGetLastError();
}

}  // namespace moe
