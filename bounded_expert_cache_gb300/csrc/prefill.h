// Library-internal declarations of the prefill path (grouped dequant-GEMM).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "internal.h"

namespace moe {

constexpr int kPrefillTok = 192;  // tokens per GEMM work item
constexpr long long kPrefillWaitCycles = 4000000000ll;  // about 2 s at the SM clock

// Tensor maps of one GEMM launch: the token operand in 32-row boxes and in
// whole-tile boxes, and the quant planes of the routed experts (4-D: bytes,
// rows, matrix, slot; the gate/up GEMM takes the gate and up planes in one
// box) and of the shared expert (one slot).
struct GemmMaps {
  CUtensorMap b32, btile, q, sq;
};

struct GemmArgs {
  const int32_t* units;     // unit table of the step
  const int32_t* items;     // int4 per work item {unit, m0, n0, 0}
  const int32_t* n_items;   // [1]
  const uint8_t* pool;      // slot pool of the layer
  int64_t slot_stride;
  const uint8_t* shared;    // shared expert payload (or nullptr)
  int64_t r_soff[3], s_soff[3];  // scale-plane offsets (routed, shared)
  int H, I, Is;
  int rows_routed;          // expert-major rows of routed assignments (T*k)
  uint16_t* h;              // bf16 [rows][ldh]
  int ldh;
  float* yp;                // fp32 [rows][H], unweighted expert outputs
  uint32_t* err;
  const uint32_t* gen;      // [S] published slot generations (fail-closed check)
  int S;
  int stages;
  long long wait_cycles;    // limit of every mbarrier wait (SM clock cycles)
  int skip_ring;            // test hook: CTA 0's producer issues no copy for
                            // this ring index (-1: off), so the consumers'
                            // wait on it runs out
};

// One prefill FFN call: gather, both GEMMs, combine. A step whose union is
// larger than the slots runs as one gather, then the GEMMs once per compute
// wave (each over that wave's unit table, after the wave's fills landed),
// then one combine; `parts` selects the pieces of one call.
enum { kPartGather = 1, kPartGemm = 2, kPartCombine = 4, kPartAll = 7 };
struct PrefillArgs {
  int parts;
  uint32_t* publish_gen;    // non-null: first publish the fills of
  const int32_t* publish_list;  // [n, (slot, generation) x n] to this array
  const void* x;
  int xt, T, k, H, I, Is, S;
  const int32_t* units;
  moe_plan_t plan;
  const uint8_t* pool;
  int64_t slot_stride;
  const uint8_t* shared;
  ExpertGeom g, gs;
  __half* x16;              // [rows][H]
  uint16_t* h;              // bf16 [rows][ldh]
  int ldh;
  float* yp;                // [rows][H]
  float* y;                 // [T][H]
  int32_t *items0, *n_items0, *items1, *n_items1;
  int max_items0, max_items1;
  int n_sm;                 // persistent GEMM grid
  uint32_t* err;
  const uint32_t* gen;
  cudaEvent_t ev[4];        // optional timing around the two GEMMs
  long long wait_cycles;    // 0: the default limit of the GEMMs' waits (about 2 s)
  int skip_ring;            // test hook of the gate/up GEMM (see GemmArgs), -1: off
};
cudaError_t prefill_ffn(const PrefillArgs& p, cudaStream_t st);

// The driver's tensor-map encoder, looked up once (cudaErrorNotSupported if
// the driver has none).
cudaError_t encoder();
// Tensor map of a 16-bit [rows][cols] row-major matrix (cols a multiple of
// 8): boxes of 64 columns x box_rows rows, 128-byte swizzle.
cudaError_t map16(CUtensorMap* m, const void* base, CUtensorMapDataType t, int64_t rows, int64_t cols,
                  int box_rows);

int gemm_stages(int phase);
size_t gemm_smem_bytes(int phase, int stages);
cudaError_t launch_gemm(int phase, const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t st);

}  // namespace moe
