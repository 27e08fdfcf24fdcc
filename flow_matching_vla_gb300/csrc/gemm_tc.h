// Host interface of the tcgen05 tensor-core GEMM (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace g3 {

struct TcPlan {
  int BN = 64;  // token columns per CTA (MMA N): 64, 128 or 256
  int S = 1;    // split-K factor = cluster size along K (power of two, <= 16)
  int CL = 1;   // persistent kernel: CTAs per cluster sharing each activation tile by multicast (1 or 2);
                // its activation map's box is BN / CL rows
};

// K-major bf16 tensor map over a [rows][cols] matrix with leading dimension
// ``ld`` elements; box = 64 columns x box_rows rows, 128-byte swizzle.
cudaError_t tc_make_map(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld,
                        int box_rows);
bool tc_supported(int M, int N, int K);
// Split-K factor: the largest power of two <= max_split that divides the K
// blocks and keeps tiles * S within the SM count (one wave); ``partial``: the
// split partials go to the next kernel instead of being reduced in-kernel.
TcPlan tc_plan(int M, int N, int K, int sm_count, int max_split, bool partial);
// Split-K partials the plan needs (fp32 elements of the workspace).
long long tc_workspace_floats(const TcPlan& p, int M, int N);
// W map: box_rows 128 over [N][K]; X map: box_rows plan.BN over [M][K].  With
// a.epi.tstore set (EPI_PARTIAL only), the split partials leave by tensor stores
// through ``to`` (from tc_make_part_map over the [S][M][ldo] partial buffer);
// ``to`` may be null otherwise.
cudaError_t gemm_tc(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap* to, const GemmArgs& a,
                    const TcPlan& p, float* ws, long long ws_floats, int* err, long long wait_limit, cudaStream_t s,
                    bool pdl);
// Split partials by tensor stores: N % 32 == 0, a 16-byte aligned buffer, ldo % 4 == 0.
bool tc_partial_tstore_ok(const Epi& e, int N);
// fp32 [S][M][N] map (row stride ld, split stride M * ld) with boxes of 32 x 32 x 1.
cudaError_t tc_make_part_map(CUtensorMap* m, const void* ptr, long long M, long long N, long long ld, int S);

// gemm_tc for one epilogue kind ``ek`` (EPI_PARTIAL, or EPI_ROPE / EPI_GEGLU /
// EPI_STORE with plan.S == 1 or plan.BN <= 128) through a kernel holding only that epilogue.
cudaError_t gemm_tc_split_spec(int ek, const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap* to,
                               const GemmArgs& a, const TcPlan& p, float* ws, int* err, long long wait_limit,
                               cudaStream_t s, bool pdl);

// E4M3 weights (uint8 codes [N][K], one fp32 scale per row in a.epi.wscale):
// K a multiple of 128; the W map from tc_make_map_e4m3 (box 128 x 128 bytes),
// the X map as above.
bool tc_supported_e4m3(int M, int N, int K);
TcPlan tc_plan_e4m3(int M, int N, int K, int sm_count, int max_split, bool partial);
cudaError_t tc_make_map_e4m3(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld);
cudaError_t gemm_tc_e4m3(const CUtensorMap& tw, const CUtensorMap& tx, const GemmArgs& a, const TcPlan& p,
                         float* ws, long long ws_floats, int* err, long long wait_limit, cudaStream_t s, bool pdl);

// Large token counts (no split, M > 64): persistent CTAs with a double-buffered
// TMEM accumulator so each tile's epilogue overlaps the next tile's MMAs;
// with plan.CL = 2, clusters of two CTAs over adjacent weight tiles share each
// activation tile by TMA multicast (X map box: BN / 2 rows).
// With a.epi.tstore set, its epilogue stages the outputs in shared memory and
// writes them with tensor stores through ``to`` (from tc_make_out_map over the
// output, cols = N for EPI_STORE / EPI_ROPE and N / 2 for EPI_GEGLU; only where
// tc_tstore_ok holds); ``to`` may be null otherwise.
bool tc_use_persistent(const TcPlan& p, int M);
cudaError_t gemm_tc_persistent_launch(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap* to,
                                      const GemmArgs& a, const TcPlan& p, int sm_count, int* err,
                                      long long wait_limit, cudaStream_t s, bool pdl);
// The epilogue kinds and layouts the tensor-store path covers: bf16 EPI_STORE
// without row remap, EPI_ROPE with hd % 32 == 0, EPI_GEGLU; N % 32 == 0, a
// 16-byte aligned output with a leading dimension of a multiple of 8 elements.
bool tc_tstore_ok(const Epi& e, int N);
// bf16 [rows][cols] output map with leading dimension ``ld``: boxes of 16 columns x 32 rows, no swizzle.
cudaError_t tc_make_out_map(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld);

}  // namespace g3
