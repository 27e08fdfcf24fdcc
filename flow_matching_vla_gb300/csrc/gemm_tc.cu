// Host side of the tensor-core GEMM: tensor-map encoding, the split-K planner
// and the launch dispatch (kernels in gemm_tc_impl.cuh; the persistent launches
// in gemm_tc_pers.cu, the epilogue-specialised split launches in gemm_tc_spec.cu).
#include "gemm_tc_impl.cuh"

namespace g3 {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

cudaError_t tc_make_map(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld,
                        int box_rows) {
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&g_encode, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !g_encode) return cudaErrorNotSupported;
  }
  if (((uintptr_t)ptr & 15) || (ld * 2) % 16 || cols % BK) return cudaErrorInvalidValue;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                        es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

TcPlan tc_plan(int M, int N, int K, int sm_count, int max_split, bool partial) {
  TcPlan p;
  p.BN = M <= 64 ? 64 : (M <= 128 ? 128 : 256);
  // unsplit GEMMs whose 256-token tiles leave more than half the SMs idle: halve
  // the tiles (still one wave) to put twice the SMs on the weights
  if (p.BN == 256 && !partial && 2LL * ((N + BM - 1) / BM) * ((M + 255) / 256) <= sm_count) p.BN = 128;
  const int KB = K / BK;
  const long long tiles = (long long)((N + BM - 1) / BM) * ((M + p.BN - 1) / p.BN);
  // a CTA fills an SM's shared memory: the split stays within one wave.  A
  // 256-token tile cannot reduce its split on chip, so it only splits when the
  // partials go to the next kernel.
  if (p.BN == 256 && !partial) max_split = 1;
  p.S = 1;
  while (p.S < 16 && 2 * p.S <= max_split && KB % (2 * p.S) == 0 && tiles * 2 * p.S <= sm_count) p.S *= 2;
  return p;
}

bool tc_supported(int M, int N, int K) { return M > 0 && N > 0 && K > 0 && K % BK == 0 && N % 2 == 0; }

bool tc_supported_e4m3(int M, int N, int K) { return M > 0 && N > 0 && K > 0 && K % (2 * BK) == 0 && N % 2 == 0; }

TcPlan tc_plan_e4m3(int M, int N, int K, int sm_count, int max_split, bool partial) {
  // a stage covers 128 K elements: plan as a bf16 GEMM of half the K blocks
  return tc_plan(M, N, K / 2, sm_count, max_split, partial);
}

cudaError_t tc_make_map_e4m3(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld) {
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&g_encode, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !g_encode) return cudaErrorNotSupported;
  }
  if (((uintptr_t)ptr & 15) || ld % 16 || cols % 128) return cudaErrorInvalidValue;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t gemm_tc_e4m3(const CUtensorMap& tw, const CUtensorMap& tx, const GemmArgs& a, const TcPlan& p,
                         float* ws, long long ws_floats, int* err, long long wait_limit, cudaStream_t s, bool pdl) {
  if (!tc_supported_e4m3(a.M, a.N, a.K) || (a.K / (2 * BK)) % p.S || !a.epi.wscale) return cudaErrorInvalidValue;
  if (a.epi.kind != EPI_PARTIAL && tc_workspace_floats(p, a.M, a.N) > ws_floats) return cudaErrorInvalidValue;
  switch (p.BN) {
    // A stages live in tensor memory (64 columns each, beside the BN-column accumulator)
    case 64: return launch_ta<64, 4, WF_E4M3>(tw, tx, a, p.S, ws, err, wait_limit, s, pdl);    // 4 x 16 KB X stages
    case 128: return launch_ta<128, 4, WF_E4M3>(tw, tx, a, p.S, ws, err, wait_limit, s, pdl);  // 4 x 32 KB
    case 256: return launch_ta<256, 2, WF_E4M3>(tw, tx, a, p.S, ws, err, wait_limit, s, pdl);  // 2 x 64 KB
    default: return cudaErrorInvalidValue;
  }
}

long long tc_workspace_floats(const TcPlan& p, int M, int N) {
  if (p.S == 1) return 0;
  const long long tiles = (long long)((N + BM - 1) / BM) * ((M + p.BN - 1) / p.BN);
  return tiles * p.S * p.BN * BM;
}

cudaError_t gemm_tc(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap* to, const GemmArgs& a,
                    const TcPlan& p, float* ws, long long ws_floats, int* err, long long wait_limit, cudaStream_t s,
                    bool pdl) {
  if (!tc_supported(a.M, a.N, a.K) || (a.K / BK) % p.S) return cudaErrorInvalidValue;
  if (a.epi.kind != EPI_PARTIAL && tc_workspace_floats(p, a.M, a.N) > ws_floats) return cudaErrorInvalidValue;
  // kernels specialised to one epilogue: residual partials, and RoPE / GeGLU / plain
  // outputs without a split or with the on-chip reduction (tiles of up to 128 tokens)
  const int k = a.epi.kind;
  if (k == EPI_PARTIAL || ((k == EPI_ROPE || k == EPI_GEGLU || k == EPI_STORE) && (p.S == 1 || p.BN <= 128)))
    return gemm_tc_split_spec(k, tw, tx, to, a, p, ws, err, wait_limit, s, pdl);
  if (a.epi.tstore) return cudaErrorInvalidValue;
  switch (p.BN) {
    case 64: return launch<64, 8>(tw, tx, tw, a, p.S, ws, err, wait_limit, s, pdl);    // 8 x 24 KB stages
    case 128: return launch<128, 6>(tw, tx, tw, a, p.S, ws, err, wait_limit, s, pdl);   // 6 x 32 KB stages
    case 256: return launch<256, 4>(tw, tx, tw, a, p.S, ws, err, wait_limit, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace g3

namespace g3 {

bool tc_use_persistent(const TcPlan& p, int M) { return p.S == 1 && M > 64; }

bool tc_partial_tstore_ok(const Epi& e, int N) {
  return e.kind == EPI_PARTIAL && N % 32 == 0 && e.out && !((uintptr_t)e.out & 15) && (e.ldo * 4) % 16 == 0;
}

cudaError_t tc_make_part_map(CUtensorMap* m, const void* ptr, long long M, long long N, long long ld, int S) {
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&g_encode, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !g_encode) return cudaErrorNotSupported;
  }
  if (((uintptr_t)ptr & 15) || (ld * 4) % 16 || N % 32 || M <= 0 || S <= 0) return cudaErrorInvalidValue;
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)S};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)(M * ld * 4)};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool tc_tstore_ok(const Epi& e, int N) {
  if (N % 32 || !e.out || ((uintptr_t)e.out & 15) || (e.ldo * 2) % 16) return false;
  switch (e.kind) {
    case EPI_STORE: return !e.out_f32 && e.rg == 0;
    case EPI_ROPE: return e.hd > 0 && e.hd % 32 == 0 && e.rope_cols % 32 == 0;
    case EPI_GEGLU: return true;
    default: return false;
  }
}

cudaError_t tc_make_out_map(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld) {
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&g_encode, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !g_encode) return cudaErrorNotSupported;
  }
  if (((uintptr_t)ptr & 15) || (ld * 2) % 16 || cols % 16 || rows <= 0) return cudaErrorInvalidValue;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace g3
