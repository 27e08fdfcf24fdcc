// Launches of the persistent tensor-core GEMM (its kernels live in
// gemm_tc_impl.cuh; compiled in a translation unit of their own so the library
// builds its GEMM kernels in parallel).
#include "gemm_tc_impl.cuh"

namespace g3 {

cudaError_t gemm_tc_persistent_launch(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap* to,
                                      const GemmArgs& a, const TcPlan& p, int sm_count, int* err,
                                      long long wait_limit, cudaStream_t s, bool pdl) {
  if (!tc_supported(a.M, a.N, a.K) || p.S != 1) return cudaErrorInvalidValue;
  if (a.epi.tstore && (!to || !tc_tstore_ok(a.epi, a.N))) return cudaErrorInvalidValue;
  const CUtensorMap& o = to ? *to : tw;   // unused unless a.epi.tstore
  // tensor-store RoPE and GeGLU epilogues (the projections of every layer) run in
  // kernels specialised to that one epilogue
  const int ek = !a.epi.tstore ? -1 : a.epi.kind == EPI_ROPE ? EPI_ROPE : a.epi.kind == EPI_GEGLU ? EPI_GEGLU : -1;
#define G3_PERS(BN_, ST_, CL_)                                                                            \
  (ek == EPI_ROPE    ? launch_persistent<BN_, ST_, CL_, EPI_ROPE>(tw, tx, o, a, sm_count, err, wait_limit, s, pdl) \
   : ek == EPI_GEGLU ? launch_persistent<BN_, ST_, CL_, EPI_GEGLU>(tw, tx, o, a, sm_count, err, wait_limit, s, pdl) \
                     : launch_persistent<BN_, ST_, CL_, -1>(tw, tx, o, a, sm_count, err, wait_limit, s, pdl))
  switch (p.BN) {
    case 128: return p.CL == 2 ? G3_PERS(128, 6, 2) : G3_PERS(128, 6, 1);
    case 256: return p.CL == 2 ? G3_PERS(256, 4, 2) : G3_PERS(256, 4, 1);
    default: return cudaErrorInvalidValue;
  }
#undef G3_PERS
}

}  // namespace g3
