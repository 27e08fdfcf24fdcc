// Launches of the split-K tensor-core GEMM specialised to one epilogue kind
// (kernels in gemm_tc_impl.cuh; a translation unit of their own so the library
// builds its GEMM kernels in parallel).
#include "gemm_tc_impl.cuh"

namespace g3 {

cudaError_t gemm_tc_split_spec(int ek, const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap* to,
                               const GemmArgs& a, const TcPlan& p, float* ws, int* err, long long wait_limit,
                               cudaStream_t s, bool pdl) {
  if (a.epi.tstore && (ek != EPI_PARTIAL || !to || !tc_partial_tstore_ok(a.epi, a.N))) return cudaErrorInvalidValue;
  const CUtensorMap& o = to ? *to : tw;   // unused unless a.epi.tstore
#define G3_SPEC(BN_, ST_)                                                                        \
  (ek == EPI_PARTIAL ? launch<BN_, ST_, EPI_PARTIAL>(tw, tx, o, a, p.S, ws, err, wait_limit, s, pdl) \
   : ek == EPI_ROPE  ? launch<BN_, ST_, EPI_ROPE>(tw, tx, o, a, p.S, ws, err, wait_limit, s, pdl)    \
   : ek == EPI_GEGLU ? launch<BN_, ST_, EPI_GEGLU>(tw, tx, o, a, p.S, ws, err, wait_limit, s, pdl)   \
                     : launch<BN_, ST_, EPI_STORE>(tw, tx, o, a, p.S, ws, err, wait_limit, s, pdl))
  if (ek != EPI_PARTIAL && ek != EPI_ROPE && ek != EPI_GEGLU && ek != EPI_STORE) return cudaErrorInvalidValue;
  if (a.epi.kind != ek) return cudaErrorInvalidValue;
  // the other kernels hold no workspace reduction: a split needs the on-chip one
  if (ek != EPI_PARTIAL && p.S > 1 && p.BN > 128) return cudaErrorInvalidValue;
  switch (p.BN) {
    case 64: return G3_SPEC(64, 8);
    case 128: return G3_SPEC(128, 6);
    case 256: return G3_SPEC(256, 4);
    default: return cudaErrorInvalidValue;
  }
#undef G3_SPEC
}

}  // namespace g3
