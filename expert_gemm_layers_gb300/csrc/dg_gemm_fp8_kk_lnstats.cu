// Instantiation unit of the tcgen05 GEMM: e4m3 A and B K-major, row/column dequantisation, bias + per-tile LayerNorm statistics.
#include "dg_internal.h"

namespace dg {

cudaError_t launch_gemm_fp8_kk_lnstats(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d,
                               const CUtensorMap& c, const GemmParams& p, int num_sms, cudaStream_t s) {
  return launch_gemm_t<true, false, false, EPI_BIAS_LNSTATS>(a, b, d, c, p, num_sms, s);
}

}  // namespace dg
