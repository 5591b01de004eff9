// Instantiation unit of the tcgen05 GEMM: e4m3 A and B K-major, D = alpha*acc + beta*C.
#include "dg_internal.h"

namespace dg {

cudaError_t launch_gemm_fp8_kk(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d,
                               const CUtensorMap& c, const GemmParams& p, int num_sms, cudaStream_t s) {
  return launch_gemm_t<true, false, false, EPI_FP8>(a, b, d, c, p, num_sms, s);
}

cudaError_t gemm_fp8_units(int num_sms, int* units) {
  return gemm_units_t<true, false, false, EPI_FP8>(num_sms, units);
}

}  // namespace dg
