// Instantiation unit of the tcgen05 GEMM: bf16 A K-major, B MN-major, plain bf16 store.
#include "dg_internal.h"

namespace dg {

cudaError_t launch_gemm_bf16_km_store(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d,
                                      const CUtensorMap& c, const GemmParams& p, int num_sms, cudaStream_t s) {
  return launch_gemm_t<false, false, true, EPI_STORE>(a, b, d, c, p, num_sms, s);
}

}  // namespace dg
