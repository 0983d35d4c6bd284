// sgemv_m1.cu -- specialised SparseGemv kernel for m = 1 (decode).
#include "sgemv_internal.cuh"

namespace sgemv {

cudaError_t launch_m1(const Layout& L, const RunArgs& a, cudaStream_t s) {
  (void)L; (void)a; (void)s;
  return cudaErrorNotSupported;
}

}  // namespace sgemv
