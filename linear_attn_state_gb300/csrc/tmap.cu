// Tensor maps (TMA descriptors) over the packed token inputs of a build.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "hypic_internal.h"

namespace hypic {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 3-D map over [n_tok][n_streams][d] with boxes of 64 tokens x 1 stream x
// `inner` elements.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t es, const void* base, int64_t n_tok,
              int n_streams, int d, uint32_t inner, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n_streams),
                        static_cast<cuuint64_t>(n_tok)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * es,
                           static_cast<cuuint64_t>(d) * es * static_cast<cuuint64_t>(n_streams)};
  cuuint32_t box[3] = {inner, 1u, 64u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_token_map(CUtensorMap* m, const void* base, int64_t n_tok, int n_streams, int d) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, n_tok, n_streams, d, 64u,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_gate_map(CUtensorMap* m, const float* base, int64_t n_tok, int n_streams, int d) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, n_tok, n_streams, d, 32u,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace hypic
