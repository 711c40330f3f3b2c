// TMA tensor maps for librpa's kernels (host side): cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point so that the library needs
// no link against libcuda.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "rpa_internal.h"

namespace rpa {
namespace {

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeFn lookup_encode_fn() {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<EncodeFn>(ptr);
  cudaGetLastError();
  return nullptr;
}

EncodeFn encode_fn() {
  static const EncodeFn fn = lookup_encode_fn();   // looked up once, thread-safe
  return fn;
}

}  // namespace

bool tmap_available() { return encode_fn() != nullptr; }

bool make_tmap_3d(CUtensorMap* m, const void* base, uint64_t d, uint64_t mid, uint64_t outer,
                  uint32_t box_mid, uint32_t box_outer) {
  EncodeFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {d, mid, outer};
  cuuint64_t strides[2] = {d * 2, d * mid * 2};
  cuuint32_t box[3] = {64, box_mid, box_outer};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_3d_u8(CUtensorMap* m, const void* base, uint64_t d, uint64_t mid, uint64_t outer,
                     uint32_t box_mid, uint32_t box_outer) {
  EncodeFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {d, mid, outer};
  cuuint64_t strides[2] = {d, d * mid};
  cuuint32_t box[3] = {128, box_mid, box_outer};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same tensor seen as 4-D, (64, mid, outer, d / 64): the 64-element
// chunks of a row become the outermost dimension (stride 128 bytes), so one
// box (64, box_mid, box_outer, d / 64) brings every chunk of box_outer rows
// and lands in shared memory as [chunk][row][128 B], the layout that d / 64
// separate 3-D boxes of (64, box_mid, box_outer) give, in one copy.
bool make_tmap_4d_chunks(CUtensorMap* m, const void* base, uint64_t d, uint64_t mid,
                         uint64_t outer, uint32_t box_mid, uint32_t box_outer, bool fp8) {
  EncodeFn fn = encode_fn();
  if (fn == nullptr) return false;
  const uint64_t esz = fp8 ? 1 : 2;
  const uint64_t inner = 128 / esz;            // elements of one 128-byte chunk
  if (d % inner != 0) return false;
  cuuint64_t dims[4] = {inner, mid, outer, d / inner};
  cuuint64_t strides[3] = {d * esz, d * mid * esz, 128};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(inner), box_mid, box_outer,
                       static_cast<cuuint32_t>(d / inner)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace rpa
