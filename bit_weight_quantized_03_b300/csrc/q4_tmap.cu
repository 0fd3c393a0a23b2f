// q4_tmap.cu -- host-side TMA tensor-map encoding shared by the GEMV and GEMM
// launchers.  cuTensorMapEncodeTiled is fetched from the driver at run time (no
// link-time dependency on libcuda).  Encoded maps depend only on address,
// sizes, strides and box -- never on the data -- so they are cached by those.
#include <mutex>

#include "q4_internal.h"

namespace q4 {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct Key {
  const void* base;
  uint64_t dim0, dim1, stride;
  uint32_t box0, box1;
  int dtype, swizzle;
  bool operator==(const Key& o) const {
    return base == o.base && dim0 == o.dim0 && dim1 == o.dim1 && stride == o.stride &&
           box0 == o.box0 && box1 == o.box1 && dtype == o.dtype && swizzle == o.swizzle;
  }
};

constexpr int kCacheSize = 256;
std::mutex cache_mu;
Key cache_keys[kCacheSize];
CUtensorMap cache_maps[kCacheSize];
bool cache_used[kCacheSize] = {false};
int cache_next = 0;

}  // namespace

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
                    uint64_t dim1, uint64_t row_stride_bytes, uint32_t box0, uint32_t box1,
                    CUtensorMapSwizzle swizzle) {
  const Key key{base, dim0, dim1, row_stride_bytes, box0, box1, static_cast<int>(dtype),
                static_cast<int>(swizzle)};
  {
    std::lock_guard<std::mutex> lk(cache_mu);
    for (int i = 0; i < kCacheSize; ++i) {
      if (cache_used[i] && cache_keys[i] == key) {
        *map = cache_maps[i];
        return true;
      }
    }
  }
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lk(cache_mu);
  cache_keys[cache_next] = key;
  cache_maps[cache_next] = *map;
  cache_used[cache_next] = true;
  cache_next = (cache_next + 1) % kCacheSize;
  return true;
}

}  // namespace q4
