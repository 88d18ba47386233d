// Host side of the TMA tensor tiles: encodes the tensor map through which the
// attention producers copy K/V page tiles.  cuTensorMapEncodeTiled comes from
// the runtime's driver entry-point lookup, so the library does not link
// against the driver library itself.
#include <cudaTypedefs.h>

#include <mutex>

#include "spg_internal.h"

namespace spg {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

bool make_kv_tmap(CUtensorMap* map, const void* pool, int kv_dtype, long long rows, int head_dim,
                  int page_size, bool* whole_page) {
  const int esz = kv_dtype == SPG_I8 ? 1 : 2;
  if (kv_dtype != SPG_F16 && kv_dtype != SPG_BF16 && kv_dtype != SPG_I8) return false;
  if ((head_dim * esz) % 128 != 0 || page_size < 8 || page_size > 256) return false;
  if (rows < 1 || rows > 0x7fffffffLL) return false;  // int32 row coordinates
  if ((reinterpret_cast<uintptr_t>(pool) & 15u) != 0) return false;
  const auto fn = encode_fn();
  if (!fn) return false;
  const CUtensorMapDataType dt = kv_dtype == SPG_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : kv_dtype == SPG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(head_dim) * esz;
  const cuuint32_t nt = static_cast<cuuint32_t>(row_bytes / 128);  // 128-byte slices of a row
  // Whole page in one copy: a 3-D view (x: the 128 bytes of a slice, y: rows,
  // z: slices), so that a box of [128 bytes][page_size rows][nt slices] lands
  // as nt tiles of [page_size rows][128 bytes], the same layout (and 128-byte
  // swizzle) as nt separate 2-D tile copies.
  {
    const cuuint64_t dims[3] = {128u / static_cast<cuuint64_t>(esz), static_cast<cuuint64_t>(rows), nt};
    const cuuint64_t strides[2] = {row_bytes, 128u};
    const cuuint32_t box[3] = {128u / esz, static_cast<cuuint32_t>(page_size), nt};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    if (fn(map, dt, 3, const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      *whole_page = true;
      return true;
    }
  }
  // else one 2-D tile of [page_size rows][128 bytes] per slice
  *whole_page = false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {128u / esz, static_cast<cuuint32_t>(page_size)};  // 128-byte rows
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = fn(map, dt, 2, const_cast<void*>(pool), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace spg
