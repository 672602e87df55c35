// etc_common.cu -- error reporting, launch accounting, TMA descriptor encoding,
// and the chain's plan entry point.
#include <cstdio>
#include <mutex>

#include "../../include/etc_moe.h"
#include "etc_host.h"

namespace etc {

namespace {
thread_local std::string t_last_error;
}

std::atomic<long long> g_launches{0};

int set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

void clear_error() { t_last_error.clear(); }
const char* last_error() { return t_last_error.c_str(); }

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                     const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                     const cuuint32_t*, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);

static PFN_encodeTiled get_encode() {
  static PFN_encodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  });
  return fn;
}

// Row-major bf16 matrix [rows, inner] with a box of [box_rows, box_inner],
// 128-byte swizzle (box_inner * 2 must be 128), zero fill out of bounds.
CUresult encode_tensor_map_2d_bf16(CUtensorMap* m, const void* base, unsigned long long inner,
                                   unsigned long long rows, unsigned box_inner,
                                   unsigned box_rows) {
  PFN_encodeTiled fn = get_encode();
  if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// 3-D map of a bf16 tensor [outer][middle][inner] (inner contiguous), same
// swizzle and fill as above; the box lands as box_outer blocks of box_mid
// rows of 128-byte swizzled rows.
CUresult encode_tensor_map_3d_bf16(CUtensorMap* m, const void* base, unsigned long long inner,
                                   unsigned long long mid, unsigned long long outer,
                                   unsigned box_inner, unsigned box_mid, unsigned box_outer) {
  PFN_encodeTiled fn = get_encode();
  if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * 2, inner * 2 * mid};
  cuuint32_t box[3] = {box_inner, box_mid, box_outer};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int sm_count(int device) {
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  return n;
}

}  // namespace etc

extern "C" {

const char* etc_last_error(void) { return etc::last_error(); }

long long etc_launch_count(void) { return etc::g_launches.load(); }

}  // extern "C"

extern "C" int etc_chain_plan(etc_plan_t* plan, const etc_moe_opts* opts, int n_blocks) {
  if (!opts) {
    etc::clear_error();
    if (plan) *plan = nullptr;
    return etc::set_error(ETC_ERR_INVALID, "opts is NULL");
  }
  etc_moe_opts o = *opts;
  o.n_blocks = n_blocks;
  return etc_moe_plan(plan, &o);
}
