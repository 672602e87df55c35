// etc_host.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <string>

namespace etc {

// Thread-local last-error message; returns `code` for tail calls.
int set_error(int code, const char* fmt, ...);
void clear_error();
const char* last_error();

// Process-wide count of kernel launches issued by the library.
extern std::atomic<long long> g_launches;

// cuTensorMapEncodeTiled obtained through the runtime's driver entry point.
CUresult encode_tensor_map_2d_bf16(CUtensorMap* m, const void* base, unsigned long long inner,
                                   unsigned long long rows, unsigned box_inner,
                                   unsigned box_rows);
CUresult encode_tensor_map_3d_bf16(CUtensorMap* m, const void* base, unsigned long long inner,
                                   unsigned long long mid, unsigned long long outer,
                                   unsigned box_inner, unsigned box_mid, unsigned box_outer);

int sm_count(int device);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace etc

#define ETC_CUDA_TRY(expr)                                                            \
  do {                                                                                \
    cudaError_t _e = (expr);                                                          \
    if (_e != cudaSuccess)                                                            \
      return ::etc::set_error(ETC_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(_e)); \
  } while (0)
