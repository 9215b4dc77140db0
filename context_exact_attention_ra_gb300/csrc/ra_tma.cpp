// Host side of the TMA loads: tensor maps over [B][rows][H][D] bf16 tensors;
// and the identity of the current CUDA context.  The CUDA driver API's
// cuTensorMapEncodeTiled, cuCtxGetCurrent and cuCtxGetId are looked up once
// through the runtime.

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ra_internal.h"

namespace ra {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(int* err) {
  static EncodeTiledFn fn = nullptr;
  static int status = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || f == nullptr)
      status = (e != cudaSuccess) ? static_cast<int>(e) : static_cast<int>(cudaErrorNotSupported);
    else
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  *err = status;
  return fn;
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CtxFns {
  CtxGetCurrentFn current = nullptr;
  CtxGetIdFn id = nullptr;
};

const CtxFns& ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess && f != nullptr)
      fns.current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess && f != nullptr)
      fns.id = reinterpret_cast<CtxGetIdFn>(f);
  });
  return fns;
}

}  // namespace

unsigned long long current_context_id() {
  const CtxFns& f = ctx_fns();
  if (f.current == nullptr || f.id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (f.current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (f.id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id + 1;   // 0 stays free for "no context"
}

// Boxes of 64 columns (128 bytes, 128-byte swizzle) x 1 head x box_rows rows;
// rows past the end of the tensor read as zeros.
int make_tma_map_bf16(CUtensorMap* map, const void* base, int B, long long rows, int H, int D,
                      int box_rows) {
  int err = 0;
  EncodeTiledFn fn = encode_fn(&err);
  if (fn == nullptr) return err ? err : static_cast<int>(cudaErrorNotSupported);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                           static_cast<cuuint64_t>(rows) * H * D * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : static_cast<int>(cudaErrorInvalidValue);
}

// The rows r, r + c, r + 2c, ... of a [B][S][H][D] bf16 tensor (the keys of
// striped shard r) as dimension 3 of a 5-D view {D, H, c, S / c, B}: a box of
// 64 columns x 1 head x 1 shard x box_rows rows x 1 loads box_rows keys of one
// shard; rows past S / c read as zeros.
int make_tma_map_bf16_strided(CUtensorMap* map, const void* base, int B, long long S, int H, int D, int c,
                              int box_rows) {
  int err = 0;
  EncodeTiledFn fn = encode_fn(&err);
  if (fn == nullptr) return err ? err : static_cast<int>(cudaErrorNotSupported);
  if (c <= 0 || S % c != 0) return static_cast<int>(cudaErrorInvalidValue);
  const cuuint64_t row = static_cast<cuuint64_t>(H) * D * 2;
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(c),
                        static_cast<cuuint64_t>(S / c), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[4] = {static_cast<cuuint64_t>(D) * 2, row, row * static_cast<cuuint64_t>(c),
                           row * static_cast<cuuint64_t>(S)};
  cuuint32_t box[5] = {64, 1, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace ra
