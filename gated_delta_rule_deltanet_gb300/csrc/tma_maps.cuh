// tma_maps.cuh -- tensor maps for the TMA copies (host side).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace kda {

// cuTensorMapEncodeTiled from the driver (the runtime is linked statically, libcuda is not)
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// An fp32 matrix of `rows` x `cols` with rows `stride` floats apart (base and stride 16-byte
// aligned), copied in boxes of 32 columns x `box_rows` rows with the 128-byte swizzle: each
// box lands as box_rows rows of 128 bytes, the K-major operand layout of kind::tf32 MMAs.
inline bool encode_f32_blocks(CUtensorMap* m, const float* base, uint64_t rows, uint64_t cols,
                              uint64_t stride, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc || rows == 0 || (reinterpret_cast<uintptr_t>(base) & 15u) || (stride & 3u)) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {stride * 4};
  const cuuint32_t box[2] = {32, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same for token rows of one head in a [T, H, cols] fp32 array: boxes of 32 columns x
// 1 head x `box_rows` tokens (zero fill past the last token).
inline bool encode_f32_token_blocks(CUtensorMap* m, const float* base, uint64_t T, uint64_t H,
                                    uint64_t cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc || T == 0 || (reinterpret_cast<uintptr_t>(base) & 15u) || (cols & 3u)) return false;
  const cuuint64_t dims[3] = {cols, H, T};
  const cuuint64_t strides[2] = {cols * 4, H * cols * 4};
  const cuuint32_t box[3] = {32, 1, box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace kda
