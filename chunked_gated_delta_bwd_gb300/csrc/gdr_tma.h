// Host side of the TMA copies: tensor maps (CUtensorMap) for bf16 tensors with the
// 128-byte shared-memory swizzle, encoded with the driver's cuTensorMapEncodeTiled,
// which is resolved once through the runtime (no link against the driver library).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <string.h>

#include <mutex>

namespace gdr {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A bf16 tensor of `rank` dimensions (dims[0] contiguous; strides[i] = byte stride of
// dimension i + 1), copied in boxes of `box` elements.  A null base leaves the map
// zeroed (a map the kernel does not use).  Returns false if the driver refuses it.
inline bool encode_bf16_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                            const cuuint64_t* strides, const cuuint32_t* box) {
    memset(m, 0, sizeof(*m));
    if (base == nullptr) return true;
    PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (fn == nullptr) return false;
    const cuuint32_t elem[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box,
              elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][cols] row-major bf16, boxes of box_rows x 64 columns
inline bool encode_rows_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    return encode_bf16_map(m, base, 2, dims, strides, box);
}

// [rows][128] row-major bf16 viewed as [2 column blocks][rows][64]: one copy moves a
// box_rows x 128 tile laid out as two SW128 column blocks ([block][row][128 B])
inline bool encode_blocked_rows_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
    const cuuint64_t dims[3] = {64, rows, 2};
    const cuuint64_t strides[2] = {256, 128};
    const cuuint32_t box[3] = {64, box_rows, 2};
    return encode_bf16_map(m, base, 3, dims, strides, box);
}

// token-major [T][H][128] bf16 activations viewed as [2 column blocks][T][H][64]: one copy
// moves 64 tokens x 128 channels of one head as two SW128 column blocks
inline bool encode_blocked_tokens_map(CUtensorMap* m, const void* base, uint64_t T, uint64_t H) {
    const cuuint64_t dims[4] = {64, H, T, 2};
    const cuuint64_t strides[3] = {256, H * 256, 128};
    const cuuint32_t box[4] = {64, 1, 64, 2};
    return encode_bf16_map(m, base, 4, dims, strides, box);
}

// token-major [T][H][D] bf16 activations, boxes of 64 tokens x 64 channels of one head
inline bool encode_tokens_map(CUtensorMap* m, const void* base, uint64_t T, uint64_t H, uint64_t D) {
    const cuuint64_t dims[3] = {D, H, T};
    const cuuint64_t strides[2] = {D * 2, H * D * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    return encode_bf16_map(m, base, 3, dims, strides, box);
}

}  // namespace gdr
