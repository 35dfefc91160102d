// Host-side helpers of the tensor-core kernels: TMA tensor-map encoding
// (through the driver entry point, no libcuda link), the SM count, and the
// one-time opt-in to large dynamic shared memory per kernel and device.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace moe {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

// Tensor map with the 128-byte swizzle; out-of-range elements of a load read
// as zero.  dims[0] is the contiguous dimension; strides_bytes[i] is the
// stride of dimension i + 1.
inline bool encode_map(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims, const uint64_t *strides_bytes,
                       const uint32_t *box, CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides_bytes[i];
  }
  return fn(m, type, (cuuint32_t)rank, const_cast<void *>(ptr), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major bf16 [rows, cols] matrix, box = box_rows x 64.
inline bool map_2d(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, uint32_t box_rows) {
  const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)cols * 2};
  const uint32_t box[2] = {64, box_rows};
  return encode_map(m, ptr, 2, dims, strides, box);
}

// The five token-tile maps of a row-major bf16 [rows, cols] matrix (box heights 256 .. 16).
inline bool map_rows(CUtensorMap *m5, const void *ptr, int64_t rows, int64_t cols) {
  for (int h = 0; h < 5; ++h)
    if (!map_2d(&m5[h], ptr, rows, cols, 256u >> h)) return false;
  return true;
}

// A row-major bf16 [rows, cols] matrix read column-block-wise (cols % 64 == 0)
// as 3-D (64, rows, cols / 64); a box (64, box_rows, nblk) lands as nblk
// blocks of box_rows rows x 128 bytes, i.e. an MN-major operand tile whose
// MN extent is the columns (64 nblk of them) and whose K extent is the rows.
inline bool map_col_blocks(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, uint32_t box_rows,
                           uint32_t nblk) {
  const uint64_t dims[3] = {64, (uint64_t)rows, (uint64_t)cols / 64};
  const uint64_t strides[2] = {(uint64_t)cols * 2, 128};
  const uint32_t box[3] = {64, box_rows, nblk};
  return encode_map(m, ptr, 3, dims, strides, box);
}

// Row-major float [rows, cols] matrix with a 32 x 32 box (128-byte rows): the
// store map of the weight-gradient epilogues.
inline bool map_f32_tile(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols) {
  const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)cols * 4};
  const uint32_t box[2] = {32, 32};
  return encode_map(m, ptr, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

// Gate/up weights [n_mat, 2*Iw, H] viewed as 5-D (H, 16, 2, Iw/16, n_mat):
// a box (64, 16, 2, groups, 1) holds, for `groups` consecutive groups of 16
// features (four groups = one 128-row M tile), the 16 gate rows followed by
// the 16 up rows of each group.
inline bool map_gate_up(CUtensorMap *m, const void *ptr, int n_mat, int Iw, int H, uint32_t groups) {
  const uint64_t dims[5] = {(uint64_t)H, 16, 2, (uint64_t)Iw / 16, (uint64_t)n_mat};
  const uint64_t strides[4] = {(uint64_t)H * 2, (uint64_t)Iw * H * 2, (uint64_t)16 * H * 2,
                               (uint64_t)2 * Iw * H * 2};
  const uint32_t box[5] = {64, 16, 2, groups, 1};
  return encode_map(m, ptr, 5, dims, strides, box);
}

// Number of SMs of the current device.
inline int device_sms() {
  static std::mutex mu;
  static int sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  int &n = sms[dev & 63];
  if (!n) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

// Opt `fn` in to `bytes` of dynamic shared memory once per device.
inline cudaError_t ensure_smem(const void *fn, int bytes) {
  static std::mutex mu;
  static const void *done[64][16] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  const void **row = done[dev & 63];
  for (int i = 0; i < 16; ++i)
    if (row[i] == fn) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < 16; ++i)
    if (!row[i]) {
      row[i] = fn;
      break;
    }
  return cudaSuccess;
}

}  // namespace moe
