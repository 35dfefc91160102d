// Shared device helpers of the MoE kernels (element conversion, status word,
// small integer utilities).  Nothing here is layer arithmetic.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace moe {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Device status codes (documented with moe_device_status in moe.h).
enum : int { STATUS_BAD_EXPERT_ID = 1, STATUS_WAIT_TIMEOUT = 2, STATUS_TMEM_ALLOC = 3, STATUS_REPEATED_EXPERT_ID = 4 };

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Record the first failed device-side check; later ones keep the first code.
__device__ inline void record_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---- element type conversion (fp32 <-> storage type) ----
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ inline float load(const float *p) { return *p; }
  static __device__ inline float to_f32(float v) { return v; }
  static __device__ inline float from_f32(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ inline float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
  static __device__ inline float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ inline __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

// 16-byte vector of storage elements: 4 floats or 8 bf16.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  static __device__ inline void load(const float *p, float (&o)[4]) {
    float4 v = *reinterpret_cast<const float4 *>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  static __device__ inline void unpack(const uint4 &v, float (&o)[4]) {
    o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
  }
  static __device__ inline void store(float *p, const float (&o)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ inline void unpack(const uint4 &v, float (&o)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // bf16 -> fp32 is a 16-bit shift
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ inline void load(const __nv_bfloat16 *p, float (&o)[8]) {
    unpack(*reinterpret_cast<const uint4 *>(p), o);
  }
  static __device__ inline void store(__nv_bfloat16 *p, const float (&o)[8]) {
    uint4 v;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
    *reinterpret_cast<uint4 *>(p) = v;
  }
};

// ---- programmatic dependent launch ----
// Kernels of the layer are launched with programmatic stream serialization:
// a kernel may be scheduled while its predecessor on the stream is still
// running, so each one first lets its own dependents launch, does only
// set-up work that touches no global memory, and waits for the predecessor
// grid to complete (and its memory to be visible) before its first global
// access.
__device__ inline void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ inline void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kernel` on `stream` with programmatic stream serialization.  The
// kernel must call griddep_wait() before reading or writing global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ inline float silu_f32(float g) { return g / (1.0f + expf(-g)); }
__device__ inline float sigmoid_f32(float z) { return 1.0f / (1.0f + expf(-z)); }

__device__ inline unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace moe
