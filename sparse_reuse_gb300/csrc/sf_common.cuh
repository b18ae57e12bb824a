// Device helpers shared by the libspecfold kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sf {

// Largest R * (B + 1) a context supports; the tree travels by value in the
// gate kernel's parameter block so a captured CUDA graph carries it.
constexpr int kMaxTreeSlots = 1024;
// Largest number of rows T = R * (B + 1) * L of one pass (the compaction of a
// layer runs in one thread block's shared memory).
constexpr int kMaxRows = 8192;

struct Tree {
  int R;
  int Bp;
  int8_t parent[kMaxTreeSlots];  // parent[r * Bp + i], -1 for the main branch
};

// Bits of the device error word.
enum : unsigned {
  kErrGate = 1u,      // gate/resolution index check
  kErrNorm = 2u,      // RMSNorm gather index check
  kErrGemm = 4u,      // GEMM argument/index check
  kErrAttn = 8u,      // attention index check
  kErrResid = 16u,    // final residual index check
  kErrTimeout = 32u,  // a bounded wait gave up
};

__device__ __forceinline__ void raise_error(unsigned* flag, unsigned bits) {
  if (flag) atomicOr(flag, bits);
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over the block (any multiple of 32 threads up to 1024); every thread
// gets the total.  `red` needs 32 floats of shared memory.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_sum(t);
}

// Load 4 consecutive elements of type T as float4 (pointer 4-element aligned).
template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}

template <typename T>
__device__ __forceinline__ void store4(T* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

}  // namespace sf

namespace sf {

// Programmatic dependent launch.  Every kernel of the pass is launched with
// programmatic stream serialisation: it may start while the previous kernel
// drains, runs its prologue, and calls pdl_wait() before its first read of
// anything an earlier kernel wrote (and before it can complete).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename Kernel, typename... Args>
cudaError_t launch_pdl_cluster(cudaStream_t st, dim3 grid, dim3 block, size_t smem, dim3 cluster, Kernel kernel,
                               Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster.x * cluster.y * cluster.z > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster.x;
    attr[1].val.clusterDim.y = cluster.y;
    attr[1].val.clusterDim.z = cluster.z;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// clusters (if any) along z
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(cudaStream_t st, dim3 grid, dim3 block, size_t smem, int cluster_z, Kernel kernel,
                       Args... args) {
  return launch_pdl_cluster(st, grid, block, smem, dim3(1, 1, cluster_z > 1 ? (unsigned)cluster_z : 1u), kernel,
                            args...);
}

}  // namespace sf
