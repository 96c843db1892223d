// psp_device.cuh -- small device helpers shared by the step's kernels:
// inline-PTX wrappers (cp.async, ldmatrix, mma.sync, movmatrix), element
// packing, shared-memory swizzles and the token -> pool-slot mapping.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>
#include <cstdint>

#include "psp_internal.h"

namespace psp {

// Raises the dynamic shared-memory limit of kernel Kern to `bytes` once per device
// (the driver call would otherwise cost host time on every step's launch).  One flag per
// device ordinal and kernel, atomic, so host threads driving different devices neither
// race nor undo each other's record; ordinals past the table set the attribute every time.
template <auto Kern>
inline cudaError_t ensure_smem_limit(int bytes) {
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> done[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < kMaxDevices;
  if (tracked && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && tracked) done[dev].store(true, std::memory_order_release);
  return e;
}

namespace dev {

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000u); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous global->shared copy; src_bytes 0 zero-fills the destination.
// Programmatic dependent launch: a prefix kernel lets the suffix kernel of the same
// step start as soon as every prefix CTA is running (the suffix CTAs then fill the
// SMs the prefix kernel leaves free).  A no-op when no dependent is launched.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
// Waits until the grids this one depends on have completed and their writes are visible.
// Pulls the line holding ptr into L2 (no register result, so nothing waits for it).
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(ptr));
}
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A(16x32, row) * B(32x8, col) + D on e4m3 operands, fp32 accumulate.
__device__ __forceinline__ void mma_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transposes an 8x8 matrix of 16-bit elements held in the warp's fragment layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two e4m3 codes (bytes 0 and 1 of x) -> f16x2 (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t x) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(x & 0xffffu), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// Two halves (an f16x2 word, first element in the low half) -> two e4m3 codes in the low
// 16 bits, first in the low byte (round to nearest even, saturating).
__device__ __forceinline__ uint32_t e4m3x2_from_f16x2(uint32_t h) {
  __half2_raw r;
  r.x = static_cast<unsigned short>(h & 0xffffu);
  r.y = static_cast<unsigned short>(h >> 16);
  return static_cast<uint32_t>(__nv_cvt_halfraw2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3));
}

// Four floats -> four e4m3 codes (round to nearest even, saturating), a in byte 0.
__device__ __forceinline__ uint32_t e4m3x4_from_floats(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xffffu) | (hi << 16);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// XOR swizzle of 16-byte chunks inside rows of CHUNKS chunks so that eight
// consecutive rows read at the same logical chunk hit distinct bank groups.
template <int CHUNKS>
__device__ __forceinline__ int swz(int row, int chunk) {
  if constexpr (CHUNKS >= 8) {
    return chunk ^ (row & 7);
  } else if constexpr (CHUNKS == 4) {
    return chunk ^ ((row >> 1) & 3);
  } else {
    return chunk ^ ((row >> 2) & 1);
  }
}

// Pool slot of logical token t of a list read at page granularity 1 << shift.
__device__ __forceinline__ int64_t slot_of(const int32_t* list, int t, int shift) {
  return (static_cast<int64_t>(__ldg(list + (t >> shift))) << shift) | (t & ((1 << shift) - 1));
}

// 2^x on the special-function unit; results below the smallest normal flush to zero
// (a probability that small adds nothing to a softmax sum of at least 1).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Max / sum over the lanes that differ only in the given xor-mask bits.
template <int FIRST, int LAST>
__device__ __forceinline__ float xor_max(float v) {
#pragma unroll
  for (int m = FIRST; m <= LAST; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
template <int FIRST, int LAST>
__device__ __forceinline__ float xor_sum(float v) {
#pragma unroll
  for (int m = FIRST; m <= LAST; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

}  // namespace dev
}  // namespace psp
