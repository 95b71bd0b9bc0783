// desc.cuh -- tcgen05 instruction and shared-memory descriptors (host + device).
//
// "tcgen05 for dummies: a B200 GEMM from scratch" (translated), sections
// "Decoding tcgen05" and "128-byte global loads and swizzle", shows the bf16 /
// fp32 instruction descriptor and the K-major 128-byte-swizzle shared-memory
// descriptor; the remaining fields (fp16 formats, fp16 accumulator, MN-major
// operands, version and swizzle codes) are the public PTX ISA encodings.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define HG_HD __host__ __device__ __forceinline__
#else
#define HG_HD inline
#endif

namespace hg {

// Instruction descriptor for tcgen05.mma kind::f16.
//   bits 4-5  D format      0 = f16, 1 = f32
//   bits 7-9  A format      0 = f16, 1 = bf16
//   bits 10-12 B format     0 = f16, 1 = bf16
//   bit 15    A major       0 = K-major, 1 = MN-major
//   bit 16    B major       0 = K-major, 1 = MN-major
//   bits 17-22 N >> 3
//   bits 24-28 M >> 4
HG_HD uint32_t make_idesc(int mma_m, int mma_n, bool in_bf16, bool acc_f32, bool a_mn_major, bool b_mn_major) {
  return (acc_f32 ? (1u << 4) : 0u) | (in_bf16 ? (1u << 7) : 0u) | (in_bf16 ? (1u << 10) : 0u) |
         (a_mn_major ? (1u << 15) : 0u) | (b_mn_major ? (1u << 16) : 0u) |
         ((uint32_t)(mma_n >> 3) << 17) | ((uint32_t)(mma_m >> 4) << 24);
}

// Swizzle codes of the shared-memory descriptor (bits 61-63).
enum : int { kSwizzleNone = 0, kSwizzle128B = 2, kSwizzle64B = 4, kSwizzle32B = 6 };

// Shared-memory matrix descriptor.
//   bits 0-13  start address >> 4 (18-bit shared address)
//   bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension byte offset >> 4
//   bits 46-48 fixed 0b001
//   bits 49-51 base offset (0: every tile starts on a swizzle-pattern boundary)
//   bits 61-63 swizzle mode
HG_HD uint64_t make_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, int swizzle) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
         ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46) | ((uint64_t)(swizzle & 7) << 61);
}

// Operand tiles as the TMA writes them with 128-byte swizzle.
//
// K-major (rows of 64 16-bit values = 128 B, the contiguous dimension is K):
// the eight 128-byte rows of a core-matrix group are contiguous, so the
// stride byte offset between 8-row groups is 1024 B; the leading offset is
// unused.  Advancing one MMA step (16 elements = 32 B) moves the start address
// by 32 B inside the swizzle atom.
constexpr uint32_t kKMajorSBO = 1024;
constexpr uint32_t kKMajorStepBytes = 32;

// MN-major (the contiguous dimension is N): each TMA box is 64 N-values wide
// (128 B) and 64 K-rows tall, rows 128 B apart.  The stride byte offset steps
// 8 K-rows (1024 B); the leading byte offset steps to the next 64-wide N block
// (the next box, 64 x 128 B = 8 KiB).  One MMA step (16 K-rows) moves the start
// address by 2048 B.
constexpr uint32_t kMNMajorSBO = 1024;
constexpr uint32_t kMNMajorLBO = 64 * 128;
constexpr uint32_t kMNMajorStepBytes = 16 * 128;

}  // namespace hg
