// Descriptors consumed by tcgen05.mma: the shared-memory matrix descriptor and the
// instruction descriptor for kind::f16.  Both are plain bit packing, usable on host
// (for tests through the C ABI helper) and device.
#pragma once
#include <cstdint>

namespace gb300 {

// Shared-memory matrix descriptor for a K-major operand stored in the 128-byte
// swizzled canonical layout that a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes:
// rows of 64 x 16-bit elements (128 B), 8-row atoms of 1024 B stacked along M (or N).
//   bits  0..13  start address >> 4
//   bits 16..29  leading-dimension byte offset >> 4 (unused for swizzled K-major; 1)
//   bits 32..45  stride-dimension byte offset >> 4 (next 8-row atom: 1024 B)
//   bits 46..48  fixed value 0b001
//   bits 49..51  base offset (0: every stage base is 1024-byte aligned)
//   bits 61..63  swizzle mode (2 = 128-byte swizzle)
// Field layout: "Optimizing GEMMs using tcgen05 - Part 1", section 2.3 (make_smem_desc)
// and section 2.2 (for a K-major swizzled operand the leading offset is unused and
// encodes as 1); the 1024-B alignment rule is section 4.1 there and "A Blackwell
// GEMM by Hand in CuTe DSL", section 6.  Moving to the next 16-deep K slice inside
// the 64-deep stage adds 32 bytes to the start address.
__host__ __device__ constexpr uint64_t smem_desc_sw128_kmajor(uint32_t smem_byte_addr) {
  return (uint64_t)((smem_byte_addr >> 4) & 0x3FFFu) | ((uint64_t)(16u >> 4) << 16) |
         ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16, fp32 accumulator, both operands K-major.
//   bits  4..5   D format (1 = fp32)
//   bits  7..9   A format (0 = fp16, 1 = bf16)
//   bits 10..12  B format (0 = fp16, 1 = bf16)
//   bit  15/16   A/B major-ness (0 = K-major)
//   bits 17..22  N >> 3
//   bits 24..28  M >> 4
// D format, B major bit, N and M positions: "Optimizing GEMMs using tcgen05 - Part 1",
// section 2.5.  The A/B format fields are not given on the pages; their positions
// and codes are those of NVIDIA's public PTX ISA instruction-descriptor table, and a
// bf16 run on non-integer inputs checks them (a wrong code fails parity outright).
__host__ __device__ constexpr uint32_t idesc_f16_kmajor(uint32_t m, uint32_t n, bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((n >> 3) << 17) |
         ((m >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with FP8 operands, fp32 accumulator, both
// operands K-major: the kind::f16 layout above with the A/B format fields holding
// 0 = E4M3 or 1 = E5M2 (NVIDIA's public PTX ISA instruction-descriptor table; an
// E5M2 run on non-integer inputs checks the code, as for bf16).
__host__ __device__ constexpr uint32_t idesc_f8_kmajor(uint32_t m, uint32_t n, bool e5m2) {
  return (1u << 4) | ((e5m2 ? 1u : 0u) << 7) | ((e5m2 ? 1u : 0u) << 10) | ((n >> 3) << 17) |
         ((m >> 4) << 24);
}

}  // namespace gb300
