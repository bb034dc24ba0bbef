// The epilogue's staging of a warp's 32 x 32 fp32 block through shared
// memory (sm_103a).
//
// After tcgen05.ld, lane l of a warp holds 32 consecutive columns of one
// row (row l of the warp's 32 TMEM lanes).  Stored straight to C, each store
// instruction would touch 32 rows.  The warp therefore writes its block to a
// 4 KB staging buffer and reads it back so that 8 lanes cover one row's 128
// bytes: each global store instruction then writes 4 whole 128-byte lines.
//
// Layout: row r occupies 128 bytes (8 chunks of 16 bytes); chunk c of row r
// is kept at chunk slot c ^ (r & 7).  A 16-byte shared-memory access is
// served 8 lanes at a time; in both directions those 8 lanes reach 8
// distinct 16-byte slots modulo 128 bytes, i.e. all 32 banks once:
//   write  lanes l .. l+7 (rows l .. l+7), chunk c: slots c ^ (l & 7), distinct;
//   read   lanes 8j .. 8j+7 (row r, chunks 0..7): slots c ^ (r & 7), distinct;
// and the 4-byte read of the scalar path (lanes 0..31 = the 32 columns of
// row r) reaches 32 distinct words of the row.
#pragma once
#include <cstdint>

namespace mpg {

__device__ __forceinline__ void stage_st16(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
__device__ __forceinline__ float4 stage_ld16(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float stage_ld4(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Byte offset of chunk `c` (16 bytes) of row `r` in the staging buffer.
__device__ __forceinline__ uint32_t stage_chunk_offset(int r, int c) {
  return (uint32_t)((r * 8 + (c ^ (r & 7))) * 16);
}

// Lane `lane` writes its row (v[0..31]) into the staging buffer at `stg`.
__device__ __forceinline__ void stage_write_row(uint32_t stg, int lane, const float* v) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    stage_st16(stg + stage_chunk_offset(lane, c), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

// Read-back for vector stores, step i of 8: this lane's row (i * 4 + lane / 8)
// and chunk (lane % 8).
__device__ __forceinline__ float4 stage_read_chunk(uint32_t stg, int lane, int i) {
  const int r = i * 4 + (lane >> 3);
  return stage_ld16(stg + stage_chunk_offset(r, lane & 7));
}

// Read-back for scalar stores: element (row r, column lane).
__device__ __forceinline__ float stage_read_elem(uint32_t stg, int lane, int r) {
  return stage_ld4(stg + stage_chunk_offset(r, lane >> 2) + (uint32_t)((lane & 3) * 4));
}

}  // namespace mpg
