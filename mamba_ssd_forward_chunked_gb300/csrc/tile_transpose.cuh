// In-place transpose of 32 x 32 fp32 tiles held in the 128-byte-swizzled
// shared-memory layout that TMA writes.
//
// Why: the TF32 tensor-core MMA reads its shared-memory operands correctly only
// in K-major order on this part (an MN-major TF32 operand produced zeros in a
// layout probe, while MN-major bf16 and K-major TF32 were exact).  The SSD
// contractions over tokens get both operands from token-major tensors, i.e.
// MN-major, so the fp32 path flips each 32-token x 32-element box in place
// before the MMA reads it.
//
// Layout of one box (4 KB, 1024-byte aligned): 32 rows of 128 bytes; the
// 16-byte chunk c of row r sits at physical chunk c ^ (r % 8).  On entry a row
// is a token and a chunk holds 4 consecutive elements; on exit a row is an
// element and a chunk holds 4 consecutive tokens.  Each of 64 threads owns a
// 4 x 4 micro-tile: it reads four 16-byte chunks (rows 4a..4a+3, chunk b),
// transposes them in registers and writes four chunks (rows 4b..4b+3,
// chunk a).  Both the reads and the writes of a warp cover 4 rows x 8 distinct
// chunk positions, so each is the minimum 4 shared-memory wavefronts.
#pragma once
#include <cstdint>

namespace ssd {

__device__ __forceinline__ void box_read_4x4(const uint8_t* box, int m, float4 (&v)[4]) {
  const int a = m >> 3, b = m & 7;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = 4 * a + q;
    v[q] = *reinterpret_cast<const float4*>(box + j * 128 + ((b ^ (j & 7)) << 4));
  }
}

__device__ __forceinline__ void box_write_4x4_transposed(uint8_t* box, int m, const float4 (&v)[4]) {
  const int a = m >> 3, b = m & 7;
  const float4 o[4] = {make_float4(v[0].x, v[1].x, v[2].x, v[3].x), make_float4(v[0].y, v[1].y, v[2].y, v[3].y),
                       make_float4(v[0].z, v[1].z, v[2].z, v[3].z), make_float4(v[0].w, v[1].w, v[2].w, v[3].w)};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = 4 * b + q;
    *reinterpret_cast<float4*>(box + e * 128 + ((a ^ (e & 7)) << 4)) = o[q];
  }
}

__device__ __forceinline__ float round_tf32(float f) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
  return __uint_as_float(r);
}

// Byte offset of element (token t, element e) of a box after the transpose.
__device__ __forceinline__ uint32_t box_t_offset(int t, int e) {
  return static_cast<uint32_t>(e * 128 + (((t >> 2) ^ (e & 7)) << 4) + (t & 3) * 4);
}

// One 32-token stage of a (batch, group) slice of Bm [B][L][G][N] written in the
// K-major TF32 box layout [B][G][Lp/32][N/32][4 KB] (what the fp32 chunk_state
// MMA reads).  256 threads: thread (a = tid / 32, e = tid % 32) of box k reads
// tokens 4a..4a+3 of column 32k+e (coalesced along e) and writes them as one
// 16-byte chunk.  Tokens past L read as 0.
__device__ __forceinline__ void b_transpose_stage(const float* __restrict__ Bm, float* __restrict__ bT, int L,
                                                  int G, int N, int Lp, int stage, int bg, int tid) {
  const int b = bg / G, g = bg % G;
  const int a = tid >> 5, e = tid & 31;
  const int nbox = N / 32;
  uint8_t* out = reinterpret_cast<uint8_t*>(bT) + (static_cast<int64_t>(bg) * (Lp / 32) + stage) * nbox * 4096;
  for (int k = 0; k < nbox; ++k) {
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int tok = stage * 32 + 4 * a + q;
      v[q] = tok < L ? round_tf32(Bm[((static_cast<int64_t>(b) * L + tok) * G + g) * N + k * 32 + e]) : 0.f;
    }
    *reinterpret_cast<float4*>(out + k * 4096 + box_t_offset(4 * a, e)) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

}  // namespace ssd
