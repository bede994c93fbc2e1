// Repacks canonical Q4 matrices into the streamed unit layout of the skinny
// GEMM phases. Runs once per context, at mk_create.
//
// A phase matrix is a vertical concatenation of canonical matrices (for
// example the Gated DeltaNet input projections qkv | z | a | b), optionally
// with the FFN gate and up rows interleaved in blocks of 8 so that one 16-row
// mma block holds gate rows f..f+7 above up rows f..f+7. Rows past the real
// count are zero (d = dmin = 0).
//
// Unit (tile t, super-block s) = rows 32t..32t+31, k 256s..256s+255:
//   bytes [0, 512): the 32 canonical 16-byte headers, row order;
//   bytes [512 + 512*kp + 16*lane + 4*w): one 32-bit word of 8 nibbles for lane
//     (g = lane/4, c = lane%4), sub-block kp, word w = (half of the tile rb =
//     w&1, k-step ks = 2kp + (w>>1)): with R0 = 16rb + g, R1 = R0 + 8 and
//     k0 = 16ks + 2c the nibbles at bits 0/16 are (R0, k0/k0+1), bits 4/20
//     (R1, k0/k0+1), bits 8/24 (R0, k0+8/k0+9), bits 12/28 (R1, k0+8/k0+9).
#include <cuda_runtime.h>

#include <cstdint>

#include "mk_internal.cuh"

namespace mk {

__device__ inline const uint8_t* pack_row_src(const PackSrc& p, int n, int nsb, int sb) {
  if (p.interleave_gate_up) {
    const int rb = n / 16, pos = n % 16;
    const int f = rb * 8 + (pos % 8);
    const int seg = pos < 8 ? 0 : 1;
    if (f >= p.row_end[seg] - p.row_begin[seg]) return nullptr;
    return p.src[seg] + ((size_t)f * nsb + sb) * 144;
  }
  for (int i = 0; i < p.n_seg; ++i)
    if (n >= p.row_begin[i] && n < p.row_end[i])
      return p.src[i] + ((size_t)(n - p.row_begin[i]) * nsb + sb) * 144;
  return nullptr;
}

__global__ void pack_units_kernel(PackSrc p, uint8_t* __restrict__ dst, int n_tiles, int nsb) {
  __shared__ uint8_t blk[32][144];
  const int unit = blockIdx.x;
  const int tile = unit / nsb, sb = unit % nsb;
  for (int i = threadIdx.x; i < 32 * 144; i += blockDim.x) {
    const int row = i / 144, b = i % 144;
    const uint8_t* s = pack_row_src(p, tile * 32 + row, nsb, sb);
    blk[row][b] = s ? s[b] : 0;
  }
  __syncthreads();
  uint8_t* out = dst + (size_t)unit * kUnitBytes;
  for (int i = threadIdx.x; i < 32 * 16; i += blockDim.x) out[i] = blk[i / 16][i % 16];
  auto code = [&](int row, int k) -> uint32_t {
    const int j = k / 32, i = k % 32;
    const uint8_t byte = blk[row][16 + 16 * j + (i % 16)];
    return i < 16 ? (byte & 15u) : (byte >> 4);
  };
  for (int wi = threadIdx.x; wi < 1024; wi += blockDim.x) {
    const int kp = wi / 128, lane = (wi / 4) % 32, w = wi % 4;
    const int rb = w & 1, ks = 2 * kp + (w >> 1);
    const int g = lane / 4, c = lane % 4;
    const int r0 = 16 * rb + g, r1 = r0 + 8, k0 = 16 * ks + 2 * c;
    const uint32_t word = code(r0, k0) | (code(r0, k0 + 1) << 16) | (code(r1, k0) << 4) |
                          (code(r1, k0 + 1) << 20) | (code(r0, k0 + 8) << 8) |
                          (code(r0, k0 + 9) << 24) | (code(r1, k0 + 8) << 12) |
                          (code(r1, k0 + 9) << 28);
    reinterpret_cast<uint32_t*>(out + kUnitHdr)[wi] = word;
  }
}

cudaError_t pack_units(const PackSrc& p, uint8_t* dst, int n_tiles, int nsb, cudaStream_t s) {
  const int units = n_tiles * nsb;
  if (units == 0) return cudaSuccess;
  pack_units_kernel<<<units, 128, 0, s>>>(p, dst, n_tiles, nsb);
  return cudaGetLastError();
}

}  // namespace mk
