// sdpa_dropout.cu — the dropout keep mask, drawn with Philox4x64-10.
//
// The SDPA node of the cuDNN 9 blog's walkthrough has a dropout option that the pages do not
// define.  Here dropout keeps each softmax probability P_ij with a mask bit and scales kept
// ones by 1/(1 - p).  The bits come from the counter-based generator Philox4x64-10 (Salmon,
// Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): element n of
// the row-major grid [b*h_q][s_q][s_kv rounded up to 128] takes 16-bit lane n % 4 of word
// (n % 16) / 4 of the block for counter (n / 16, offset, 0, 0) and key (seed, 0); it is kept
// iff that 16-bit value is >= the threshold round(p * 65536).
//
// One kernel writes the bits twice: row-major for the forward pass (a thread owns a query
// row) and transposed for the backward pass (a thread owns a key row), so neither attention
// kernel runs the generator.  In the transposed words the two rows of an even/odd pair sit
// 16 bits apart (row i at bit 16 * (i % 2) + (i % 32) / 2 of word i / 32): the backward pass
// keeps or drops a packed pair of 16-bit values with one shift and one byte permute.
#include <cstdint>

#include "sdpa_internal.h"

namespace sdpa {
namespace {

constexpr uint64_t kPhiloxM0 = 0xD2E7470EE14C6C93ull;   // round multipliers
constexpr uint64_t kPhiloxM1 = 0xCA5A826395121157ull;
constexpr uint64_t kPhiloxW0 = 0x9E3779B97F4A7C15ull;   // Weyl key increments
constexpr uint64_t kPhiloxW1 = 0xBB67AE8584CAA73Bull;

struct U64x4 {
  uint64_t x[4];
};

__device__ __forceinline__ U64x4 philox4x64_10(uint64_t c0, uint64_t c1, uint64_t k0, uint64_t k1) {
  uint64_t x0 = c0, x1 = c1, x2 = 0, x3 = 0;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kPhiloxW0;
      k1 += kPhiloxW1;
    }
    const uint64_t hi0 = __umul64hi(kPhiloxM0, x0), lo0 = kPhiloxM0 * x0;
    const uint64_t hi1 = __umul64hi(kPhiloxM1, x2), lo1 = kPhiloxM1 * x2;
    x0 = hi1 ^ x1 ^ k0;
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
  }
  return U64x4{{x0, x1, x2, x3}};
}

// 16 keep bits (bit e = element 16g + e) of counter block g.
__device__ __forceinline__ uint32_t keep16(uint64_t g, const DropoutParams& p) {
  const U64x4 w = philox4x64_10(g, p.offset, p.seed, 0);
  uint32_t bits = 0;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint32_t u = static_cast<uint32_t>(w.x[e / 4] >> (16 * (e % 4))) & 0xFFFFu;
    bits |= (u >= p.threshold ? 1u : 0u) << e;
  }
  return bits;
}

// One CTA of 128 threads per (b*h_q, 128-row query block, 128-key block).  Lane L of warp w
// draws row 32w + L: 8 Philox blocks give its 128 bits, stored as four row-major words.  The
// transposed words come from 32 ballots per 32x32 bit block and a 2 KB exchange.
__global__ void __launch_bounds__(128) dropout_mask_kernel(const DropoutParams p) {
  __shared__ uint32_t tile[128][4];   // [key within block][query word]
  const int kb = blockIdx.x, qb = blockIdx.y, bh = blockIdx.z;
  // Under a causal mask no row of this tile sees any of its keys: nothing reads these bits.
  if (p.skip_above && kb * 128 > qb * 128 + 127 + p.diag_off) return;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row = qb * 128 + threadIdx.x;
  const int64_t row_pitch = static_cast<int64_t>(p.kv_words) * 32;    // s_kv rounded up to 128
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if (row < p.s_q) {
    const uint64_t g0 = static_cast<uint64_t>((static_cast<int64_t>(bh) * p.s_q + row) * row_pitch +
                                              kb * 128) / 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = keep16(g0 + 2 * i, p) | (keep16(g0 + 2 * i + 1, p) << 16);
    if (p.rows != nullptr) {
      uint4* dst = reinterpret_cast<uint4*>(p.rows + (static_cast<int64_t>(bh) * p.s_q + row) * p.kv_words +
                                            kb * 4);
      *dst = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  if (p.cols == nullptr) return;   // uniform over the grid
  // Transpose: bit c of ballot c' over the warp's 32 rows is key 32i + c's bit for row 32w + lane.
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t mine = 0;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const uint32_t col = __ballot_sync(0xffffffffu, (w[i] >> c) & 1u);
      if (lane == c) mine = col;
    }
    // Unshuffle: even rows to the low half, odd rows to the high half (four delta swaps).
    uint32_t t = (mine ^ (mine >> 1)) & 0x22222222u;
    mine ^= t ^ (t << 1);
    t = (mine ^ (mine >> 2)) & 0x0C0C0C0Cu;
    mine ^= t ^ (t << 2);
    t = (mine ^ (mine >> 4)) & 0x00F000F0u;
    mine ^= t ^ (t << 4);
    t = (mine ^ (mine >> 8)) & 0x0000FF00u;
    mine ^= t ^ (t << 8);
    tile[32 * i + lane][warp] = mine;
  }
  __syncthreads();
  const int key = kb * 128 + threadIdx.x;
  if (key < p.s_kv) {
    uint4* dst = reinterpret_cast<uint4*>(p.cols + (static_cast<int64_t>(bh) * p.s_kv + key) * p.q_words +
                                          qb * 4);
    *dst = make_uint4(tile[threadIdx.x][0], tile[threadIdx.x][1], tile[threadIdx.x][2], tile[threadIdx.x][3]);
  }
}

}  // namespace

cudaError_t launch_dropout_mask(const DropoutParams& p, int bh, cudaStream_t st) {
  dim3 grid(p.kv_words / 4, p.q_words / 4, bh);
  dropout_mask_kernel<<<grid, 128, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sdpa
