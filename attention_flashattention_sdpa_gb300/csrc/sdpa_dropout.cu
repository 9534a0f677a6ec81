// sdpa_dropout.cu — the dropout keep mask, drawn with Philox4x32-10.
//
// The SDPA node of the cuDNN 9 blog's walkthrough has a dropout option that the pages do not
// define.  Here dropout keeps each softmax probability P_ij with a mask bit and scales kept
// ones by 1/(1 - p).  The bits come from the counter-based generator Philox4x32-10 (Salmon,
// Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): element n of
// the row-major grid [b*h_q][s_q][s_kv rounded up to 128] takes the 16-bit half n % 2 (0 =
// low) of word (n % 8) / 2 of the block for the 128-bit counter (n / 8, offset) and the 64-bit
// key seed (each as 32-bit words, low word first); it is kept iff that 16-bit value is >= the
// threshold round(p * 65536).  Each round needs two 32 x 32 -> 64-bit products.
//
// One kernel writes the bits twice: row-major for the forward pass (a thread owns a query
// row) and transposed for the backward pass (a thread owns a key row), so neither attention
// kernel runs the generator.  In both, the two elements of an even/odd pair sit 16 bits apart
// (key j of a row at bit 16 * (j % 2) + (j % 32) / 2 of word j / 32; row i of a key likewise):
// the attention kernels keep or drop a packed pair of 16-bit values with one shift and one
// byte permute.
#include <cstdint>

#include "sdpa_internal.h"

namespace sdpa {
namespace {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;   // round multipliers
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;   // Weyl key increments
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// The ten round keys of a 64-bit key (the same for every block of a draw).
struct RoundKeys {
  uint32_t k0[10], k1[10];
};

__device__ __forceinline__ RoundKeys round_keys(uint64_t seed) {
  RoundKeys rk;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    rk.k0[r] = k0;
    rk.k1[r] = k1;
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return rk;
}

// 8 keep bits of counter block g, in the paired order: element 8g + e at bit e / 2 for even e
// and at bit 16 + e / 2 for odd e.  Keep iff the 16-bit draw u is at least the threshold T,
// i.e. iff u + (65536 - T) reaches bit 16.
__device__ __forceinline__ uint32_t keep8(uint64_t g, uint32_t off_lo, uint32_t off_hi, const RoundKeys& rk,
                                          uint32_t c) {
  uint32_t x0 = static_cast<uint32_t>(g), x1 = static_cast<uint32_t>(g >> 32), x2 = off_lo, x3 = off_hi;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = static_cast<uint64_t>(kPhiloxM0) * x0;
    const uint64_t p1 = static_cast<uint64_t>(kPhiloxM1) * x2;
    x0 = static_cast<uint32_t>(p1 >> 32) ^ x1 ^ rk.k0[r];
    x1 = static_cast<uint32_t>(p1);
    x2 = static_cast<uint32_t>(p0 >> 32) ^ x3 ^ rk.k1[r];
    x3 = static_cast<uint32_t>(p0);
  }
  const uint32_t w[4] = {x0, x1, x2, x3};
  uint32_t bits = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) bits |= (((w[e / 2] >> (16 * (e % 2))) & 0xFFFFu) + c) >> 16 << (16 * (e % 2) + e / 2);
  return bits;
}

// Transposes the 32 x 32 bit matrix a warp holds (bit c of lane l's word = M[l][c]) so that
// bit l of lane c's word = M[l][c]: five exchange stages, each swapping the off-diagonal k x k
// blocks (k = 16, 8, 4, 2, 1) between lanes l and l ^ k.
// Even bits of x to the low half, odd bits to the high half (bit 2k -> k, 2k + 1 -> 16 + k):
// four delta swaps.
__device__ __forceinline__ uint32_t unshuffle_pairs(uint32_t x) {
  uint32_t t = (x ^ (x >> 1)) & 0x22222222u;
  x ^= t ^ (t << 1);
  t = (x ^ (x >> 2)) & 0x0C0C0C0Cu;
  x ^= t ^ (t << 2);
  t = (x ^ (x >> 4)) & 0x00F000F0u;
  x ^= t ^ (t << 4);
  t = (x ^ (x >> 8)) & 0x0000FF00u;
  x ^= t ^ (t << 8);
  return x;
}

__device__ __forceinline__ uint32_t transpose32(uint32_t x, int lane) {
  constexpr uint32_t kMask[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int k = 16 >> st;
    const uint32_t m = kMask[st];
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, k);
    x = (lane & k) ? ((x & ~m) | ((y >> k) & m)) : ((x & m) | ((y << k) & ~m));
  }
  return x;
}

// One CTA of 128 threads per (b*h_q, 128-row query block, 128-key block).  Lane L of warp w
// draws row 32w + L: 16 Philox blocks give its 128 bits, stored as four row-major words (keys
// paired 16 bits apart).  The
// transposed words come from a five-stage shuffle transpose of each 32x32 bit block and a 2 KB
// exchange.
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
                                              kb * 128) / 8;
    const RoundKeys rk = round_keys(p.seed);
    const uint32_t off_lo = static_cast<uint32_t>(p.offset), off_hi = static_cast<uint32_t>(p.offset >> 32);
    const uint32_t c = 65536u - p.threshold;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = keep8(g0 + 4 * i, off_lo, off_hi, rk, c) | (keep8(g0 + 4 * i + 1, off_lo, off_hi, rk, c) << 4) |
             (keep8(g0 + 4 * i + 2, off_lo, off_hi, rk, c) << 8) | (keep8(g0 + 4 * i + 3, off_lo, off_hi, rk, c) << 12);
    if (p.rows != nullptr) {
      uint4* dst = reinterpret_cast<uint4*>(p.rows + (static_cast<int64_t>(bh) * p.s_q + row) * p.kv_words +
                                            kb * 4);
      *dst = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  if (p.cols == nullptr) return;   // uniform over the grid
  // Transpose each 32 x 32 bit block: lane c then holds the bits of the key at bit position c
  // of the row words, key 32i + 2 (c % 16) + c / 16 (paired order), for the warp's rows
  // 32w .. 32w + 31 (bit l = row 32w + l); the rows are then paired the same way (even rows to
  // the low half, odd rows to the high half).
#pragma unroll
  for (int i = 0; i < 4; ++i)
    tile[32 * i + 2 * (lane % 16) + lane / 16][warp] = unshuffle_pairs(transpose32(w[i], lane));
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
