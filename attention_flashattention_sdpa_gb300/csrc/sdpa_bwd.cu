// sdpa_bwd.cu — SDPA backward pass for sm_103a: dQ, dK, dV from Q, K, V, O, dO and the
// per-row LSE kept by the forward pass.
//
// The pages show that a backward graph exists next to the forward one (cuDNN 9 blog,
// "SDPA performance", Fig. 2 "forward + backward"; "SDPA as a cuDNN graph": backward
// graphs offer the same flexibility) but print no formula; the derivative used here is
// the analytic one of O = softmax(scale·QKᵀ + mask)·V:
//     P = exp(scale·QKᵀ − LSE)            (recomputed from the forward's statistics)
//     dV = Pᵀ·dO,  dP = dO·Vᵀ,  Delta_i = Σ_d dO_id·O_id  (= Σ_j P_ij·dP_ij)
//     dS = P ∘ (dP − Delta),  dQ = scale·dS·K,  dK = scale·dSᵀ·Q
// with dK, dV summed over the query heads of each KV group.
//
// Three launches (the pages note an engine may be "a small set of cooperating kernels"):
//   1. bwd_pre:   -Delta_i, -LSE_i·log2(e) and a zeroed fp32 dQ accumulator (workspace).
//   2. bwd_main:  one CTA per (batch, KV head, 128-row KV block); K and V stay in shared
//                 memory while the CTA walks every (query head of the group, 128-row query
//                 block) it can see.  Per step five tcgen05 MMAs (Sᵀ = K·Qᵀ, dPᵀ = V·dOᵀ,
//                 dV += Pᵀ·dO, dK += dSᵀ·Q, dQ = dS·K) with dV and dK accumulating in TMEM
//                 for the whole walk, and dQ drained by a dedicated warpgroup from TMEM through
//                 shared memory into the fp32 accumulator with TMA reduce-add.
//   3. bwd_dq:    dQ = scale·accumulator, rounded to the output dtype in the caller's strides.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "ptx.cuh"
#include "sdpa_internal.h"

namespace sdpa {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float to_f32(const __half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(const __nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ uint32_t pack2(float a, float b, int dt) {
  if (dt == kBF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack2(uint32_t u, int dt) {
  if (dt == kBF16) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(h);
  }
  __half2 h = *reinterpret_cast<__half2*>(&u);
  return __half22float2(h);
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// 1. preprocess: Delta, LSE·log2 e, zeroed dQ accumulator
// ---------------------------------------------------------------------------

// Scale factors of the backward pass.  With FP8 inputs the kernels read widened copies of
// the stored codes, so the per-tensor descales enter here: S = scale·d_q·d_k·Q'K'ᵀ,
// dP = d_do·d_v·dO'V'ᵀ, dV = d_do·Pᵀ dO', dK = scale·d_q·dSᵀ Q', dQ = scale·d_k·dS K',
// Delta = d_do·rowsum(dO'∘O); dropout's 1/(1 - p) multiplies dP and dV.
struct BwdScales {
  float s_log2, dp, dv, dk, dq, delta;
};

__device__ __forceinline__ BwdScales bwd_scales(const BwdParams& p) {
  float dq = 1.f, dk = 1.f, dv = 1.f, ddo = 1.f;
  if (p.descale_q != nullptr) {
    dq = __ldg(p.descale_q);
    dk = __ldg(p.descale_k);
    dv = __ldg(p.descale_v);
    ddo = __ldg(p.descale_do);
  }
  BwdScales s;
  s.s_log2 = p.scale_log2 * dq * dk;
  s.dp = ddo * dv * p.drop_scale;
  s.dv = ddo * p.drop_scale;
  s.dk = p.scale * dq;
  s.dq = p.scale * dk;
  s.delta = ddo;
  return s;
}

// The transposed bias copy and the bias-gradient accumulator are stored in 128 x 128 tiles
// (key block kb, query block qb) ordered [nb][nh][kb][qb].  Inside a tile, for each half of
// the 64 queries (hq2) and each quarter of 32 key rows (one warp's TMEM lanes), the 16-byte
// chunks of a key row follow one another 32 rows apart: chunk e of key row 32·quad + lane is
// 16-byte unit (hq2·4 + quad)·U·32 + e·32 + lane, U = 8 chunks of eight 16-bit values (copy)
// or 16 chunks of four fp32 values (accumulator).  A warp that loads or reduce-adds chunk e of
// its 32 key rows then touches one contiguous 512-byte run instead of 32 rows.
__device__ __forceinline__ int64_t bias_tile_elems(const BwdParams& p, int bi, int hq, int kv_row, int q0) {
  const int nb = p.bias_nb > 1 ? bi : 0, nh = p.bias_nh > 1 ? hq : 0;
  const int n_kvb = (p.s_kv + kBlockN - 1) / kBlockN, n_qb = p.s_q_pad / kBlockM;
  return ((static_cast<int64_t>(nb) * p.bias_nh + nh) * n_kvb + kv_row / kBlockN) * n_qb * 16384 +
         static_cast<int64_t>(q0 / kBlockM) * 16384;
}

// 8·NV bias values of key row kv_row for queries q0.. (q0 a multiple of 8·NV within a 64-query
// half) from the tiled copy; zero for a key row beyond s_kv, which sees nothing anyway.
template <int NV>
__device__ __forceinline__ void load_bias_t(const BwdParams& p, int bi, int hq, int kv_row, int q0, uint4 (&bz)[NV]) {
  if (kv_row >= p.s_kv) {
#pragma unroll
    for (int e = 0; e < NV; ++e) bz[e] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const int r = kv_row % kBlockN, hq2 = (q0 % kBlockM) / 64, e0 = (q0 % 64) / 8;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.bias_t) +
                                                    bias_tile_elems(p, bi, hq, kv_row, q0)) +
                     ((hq2 * 4 + r / 32) * 8 + e0) * 32 + r % 32;
#pragma unroll
  for (int e = 0; e < NV; ++e) bz[e] = __ldg(src + e * 32);
}

// Starts moving a later step's bias chunks of this warp's 32 key rows (4 KB, one 128-byte
// line per lane) into L2, so that load_bias_t then hits there.
__device__ __forceinline__ void prefetch_bias_t(const BwdParams& p, int bi, int hq, int kv_row, int q0) {
  if (kv_row >= p.s_kv) return;
  const int r = kv_row % kBlockN, hq2 = (q0 % kBlockM) / 64;
  const uint4* run = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.bias_t) +
                                                    bias_tile_elems(p, bi, hq, kv_row, q0)) +
                     (hq2 * 4 + r / 32) * 8 * 32;
  prefetch_l2(run + (r % 32) * 8);
}

// This thread's first accumulator chunk for key row kv_row and queries q0.. (q0 a multiple of
// 4 within a 64-query half); chunk k of the thread is 128 floats further (nullptr past s_kv).
__device__ __forceinline__ float* dbias_row(const BwdParams& p, int bi, int hq, int kv_row, int q0) {
  if (kv_row >= p.s_kv) return nullptr;
  const int r = kv_row % kBlockN, hq2 = (q0 % kBlockM) / 64, e0 = (q0 % 64) / 4;
  return p.dbias_acc + bias_tile_elems(p, bi, hq, kv_row, q0) +
         static_cast<int64_t>(((hq2 * 4 + r / 32) * 16 + e0) * 32 + r % 32) * 4;
}

// dS of columns c, c+1 into the accumulator, four at a time (c is a compile-time constant).
__device__ __forceinline__ void dbias_emit(float* row, int c, float2 dd, float2& hold) {
  if (c % 4 == 0) {
    hold = dd;
  } else if (row != nullptr) {
    red_add_v4(row + (c / 4) * 128, hold.x, hold.y, dd.x, dd.y);
  }
}

// Columns c, c+1 of NV packed 16-bit bias vectors (eight values each), as fp32.
template <int DT, int NV>
__device__ __forceinline__ float2 bias_pair(const uint4 (&bz)[NV], int c) {
  const uint4 v = bz[c / 8];
  const uint32_t w = (c % 8 == 0) ? v.x : (c % 8 == 2) ? v.y : (c % 8 == 4) ? v.z : v.w;
  return unpack2(w, DT);
}

// One group of D/8 threads per row; each thread reads 8 elements (16 bytes) of O and dO.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdParams p) {
  // The main kernel may start its set-up and its K/V loads now; it waits for this grid before
  // it reads Delta, -LSE·log2 e or the zeroed dQ accumulator.
  griddep_launch_dependents();
  constexpr int TPR = D / 8;              // threads per row
  constexpr int ROWS = 256 / TPR;         // rows per block
  const int bh = blockIdx.y;
  const int bi = bh / p.h_q, hq = bh % p.h_q;
  const int row = blockIdx.x * ROWS + threadIdx.x / TPR;
  const int part = threadIdx.x % TPR;
  float acc = 0.f;
  const bool valid = row < batch_lens(p, bi).len_q;   // padded rows take no part
  if (valid) {
    const T* o = reinterpret_cast<const T*>(p.o) + bi * p.o_sb + hq * p.o_sh + row * p.o_ss + part * 8;
    const T* g = reinterpret_cast<const T*>(p.dout) + bi * p.do_sb + hq * p.do_sh + row * p.do_ss + part * 8;
    const uint4 ov = *reinterpret_cast<const uint4*>(o);
    const uint4 gv = *reinterpret_cast<const uint4*>(g);
    const T* oe = reinterpret_cast<const T*>(&ov);
    const T* ge = reinterpret_cast<const T*>(&gv);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc += to_f32(oe[i]) * to_f32(ge[i]);
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  const int64_t vrow = static_cast<int64_t>(bh) * p.s_q_pad + row;
  if (row < p.s_q_pad) {
    float* dq = p.dq_acc + vrow * D + part * 8;
    reinterpret_cast<float4*>(dq)[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(dq)[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (part == 0) {
      // Stored negated, so the main kernel adds them with paired fp32 instructions.
      p.delta[vrow] = valid ? -acc * bwd_scales(p).delta : 0.f;
      // Rows with no visible key (LSE = -inf) and padded rows get P = 0 everywhere.
      const float lse = valid ? p.lse[static_cast<int64_t>(bh) * p.s_q + row] : -INFINITY;
      // ALiBi's bias slope * (key - row - off) is split: -slope * (row mod 128) joins this
      // per-row term, and slope * (key - 128-aligned block start - off) is added per key row.
      const float col_bias = p.alibi ? alibi_slope_log2(p, hq) * static_cast<float>(row % kBlockM) : 0.f;
      p.lse2[vrow] = (lse == -INFINITY) ? -INFINITY : -lse * kLog2e - col_bias;
    }
  }
}

// ---------------------------------------------------------------------------
// 3. dQ = scale * accumulator, in the output dtype and strides
// ---------------------------------------------------------------------------

template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const BwdParams p) {
  griddep_wait();   // the main kernel's reduce-adds into the accumulator are complete
  constexpr int TPR = D / 8;
  constexpr int ROWS = 256 / TPR;
  const int bh = blockIdx.y;
  const int bi = bh / p.h_q, hq = bh % p.h_q;
  const int row = blockIdx.x * ROWS + threadIdx.x / TPR;
  const int part = threadIdx.x % TPR;
  if (row >= p.s_q) return;
  const float* src = p.dq_acc + (static_cast<int64_t>(bh) * p.s_q_pad + row) * D + part * 8;
  const float4 a = reinterpret_cast<const float4*>(src)[0];
  const float4 b = reinterpret_cast<const float4*>(src)[1];
  const float s = bwd_scales(p).dq;
  const int dt = sizeof(T) == 2 && std::is_same<T, __nv_bfloat16>::value ? kBF16 : kF16;
  uint4 w;
  w.x = pack2(a.x * s, a.y * s, dt);
  w.y = pack2(a.z * s, a.w * s, dt);
  w.z = pack2(b.x * s, b.y * s, dt);
  w.w = pack2(b.z * s, b.w * s, dt);
  T* dst = reinterpret_cast<T*>(p.dq) + bi * p.dq_sb + hq * p.dq_sh + row * p.dq_ss + part * 8;
  *reinterpret_cast<uint4*>(dst) = w;
}

// Split groups only: zero the fp32 dK/dV accumulators before the main kernel, and write
// dK, dV in the output dtype and strides after it.
// Split groups add dK and dV shares into fp32 accumulators [b][h_kv] x 128-row key blocks of
// D columns.  Inside a block, chunk e (four columns) of key row 32·quad + lane is float4 unit
// (quad·D/4 + e)·32 + lane, so a warp's reduction of one chunk of its 32 rows is one contiguous
// 512-byte run.  This returns the float offset of chunk 0 of key row kv_row; chunk e is 128
// floats further.
__device__ __forceinline__ int64_t kv_acc_offset(const BwdParams& p, int bi, int hk, int kv_row, int D) {
  const int r = kv_row % kBlockN;
  return ((static_cast<int64_t>(bi) * p.h_kv + hk) * p.s_kv_pad + (kv_row - r)) * D +
         static_cast<int64_t>((r / 32) * (D / 4) * 32 + r % 32) * 4;
}

// Zeros for columns [c0, c0 + ncols) of the dK and dV rows of key block j of (bi, hk) that lie
// below s_kv: what a CTA whose key block no query sees contributes (16-bit zeros are zero bits).
__device__ __forceinline__ void zero_kv_block(const BwdParams& p, int bi, int hk, int j, int c0, int ncols) {
  const int chunks = ncols / 8;
  for (int i = threadIdx.x; i < kBlockN * chunks; i += blockDim.x) {
    const int row = j * kBlockN + i / chunks, col = c0 + (i % chunks) * 8;
    if (row >= p.s_kv) continue;
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dk) + bi * p.dk_sb + hk * p.dk_sh + row * p.dk_ss + col) =
        make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dv) + bi * p.dv_sb + hk * p.dv_sh + row * p.dv_ss + col) =
        make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(256) bwd_zero_kv_kernel(const BwdParams p) {
  const int64_t n4 = static_cast<int64_t>(p.b) * p.h_kv * p.s_kv_pad * p.d / 4;
  float4* a = reinterpret_cast<float4*>(p.dk_acc);
  float4* b = reinterpret_cast<float4*>(p.dv_acc);
  for (int64_t i = blockIdx.x * 256ll + threadIdx.x; i < n4; i += 256ll * gridDim.x) {
    a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    b[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_kv_convert_kernel(const BwdParams p) {
  constexpr int TPR = D / 8;
  constexpr int ROWS = 256 / TPR;
  const int bh = blockIdx.y;
  const int bi = bh / p.h_kv, hk = bh % p.h_kv;
  const int row = blockIdx.x * ROWS + threadIdx.x / TPR;
  const int part = threadIdx.x % TPR;
  if (row >= p.s_kv) return;
  const int dt = std::is_same<T, __nv_bfloat16>::value ? kBF16 : kF16;
  const int64_t off = kv_acc_offset(p, bi, hk, row, D) + static_cast<int64_t>(2 * part) * 128;
  for (int which = 0; which < 2; ++which) {
    const float* src = (which == 0 ? p.dk_acc : p.dv_acc) + off;
    const float4 a = reinterpret_cast<const float4*>(src)[0];         // columns 8·part ..
    const float4 c = reinterpret_cast<const float4*>(src + 128)[0];   // 8·part + 4 ..
    uint4 w;
    w.x = pack2(a.x, a.y, dt);
    w.y = pack2(a.z, a.w, dt);
    w.z = pack2(c.x, c.y, dt);
    w.w = pack2(c.z, c.w, dt);
    T* dst = which == 0
                 ? reinterpret_cast<T*>(p.dk) + bi * p.dk_sb + hk * p.dk_sh + row * p.dk_ss + part * 8
                 : reinterpret_cast<T*>(p.dv) + bi * p.dv_sb + hk * p.dv_sh + row * p.dv_ss + part * 8;
    *reinterpret_cast<uint4*>(dst) = w;
  }
}

// ---------------------------------------------------------------------------
// 2. main kernel
// ---------------------------------------------------------------------------

template <int D>
struct BwdCfg {
  static constexpr int TILE = kBlockM * D * 2;        // one 128-row tile of Q, K, V or dO
  static constexpr int NCHUNK = D / 64;               // 128-byte chunks along d
  // Q / dO tiles: slots 0 and 1 hold Q of alternate steps (Q is read until dK of its step),
  // the remaining NDO slots hold dO (read until dV, early in its step), so the next step's dO
  // can load while the current step's dQ and dK run.
  static constexpr int NSLOT = (D == 64) ? 4 : 3;
  static constexpr int NDO = NSLOT - 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_RING = 2 * TILE;
  static constexpr int OFF_DS = OFF_RING + NSLOT * TILE;
  static constexpr int DS_BYTES = kBlockM * kBlockN * 2;
  static constexpr int OFF_DQ = OFF_DS + DS_BYTES;    // dQ staging: two 32-column fp32 chunks
  static constexpr int DQ_BYTES = 2 * 16384;
  static constexpr int OFF_VEC = OFF_DQ + DQ_BYTES;   // [2 buffers][LSE2, Delta][128] fp32
  static constexpr int OFF_BAR = OFF_VEC + 2 * 2 * 128 * 4;
  static constexpr int SMEM_BYTES = OFF_BAR + 512;
  static constexpr int THREADS = 512;
  static constexpr int KSTEPS_D = D / 16;             // MMAs over a d reduction
  static constexpr int R_COL = 0;                     // regions R0 = [0,128), R1 = [128,256)
  static constexpr int DV_COL = 256;
  static constexpr int DK_COL = 256 + D;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(DK_COL + D <= 512, "TMEM budget");
};

struct alignas(8) BwdBarriers {
  uint64_t kv_full;
  uint64_t ring_full[4];
  uint64_t ring_empty[4];
  uint64_t s_full[2];
  uint64_t dp_full[2];
  uint64_t p_full[2];
  uint64_t ds_full[2];
  uint64_t dq_full[2];
  uint64_t dq_free[2];
  uint64_t acc_full;
  uint64_t drain;
  uint64_t epi_ready[2];
  uint64_t dp_consumed[2];  // the compute warps have read dPᵀ out of TMEM
  uint64_t dsbuf_free[2];   // the dQ and dK MMAs of a step have read the dS buffer
  uint64_t stage_full[2];   // dQ staging buffer written by the 128 drain threads
  uint64_t stage_free[2];   // the reduce-add of that buffer has read shared memory
  uint32_t tmem_base;
  int abort;
};

// First query block (of `bq` rows) that can see key block j of a batch: with a causal mask
// key row kv is visible to query i iff kv <= i + off.
__device__ __forceinline__ int first_q_block(const BwdParams& p, const Lens& L, int j, int bq) {
  if (!p.causal) return 0;
  const int r0 = j * kBlockN - L.off;
  return r0 <= 0 ? 0 : r0 / bq;
}

template <int D, int DT, int FEAT>
__global__ void __launch_bounds__(512, 1) bwd_main_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  constexpr bool ALIBI = (FEAT & kFeatAlibi) != 0;
  constexpr bool DROP = (FEAT & kFeatDropout) != 0;
  constexpr bool BIAS = (FEAT & kFeatBias) != 0;
  constexpr bool DBIAS = (FEAT & kFeatDBias) != 0;
  extern __shared__ __align__(1024) uint8_t smem[];
  // The dQ conversion kernel may be launched now; it waits for this grid to complete.  This
  // grid in turn may run alongside the pre-pass (Delta, -LSE·log2 e, the zeroed dQ
  // accumulator): the producer waits for it (griddep_wait) before it loads the first vectors,
  // and every other read of those results follows from that load (the vectors reach the
  // compute warps through shared memory, the dQ reduce-adds follow the MMAs that follow the
  // Q tiles).  The producer waits again at its exit, so a CTA that gave up early still
  // completes after the pre-pass.
  griddep_launch_dependents();
  BwdBarriers& bars = *reinterpret_cast<BwdBarriers*>(smem + C::OFF_BAR);
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sRing = smem + C::OFF_RING;
  uint8_t* sDS = smem + C::OFF_DS;
  uint8_t* sDQ = smem + C::OFF_DQ;
  float* sVec = reinterpret_cast<float*>(smem + C::OFF_VEC);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // Launch order: units (batch, KV head, share) in groups whose Q and dO together take about
  // 32 MB, so that resident CTAs share them in L2; within a group the heaviest KV blocks of
  // all its units go first (for causal, the first blocks), then the next block index, which
  // shortens the tail of long CTAs.  Units of 8 MB or more go one at a time (head-major).
  const int n_kvb = (p.s_kv + kBlockN - 1) / kBlockN;
  const int n_units = p.b * p.h_kv * p.kv_split;
  const long long unit_bytes = 4ll * p.heads_per_split * p.s_q_pad * p.d;
  int G = static_cast<int>((32ll << 20) / (unit_bytes > 0 ? unit_bytes : 1));
  G = (unit_bytes >= (8ll << 20) || G < 1) ? 1 : (G > n_units ? n_units : G);
  const int grp = blockIdx.x / (G * n_kvb);
  const int gsz = min(G, n_units - grp * G);
  const int rem = blockIdx.x - grp * G * n_kvb;
  const int j = rem / gsz;                                  // KV block
  const int unit = grp * G + rem % gsz;
  const int split = unit % p.kv_split;                      // share of the KV group's heads
  const int bhk = unit / p.kv_split;
  const int bi = bhk / p.h_kv;
  const int hk = bhk % p.h_kv;
  const Lens L = batch_lens(p, bi);
  const int n_qb = (L.len_q + kBlockM - 1) / kBlockM;
  const int q_first = first_q_block(p, L, j, kBlockM);
  const bool kv_live = j * kBlockN < L.len_kv;              // this block holds a valid key
  const int per_head = (kv_live && q_first < n_qb) ? n_qb - q_first : 0;
  const int head0 = hk * p.group + split * p.heads_per_split;
  const int n_heads = max(0, min(p.heads_per_split, (hk + 1) * p.group - head0));
  const int n_iter = per_head * n_heads;
  // No query sees this key block (it lies beyond len_kv, or above a causal diagonal): its dK
  // and dV rows are zero (split groups: the zeroed accumulators already hold its share), and
  // the CTA needs neither its K/V tiles nor tensor memory.
  if (n_iter == 0) {
    griddep_wait();
    if (p.kv_split == 1) zero_kv_block(p, bi, hk, j, 0, D);
    return;
  }

  // The 128-byte swizzle of every tile assumes a 1024-byte aligned base (the budget leaves
  // no room for manual alignment).  If that ever fails, report it and do nothing.
  if (smem_u32(smem) & 1023u) {
    griddep_wait();
    if (threadIdx.x == 0) atomicOr(&g_device_error, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars.kv_full, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars.ring_full[s], 1);
      mbar_init(&bars.ring_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.s_full[b], 1);
      mbar_init(&bars.dp_full[b], 1);
      mbar_init(&bars.dq_full[b], 1);
      mbar_init(&bars.p_full[b], 256);
      mbar_init(&bars.ds_full[b], 256);
      mbar_init(&bars.dq_free[b], 128);
    }
    mbar_init(&bars.acc_full, 1);
    mbar_init(&bars.drain, 1);
    mbar_init(&bars.epi_ready[0], 128);
    mbar_init(&bars.epi_ready[1], 128);
    mbar_init(&bars.dp_consumed[0], 256);
    mbar_init(&bars.dp_consumed[1], 256);
    mbar_init(&bars.dsbuf_free[0], 1);
    mbar_init(&bars.dsbuf_free[1], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.stage_full[i], 128);
      mbar_init(&bars.stage_free[i], 1);
    }
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort_flag = &bars.abort;
  const Waiter wt{abort_flag, p.wait_limit};

  // iteration n -> (query head, query block)
  auto iter_head = [&](int n) { return head0 + n / per_head; };
  auto iter_qblk = [&](int n) { return q_first + n % per_head; };

  // Copies the producer has issued (for the drain at the end, should a role give up).
  bool producer = false;
  int nq = 0, nd = 0;   // Q and dO tiles issued

  // Register budget per thread: 64 for the producer / MMA warpgroup, 152 for each compute
  // warpgroup, 144 for the dQ drain (64 + 2 x 152 + 144 = 4 x 128, the launch's budget).
  if (warp < 4) {
  regs_dec<64>();
  if (warp == 0) {
    // ================================ TMA producer ====================================
    if (elect_one_sync()) {
      producer = true;
      mbar_arrive_expect_tx(&bars.kv_full, 2 * C::TILE);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_4d(sK + c * 16384, &p.tm_k, &bars.kv_full, c * 64, j * kBlockN, hk, bi);
        tma_load_4d(sV + c * 16384, &p.tm_v, &bars.kv_full, c * 64, j * kBlockN, hk, bi);
      }
      bool ok = true;
      for (int n = 0; n < n_iter && ok; ++n) {
        const int hq = iter_head(n), qb = iter_qblk(n);
        const int64_t vrow = (static_cast<int64_t>(bi) * p.h_q + hq) * p.s_q_pad + qb * kBlockM;
        for (int which = 0; which < 2 && ok; ++which) {
          // Q(n) -> slot n % 2 (use n / 2); dO(n) -> slot 2 + n % NDO (use n / NDO).
          const int slot = which == 0 ? (n & 1) : 2 + n % C::NDO;
          const int use = which == 0 ? (n >> 1) : n / C::NDO;
          if (!mbar_wait(&bars.ring_empty[slot], (use & 1) ^ 1, wt)) {
            ok = false;
            break;
          }
          // Both per-row vectors (-LSE·log2 e and -Delta) travel with Q: the compute warps then
          // wait for no dO tile, whose slot is refilled only once dV of the previous step ran.
          mbar_arrive_expect_tx(&bars.ring_full[slot], which == 0 ? C::TILE + 1024 : C::TILE);
          const CUtensorMap* map = which == 0 ? &p.tm_q : &p.tm_do;
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_4d(sRing + slot * C::TILE + c * 16384, map, &bars.ring_full[slot], c * 64,
                        qb * kBlockM, hq, bi);
          if (which == 0) {
            if (n == 0) griddep_wait();   // K/V and the first Q tile are already on their way
            bulk_load(sVec + (n & 1) * 256, p.lse2 + vrow, 512, &bars.ring_full[slot]);
            bulk_load(sVec + (n & 1) * 256 + 128, p.delta + vrow, 512, &bars.ring_full[slot]);
          }
          if (which == 0) ++nq; else ++nd;
        }
      }
    }
  } else if (warp == 1) {
    // ================================ MMA issuer ======================================
    if (elect_one_sync()) {
      const uint32_t fmt = (DT == kBF16) ? 1u : 0u;
      const uint32_t idesc_sq = make_idesc(fmt, 128, 128, false, false);     // Sᵀ, dPᵀ
      const uint32_t idesc_acc = make_idesc(fmt, 128, D, false, true);       // dV, dK
      const uint32_t idesc_dq = make_idesc(fmt, 128, D, true, true);         // dQ
      const uint32_t kA = smem_u32(sK), vA = smem_u32(sV), dsA = smem_u32(sDS);
      bool ok = mbar_wait(&bars.kv_full, 0, wt);
      tc_fence_after();
      // Sᵀ = K·Qᵀ of step m into region `reg` (Q of step m is in slot m % 2).
      auto issue_s = [&](int reg, int m, int& qslot) -> bool {
        qslot = m & 1;
        if (!mbar_wait(&bars.ring_full[qslot], (m >> 1) & 1, wt)) return false;
        tc_fence_after();
        const uint32_t qB = smem_u32(sRing + qslot * C::TILE);
#pragma unroll
        for (int k = 0; k < C::KSTEPS_D; ++k) {
          const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
          mma_ss(tmem + C::R_COL + reg * 128, make_sdesc_sw128(kA + off, 16, 1024),
                 make_sdesc_sw128(qB + off, 16, 1024), idesc_sq, k > 0, false);
        }
        tc_commit(&bars.s_full[reg]);
        return true;
      };
      int qslot = 0, qslot_next = 0;
      if (ok && n_iter > 0) ok = issue_s(0, 0, qslot);
      for (int n = 0; n < n_iter && ok; ++n) {
        const int b = n & 1;
        const uint32_t par = (n >> 1) & 1;
        const uint32_t X = tmem + C::R_COL + b * 128;         // Sᵀ, Pᵀ, then dQ of step n
        const uint32_t Y = tmem + C::R_COL + (b ^ 1) * 128;   // dPᵀ of step n, then Sᵀ of n+1
        const uint32_t qB = smem_u32(sRing + qslot * C::TILE);
        // ---- dPᵀ = V·dOᵀ (into the region dQ of the previous step used) ----
        const int gslot = 2 + n % C::NDO;
        if (!mbar_wait(&bars.ring_full[gslot], (n / C::NDO) & 1, wt)) { ok = false; break; }
        if (n >= 1 && !mbar_wait(&bars.dq_free[b ^ 1], ((n - 1) >> 1) & 1, wt)) { ok = false; break; }
        tc_fence_after();
        const uint32_t gB = smem_u32(sRing + gslot * C::TILE);
#pragma unroll
        for (int k = 0; k < C::KSTEPS_D; ++k) {
          const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
          mma_ss(Y, make_sdesc_sw128(vA + off, 16, 1024), make_sdesc_sw128(gB + off, 16, 1024),
                 idesc_sq, k > 0, false);
        }
        tc_commit(&bars.dp_full[b]);
        // ---- dV += Pᵀ·dO  (Pᵀ in TMEM: q 0..63 at X+0.., q 64..127 at X+64..) ----
        if (!mbar_wait(&bars.p_full[b], par, wt)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t a_col = (k < 4) ? k * 8 : 64 + (k - 4) * 8;
          mma_ts(tmem + C::DV_COL, X + a_col, make_sdesc_sw128(gB + k * 2048, 16384, 1024),
                 idesc_acc, (n > 0 || k > 0) ? 1u : 0u, false);
        }
        tc_commit(&bars.ring_empty[gslot]);
        // ---- Sᵀ of the next step, as soon as dPᵀ has left region Y ----
        if (n + 1 < n_iter) {
          if (!mbar_wait(&bars.dp_consumed[b], par, wt)) { ok = false; break; }
          if (!issue_s(b ^ 1, n + 1, qslot_next)) { ok = false; break; }
        }
        // ---- dQ = dS·K first (its drain gates the next dPᵀ), then dK += dSᵀ·Q (dS read
        //      K-major from shared memory) ----
        if (!mbar_wait(&bars.ds_full[b], par, wt)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          mma_ss(X, make_sdesc_sw128(dsA + k * 2048, 16384, 1024),
                 make_sdesc_sw128(kA + k * 2048, 16384, 1024), idesc_dq, k > 0, false);
        }
        tc_commit(&bars.dq_full[b]);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
          mma_ss(tmem + C::DK_COL, make_sdesc_sw128(dsA + off, 16, 1024),
                 make_sdesc_sw128(qB + k * 2048, 16384, 1024), idesc_acc,
                 (n > 0 || k > 0) ? 1u : 0u, false);
        }
        tc_commit(&bars.dsbuf_free[b]);
        tc_commit(&bars.ring_empty[qslot]);
        qslot = qslot_next;
      }
      tc_commit(&bars.acc_full);
      tc_commit(&bars.drain);
      mbar_wait_drain(&bars.drain, 0);
    }
  }
  } else if (warp < 12) {
    regs_inc<152>();
    // ============================ Pᵀ / dSᵀ (two column halves) ========================
    const int h = (warp - 4) / 4;                         // query columns [64h, 64h+64)
    const int quad = warp % 4;
    const int r = quad * 32 + lane;                       // key row within the block (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int kv_row = j * kBlockN + r;
    const BwdScales bs = bwd_scales(p);
    // Dropout: keep bits of this key row for step n's 64 query columns (transposed mask).
    // They are loaded one step ahead: a step outlasts the latency of the (uncoalesced) load.
    auto load_keep = [&](int n) {
      if (!DROP || kv_row >= p.s_kv || n >= n_iter) return make_uint2(0u, 0u);
      return __ldg(reinterpret_cast<const uint2*>(
          p.drop_cols + ((static_cast<int64_t>(bi) * p.h_q + iter_head(n)) * p.s_kv + kv_row) * p.drop_q_words +
          (iter_qblk(n) * kBlockM + 64 * h) / 32));
    };
    uint2 keep_next = load_keep(0);
    if (BIAS && n_iter > 0) prefetch_bias_t(p, bi, iter_head(0), kv_row, iter_qblk(0) * kBlockM + 64 * h);
    bool ok = true;
    for (int n = 0; n < n_iter; ++n) {
      const int b = n & 1;
      const uint32_t par = (n >> 1) & 1;
      const uint32_t X = tmem + lane_off + C::R_COL + b * 128;
      const uint32_t Y = tmem + lane_off + C::R_COL + (b ^ 1) * 128;
      const int q0 = iter_qblk(n) * kBlockM + 64 * h;     // first query column of this half
      const uint2 keep = keep_next;
      if constexpr (DROP) keep_next = load_keep(n + 1);
      // Additive bias of this key row for the 64 query columns (transposed copy); the next
      // step's row is sent to L2 first.
      uint4 bz[BIAS ? 8 : 1];
      if constexpr (BIAS) {
        if (n + 1 < n_iter)
          prefetch_bias_t(p, bi, iter_head(n + 1), kv_row, iter_qblk(n + 1) * kBlockM + 64 * h);
        load_bias_t(p, bi, iter_head(n), kv_row, q0, bz);
      }
      // Bias gradient: this key row's 64 query columns of the transposed accumulator.
      float* dbrow = DBIAS ? dbias_row(p, bi, iter_head(n), kv_row, q0) : nullptr;
      const float* nlse2 = sVec + (b * 2 + 0) * 128 + 64 * h;    // -LSE·log2 e per column
      const float* ndelta = sVec + (b * 2 + 1) * 128 + 64 * h;   // -Delta per column
      // Pᵀ = exp2(Sᵀ·scale·log2e − LSE·log2e), masked where key > query
      // This step's -LSE and -Delta vectors arrive with its Q tile.  Q's slot is refilled only
      // after dK of this step, which needs every thread's dS, so the refill cannot overtake
      // this wait, and both vectors stay in place until this step's dS is stored.
      if (!mbar_wait_warp(&bars.ring_full[n & 1], (n >> 1) & 1, wt)) { ok = false; break; }
      if (!mbar_wait_warp(&bars.s_full[b], par, wt)) { ok = false; break; }
      tc_fence_after();
      // With dropout, a bias or ALiBi (more work per score) the first 32 columns of Sᵀ are computed
      // while the second 32 are read from TMEM, and their Pᵀ is stored while the second 32
      // are computed; the plain instance reads all 64 at once (measured no faster split).
      constexpr bool SPLIT = DROP || BIAS || ALIBI;
      uint32_t sv[64];
      tmem_ld32(X + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      if constexpr (SPLIT) {
        tmem_ld_wait();
        reg_fence32(&sv[0]);
      }
      tmem_ld32(X + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      if constexpr (!SPLIT) tmem_ld_wait();
      // Query column c is visible to key row kv_row iff c >= lim (causal: kv <= q + off);
      // keys beyond len_kv see nothing.  Padded query columns already have P = 0.
      const bool need_mask = (p.causal && (q0 + L.off < j * kBlockN + kBlockN - 1)) ||
                             (j * kBlockN + kBlockN > L.len_kv);
      int lim = p.causal ? kv_row - q0 - L.off : -(1 << 30);
      if (kv_row >= L.len_kv) lim = 1 << 30;
      uint32_t pk[32], pm[DROP ? 32 : 1];
      const float2 sc2 = make_float2(bs.s_log2, bs.s_log2);
      // ALiBi: the key-row part of the bias (the column part is in the -LSE vector).
      const float kr = ALIBI ? alibi_slope_log2(p, iter_head(n)) *
                                   static_cast<float>(kv_row - iter_qblk(n) * kBlockM - L.off) : 0.f;
      const float2 kr2 = make_float2(kr, kr);
      float4 nl4;
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        if (SPLIT && c == 32) {
          // First half of Pᵀ to TMEM; the second half of Sᵀ has landed.
          if constexpr (DROP) {
            tmem_st16(X + 64 * h, *reinterpret_cast<uint32_t(*)[16]>(&pm[0]));
          } else {
            tmem_st16(X + 64 * h, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
          }
          tmem_ld_wait();
          reg_fence32(&sv[32]);
        }
        if ((c & 3) == 0) nl4 = *reinterpret_cast<const float4*>(nlse2 + c);
        float2 nl = (c & 3) ? make_float2(nl4.z, nl4.w) : make_float2(nl4.x, nl4.y);
        if constexpr (ALIBI) nl = add2(nl, kr2);
        if constexpr (BIAS) nl = fma2(bias_pair<DT>(bz, c), make_float2(kLog2e, kLog2e), nl);
        const float2 x = fma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, nl);
        float p0 = ex2(x.x);
        float p1 = ex2(x.y);
        if (need_mask) {
          if (c < lim) p0 = 0.f;
          if (c + 1 < lim) p1 = 0.f;
        }
        pk[c / 2] = pack2(p0, p1, DT);
        if constexpr (DROP) {
          // dV takes the kept P only; dS below takes every P.  A zero of either 16-bit type
          // is all zero bits, so the kept pair is the packed pair with dropped halves cleared.
          // The pair's keep bits sit at bits i and i + 16 of its word: shifted to bits 15 and
          // 31, a sign-replicating byte permute spreads them to the two 16-bit lanes.
          const uint32_t w = (c < 32) ? keep.x : keep.y;
          pm[c / 2] = pk[c / 2] & prmt(w << (15 - (c % 32) / 2), 0u, 0xBB99u);
        }
      }
      if constexpr (SPLIT) {
        if constexpr (DROP) {
          tmem_st16(X + 64 * h + 16, *reinterpret_cast<uint32_t(*)[16]>(&pm[16]));
        } else {
          tmem_st16(X + 64 * h + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
        }
      } else {
        tmem_st32(X + 64 * h, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_full[b]);
      // dSᵀ = Pᵀ ∘ (dPᵀ − Delta)
      if (!mbar_wait_warp(&bars.dp_full[b], par, wt)) { ok = false; break; }
      tc_fence_after();
      uint32_t ds[32];
      float2 dbhold = make_float2(0.f, 0.f);   // pairs of dS awaiting a 4-wide reduce-add
      if constexpr (DROP) {
        // dP = keep / (1 - p) * dO·Vᵀ.  Half the columns at a time (fewer live registers):
        // the second half is read before region Y is released.
        const float2 rk2 = make_float2(bs.dp, bs.dp);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tmem_ld32(Y + 64 * h + 32 * half, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
          tmem_ld_wait();
          if (half == 1) {
            tc_fence_before();
            mbar_arrive(&bars.dp_consumed[b]);   // region Y may now take the next step's Sᵀ
          }
          const uint32_t w = half == 0 ? keep.x : keep.y;
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 nd = *reinterpret_cast<const float2*>(ndelta + 32 * half + c);
            // The pair's keep bits (bits c/2 and c/2 + 16) as two all-ones / all-zeros masks.
            const uint32_t kx = w << (15 - c / 2);
            const float2 dpv = make_float2(__uint_as_float(sv[c] & prmt(kx, 0u, 0x9999u)),
                                           __uint_as_float(sv[c + 1] & prmt(kx, 0u, 0xBBBBu)));
            const float2 dd = mul2(unpack2(pk[16 * half + c / 2], DT), fma2(dpv, rk2, nd));
            ds[16 * half + c / 2] = pack2(dd.x, dd.y, DT);
            if constexpr (DBIAS) dbias_emit(dbrow, 32 * half + c, dd, dbhold);
          }
        }
      } else {
        tmem_ld32(Y + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(Y + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bars.dp_consumed[b]);   // region Y may now take the next step's Sᵀ
        const float2 dp2 = make_float2(bs.dp, bs.dp);
        float4 nd4;
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          if ((c & 3) == 0) nd4 = *reinterpret_cast<const float4*>(ndelta + c);
          const float2 nd = (c & 3) ? make_float2(nd4.z, nd4.w) : make_float2(nd4.x, nd4.y);
          const float2 dd = mul2(unpack2(pk[c / 2], DT),
                                 fma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), dp2, nd));
          ds[c / 2] = pack2(dd.x, dd.y, DT);
          if constexpr (DBIAS) dbias_emit(dbrow, c, dd, dbhold);
        }
      }
      // dS in shared memory, one 128-byte swizzled row per key row r, chunk h holding query
      // columns 64h..64h+63: read K-major (rows = keys) as the A operand of dK += dSᵀ·Q and
      // MN-major (rows = queries) as the A operand of dQ = dS·K.  The previous step's dQ and
      // dK MMAs must have finished reading it.
      if (n >= 1 && !mbar_wait_warp(&bars.dsbuf_free[b ^ 1], ((n - 1) >> 1) & 1, wt)) { ok = false; break; }
      uint8_t* rowp = sDS + h * 16384 + r * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint4 w = make_uint4(ds[u * 4 + 0], ds[u * 4 + 1], ds[u * 4 + 2], ds[u * 4 + 3]);
        *reinterpret_cast<uint4*>(rowp + ((u ^ (r & 7)) * 16)) = w;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars.ds_full[b]);
    }
    // ---- epilogue: dV (h = 0) or dK (h = 1) through shared memory and a TMA store ----
    ok = ok && mbar_wait_warp(&bars.acc_full, 0, wt);
    uint8_t* stage = sRing + h * C::TILE;
    if (ok && p.kv_split > 1) {
      // Split group: add this CTA's share into the fp32 accumulator (once per CTA).
      tc_fence_after();
      const uint32_t acc = tmem + lane_off + (h == 0 ? C::DV_COL : C::DK_COL);
      const float mul = (h == 0) ? bs.dv : bs.dk;
      float* dst = (h == 0 ? p.dv_acc : p.dk_acc) + kv_acc_offset(p, bi, hk, kv_row, D);
#pragma unroll 1
      for (int c = 0; c < D / 32 && n_iter > 0; ++c) {
        uint32_t v[32];
        tmem_ld32(acc + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 8; ++u)
          red_add_v4(dst + (c * 8 + u) * 128, __uint_as_float(v[u * 4]) * mul,
                     __uint_as_float(v[u * 4 + 1]) * mul, __uint_as_float(v[u * 4 + 2]) * mul,
                     __uint_as_float(v[u * 4 + 3]) * mul);
      }
    } else if (ok) {
      tc_fence_after();
      const uint32_t acc = tmem + lane_off + (h == 0 ? C::DV_COL : C::DK_COL);
      const float mul = (h == 0) ? bs.dv : bs.dk;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[64];
        if (n_iter > 0) {
          tmem_ld32(acc + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(acc + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = 0u;
        }
        uint8_t* rowp = stage + c * 16384 + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint4 w;
          w.x = pack2(__uint_as_float(v[u * 8 + 0]) * mul, __uint_as_float(v[u * 8 + 1]) * mul, DT);
          w.y = pack2(__uint_as_float(v[u * 8 + 2]) * mul, __uint_as_float(v[u * 8 + 3]) * mul, DT);
          w.z = pack2(__uint_as_float(v[u * 8 + 4]) * mul, __uint_as_float(v[u * 8 + 5]) * mul, DT);
          w.w = pack2(__uint_as_float(v[u * 8 + 6]) * mul, __uint_as_float(v[u * 8 + 7]) * mul, DT);
          *reinterpret_cast<uint4*>(rowp + ((u ^ (r & 7)) * 16)) = w;
        }
      }
      fence_proxy_async_smem();
    }
    // Every thread of the warpgroup arrives exactly once, so the bounded wait below can only
    // end by completion or timeout.
    mbar_arrive(&bars.epi_ready[h]);
    if (r == 0) {
      const bool all_ok = mbar_wait(&bars.epi_ready[h], 0, wt) && ok && !*abort_flag;
      if (all_ok && p.kv_split == 1) {
        const CUtensorMap* map = (h == 0) ? &p.tm_dv : &p.tm_dk;
        for (int c = 0; c < D / 64; ++c)
          tma_store_4d(map, stage + c * 16384, c * 64, j * kBlockN, hk, bi);
        tma_store_commit();
        tma_store_wait_read_all();
      }
    }
  } else {
    regs_inc<144>();
    // ===================== dQ drain: TMEM -> shared memory -> TMA reduce-add ===========
    // dQ of a step sits in TMEM (query row r = lane r, d columns).  All of it is read into
    // registers first, so the region goes back to the next step's dPᵀ MMA at once; it then
    // leaves as 32-column fp32 chunks (128 rows x 128 bytes, 128-byte swizzled) through two
    // staging buffers, so that two TMA reduce-adds into the fp32 accumulator are in flight.
    const int quad = warp % 4;
    const int r = quad * 32 + lane;                       // query row within the block
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    constexpr int NCH = D / 32;                           // 32-column chunks per step
    bool ok = true;
    int use[2] = {0, 0};                                  // times each buffer has been filled
    for (int n = 0; n < n_iter && ok; ++n) {
      const int b = n & 1;
      if (!mbar_wait_warp(&bars.dq_full[b], (n >> 1) & 1, wt)) { ok = false; break; }
      tc_fence_after();
      const int hq = iter_head(n);
      const int row0 = (bi * p.h_q + hq) * p.s_q_pad + iter_qblk(n) * kBlockM;
      const uint32_t X = tmem + lane_off + C::R_COL + b * 128;
      uint32_t v[D];
#pragma unroll
      for (int c = 0; c < NCH; ++c)
        tmem_ld32(X + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[c * 32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars.dq_free[b]);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int buf = c & 1;
        // Buffer `buf` is free once the reduce-add of its previous fill has read it.
        if (use[buf] > 0 && !mbar_wait_warp(&bars.stage_free[buf], (use[buf] - 1) & 1, wt)) {
          ok = false;
          break;
        }
        uint8_t* rowp = sDQ + buf * 16384 + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(rowp + ((u ^ (r & 7)) * 16)) =
              make_uint4(v[c * 32 + u * 4], v[c * 32 + u * 4 + 1], v[c * 32 + u * 4 + 2],
                         v[c * 32 + u * 4 + 3]);
        fence_proxy_async_smem();
        mbar_arrive(&bars.stage_full[buf]);
        if (r == 0) {
          if (!mbar_wait(&bars.stage_full[buf], use[buf] & 1, wt)) ok = false;
          if (ok) {
            tma_reduce_add_2d(&p.tm_dqacc, sDQ + buf * 16384, c * 32, row0);
            tma_store_commit();
            bulk_wait_read<1>();                          // the other buffer's reduce has read
          }
          if (use[buf ^ 1] > 0 || c > 0) mbar_arrive(&bars.stage_free[buf ^ 1]);
        }
        ++use[buf];
      }
    }
    if (r == 0) {
      bulk_wait_read<0>();
      tma_store_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  // Every role is done.  If one gave up (the abort flag, visible to all after the barrier),
  // copies the producer issued may still be in flight: let them land before the CTA's shared
  // memory is released.  (Each ring slot holds at most one copy in flight.)
  if (producer) griddep_wait();   // returns at once unless the producer gave up before its wait
  if (producer && *abort_flag) {
    mbar_wait_drain(&bars.kv_full, 0);
    for (int m = (nq > 2 ? nq - 2 : 0); m < nq; ++m) mbar_wait_drain(&bars.ring_full[m & 1], (m >> 1) & 1);
    for (int m = (nd > C::NDO ? nd - C::NDO : 0); m < nd; ++m)
      mbar_wait_drain(&bars.ring_full[2 + m % C::NDO], (m / C::NDO) & 1);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// d = 256
// ---------------------------------------------------------------------------
// dK and dV of a 128-row KV block at d = 256 would fill all 512 TMEM columns, and K and V
// alone take 128 KB of shared memory.  So a CTA owns one half of d of dK and dV, walks
// 64-row query blocks, and computes its half of dQ transposed (dQᵀ = Kᵀ·dSᵀ: rows = its 128
// d indices, so M stays 128) into a transposed fp32 accumulator [b·h_q][d][s_q_pad].  Both
// halves compute the full-d reductions Sᵀ = K·Qᵀ and dPᵀ = V·dOᵀ.
//
// The roles are those of the d = 128 kernel, linked by mbarriers: one thread loads, one
// issues the MMAs, two warpgroups compute Pᵀ and dSᵀ (32 query columns each) and one
// warpgroup drains dQᵀ.  Per step the MMAs run Sᵀ, dPᵀ, dV += Pᵀ·dO, then the next step's
// Sᵀ while dS is computed, then dK += dSᵀ·Q and dQᵀ.  The own d-half of Q is double-buffered
// (the next step's lands while this step's dK still reads it); the far half of Q and both
// halves of dO are refilled as soon as the MMAs that read them are done.  Half of dQᵀ (32
// fp32 columns) leaves through the dS buffer as one TMA reduce-add, which then takes the
// next step's dS; the other half goes from registers as vector reductions at the same time
// (the dS buffer holds one chunk, and TMA reduce-adds of one SM drain at a bounded rate).
struct D256 {
  static constexpr int BQ = 64;                  // query rows per step
  static constexpr int OFF_K = 0;                // 128 x 256: four 16 KB chunks of 64 columns
  static constexpr int OFF_V = 65536;
  static constexpr int OFF_QF = 131072;          // the other d-half of Q: two 8 KB chunks
  static constexpr int OFF_QN = 147456;          // own d-half of Q: two buffers of 16 KB
  static constexpr int OFF_DO = 180224;          // dO, 64 x 256: four 8 KB chunks
  static constexpr int OFF_DS = 212992;          // dS (128 key rows x 64 queries), then dQᵀ
  static constexpr int OFF_VEC = 229376;         // [2][-LSE·log2e, -Delta][64] fp32
  static constexpr int OFF_BAR = OFF_VEC + 1024;
  static constexpr int SMEM_BYTES = OFF_BAR + 256;
  static constexpr int THREADS = 512;
  // Sᵀ/Pᵀ alternates between two regions by step parity, so the next step's Sᵀ never
  // overwrites the Pᵀ that this step's dV MMAs read.
  static constexpr int COL_S0 = 0, COL_DP = 64, COL_DQ = 128, COL_S1 = 192, COL_DV = 256, COL_DK = 384;
  static constexpr int col_s(int n) { return (n & 1) ? COL_S1 : COL_S0; }
};
static_assert(D256::SMEM_BYTES <= 232448, "shared memory budget");

struct alignas(8) D256Barriers {
  uint64_t kv_full, qf_full, qf_empty, qn_full[2], qn_empty[2], df_full, df_empty, dn_full, dn_empty;
  uint64_t s_full, p_full, dp_full, dp_consumed, ds_full, dq_full, ds_free, stage_full;
  uint64_t acc_full, drain, epi_ready[2];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(D256Barriers) <= 256, "barrier block");

template <int DT, int FEAT>
__global__ void __launch_bounds__(512, 1) bwd_d256_kernel(const __grid_constant__ BwdParams p) {
  using C = D256;
  constexpr bool ALIBI = (FEAT & kFeatAlibi) != 0;
  constexpr bool DROP = (FEAT & kFeatDropout) != 0;
  constexpr bool BIAS = (FEAT & kFeatBias) != 0;
  constexpr bool DBIAS = (FEAT & kFeatDBias) != 0;
  extern __shared__ __align__(1024) uint8_t smem[];
  // Programmatic dependent launch, as in the d <= 128 kernel: the dQ conversion may launch now,
  // and the producer waits for the pre-pass before it loads the first vectors (every other
  // use of the pre-pass's results follows from that load) and again at its exit.
  griddep_launch_dependents();
  if (smem_u32(smem) & 1023u) {
    griddep_wait();
    if (threadIdx.x == 0) atomicOr(&g_device_error, kErrSmemAlign);
    return;
  }
  D256Barriers& bars = *reinterpret_cast<D256Barriers*>(smem + C::OFF_BAR);
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQF = smem + C::OFF_QF;
  uint8_t* sQN = smem + C::OFF_QN;
  uint8_t* sdO = smem + C::OFF_DO;
  uint8_t* sDS = smem + C::OFF_DS;
  float* sVec = reinterpret_cast<float*>(smem + C::OFF_VEC);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // Launch order: the two d-halves of a KV block side by side; units (batch, KV head, share)
  // in groups whose Q and dO together take about 32 MB, so that resident CTAs share them in
  // L2; within a group the heaviest KV blocks of all its units first (for causal, the first
  // blocks), then the next block index.  Units of 8 MB or more go one at a time.
  const int dh = blockIdx.x & 1;                 // own d-half: chunks 2dh, 2dh + 1
  const int fh = 1 - dh;                         // the other half
  const int rest = blockIdx.x >> 1;
  const int units = p.b * p.h_kv * p.kv_split;
  const int n_kvb = (p.s_kv + kBlockN - 1) / kBlockN;
  const long long unit_bytes = 4ll * p.heads_per_split * p.s_q_pad * 256;
  int G = static_cast<int>((32ll << 20) / (unit_bytes > 0 ? unit_bytes : 1));
  G = (unit_bytes >= (8ll << 20) || G < 1) ? 1 : (G > units ? units : G);
  const int grp = rest / (G * n_kvb);
  const int gsz = min(G, units - grp * G);
  const int grem = rest - grp * G * n_kvb;
  const int j = grem / gsz;                      // KV block
  const int unit = grp * G + grem % gsz;
  const int split = unit % p.kv_split;
  const int bhk = unit / p.kv_split;
  const int bi = bhk / p.h_kv;
  const int hk = bhk % p.h_kv;
  const Lens L = batch_lens(p, bi);
  const int n_qb = (L.len_q + C::BQ - 1) / C::BQ;
  const int q_first = first_q_block(p, L, j, C::BQ);
  const bool kv_live = j * kBlockN < L.len_kv;
  const int per_head = (kv_live && q_first < n_qb) ? n_qb - q_first : 0;
  const int head0 = hk * p.group + split * p.heads_per_split;
  const int n_heads = max(0, min(p.heads_per_split, (hk + 1) * p.group - head0));
  const int n_iter = per_head * n_heads;
  if (n_iter == 0) {   // no query sees this key block: zero dK/dV rows of this half of d
    griddep_wait();
    if (p.kv_split == 1) zero_kv_block(p, bi, hk, j, dh * 128, 128);
    return;
  }
  auto iter_head = [&](int n) { return head0 + n / per_head; };
  auto iter_q0 = [&](int n) { return (q_first + n % per_head) * C::BQ; };

  if (threadIdx.x == 0) {
    mbar_init(&bars.kv_full, 1);
    mbar_init(&bars.qf_full, 1);
    mbar_init(&bars.qf_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.qn_full[b], 1);
      mbar_init(&bars.qn_empty[b], 1);
      mbar_init(&bars.epi_ready[b], 128);
    }
    mbar_init(&bars.df_full, 1);
    mbar_init(&bars.df_empty, 1);
    mbar_init(&bars.dn_full, 1);
    mbar_init(&bars.dn_empty, 1);
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.p_full, 256);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.dp_consumed, 256);
    mbar_init(&bars.ds_full, 256);
    mbar_init(&bars.dq_full, 1);
    mbar_init(&bars.ds_free, 1);
    mbar_init(&bars.stage_full, 128);
    mbar_init(&bars.acc_full, 1);
    mbar_init(&bars.drain, 1);
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort_flag = &bars.abort;
  const Waiter wt{abort_flag, p.wait_limit};

  // Loads the producer has issued on each barrier (for the drain should a role give up).
  bool producer = false;
  int n_qf = 0, n_qn = 0, n_df = 0, n_dn = 0;

  if (warp == 0) {
    // ================================ TMA producer ====================================
    if (lane == 0) {
      producer = true;
      mbar_arrive_expect_tx(&bars.kv_full, 2 * 65536);
      for (int c = 0; c < 4; ++c) {
        tma_load_4d(sK + c * 16384, &p.tm_k, &bars.kv_full, c * 64, j * kBlockN, hk, bi);
        tma_load_4d(sV + c * 16384, &p.tm_v, &bars.kv_full, c * 64, j * kBlockN, hk, bi);
      }
      // In the order the MMAs free the buffers: Q far (after Sᵀ of the previous step), Q own
      // half (after dK two steps back), dO far (after dPᵀ), dO own half (after dV).
      for (int n = 0; n < n_iter; ++n) {
        const int hq = iter_head(n), q0 = iter_q0(n);
        if (n > 0 && !mbar_wait(&bars.qf_empty, (n - 1) & 1, wt)) break;
        mbar_arrive_expect_tx(&bars.qf_full, 16384);
        for (int c = 2 * fh; c < 2 * fh + 2; ++c)
          tma_load_4d(sQF + (c - 2 * fh) * 8192, &p.tm_q, &bars.qf_full, c * 64, q0, hq, bi);
        ++n_qf;
        const int b = n & 1;
        if (n > 1 && !mbar_wait(&bars.qn_empty[b], ((n - 2) >> 1) & 1, wt)) break;
        mbar_arrive_expect_tx(&bars.qn_full[b], 16384 + 512);
        for (int c = 2 * dh; c < 2 * dh + 2; ++c)
          tma_load_4d(sQN + b * 16384 + (c - 2 * dh) * 8192, &p.tm_q, &bars.qn_full[b], c * 64, q0, hq, bi);
        const int64_t vrow = (static_cast<int64_t>(bi) * p.h_q + hq) * p.s_q_pad + q0;
        if (n == 0) griddep_wait();   // K/V and the first Q tiles are already on their way
        bulk_load(sVec + b * 128, p.lse2 + vrow, 256, &bars.qn_full[b]);
        bulk_load(sVec + b * 128 + 64, p.delta + vrow, 256, &bars.qn_full[b]);
        ++n_qn;
        if (n > 0 && !mbar_wait(&bars.df_empty, (n - 1) & 1, wt)) break;
        mbar_arrive_expect_tx(&bars.df_full, 16384);
        for (int c = 2 * fh; c < 2 * fh + 2; ++c)
          tma_load_4d(sdO + c * 8192, &p.tm_do, &bars.df_full, c * 64, q0, hq, bi);
        ++n_df;
        if (n > 0 && !mbar_wait(&bars.dn_empty, (n - 1) & 1, wt)) break;
        mbar_arrive_expect_tx(&bars.dn_full, 16384);
        for (int c = 2 * dh; c < 2 * dh + 2; ++c)
          tma_load_4d(sdO + c * 8192, &p.tm_do, &bars.dn_full, c * 64, q0, hq, bi);
        ++n_dn;
      }
    }
  } else if (warp == 1) {
    // ================================ MMA issuer ======================================
    if (lane == 0) {
      const uint32_t fmt = (DT == kBF16) ? 1u : 0u;
      const uint32_t idesc_s = make_idesc(fmt, 128, C::BQ, false, false);    // Sᵀ, dPᵀ
      const uint32_t idesc_acc = make_idesc(fmt, 128, 128, false, true);     // dV, dK
      const uint32_t idesc_dq = make_idesc(fmt, 128, C::BQ, true, true);     // dQᵀ
      const uint32_t kA = smem_u32(sK), vA = smem_u32(sV), qF = smem_u32(sQF), qN = smem_u32(sQN);
      const uint32_t gA = smem_u32(sdO), dsA = smem_u32(sDS);
      bool ok = mbar_wait(&bars.kv_full, 0, wt);
      // Sᵀ = K·Qᵀ of step m over all of d (Q's own half in buffer m % 2, the other half in QF).
      auto issue_s = [&](int m) -> bool {
        if (!mbar_wait(&bars.qf_full, m & 1, wt)) return false;
        if (!mbar_wait(&bars.qn_full[m & 1], (m >> 1) & 1, wt)) return false;
        tc_fence_after();
        const uint32_t qn = qN + (m & 1) * 16384;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int c = k / 4;
          const uint32_t b = ((c >> 1) == dh ? qn + (c - 2 * dh) * 8192 : qF + (c - 2 * fh) * 8192) + (k % 4) * 32;
          mma_ss(tmem + C::col_s(m), make_sdesc_sw128(kA + c * 16384 + (k % 4) * 32, 16, 1024),
                 make_sdesc_sw128(b, 16, 1024), idesc_s, k > 0, false);
        }
        tc_commit(&bars.s_full);
        tc_commit(&bars.qf_empty);
        return true;
      };
      if (ok && n_iter > 0) ok = issue_s(0);
      for (int n = 0; n < n_iter && ok; ++n) {
        // ---- dPᵀ = V·dOᵀ over all of d, once the compute warps have read the last one ----
        if (!mbar_wait(&bars.df_full, n & 1, wt) || !mbar_wait(&bars.dn_full, n & 1, wt) ||
            (n > 0 && !mbar_wait(&bars.dp_consumed, (n - 1) & 1, wt))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint32_t off_a = (k / 4) * 16384 + (k % 4) * 32, off_b = (k / 4) * 8192 + (k % 4) * 32;
          mma_ss(tmem + C::COL_DP, make_sdesc_sw128(vA + off_a, 16, 1024),
                 make_sdesc_sw128(gA + off_b, 16, 1024), idesc_s, k > 0, false);
        }
        tc_commit(&bars.dp_full);
        tc_commit(&bars.df_empty);
        // ---- dV_h += Pᵀ·dO_h (Pᵀ in TMEM: queries 0..31 at S+0.., 32..63 at S+32..) ----
        if (!mbar_wait(&bars.p_full, n & 1, wt)) { ok = false; break; }
        tc_fence_after();
        const uint32_t gh = gA + dh * 2 * 8192;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t a_col = (k < 2) ? k * 8 : 32 + (k - 2) * 8;
          mma_ts(tmem + C::COL_DV, tmem + C::col_s(n) + a_col, make_sdesc_sw128(gh + k * 2048, 8192, 1024),
                 idesc_acc, (n > 0 || k > 0) ? 1u : 0u, false);
        }
        tc_commit(&bars.dn_empty);
        // ---- the next step's Sᵀ, into the other Sᵀ region ----
        if (n + 1 < n_iter && !issue_s(n + 1)) { ok = false; break; }
        // ---- dK_h += dSᵀ·Q_h, then dQᵀ_h = K_hᵀ·dSᵀ ----
        if (!mbar_wait(&bars.ds_full, n & 1, wt)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qn = qN + (n & 1) * 16384;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem + C::COL_DK, make_sdesc_sw128(dsA + k * 32, 16, 1024),
                 make_sdesc_sw128(qn + k * 2048, 8192, 1024), idesc_acc, (n > 0 || k > 0) ? 1u : 0u,
                 false);
        tc_commit(&bars.qn_empty[n & 1]);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss(tmem + C::COL_DQ, make_sdesc_sw128(kA + dh * 2 * 16384 + k * 2048, 16384, 1024),
                 make_sdesc_sw128(dsA + k * 2048, 8192, 1024), idesc_dq, k > 0, false);
        tc_commit(&bars.dq_full);
      }
      tc_commit(&bars.acc_full);
      tc_commit(&bars.drain);
      mbar_wait_drain(&bars.drain, 0);
    }
  } else if (warp >= 4 && warp < 12) {
    // ============================ Pᵀ / dSᵀ (two column halves) ========================
    const int h = (warp - 4) / 4;                         // query columns [32h, 32h+32)
    const int quad = warp % 4;
    const int r = quad * 32 + lane;                       // key row within the block (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int kv_row = j * kBlockN + r;
    const BwdScales bs = bwd_scales(p);
    bool ok = true;
    for (int n = 0; n < n_iter; ++n) {
      const int hq = iter_head(n);
      const int qb = iter_q0(n);                          // first query row of the block
      const int q0 = qb + 32 * h;                         // first query column of this half
      // Dropout: keep bits of this key row for the 32 query columns (transposed mask).
      uint32_t keep = 0u;
      if (DROP && kv_row < p.s_kv)
        keep = __ldg(p.drop_cols + ((static_cast<int64_t>(bi) * p.h_q + hq) * p.s_kv + kv_row) * p.drop_q_words +
                     q0 / 32);
      uint4 bz[BIAS ? 4 : 1];
      if constexpr (BIAS) load_bias_t(p, bi, hq, kv_row, q0, bz);
      const float* nlse2 = sVec + (n & 1) * 128 + 32 * h;
      const float* ndelta = sVec + (n & 1) * 128 + 64 + 32 * h;
      // The vectors arrive with Q's own half; its buffer is refilled only after dK of this
      // step, which needs every thread's dS, so the refill cannot overtake this wait.
      if (!mbar_wait_warp(&bars.qn_full[n & 1], (n >> 1) & 1, wt)) { ok = false; break; }
      if (!mbar_wait_warp(&bars.s_full, n & 1, wt)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(tmem + lane_off + C::col_s(n) + 32 * h, sv);
      tmem_ld_wait();
      const bool need_mask = (p.causal && (qb + L.off < j * kBlockN + kBlockN - 1)) ||
                             (j * kBlockN + kBlockN > L.len_kv);
      int lim = p.causal ? kv_row - q0 - L.off : -(1 << 30);   // column c visible iff c >= lim
      if (kv_row >= L.len_kv) lim = 1 << 30;
      const float2 sc2 = make_float2(bs.s_log2, bs.s_log2);
      // ALiBi: the key-row part of the bias (the column part is in the -LSE vector, relative
      // to the 128-aligned block that holds this query block).
      const float kr = ALIBI ? alibi_slope_log2(p, hq) *
                                   static_cast<float>(kv_row - (qb / kBlockM) * kBlockM - L.off) : 0.f;
      const float2 kr2 = make_float2(kr, kr);
      float pf[32];                                      // every P (dS takes all of them)
      uint32_t pk[16];                                   // dV's operand: the kept P
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float2 nl = *reinterpret_cast<const float2*>(nlse2 + c);
        if constexpr (ALIBI) nl = add2(nl, kr2);
        if constexpr (BIAS) nl = fma2(bias_pair<DT>(bz, c), make_float2(kLog2e, kLog2e), nl);
        const float2 x = fma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, nl);
        float p0 = ex2(x.x), p1 = ex2(x.y);
        if (need_mask) {
          if (c < lim) p0 = 0.f;
          if (c + 1 < lim) p1 = 0.f;
        }
        pf[c] = p0;
        pf[c + 1] = p1;
        if constexpr (DROP) {
          // The pair's keep bits sit at bits c/2 and c/2 + 16 of the word.
          pk[c / 2] = pack2((keep >> (c / 2)) & 1u ? p0 : 0.f, (keep >> (c / 2 + 16)) & 1u ? p1 : 0.f, DT);
        } else {
          pk[c / 2] = pack2(p0, p1, DT);
        }
      }
      tmem_st16(tmem + lane_off + C::col_s(n) + 32 * h, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_full);
      // ---- dSᵀ = Pᵀ ∘ (dPᵀ − Delta) ----
      if (!mbar_wait_warp(&bars.dp_full, n & 1, wt)) { ok = false; break; }
      tc_fence_after();
      tmem_ld32(tmem + lane_off + C::COL_DP + 32 * h, sv);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars.dp_consumed);
      const float2 rk2 = make_float2(bs.dp, bs.dp);
      // Both d-halves compute the same dS: the first half alone adds it to the bias gradient.
      float* dbrow = (DBIAS && dh == 0) ? dbias_row(p, bi, hq, kv_row, q0) : nullptr;
      float2 dbhold = make_float2(0.f, 0.f);
      uint32_t ds[16];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float2 dp = make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
        const float2 nd = *reinterpret_cast<const float2*>(ndelta + c);
        if constexpr (DROP) {
          // dS = P * (keep / (1 - p) * dO·Vᵀ - Delta) takes every P.
          dp.x = (keep >> (c / 2)) & 1u ? dp.x : 0.f;
          dp.y = (keep >> (c / 2 + 16)) & 1u ? dp.y : 0.f;
        }
        const float2 dd = mul2(make_float2(pf[c], pf[c + 1]), fma2(dp, rk2, nd));
        ds[c / 2] = pack2(dd.x, dd.y, DT);
        if constexpr (DBIAS) dbias_emit(dbrow, c, dd, dbhold);
      }
      // dS row r (128 bytes, 128-byte swizzled), this half in 16-byte units 4h..4h+3: read
      // K-major as dK's A operand and MN-major as dQᵀ's B operand.  The buffer is free once
      // the previous step's dQᵀ has left it.
      if (n > 0 && !mbar_wait_warp(&bars.ds_free, (n - 1) & 1, wt)) { ok = false; break; }
      uint8_t* rowp = sDS + r * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        *reinterpret_cast<uint4*>(rowp + (((4 * h + u) ^ (r & 7)) * 16)) =
            make_uint4(ds[u * 4], ds[u * 4 + 1], ds[u * 4 + 2], ds[u * 4 + 3]);
      fence_proxy_async_smem();
      mbar_arrive(&bars.ds_full);
    }
    // ---- epilogue: dV_h (h = 0) or dK_h (h = 1) ----
    ok = ok && mbar_wait_warp(&bars.acc_full, 0, wt);
    uint8_t* stage = sQF + h * 32768;                     // Q and dO buffers: all read by now
    tc_fence_after();
    const uint32_t acc = tmem + lane_off + (h == 0 ? C::COL_DV : C::COL_DK);
    const float mul = (h == 0) ? bs.dv : bs.dk;
    if (ok && p.kv_split > 1) {
      if (n_iter > 0) {
        float* dst = (h == 0 ? p.dv_acc : p.dk_acc) + kv_acc_offset(p, bi, hk, kv_row, 256);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(acc + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 8; ++u)
            red_add_v4(dst + (dh * 32 + c * 8 + u) * 128, __uint_as_float(v[u * 4]) * mul,
                       __uint_as_float(v[u * 4 + 1]) * mul, __uint_as_float(v[u * 4 + 2]) * mul,
                       __uint_as_float(v[u * 4 + 3]) * mul);
        }
      }
    } else if (ok) {
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t v[64];
        if (n_iter > 0) {
          tmem_ld32(acc + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(acc + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = 0u;
        }
        uint8_t* rowp = stage + c * 16384 + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint4 w;
          w.x = pack2(__uint_as_float(v[u * 8 + 0]) * mul, __uint_as_float(v[u * 8 + 1]) * mul, DT);
          w.y = pack2(__uint_as_float(v[u * 8 + 2]) * mul, __uint_as_float(v[u * 8 + 3]) * mul, DT);
          w.z = pack2(__uint_as_float(v[u * 8 + 4]) * mul, __uint_as_float(v[u * 8 + 5]) * mul, DT);
          w.w = pack2(__uint_as_float(v[u * 8 + 6]) * mul, __uint_as_float(v[u * 8 + 7]) * mul, DT);
          *reinterpret_cast<uint4*>(rowp + ((u ^ (r & 7)) * 16)) = w;
        }
      }
      fence_proxy_async_smem();
    }
    // Every thread of the warpgroup arrives exactly once.
    mbar_arrive(&bars.epi_ready[h]);
    if (r == 0) {
      const bool all_ok = mbar_wait(&bars.epi_ready[h], 0, wt) && ok && !*abort_flag;
      if (all_ok && p.kv_split == 1) {
        const CUtensorMap* map = (h == 0) ? &p.tm_dv : &p.tm_dk;
        for (int c = 0; c < 2; ++c)
          tma_store_4d(map, stage + c * 16384, (dh * 2 + c) * 64, j * kBlockN, hk, bi);
        tma_store_commit();
        tma_store_wait_read_all();
      }
    }
  } else if (warp >= 12) {
    // ===================== dQᵀ drain: TMEM -> fp32 accumulator =======================
    // Row r of this half of d, 64 query columns, read at once (TMEM is then free for the
    // next dQᵀ).
    const int quad = warp % 4;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = true;
    for (int n = 0; n < n_iter && ok; ++n) {
      const int hq = iter_head(n), q0 = iter_q0(n);
      const int drow = (bi * p.h_q + hq) * 256 + dh * 128;
      if (!mbar_wait_warp(&bars.dq_full, n & 1, wt)) { ok = false; break; }
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(tmem + lane_off + C::COL_DQ, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(tmem + lane_off + C::COL_DQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait();
      tc_fence_before();
      // Columns 0..31 leave through the dS buffer as one TMA reduce-add; columns 32..63 go
      // straight from registers as vector reductions, while the first chunk is read.
      {
        uint8_t* rowp = sDS + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(rowp + ((u ^ (r & 7)) * 16)) =
              make_uint4(v[u * 4], v[u * 4 + 1], v[u * 4 + 2], v[u * 4 + 3]);
        fence_proxy_async_smem();
        mbar_arrive(&bars.stage_full);                    // phase n
        float* dst = p.dq_acc + (static_cast<int64_t>(drow) + r) * p.s_q_pad + q0 + 32;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          red_add_v4(dst + u * 4, __uint_as_float(v[32 + u * 4]), __uint_as_float(v[32 + u * 4 + 1]),
                     __uint_as_float(v[32 + u * 4 + 2]), __uint_as_float(v[32 + u * 4 + 3]));
        bool issued = true;
        if (r == 0) {
          issued = mbar_wait(&bars.stage_full, n & 1, wt);
          if (issued) {
            tma_reduce_add_2d(&p.tm_dqacc, sDS, q0, drow);
            tma_store_commit();
            bulk_wait_read<0>();
            mbar_arrive(&bars.ds_free);
          }
        }
        ok = __all_sync(0xffffffffu, issued) != 0;
      }
    }
    if (r == 0) {
      bulk_wait_read<0>();
      tma_store_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  // Every role is done.  If one gave up, copies the producer issued may still be in flight:
  // let them land before the CTA's shared memory is released.
  if (producer) griddep_wait();   // returns at once unless the producer gave up before its wait
  if (producer && *abort_flag) {
    mbar_wait_drain(&bars.kv_full, 0);
    if (n_qf > 0) mbar_wait_drain(&bars.qf_full, (n_qf - 1) & 1);
    for (int m = (n_qn > 2 ? n_qn - 2 : 0); m < n_qn; ++m) mbar_wait_drain(&bars.qn_full[m & 1], (m >> 1) & 1);
    if (n_df > 0) mbar_wait_drain(&bars.df_full, (n_df - 1) & 1);
    if (n_dn > 0) mbar_wait_drain(&bars.dn_full, (n_dn - 1) & 1);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dQ = scale · (transposed accumulator)ᵀ for d = 256, through 32 x 32 shared-memory tiles.
template <typename T>
__global__ void __launch_bounds__(256) bwd_dqT_kernel(const BwdParams p) {
  griddep_wait();   // the main kernel's reduce-adds into the accumulator are complete
  __shared__ float tile[32][33];
  const int bh = blockIdx.z;
  const int bi = bh / p.h_q, hq = bh % p.h_q;
  const int i0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  for (int k = ty; k < 32; k += 8)
    tile[k][tx] = p.dq_acc[(static_cast<int64_t>(bh) * 256 + c0 + k) * p.s_q_pad + i0 + tx];
  __syncthreads();
  for (int k = ty; k < 32; k += 8) {
    const int i = i0 + k;
    if (i >= p.s_q) continue;
    const float v = tile[tx][k] * bwd_scales(p).dq;
    T* dst = reinterpret_cast<T*>(p.dq) + bi * p.dq_sb + hq * p.dq_sh + i * p.dq_ss + c0 + tx;
    if constexpr (std::is_same<T, __nv_bfloat16>::value) *dst = __float2bfloat16_rn(v);
    else *dst = __float2half_rn(v);
  }
}

// Launches `kern` so that it may start while the kernel ahead of it on the stream is still
// running (programmatic dependent launch); the kernel waits (griddep_wait) before it touches
// that kernel's results.
cudaError_t launch_dependent(void (*kern)(BwdParams), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             const BwdParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int DT>
cudaError_t launch_d256(const BwdParams& p, cudaStream_t st) {
  using T = typename std::conditional<DT == kBF16, __nv_bfloat16, __half>::type;
  constexpr int ROWS = 256 / (256 / 8);
  const int bh = p.b * p.h_q;
  dim3 gpre((p.s_q_pad + ROWS - 1) / ROWS, bh);
  bwd_pre_kernel<T, 256><<<gpre, 256, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.kv_split > 1) {
    bwd_zero_kv_kernel<<<1024, 256, 0, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int feat = (p.alibi ? kFeatAlibi : 0) | (p.drop_cols ? kFeatDropout : 0) | (p.bias_t ? kFeatBias : 0) |
                   (p.dbias_acc ? kFeatDBias : 0);
  auto kern = bwd_d256_kernel<DT, 0>;
  if (feat == kFeatAlibi) kern = bwd_d256_kernel<DT, kFeatAlibi>;
  if (feat == kFeatDropout) kern = bwd_d256_kernel<DT, kFeatDropout>;
  if (feat == (kFeatAlibi | kFeatDropout)) kern = bwd_d256_kernel<DT, kFeatAlibi | kFeatDropout>;
  if (feat == kFeatBias) kern = bwd_d256_kernel<DT, kFeatBias>;
  if (feat == (kFeatBias | kFeatDropout)) kern = bwd_d256_kernel<DT, kFeatBias | kFeatDropout>;
  if (feat == (kFeatBias | kFeatDBias)) kern = bwd_d256_kernel<DT, kFeatBias | kFeatDBias>;
  if (feat == (kFeatBias | kFeatDBias | kFeatDropout)) kern = bwd_d256_kernel<DT, kFeatBias | kFeatDBias | kFeatDropout>;
  e = set_smem_once(reinterpret_cast<const void*>(kern), D256::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const unsigned grid = 2u * p.b * p.h_kv * p.kv_split * ((p.s_kv + kBlockN - 1) / kBlockN);
  e = launch_dependent(kern, dim3(grid), dim3(D256::THREADS), D256::SMEM_BYTES, st, p);
  if (e != cudaSuccess) return e;
  dim3 gdq(p.s_q_pad / 32, 256 / 32, bh);
  e = launch_dependent(bwd_dqT_kernel<T>, gdq, dim3(256), 0, st, p);
  if (e != cudaSuccess || p.kv_split == 1) return e;
  dim3 gkv((p.s_kv + ROWS - 1) / ROWS, p.b * p.h_kv);
  bwd_kv_convert_kernel<T, 256><<<gkv, 256, 0, st>>>(p);
  return cudaGetLastError();
}

template <int D, int DT>
cudaError_t launch_t(const BwdParams& p, cudaStream_t st) {
  using T = typename std::conditional<DT == kBF16, __nv_bfloat16, __half>::type;
  using C = BwdCfg<D>;
  constexpr int ROWS = 256 / (D / 8);
  const int bh = p.b * p.h_q;
  dim3 gpre((p.s_q_pad + ROWS - 1) / ROWS, bh);
  bwd_pre_kernel<T, D><<<gpre, 256, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.kv_split > 1) {
    bwd_zero_kv_kernel<<<1024, 256, 0, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int feat = (p.alibi ? kFeatAlibi : 0) | (p.drop_cols ? kFeatDropout : 0) | (p.bias_t ? kFeatBias : 0) |
                   (p.dbias_acc ? kFeatDBias : 0);
  auto kern = bwd_main_kernel<D, DT, 0>;
  if (feat == kFeatAlibi) kern = bwd_main_kernel<D, DT, kFeatAlibi>;
  if (feat == kFeatDropout) kern = bwd_main_kernel<D, DT, kFeatDropout>;
  if (feat == (kFeatAlibi | kFeatDropout)) kern = bwd_main_kernel<D, DT, kFeatAlibi | kFeatDropout>;
  if (feat == kFeatBias) kern = bwd_main_kernel<D, DT, kFeatBias>;
  if (feat == (kFeatBias | kFeatDropout)) kern = bwd_main_kernel<D, DT, kFeatBias | kFeatDropout>;
  if (feat == (kFeatBias | kFeatDBias)) kern = bwd_main_kernel<D, DT, kFeatBias | kFeatDBias>;
  if (feat == (kFeatBias | kFeatDBias | kFeatDropout)) kern = bwd_main_kernel<D, DT, kFeatBias | kFeatDBias | kFeatDropout>;
  e = set_smem_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const unsigned gmain = static_cast<unsigned>(p.b) * p.h_kv * p.kv_split * ((p.s_kv + kBlockN - 1) / kBlockN);
  e = launch_dependent(kern, dim3(gmain), dim3(C::THREADS), C::SMEM_BYTES, st, p);
  if (e != cudaSuccess) return e;
  dim3 gdq((p.s_q + ROWS - 1) / ROWS, bh);
  e = launch_dependent(bwd_dq_kernel<T, D>, gdq, dim3(256), 0, st, p);
  if (e != cudaSuccess || p.kv_split == 1) return e;
  dim3 gkv((p.s_kv + ROWS - 1) / ROWS, p.b * p.h_kv);
  bwd_kv_convert_kernel<T, D><<<gkv, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

int bwd_kv_split(int b, int h_q, int h_kv, int s_kv) {
  // Aim for at least ~8 waves of CTAs on a 152-SM part; never split finer than one head.
  // (A/B on GB300: 8 waves beat 4 by 4-7% on GQA/MQA 70B shapes; 16 was no better.)
  constexpr long kTargetCtas = 1216;
  const int group = h_q / h_kv;
  const long ctas = static_cast<long>(b) * h_kv * ((s_kv + 127) / 128);
  if (group == 1 || ctas >= kTargetCtas) return 1;
  int want = static_cast<int>((kTargetCtas + ctas - 1) / ctas);
  if (want > group) want = group;
  const int per = (group + want - 1) / want;   // heads per CTA
  return (group + per - 1) / per;
}

size_t bwd_workspace_bytes(int b, int h_q, int h_kv, int s_q, int s_kv, int d) {
  const size_t pad = static_cast<size_t>((s_q + 127) / 128) * 128;
  const size_t kv_pad = static_cast<size_t>((s_kv + 127) / 128) * 128;
  auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t n = a(static_cast<size_t>(b) * h_q * pad * d * 4) + 2 * a(static_cast<size_t>(b) * h_q * pad * 4);
  if (bwd_kv_split(b, h_q, h_kv, s_kv) > 1) n += 2 * a(static_cast<size_t>(b) * h_kv * kv_pad * d * 4);
  return n;
}

cudaError_t launch_bwd(const BwdParams& p, int dtype, cudaStream_t st) {
  if (dtype == kBF16) {
    if (p.d == 64) return launch_t<64, kBF16>(p, st);
    if (p.d == 128) return launch_t<128, kBF16>(p, st);
    if (p.d == 256) return launch_d256<kBF16>(p, st);
  } else if (dtype == kF16) {
    if (p.d == 64) return launch_t<64, kF16>(p, st);
    if (p.d == 128) return launch_t<128, kF16>(p, st);
    if (p.d == 256) return launch_d256<kF16>(p, st);
  }
  return cudaErrorInvalidValue;
}

namespace {

// Sixteen FP8 codes (one 16-byte load along d) -> sixteen F16 or BF16 values (32 bytes),
// exact: every E4M3 and E5M2 value is representable in both.
template <typename T>
__global__ void __launch_bounds__(256) fp8_widen_kernel(const uint8_t* src, int64_t sb, int64_t sh, int64_t ss,
                                                        int b, int h, int s, int d, int e5m2, T* dst) {
  const int per_row = d / 16;
  const int64_t n = static_cast<int64_t>(b) * h * s * per_row;
  const __nv_fp8_interpretation_t fmt = e5m2 ? __NV_E5M2 : __NV_E4M3;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int part = static_cast<int>(t % per_row);
    int64_t r = t / per_row;
    const int si = static_cast<int>(r % s);
    r /= s;
    const int hi = static_cast<int>(r % h);
    const int bi = static_cast<int>(r / h);
    const uint4 v = *reinterpret_cast<const uint4*>(src + bi * sb + hi * sh + si * ss + part * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>((w[i / 2] >> (16 * (i % 2))) & 0xFFFFu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, fmt);
      if constexpr (std::is_same<T, __half>::value) {
        o[i] = static_cast<uint32_t>(hr.x) | (static_cast<uint32_t>(hr.y) << 16);
      } else {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        const __nv_bfloat162 bb = __floats2bfloat162_rn(f.x, f.y);
        o[i] = *reinterpret_cast<const uint32_t*>(&bb);
      }
    }
    uint4* out = reinterpret_cast<uint4*>(dst + ((static_cast<int64_t>(bi) * h + hi) * s + si) * d + part * 16);
    out[0] = make_uint4(o[0], o[1], o[2], o[3]);
    out[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace

namespace {

// [nb][nh][s_q][s_kv] (strided, 16-bit) -> the tiled transposed copy (see bias_tile_elems):
// one 128 x 128 tile per CTA through shared memory, 16-byte loads and stores; query rows
// beyond s_q and keys beyond s_kv get zeros.  With skip_above, tiles whose keys all lie beyond
// every query's causal limit (key > query + diag_off) are not written: the backward pass
// never reads them.
__global__ void __launch_bounds__(256) bias_transpose_kernel(const uint16_t* src, int64_t sb, int64_t sh,
                                                             int64_t ss, int nh, int s_q, int s_kv, int s_q_pad,
                                                             int skip_above, int diag_off, uint16_t* dst) {
  __shared__ uint16_t tile[128][136];   // [query][key], rows padded against bank conflicts
  const int z = blockIdx.z;
  const int nbi = z / nh, nhi = z % nh;
  const int i0 = blockIdx.x * 128, j0 = blockIdx.y * 128;
  if (skip_above && j0 > i0 + 127 + diag_off) return;
  const uint16_t* s = src + nbi * sb + nhi * sh;
  for (int t = threadIdx.x; t < 2048; t += 256) {   // 128 query rows x 16 chunks of 8 keys
    const int r = t / 16, c = t % 16;
    const int i = i0 + r, j = j0 + 8 * c;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (i < s_q) {
      const uint16_t* row = s + static_cast<int64_t>(i) * ss + j;
      if (j + 8 <= s_kv) {
        v = __ldg(reinterpret_cast<const uint4*>(row));
      } else {
        uint32_t h[4] = {0u, 0u, 0u, 0u};
        for (int u = 0; u < 8 && j + u < s_kv; ++u) h[u / 2] |= static_cast<uint32_t>(row[u]) << (16 * (u % 2));
        v = make_uint4(h[0], h[1], h[2], h[3]);
      }
    }
    *reinterpret_cast<uint4*>(&tile[r][8 * c]) = v;
  }
  __syncthreads();
  const int n_qb = s_q_pad / 128;
  uint4* d = reinterpret_cast<uint4*>(dst + ((static_cast<int64_t>(z) * gridDim.y + blockIdx.y) * n_qb + blockIdx.x) * 16384);
  for (int o = threadIdx.x; o < 2048; o += 256) {   // 16-byte unit ((hq2 * 4 + quad) * 8 + e) * 32 + lane
    const int lane = o % 32, e = (o / 32) % 8, quad = (o / 256) % 4, hq2 = o / 1024;
    const int key = quad * 32 + lane, q = hq2 * 64 + e * 8;
    uint32_t h[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      h[u] = static_cast<uint32_t>(tile[q + 2 * u][key]) | (static_cast<uint32_t>(tile[q + 2 * u + 1][key]) << 16);
    d[o] = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

}  // namespace

cudaError_t launch_bias_transpose(const void* src, int64_t sb, int64_t sh, int64_t ss, int nb, int nh,
                                  int s_q, int s_kv, int s_q_pad, int skip_above, int diag_off, void* dst,
                                  cudaStream_t st) {
  dim3 grid(s_q_pad / 128, (s_kv + 127) / 128, nb * nh);
  bias_transpose_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(src), sb, sh, ss, nh, s_q, s_kv,
                                              s_q_pad, skip_above, diag_off, static_cast<uint16_t*>(dst));
  return cudaGetLastError();
}

namespace {

// Tiled fp32 accumulator (see bias_tile_elems) -> dbias [nb][nh][s_q][s_kv] (16-bit, caller
// strides): one CTA per 64 queries (one half, hq2) of a 128 x 128 tile, through shared memory.
template <typename T>
__global__ void __launch_bounds__(256) dbias_convert_kernel(const float* acc, int nh, int s_q, int s_kv,
                                                            int s_q_pad, T* dst, int64_t sb, int64_t sh,
                                                            int64_t ss) {
  __shared__ float tile[64][129];   // [query][key]
  const int z = blockIdx.z;
  const int nbi = z / nh, nhi = z % nh;
  const int qb = blockIdx.x / 2, hq2 = blockIdx.x % 2, kb = blockIdx.y;
  const int i0 = qb * 128 + hq2 * 64, j0 = kb * 128;
  if (i0 >= s_q) return;
  const int n_qb = s_q_pad / 128;
  const float4* a = reinterpret_cast<const float4*>(acc + ((static_cast<int64_t>(z) * gridDim.y + kb) * n_qb + qb) * 16384) +
                    hq2 * 2048;
  for (int o = threadIdx.x; o < 2048; o += 256) {   // float4 unit (quad * 16 + e) * 32 + lane of this half
    const int lane = o % 32, e = (o / 32) % 16, quad = o / 512;
    const float4 v = a[o];
    const int key = quad * 32 + lane, q = e * 4;
    tile[q][key] = v.x;
    tile[q + 1][key] = v.y;
    tile[q + 2][key] = v.z;
    tile[q + 3][key] = v.w;
  }
  __syncthreads();
  T* d = dst + nbi * sb + nhi * sh;
  for (int t = threadIdx.x; t < 1024; t += 256) {   // 64 query rows x 16 chunks of 8 keys
    const int r = t / 16, c = t % 16;
    const int i = i0 + r, j = j0 + 8 * c;
    if (i >= s_q || j >= s_kv) continue;
    T* row = d + static_cast<int64_t>(i) * ss + j;
    if (j + 8 <= s_kv) {
      uint32_t h[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        T lo, hi;
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
          lo = __float2bfloat16_rn(tile[r][8 * c + 2 * u]);
          hi = __float2bfloat16_rn(tile[r][8 * c + 2 * u + 1]);
        } else {
          lo = __float2half_rn(tile[r][8 * c + 2 * u]);
          hi = __float2half_rn(tile[r][8 * c + 2 * u + 1]);
        }
        h[u] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&lo)) |
               (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&hi)) << 16);
      }
      *reinterpret_cast<uint4*>(row) = make_uint4(h[0], h[1], h[2], h[3]);
    } else {
      for (int u = 0; j + u < s_kv; ++u) {
        if constexpr (std::is_same<T, __nv_bfloat16>::value) row[u] = __float2bfloat16_rn(tile[r][8 * c + u]);
        else row[u] = __float2half_rn(tile[r][8 * c + u]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_dbias_convert(const float* acc, int nb, int nh, int s_q, int s_kv, int s_q_pad, void* dst,
                                 int64_t sb, int64_t sh, int64_t ss, int dtype, cudaStream_t st) {
  dim3 grid(s_q_pad / 128 * 2, (s_kv + 127) / 128, nb * nh);
  if (dtype == kBF16)
    dbias_convert_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(acc, nh, s_q, s_kv, s_q_pad,
                                                              static_cast<__nv_bfloat16*>(dst), sb, sh, ss);
  else
    dbias_convert_kernel<__half><<<grid, 256, 0, st>>>(acc, nh, s_q, s_kv, s_q_pad, static_cast<__half*>(dst),
                                                       sb, sh, ss);
  return cudaGetLastError();
}

cudaError_t launch_fp8_widen(const void* src, int64_t sb, int64_t sh, int64_t ss, int b, int h, int s,
                             int d, int src_e5m2, void* dst, int dst_dtype, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(b) * h * s * (d / 16);
  const int64_t want = (n + 255) / 256;
  const unsigned grid = static_cast<unsigned>(want < 152 * 16 ? want : 152 * 16);
  const uint8_t* p8 = static_cast<const uint8_t*>(src);
  if (dst_dtype == kBF16)
    fp8_widen_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p8, sb, sh, ss, b, h, s, d, src_e5m2,
                                                          static_cast<__nv_bfloat16*>(dst));
  else
    fp8_widen_kernel<__half><<<grid, 256, 0, st>>>(p8, sb, sh, ss, b, h, s, d, src_e5m2, static_cast<__half*>(dst));
  return cudaGetLastError();
}

uint32_t bwd_take_device_error() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, ptx::g_device_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(ptx::g_device_error, &z, sizeof(z));
  return v;
}

}  // namespace sdpa
