// sdpa_fwd.cu — fused SDPA forward pass for sm_103a.
//
// Computes, per (batch, query head) and per 128-row query tile, O = softmax(scale·QKᵀ +
// mask)·V and LSE = log Σ exp(scale·QKᵀ) without materialising the score matrix
// [attention codelab, §1 "How attention works" and §5/§6 (the fused kernel never writes
// the (B, N, T, S) weights); cuDNN 9 blog, "SDPA as a cuDNN graph", Fig. 4: BMM1 → scale →
// causal mask → softmax → BMM2 fused into one engine].
//
// One CTA owns NQT query tiles (NQT = 2 for 16-bit inputs with d <= 128, else 1) of one
// (batch, head) and walks the key/value blocks it can see:
//   warp 0       TMA producer: Q tiles once, then K/V blocks through an NS-slot ring.
//   warp 1       MMA issuer (one thread): S = Q·Kᵀ into TMEM, O += P·V with P read from
//                TMEM, completion signalled with tcgen05.commit.
//   warps 4..    one softmax warpgroup per Q tile; thread r owns query row r (TMEM lane r):
//                online softmax in the exp2 domain with the scale folded in, P written back
//                to TMEM over its own scores, O rescaled in TMEM only when the running max
//                grows by more than a threshold, and the epilogue (O / l via a TMA store,
//                LSE).
// Causal: key blocks wholly above a tile's diagonal are never loaded; only blocks that cross
// the diagonal (or the ragged end of the keys) are masked element-wise [codelab §7: key j
// is visible to query i iff j <= i].
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "ptx.cuh"
#include "sdpa_internal.h"

namespace sdpa {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Two 16-bit values (F16 or BF16) of a 32-bit word as fp32.
__device__ __forceinline__ float2 unpack16x2(uint32_t w, int dt) {
  if (dt == kBF16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

template <int D, int DT, bool ONE = false, bool PERSIST = false, bool TMA_BIAS = false>
struct FwdCfg {
  static constexpr int ES = (DT == kE4M3) ? 1 : 2;               // input element bytes
  static constexpr int NQT = (!ONE && D <= 128) ? 2 : 1;         // Q tiles per work unit
  static constexpr int CHUNK_ELEMS = 128 / ES;                    // elements per 128-byte row chunk
  static constexpr int NCHUNK = D * ES / 128;                     // 128-byte chunks along d
  static constexpr int TILE_BYTES = kBlockM * D * ES;             // one Q or K or V tile
  static constexpr int Q_BYTES = NQT * TILE_BYTES;
  static constexpr int OUT_TILE = kBlockM * D * 2;                // one 16-bit O tile
  // Where the epilogue stages O for its TMA store.  A CTA that walks several work units
  // (persistent) loads the next unit's Q and K/V while it stores this unit's O, so it stages
  // in a buffer of its own; a CTA with one unit stages two Q tiles in their own Q buffers
  // (unless those are smaller: E4M3 inputs) and one Q tile in the K/V ring.
  static constexpr bool OWN_STAGE = PERSIST || (NQT == 2 && TILE_BYTES < OUT_TILE);
  static constexpr int STAGE_BYTES = OWN_STAGE ? NQT * OUT_TILE : 0;
  // Additive bias (one Q tile, d <= 128): two stages of the 128 x 128 bias tile of a key
  // block, loaded by TMA as two 64-key halves (one per softmax warpgroup).
  static constexpr int BIAS_STAGE = kBlockM * kBlockN * 2;
  static constexpr int BIAS_BYTES = TMA_BIAS ? 2 * BIAS_STAGE : 0;
  // Shared memory: the per-SM limit (227 KB) less the static arrays (the barriers, and with
  // one Q tile the column halves' exchange arrays) and the 1 KB alignment slack.
  static constexpr int STATIC_BYTES = NQT == 2 ? 512 : 3584;
  static constexpr int RING_BUDGET =
      (PERSIST ? 232448 - STATIC_BYTES - 1024 : 196608) - Q_BYTES - STAGE_BYTES - BIAS_BYTES;
  static constexpr int NS = (RING_BUDGET / TILE_BYTES) > 8 ? 8 : (RING_BUDGET / TILE_BYTES);
  static constexpr int RING_BYTES = NS * TILE_BYTES;
  static constexpr int OUT_TILE_BYTES = kBlockM * D * 2;          // 16-bit output tile
  static constexpr int SMEM_BYTES = Q_BYTES + RING_BYTES + STAGE_BYTES + BIAS_BYTES + 1024 /*align slack*/;
  // Two softmax warpgroups: one per Q tile, or, with one Q tile, one per half of the 128
  // score columns of a key block.
  static constexpr int THREADS = 384;
  static constexpr int KSTEPS_S = D * ES / 32;                    // QKᵀ: 32 bytes of d per MMA
  static constexpr int PV_ROWS = 32 / ES;                         // PV: kv rows per MMA
  static constexpr int KSTEPS_PV = kBlockN / PV_ROWS;
  static constexpr int P_COLS = kBlockN * ES / 4;                 // TMEM columns holding P
  static constexpr int SCOLS = (NQT == 2) ? kBlockN : kBlockN / 2;  // score columns per thread
  static constexpr int PW = P_COLS * SCOLS / kBlockN;             // P words per thread
  static constexpr int O_COL0 = 256;                              // S slots at 0 and 128
  static constexpr float THRESH = (DT == kE4M3) ? 0.8f : 8.0f;    // lazy-rescale threshold
  static constexpr float P_OFFSET = (DT == kE4M3) ? 8.0f : 0.0f;  // P scaled by 2^8 for E4M3
  static_assert(NS >= 2, "K/V ring needs at least two slots");
  static_assert(!TMA_BIAS || (NQT == 1 && !PERSIST && D <= 128), "bias tiles: one Q tile, d <= 128");
  static_assert(SMEM_BYTES + STATIC_BYTES <= 232448, "shared memory budget");
  static_assert(O_COL0 + NQT * D <= 512, "TMEM budget");
  static_assert(OWN_STAGE || NQT == 2 || OUT_TILE_BYTES <= RING_BYTES, "epilogue staging");
};

struct alignas(8) FwdBarriers {
  uint64_t q_full[2];
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t o_empty[2];    // the epilogue has read O out of TMEM (the next unit may overwrite it)
  uint64_t q_empty;       // the last QKᵀ MMAs of a unit are done (its Q buffer may be refilled)
  uint64_t stage_free[2]; // the TMA store of the staged O has read shared memory
  uint64_t pv_done;
  uint64_t drain;
  uint64_t epi_ready[2];
  uint64_t mx_ready[2];   // column halves: row-max candidates exchanged (per block parity)
  uint64_t l_ready;       // column halves: row sums exchanged (once per unit)
  uint64_t bias_full[2];  // bias tile of a key block landed (by stage)
  uint64_t bias_empty[2]; // both softmax warpgroups have read it
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint32_t pack2(float a, float b, int dt) {
  if (dt == kBF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

// Number of key blocks the query rows [m0, m0 + rows) of a batch must visit (0 when none of
// them has a visible key).
__device__ __forceinline__ int kv_blocks_for(const FwdParams& p, const Lens& L, int m0, int rows) {
  if (m0 >= L.len_q) return 0;
  const int last_row = min(m0 + rows, L.len_q) - 1;
  int lim = L.len_kv - 1;                         // last visible key of any of these rows
  if (p.causal) lim = min(lim, last_row + L.off);
  return lim < 0 ? 0 : lim / kBlockN + 1;
}

// One work unit: NQT query tiles of one (batch, query head).
struct FwdUnit {
  int bi, hq, hk, m0, n_blocks;
  Lens L;
};

template <int D, int DT, int OUT_DT, int FEAT>
__global__ void __launch_bounds__(FwdCfg<D, DT>::THREADS, 1)
    sdpa_fwd_kernel(const __grid_constant__ FwdParams p) {
  constexpr bool PERSIST = (FEAT & kFeatPersist) != 0;
  constexpr bool BIAS = (FEAT & kFeatBias) != 0;
  // d <= 128: the bias reaches the softmax threads as TMA tiles in shared memory (coalesced
  // bulk copies; per-thread row loads of 16 bytes kept the L1 pipeline ~80% busy).  d = 256
  // has no room for them and loads its rows per thread.
  constexpr bool TMA_BIAS = BIAS && D <= 128;
  using C = FwdCfg<D, DT, (FEAT & kFeatOneTile) != 0, PERSIST, TMA_BIAS>;
  constexpr bool ALIBI = (FEAT & kFeatAlibi) != 0;
  constexpr bool DROP = (FEAT & kFeatDropout) != 0;
  constexpr int NQT = C::NQT;
  constexpr int NS = C::NS;
  constexpr bool FP8 = (DT == kE4M3);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::Q_BYTES;
  uint8_t* sStage = sRing + C::RING_BYTES;   // STAGE_BYTES of its own (OWN_STAGE only)
  uint8_t* sBias = sStage + C::STAGE_BYTES;  // BIAS_BYTES (TMA_BIAS only)
  __shared__ FwdBarriers bars;
  // Column halves (one Q tile): per-row exchange of the row-max candidate (by block parity)
  // and, at the end of a unit, of the row sums.
  __shared__ float xch[NQT == 1 ? 2 : 1][2][NQT == 1 ? kBlockM : 1];
  __shared__ float xl[2][NQT == 1 ? kBlockM : 1];
  static_assert(sizeof(FwdBarriers) + sizeof(xch) + sizeof(xl) <= C::STATIC_BYTES, "static shared memory");

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- work units ------------------------------------------------------------------------
  // Unit order: longest first — the heaviest query tile(s) (the latest, for causal) of every
  // (batch, head) pair, then the next heaviest, and so on.  When the heads' K and V together
  // exceed ~64 MB (they would stream from HBM once per tile), this runs over groups of query
  // heads whose K and V take ~32 MB instead, one group after another, so that a group's K/V
  // stays in L2 while all its tiles run.  CTA c takes units c, 2G - 1 - c, 2G + c, ... of that
  // order (G CTAs; back and forth, so that the longest and the shortest units pair up): with
  // one CTA per unit that is unit c alone; with fewer CTAs (persistent) each walks several
  // units and loads the next unit's tiles while it finishes the current one.
  const int n_bh = p.b * p.h_q;
  const long long kv_bytes = 2ll * p.s_kv * D * C::ES;             // K and V of one KV head
  int G = n_bh;                                                     // query heads per group
  if (kv_bytes * (n_bh / p.group) > (64ll << 20)) {
    G = static_cast<int>((32ll << 20) / kv_bytes) * p.group;
    G = G < p.group ? p.group : (G > n_bh ? n_bh : G);
  }
  const int n_units = n_bh * p.num_m_blocks;
  // Units of this CTA: k-th unit, or >= n_units when there are no more.  Without PERSIST the
  // CTA has exactly one (unit blockIdx.x), and every loop over units runs once.
  constexpr int kMaxUnits = PERSIST ? 0x7fffffff : 1;
  auto unit_at = [&](int k) -> int {
    const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    if constexpr (!PERSIST) return c;
    return k * g + ((k & 1) ? g - 1 - c : c);
  };
  auto decode = [&](int u) -> FwdUnit {
    FwdUnit w;
    const int grp = u / (G * p.num_m_blocks);
    const int gsz = min(G, n_bh - grp * G);
    const int rem = u - grp * G * p.num_m_blocks;
    const int bh = grp * G + rem % gsz;
    w.bi = bh / p.h_q;
    w.hq = bh % p.h_q;
    w.hk = w.hq / p.group;
    w.m0 = (p.num_m_blocks - 1 - rem / gsz) * kBlockM * NQT;
    w.L = batch_lens(p, w.bi);
    w.n_blocks = kv_blocks_for(p, w.L, w.m0, kBlockM * NQT);
    return w;
  };
  // The first unit, decoded once for every role (a CTA without PERSIST has no other).
  const FwdUnit first = decode(unit_at(0) < n_units ? unit_at(0) : 0);
  auto unit = [&](int k, int u) -> FwdUnit { return (!PERSIST || k == 0) ? first : decode(u); };
  // Key block visited at step j of a unit with n key blocks.  With ALiBi the bias of a row
  // only falls with distance from its diagonal, so the blocks go from the last one down: the
  // first block holds the row maximum (nearly) and the running max seldom has to rescale O.
  auto kv_block = [&](int j, int n) { return ALIBI ? n - 1 - j : j; };

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.q_full[t], 1);
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], NQT == 2 ? 128 : 256);
      mbar_init(&bars.o_full[t], 1);
      mbar_init(&bars.o_empty[t], NQT == 2 ? 128 : 256);
      mbar_init(&bars.stage_free[t], 1);
    }
    for (int s = 0; s < 8; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    mbar_init(&bars.q_empty, 1);
    mbar_init(&bars.pv_done, 1);
    mbar_init(&bars.drain, 1);
    mbar_init(&bars.epi_ready[0], NQT == 2 ? 128 : 256);
    mbar_init(&bars.epi_ready[1], 128);
    mbar_init(&bars.mx_ready[0], 256);
    mbar_init(&bars.mx_ready[1], 256);
    mbar_init(&bars.l_ready, 256);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.bias_full[b], 1);
      mbar_init(&bars.bias_empty[b], 256);
    }
    bars.abort = 0;
    fence_mbar_init();
    // The first unit's Q tiles and first K block go out before the CTA's set-up (TMEM
    // allocation, the block barrier): their latency from HBM overlaps it.  Thread 0 is the
    // producer and carries on from there.
    if (unit_at(0) < n_units && first.n_blocks > 0) {
      for (int t = 0; t < NQT; ++t) {
        mbar_arrive_expect_tx(&bars.q_full[t], C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_4d(sQ + t * C::TILE_BYTES + c * 16384, &p.tm_q, &bars.q_full[t], c * C::CHUNK_ELEMS,
                      first.m0 + t * kBlockM, first.hq, first.bi);
      }
      mbar_arrive_expect_tx(&bars.kv_full[0], C::TILE_BYTES);
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_4d(sRing + c * 16384, &p.tm_k, &bars.kv_full[0], c * C::CHUNK_ELEMS,
                    kv_block(0, first.n_blocks) * kBlockN, first.hk, first.bi);
    }
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

  // Copies the producer has issued (for the drain at the end, should a role give up).
  bool producer = false;
  int q_issued = 0, kv_issued = 0, bias_issued = 0;

  // Registers (384 threads, 168 each at launch): the producer / MMA warpgroup gives some to
  // the two softmax warpgroups, 88 + 2 x 200 <= 3 x 168; a bias row needs 8 more per softmax
  // thread (80 + 2 x 208).
  constexpr int kRegsProd = BIAS ? 80 : 88;
  constexpr int kRegsSoftmax = BIAS ? 208 : 200;
  if (warp < 4) {
  regs_dec<kRegsProd>();
  if (warp == 0) {
    // ================================ TMA producer ====================================
    if (lane == 0) {
      producer = true;
      tma_prefetch_desc(&p.tm_v);
      // The first unit's Q and first K block were issued before the set-up.
      bool early = unit_at(0) < n_units && first.n_blocks > 0;
      int it = early ? 1 : 0, qn = 0;
      q_issued = kv_issued = it;
      bool ok = true;
      for (int k = 0; ok && k < kMaxUnits; ++k) {
        const int u = unit_at(k);
        if (u >= n_units) break;
        const FwdUnit w = unit(k, u);
        const int nb = w.n_blocks;
        if (nb == 0) continue;
        if (k == 0 && early) {
          q_issued = ++qn;
        } else {
          // Q of this unit goes where the previous unit's Q was: wait until its last QKᵀ
          // MMAs have read it.
          if (PERSIST && qn > 0 && !mbar_wait(&bars.q_empty, (qn - 1) & 1, wt)) { ok = false; break; }
          for (int t = 0; t < NQT; ++t) {
            mbar_arrive_expect_tx(&bars.q_full[t], C::TILE_BYTES);
            for (int c = 0; c < C::NCHUNK; ++c)
              tma_load_4d(sQ + t * C::TILE_BYTES + c * 16384, &p.tm_q, &bars.q_full[t],
                          c * C::CHUNK_ELEMS, w.m0 + t * kBlockM, w.hq, w.bi);
          }
          q_issued = ++qn;
        }
        auto load = [&](const CUtensorMap* map, int j) {
          if (early) {          // K of the first block: issued before the set-up
            early = false;
            return true;
          }
          const int slot = it % NS;
          const uint32_t ph = (it / NS) & 1;
          if (!mbar_wait(&bars.kv_empty[slot], ph ^ 1, wt)) return false;
          mbar_arrive_expect_tx(&bars.kv_full[slot], C::TILE_BYTES);
          uint8_t* dst = sRing + slot * C::TILE_BYTES;
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_4d(dst + c * 16384, map, &bars.kv_full[slot], c * C::CHUNK_ELEMS,
                        kv_block(j, nb) * kBlockN, w.hk, w.bi);
          kv_issued = ++it;
          return true;
        };
        // The bias tile of key block j (rows of this unit's Q tile, 128 keys) into stage
        // bias_issued % 2, as two 64-key halves.
        auto load_bias = [&](int j) {
          const int b = bias_issued & 1;
          if (!mbar_wait(&bars.bias_empty[b], ((bias_issued >> 1) & 1) ^ 1, wt)) return false;
          mbar_arrive_expect_tx(&bars.bias_full[b], C::BIAS_STAGE);
          for (int c = 0; c < 2; ++c)
            tma_load_4d(sBias + b * C::BIAS_STAGE + c * (C::BIAS_STAGE / 2), &p.tm_bias, &bars.bias_full[b],
                        kv_block(j, nb) * kBlockN + 64 * c, w.m0, p.bias_sh != 0 ? w.hq : 0,
                        p.bias_sb != 0 ? w.bi : 0);
          ++bias_issued;
          // The tiles two and three key blocks ahead start towards L2 (HBM latency is long
          // against two 32 KB stages): j + 2 and j + 3 from the first block, then j + 3.
          for (int a = (j == 0 ? 2 : 3); a <= 3; ++a)
            if (j + a < nb)
              for (int c = 0; c < 2; ++c)
                tma_prefetch_4d(&p.tm_bias, kv_block(j + a, nb) * kBlockN + 64 * c, w.m0,
                                p.bias_sh != 0 ? w.hq : 0, p.bias_sb != 0 ? w.bi : 0);
          return true;
        };
        if (NQT == 2) {
          for (int j = 0; j < nb && ok; ++j) {
            ok = load(&p.tm_k, j);
            if (ok) ok = load(&p.tm_v, j);
          }
        } else {
          ok = load(&p.tm_k, 0);
          for (int j = 0; j < nb && ok; ++j) {
            if (j + 1 < nb) ok = load(&p.tm_k, j + 1);
            if (ok) ok = load(&p.tm_v, j);
            if (TMA_BIAS && ok) ok = load_bias(j);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ================================ MMA issuer ======================================
    if (elect_one_sync()) {
      const uint32_t fmt = (DT == kBF16) ? 1u : 0u;
      uint32_t idesc_s = make_idesc(fmt, kBlockM, kBlockN, false, false);
      if (p.negate_scores) idesc_s |= (1u << 13);
      const uint32_t idesc_pv = make_idesc(fmt, kBlockM, D, false, true);
      int it = 0;
      bool ok = true;
      auto wait_full = [&]() -> int {
        const int slot = it % NS;
        if (!mbar_wait(&bars.kv_full[slot], (it / NS) & 1, wt)) return -1;
        ++it;
        tc_fence_after();
        return slot;
      };
      auto issue_s = [&](int t_q, int s_slot, int kslot) {
        const uint32_t qa = smem_u32(sQ + t_q * C::TILE_BYTES);
        const uint32_t kb = smem_u32(sRing + kslot * C::TILE_BYTES);
#pragma unroll
        for (int k = 0; k < C::KSTEPS_S; ++k) {
          const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
          mma_ss(tmem + s_slot * 128, make_sdesc_sw128(qa + off, 16, 1024),
                 make_sdesc_sw128(kb + off, 16, 1024), idesc_s, k > 0, FP8);
        }
        tc_commit(&bars.s_full[s_slot]);
      };
      auto issue_pv = [&](int t_q, int s_slot, int vslot, bool first) {
        const uint32_t vb = smem_u32(sRing + vslot * C::TILE_BYTES);
        const uint32_t o_col = tmem + C::O_COL0 + t_q * D;
#pragma unroll
        for (int k = 0; k < C::KSTEPS_PV; ++k) {
          mma_ts(o_col, tmem + s_slot * 128 + k * 8,
                 make_sdesc_sw128(vb + k * C::PV_ROWS * 128, 16384, 1024), idesc_pv,
                 (!first || k > 0) ? 1u : 0u, FP8);
        }
      };
      // Before the first P·V of a unit overwrites O of tile t, the previous unit's epilogue
      // must have read it out of TMEM.
      auto o_free = [&](int t, int qn) {
        if (!PERSIST || qn == 0) return true;
        if (!mbar_wait(&bars.o_empty[t], (qn - 1) & 1, wt)) return false;
        tc_fence_after();
        return true;
      };
      int qn = 0, jb = 0;   // units with key blocks so far; key blocks so far
      for (int k = 0; ok && k < kMaxUnits; ++k) {
        const int u = unit_at(k);
        if (u >= n_units) break;
        const int nb = unit(k, u).n_blocks;
        if (nb == 0) continue;
        for (int t = 0; t < NQT && ok; ++t) ok = mbar_wait(&bars.q_full[t], qn & 1, wt);
        if (!ok) break;
        tc_fence_after();
        if (NQT == 2) {
          const int kslot = wait_full();
          if (kslot < 0) { ok = false; break; }
          issue_s(0, 0, kslot);
          issue_s(1, 1, kslot);
          tc_commit(&bars.kv_empty[kslot]);
          if (PERSIST && nb == 1) tc_commit(&bars.q_empty);
          for (int j = 0; j < nb && ok; ++j) {
            const int vslot = wait_full();
            if (vslot < 0) { ok = false; break; }
            const uint32_t ph = (jb + j) & 1;
            // tile 0
            if (!mbar_wait(&bars.p_full[0], ph, wt)) { ok = false; break; }
            tc_fence_after();
            if (j == 0 && !o_free(0, qn)) { ok = false; break; }
            issue_pv(0, 0, vslot, j == 0);
            if (j + 1 == nb) tc_commit(&bars.o_full[0]);
            int nk = -1;
            if (j + 1 < nb) {
              nk = wait_full();
              if (nk < 0) { ok = false; break; }
              issue_s(0, 0, nk);
            }
            // tile 1
            if (!mbar_wait(&bars.p_full[1], ph, wt)) { ok = false; break; }
            tc_fence_after();
            if (j == 0 && !o_free(1, qn)) { ok = false; break; }
            issue_pv(1, 1, vslot, j == 0);
            if (j + 1 == nb) tc_commit(&bars.o_full[1]);
            tc_commit(&bars.kv_empty[vslot]);
            if (nk >= 0) {
              issue_s(1, 1, nk);
              tc_commit(&bars.kv_empty[nk]);
              if (PERSIST && j + 2 == nb) tc_commit(&bars.q_empty);
            }
          }
        } else {
          const int k0 = wait_full();
          if (k0 < 0) { ok = false; break; }
          issue_s(0, jb & 1, k0);
          tc_commit(&bars.kv_empty[k0]);
          if (PERSIST && nb == 1) tc_commit(&bars.q_empty);
          for (int j = 0; j < nb && ok; ++j) {
            const int jg = jb + j;
            if (j + 1 < nb) {
              const int nk = wait_full();
              if (nk < 0) { ok = false; break; }
              issue_s(0, (jg + 1) & 1, nk);
              tc_commit(&bars.kv_empty[nk]);
              if (PERSIST && j + 2 == nb) tc_commit(&bars.q_empty);
            }
            const int vslot = wait_full();
            if (vslot < 0) { ok = false; break; }
            if (!mbar_wait(&bars.p_full[jg & 1], (jg >> 1) & 1, wt)) { ok = false; break; }
            tc_fence_after();
            if (j == 0 && !o_free(0, qn)) { ok = false; break; }
            issue_pv(0, jg & 1, vslot, j == 0);
            tc_commit(&bars.pv_done);
            if (j + 1 == nb) tc_commit(&bars.o_full[0]);
            tc_commit(&bars.kv_empty[vslot]);
          }
        }
        jb += nb;
        ++qn;
      }
      // Whatever happened, wait for the tensor core to finish before TMEM is released.
      tc_commit(&bars.drain);
      mbar_wait_drain(&bars.drain, 0);
    }
  }
  } else {
    regs_inc<kRegsSoftmax>();
    // ============================ softmax / epilogue ==================================
    constexpr int SC = C::SCOLS;
    const int t = (NQT == 2) ? (warp - 4) / 4 : 0;         // Q tile of this warpgroup
    const int hc = (NQT == 1) ? (warp - 4) / 4 : 0;        // column half (one Q tile)
    const int col0 = hc * SC;                                // first score column of this thread
    const int quad = warp % 4;                               // TMEM lane quadrant
    const int r = quad * 32 + lane;                          // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool storer = (r == 0 && hc == 0);                 // issues this tile's O store

    float c_scale = p.scale_log2;
    float v_scale = 1.f;
    if (FP8) {
      c_scale *= __ldg(p.descale_q) * __ldg(p.descale_k);
      v_scale = __ldg(p.descale_v);
    }
    if (DROP) v_scale *= p.drop_scale;
    const float u_scale_base = c_scale;
    bool ok = true;
    int jb = 0, qn = 0, ue = 0;   // key blocks, units with key blocks, epilogues so far

    for (int k = 0; ok && k < kMaxUnits; ++k) {
      const int u = unit_at(k);
      if (u >= n_units) break;
      const FwdUnit w = unit(k, u);
      const int bi = w.bi, hq = w.hq, m0 = w.m0, n_blocks = w.n_blocks;
      const Lens& L = w.L;
      const int q_row = m0 + t * kBlockM + r;
      const int tile_row0 = m0 + t * kBlockM;
      // Additive bias: this row of the bias tensor (16-bit, 16-byte aligned rows).
      const uint16_t* bias_row = nullptr;
      if (BIAS && q_row < p.s_q)
        bias_row = static_cast<const uint16_t*>(p.bias) + bi * p.bias_sb + hq * p.bias_sh +
                   static_cast<int64_t>(q_row) * p.bias_ss;
      // Dropout: this row's keep bits (4 words per key block); kept P are scaled at the end.
      const uint4* drop_row = nullptr;
      if (DROP && q_row < p.s_q)
        drop_row = reinterpret_cast<const uint4*>(
            p.drop_rows + (static_cast<int64_t>(bi) * p.h_q * p.s_q + static_cast<int64_t>(hq) * p.s_q + q_row) *
                              p.drop_kv_words);
      // Highest key index this row may see (-1: none, e.g. a padded row).
      int row_limit = L.len_kv - 1;
      if (p.causal) row_limit = min(row_limit, q_row + L.off);
      if (q_row >= L.len_q) row_limit = -1;
      // ALiBi slope of this head in the log2 domain, kept away from 0 so that the scores can
      // be carried divided by it (a slope below 1e-20 adds at most ~1e-15 to any score).
      const float sl2 = ALIBI ? fmaxf(alibi_slope_log2(p, hq), 1e-20f) : 0.f;
      const float u_scale = ALIBI ? u_scale_base / sl2 : 0.f;

      float m_ref = -INFINITY;   // running max (log2 domain, scale folded in)
      float l = 0.f;             // running sum of exp2(x - m_ref + P_OFFSET)

      for (int j = 0; j < n_blocks; ++j) {
        const int jg = jb + j;   // key block index over every unit of this CTA
        const int slot = (NQT == 2) ? t : (jg & 1);
        const uint32_t ph = (NQT == 2) ? (jg & 1) : ((jg >> 1) & 1);
        uint4 keep = make_uint4(0u, 0u, 0u, 0u);
        if (DROP && drop_row != nullptr) keep = __ldg(drop_row + kv_block(j, n_blocks));
        // The bias of this row and key block, loaded before the scores arrive; the next key
        // block's part of the row is sent to L2 first, so those loads find it there.
        uint4 bz[BIAS ? SC / 8 : 1];
        if constexpr (TMA_BIAS) {
          // This row's 64 keys of the key block's bias tile (128-byte rows, 128-byte swizzle).
          const int bs = jg & 1;
          if (!mbar_wait_warp(&bars.bias_full[bs], (jg >> 1) & 1, wt)) { ok = false; break; }
          const uint8_t* rowp = sBias + bs * C::BIAS_STAGE + hc * (C::BIAS_STAGE / 2) + r * 128;
#pragma unroll
          for (int e = 0; e < SC / 8; ++e) bz[e] = *reinterpret_cast<const uint4*>(rowp + ((e ^ (r & 7)) * 16));
          mbar_arrive(&bars.bias_empty[bs]);
        } else if constexpr (BIAS) {
          if (bias_row != nullptr && j + 1 < n_blocks) {
            const int kn = kv_block(j + 1, n_blocks) * kBlockN + col0;
            if (kn + SC <= p.s_kv) {
#pragma unroll
              for (int o = 0; o < SC; o += 64) prefetch_l2(bias_row + kn + o);
              prefetch_l2(bias_row + kn + SC - 1);
            }
          }
          const int kb0 = kv_block(j, n_blocks) * kBlockN + col0;
#pragma unroll
          for (int e = 0; e < SC / 8; ++e) {
            const int k0 = kb0 + 8 * e;
            if (bias_row != nullptr && k0 + 8 <= p.s_kv) {
              bz[e] = __ldg(reinterpret_cast<const uint4*>(bias_row + k0));
            } else {
              uint32_t h[4] = {0u, 0u, 0u, 0u};
              for (int uu = 0; bias_row != nullptr && uu < 8 && k0 + uu < p.s_kv; ++uu)
                h[uu / 2] |= static_cast<uint32_t>(bias_row[k0 + uu]) << (16 * (uu % 2));
              bz[e] = make_uint4(h[0], h[1], h[2], h[3]);
            }
          }
        }
        if (!mbar_wait_warp(&bars.s_full[slot], ph, wt)) { ok = false; break; }
        tc_fence_after();
        const uint32_t s_addr = tmem + lane_off + slot * 128;

        uint32_t sv[SC];
#pragma unroll
        for (int c = 0; c < SC / 32; ++c)
          tmem_ld32(s_addr + col0 + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
        tmem_ld_wait();

        const int kv0 = kv_block(j, n_blocks) * kBlockN;
        const bool need_mask = (kv0 + kBlockN - 1 > L.len_kv - 1) ||
                               (p.causal && kv0 + kBlockN - 1 > tile_row0 + L.off) ||
                               (tile_row0 + kBlockM > L.len_q);
        if (need_mask) {
          const int lim = row_limit - kv0 - col0;
#pragma unroll
          for (int c = 0; c < SC; ++c)
            if (c > lim) sv[c] = __float_as_uint(-INFINITY);
        }
        if constexpr (BIAS) {
          // y = s * |scale| + bias in natural-log units; the max and the exponent scale by log2 e.
          const float2 sn2 = make_float2(c_scale / kLog2e, c_scale / kLog2e);
#pragma unroll
          for (int c = 0; c < SC; c += 2) {
            const uint32_t wd = (c % 8 == 0) ? bz[c / 8].x : (c % 8 == 2) ? bz[c / 8].y
                              : (c % 8 == 4) ? bz[c / 8].z : bz[c / 8].w;
            const float2 y = fma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sn2,
                                  unpack16x2(wd, DT));
            sv[c] = __float_as_uint(y.x);
            sv[c + 1] = __float_as_uint(y.y);
          }
        }
        if constexpr (ALIBI) {
          // ALiBi splits slope * (key - row - off) into a column part slope * c and a row part
          // slope * (kv0 - row - off) folded into the max.  The scores are carried divided by
          // the slope, u = s * scale / slope + c (c an immediate: nothing to keep in registers),
          // and scaled back by the slope in the max and the exponent.
#pragma unroll
          for (int c = 0; c < SC; ++c)
            sv[c] = __float_as_uint(fmaf(__uint_as_float(sv[c]), u_scale, static_cast<float>(c)));
        }
        // Row max over four independent chains of three-input max.
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < SC; c += 8) {
          mx0 = max3(mx0, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
          mx1 = max3(mx1, __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
          mx2 = max3(mx2, __uint_as_float(sv[c + 4]), __uint_as_float(sv[c + 5]));
          mx3 = max3(mx3, __uint_as_float(sv[c + 6]), __uint_as_float(sv[c + 7]));
        }
        const float mx = max3(mx0, mx1, fmaxf(mx2, mx3));
        // ALiBi row part of this key block: slope * (kv0 + col0 - q_row - off).
        const float row_bias = ALIBI ? sl2 * static_cast<float>(kv0 + col0 - q_row - L.off) : 0.f;
        float m_cand = ALIBI ? sl2 * mx + row_bias : BIAS ? mx * kLog2e : mx * c_scale;
        if constexpr (NQT == 1) {
          // Both column halves take the larger of their two candidates, so they keep the same
          // running max (and rescale O together).
          xch[jg & 1][hc][r] = m_cand;
          mbar_arrive(&bars.mx_ready[jg & 1]);
          if (!mbar_wait_warp(&bars.mx_ready[jg & 1], (jg >> 1) & 1, wt)) { ok = false; break; }
          m_cand = fmaxf(m_cand, xch[jg & 1][hc ^ 1][r]);
        }
        float alpha = 1.f;
        if (m_cand > m_ref + C::THRESH) {
          alpha = ex2(m_ref - m_cand);
          m_ref = m_cand;
        }
        // A row that has seen no visible key yet keeps m_ref = -inf and all its P are 0.
        const float neg_m = (m_ref == -INFINITY) ? 0.f : C::P_OFFSET - m_ref;

        // x = s * scale - m in pairs; P = 2^x; row sums in pairs.
        const float cs = ALIBI ? sl2 : BIAS ? kLog2e : c_scale;   // ALiBi: scores carried as u
        const float nm = ALIBI ? neg_m + row_bias : neg_m;
        const float2 cs2 = make_float2(cs, cs);
        const float2 nm2 = make_float2(nm, nm);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
        uint32_t pk[C::PW];
#pragma unroll
        for (int c = 0; c < SC; c += 4) {
          const float2 x01 = fma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), cs2, nm2);
          const float2 x23 = fma2(make_float2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), cs2, nm2);
          float2 p01 = make_float2(ex2(x01.x), ex2(x01.y));
          float2 p23 = make_float2(ex2(x23.x), ex2(x23.y));
          acc0 = add2(acc0, p01);
          acc1 = add2(acc1, p23);
          if (FP8) {
            pk[c / 4] = pack4_e4m3(p01.x, p01.y, p23.x, p23.y);
          } else {
            pk[c / 2] = pack2(p01.x, p01.y, DT);
            pk[c / 2 + 1] = pack2(p23.x, p23.y, DT);
          }
          if constexpr (DROP && !FP8) {
            // Row sums take every P; P·V only the kept ones.  A pair's keep bits sit at bits
            // e/2 and e/2 + 16 of its word (e = its even column within the word): shifted to
            // bits 15 and 31, a sign-replicating byte permute spreads them to the two 16-bit
            // lanes, and a 16-bit zero is all zero bits.
            const int cg = c + col0;   // column within the key block
            const uint32_t wd = (cg < 32) ? keep.x : (cg < 64) ? keep.y : (cg < 96) ? keep.z : keep.w;
            const int e = cg % 32;
            pk[c / 2] &= prmt(wd << (15 - e / 2), 0u, 0xBB99u);
            pk[c / 2 + 1] &= prmt(wd << (14 - e / 2), 0u, 0xBB99u);
          }
        }
        const float rowsum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
        // P over this thread's columns (P words start at col0 * bytes per element / 4).
        const uint32_t p_addr = s_addr + col0 * C::ES / 4;
        if constexpr (C::PW % 32 == 0) {
#pragma unroll
          for (int c = 0; c < C::PW / 32; ++c)
            tmem_st32(p_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[c * 32]));
        } else {
          static_assert(C::PW == 16, "P words per thread");
          tmem_st16(p_addr, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
        }
        l = l * alpha + rowsum;

        if (NQT == 1 && j > 0) {
          // O is still being accumulated by the previous block's P·V.
          if (!mbar_wait_warp(&bars.pv_done, (jg - 1) & 1, wt)) { ok = false; break; }
          tc_fence_after();
        }
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // Each column half rescales its half of O.
          constexpr int OC = (NQT == 2) ? D : D / 2;
          const uint32_t o_addr = tmem + lane_off + C::O_COL0 + t * D + hc * OC;
#pragma unroll 1
          for (int c = 0; c < OC / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(o_addr + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(o_addr + c * 32, ov);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars.p_full[slot]);
      }
      jb += n_blocks;

      // ---- epilogue: O / l through shared memory and a TMA store; LSE ------------------
      // A unit whose rows see no key at all (padding) skips the pipeline and writes zeros.
      ok = ok && (n_blocks == 0 || mbar_wait_warp(&bars.o_full[t], qn & 1, wt));
      uint8_t* stage = C::OWN_STAGE ? sStage + t * C::OUT_TILE
                       : (NQT == 1) ? sRing : sQ + t * C::TILE_BYTES;
      if constexpr (NQT == 1) {
        // The row sum is the sum of the two halves' partial sums.  Both halves arrive whatever
        // happened, so the bounded wait can only fail through a timeout.
        xl[hc][r] = l;
        mbar_arrive(&bars.l_ready);
        ok = ok && mbar_wait_warp(&bars.l_ready, ue & 1, wt);
        if (ok) l += xl[hc ^ 1][r];
      }
      if constexpr (C::OWN_STAGE) {
        // The staging buffer is free once the previous unit's store has read it.
        if (ue > 0) {
          if (storer) {
            bulk_wait_read<0>();
            mbar_arrive(&bars.stage_free[t]);
          }
          ok = ok && mbar_wait_warp(&bars.stage_free[t], (ue - 1) & 1, wt);
        }
      }
      if (ok) {
        tc_fence_after();
        const float inv_l = (l > 0.f) ? v_scale / l : 0.f;   // rows without a visible key: O = 0
        const uint32_t o_addr = tmem + lane_off + C::O_COL0 + t * D;
        // O leaves in 64-column chunks; with column halves each writes half of them (at d = 64
        // the single chunk is the first half's).
        constexpr int NCK = (NQT == 2) ? D / 64 : (D / 128 > 0 ? D / 128 : 1);
        const int c_end = min((hc + 1) * NCK, D / 64);
#pragma unroll 1
        for (int c = hc * NCK; c < c_end; ++c) {
          uint32_t ov[64];
          if (n_blocks > 0) {
            tmem_ld32(o_addr + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
            tmem_ld32(o_addr + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) ov[i] = 0u;
          }
          uint8_t* rowp = stage + c * 16384 + r * 128;
#pragma unroll
          for (int uu = 0; uu < 8; ++uu) {
            uint4 wv;
            wv.x = pack2(__uint_as_float(ov[uu * 8 + 0]) * inv_l, __uint_as_float(ov[uu * 8 + 1]) * inv_l, OUT_DT);
            wv.y = pack2(__uint_as_float(ov[uu * 8 + 2]) * inv_l, __uint_as_float(ov[uu * 8 + 3]) * inv_l, OUT_DT);
            wv.z = pack2(__uint_as_float(ov[uu * 8 + 4]) * inv_l, __uint_as_float(ov[uu * 8 + 5]) * inv_l, OUT_DT);
            wv.w = pack2(__uint_as_float(ov[uu * 8 + 6]) * inv_l, __uint_as_float(ov[uu * 8 + 7]) * inv_l, OUT_DT);
            *reinterpret_cast<uint4*>(rowp + ((uu ^ (r & 7)) * 16)) = wv;
          }
        }
        fence_proxy_async_smem();
        if (p.lse != nullptr && q_row < p.s_q && hc == 0)
          p.lse[(static_cast<int64_t>(bi) * p.h_q + hq) * p.s_q + q_row] =
              (l > 0.f) ? (m_ref - C::P_OFFSET + __log2f(l)) * kLn2 : -INFINITY;
      }
      if (n_blocks > 0) {
        // O has left TMEM (or never will, after a failure): the next unit may overwrite it.
        if constexpr (PERSIST) {
          tc_fence_before();
          mbar_arrive(&bars.o_empty[t]);
        }
        ++qn;
      }
      // Every thread of the warpgroup arrives exactly once per unit, whatever happened above,
      // so the bounded wait below can only fail through a timeout, never deadlock.
      mbar_arrive(&bars.epi_ready[t]);
      if (storer) {
        const bool all_ok = mbar_wait(&bars.epi_ready[t], ue & 1, wt) && ok && !*abort_flag;
        if (all_ok) {
          for (int c = 0; c < D / 64; ++c)
            tma_store_4d(&p.tm_o, stage + c * 16384, c * 64, tile_row0, hq, bi);
          tma_store_commit();
          // A CTA with its own staging buffer lets the store run while it goes on to the next
          // unit; otherwise the buffer is the Q tile or the ring, released at the exit.
          if constexpr (!C::OWN_STAGE) tma_store_wait_read_all();
        }
      }
      ++ue;
    }
    if (storer) tma_store_wait_read_all();
  }

  tc_fence_before();
  __syncthreads();
  // Every role is done.  If one gave up (the abort flag, visible to all after the barrier),
  // copies the producer issued may still be in flight: let them land before the CTA's shared
  // memory is released.  (Q and each ring slot hold at most one copy in flight.)
  if (producer && *abort_flag) {
    if (q_issued > 0)
      for (int t = 0; t < NQT; ++t) mbar_wait_drain(&bars.q_full[t], (q_issued - 1) & 1);
    for (int k = (kv_issued > NS ? kv_issued - NS : 0); k < kv_issued; ++k)
      mbar_wait_drain(&bars.kv_full[k % NS], (k / NS) & 1);
    for (int k = (bias_issued > 2 ? bias_issued - 2 : 0); k < bias_issued; ++k)
      mbar_wait_drain(&bars.bias_full[k & 1], (k >> 1) & 1);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int DT, int OUT_DT>
cudaError_t launch_t(const FwdParams& p, cudaStream_t st) {
  int smem = FwdCfg<D, DT>::SMEM_BYTES;
  auto kern = sdpa_fwd_kernel<D, DT, OUT_DT, 0>;
  if constexpr (DT != kE4M3 && D <= 128) {
    if (p.one_tile) {
      kern = p.ctas ? sdpa_fwd_kernel<D, DT, OUT_DT, kFeatOneTile | kFeatPersist>
                    : sdpa_fwd_kernel<D, DT, OUT_DT, kFeatOneTile>;
      smem = p.ctas ? FwdCfg<D, DT, true, true>::SMEM_BYTES : FwdCfg<D, DT, true>::SMEM_BYTES;
    } else if (p.ctas) {
      kern = sdpa_fwd_kernel<D, DT, OUT_DT, kFeatPersist>;
      smem = FwdCfg<D, DT, false, true>::SMEM_BYTES;
    }
  }
  if constexpr (DT != kE4M3) {
    const int feat = (p.alibi ? kFeatAlibi : 0) | (p.drop_rows ? kFeatDropout : 0) | (p.bias ? kFeatBias : 0);
    if (feat == kFeatAlibi) kern = sdpa_fwd_kernel<D, DT, OUT_DT, kFeatAlibi>;
    if (feat == kFeatDropout) kern = sdpa_fwd_kernel<D, DT, OUT_DT, kFeatDropout>;
    if (feat == (kFeatAlibi | kFeatDropout)) kern = sdpa_fwd_kernel<D, DT, OUT_DT, kFeatAlibi | kFeatDropout>;
    // With d <= 128 the bias instances run one Q tile per CTA (the bias tiles take the
    // shared memory of the second one; the caller sizes the grid accordingly).
    constexpr int kBiasTile = D <= 128 ? kFeatOneTile : 0;
    if (feat == kFeatBias) kern = sdpa_fwd_kernel<D, DT, OUT_DT, kFeatBias | kBiasTile>;
    if (feat == (kFeatBias | kFeatDropout)) kern = sdpa_fwd_kernel<D, DT, OUT_DT, kFeatBias | kFeatDropout | kBiasTile>;
    if constexpr (D <= 128) {
      if (feat & kFeatBias) smem = FwdCfg<D, DT, true, false, true>::SMEM_BYTES;
    }
  }
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = p.ctas ? static_cast<unsigned>(p.ctas) : static_cast<unsigned>(p.b) * p.h_q * p.num_m_blocks;
  kern<<<grid, FwdCfg<D, DT>::THREADS, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

int fwd_persistent_ctas(long long units, int s_kv, int d, int in_dtype, bool plain, int num_sms) {
  if (!plain || in_dtype == kE4M3 || d > 128) return 0;
  if (units <= num_sms || units >= 4ll * num_sms) return 0;
  // Long units amortise their set-up anyway and keep the deeper K/V ring of the one-unit
  // schedule (a 2K-query chunk against 8K keys: 1366 persistent vs 1430 TFLOP/s).
  if (s_kv > 4096) return 0;
  return num_sms;
}

bool fwd_prefer_one_tile(int b, int h_q, int s_q, int d, int in_dtype, bool plain, int num_sms) {
  if (!plain || in_dtype == kE4M3 || d > 128) return false;
  const long long two_tile_ctas = static_cast<long long>(b) * h_q * ((s_q + 255) / 256);
  return two_tile_ctas < num_sms;
}

int fwd_q_tiles(int d, int in_dtype) {
  (void)in_dtype;
  return d <= 128 ? 2 : 1;
}

cudaError_t launch_fwd(const FwdParams& p, int d, int in_dtype, int out_dtype, cudaStream_t st) {
  if (in_dtype == kF16) {
    if (d == 64) return launch_t<64, kF16, kF16>(p, st);
    if (d == 128) return launch_t<128, kF16, kF16>(p, st);
    if (d == 256) return launch_t<256, kF16, kF16>(p, st);
  } else if (in_dtype == kBF16) {
    if (d == 64) return launch_t<64, kBF16, kBF16>(p, st);
    if (d == 128) return launch_t<128, kBF16, kBF16>(p, st);
    if (d == 256) return launch_t<256, kBF16, kBF16>(p, st);
  } else if (in_dtype == kE4M3) {
    if (out_dtype == kBF16) {
      if (d == 128) return launch_t<128, kE4M3, kBF16>(p, st);
      if (d == 256) return launch_t<256, kE4M3, kBF16>(p, st);
    } else {
      if (d == 128) return launch_t<128, kE4M3, kF16>(p, st);
      if (d == 256) return launch_t<256, kE4M3, kF16>(p, st);
    }
  }
  return cudaErrorInvalidValue;
}

uint32_t fwd_take_device_error() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, ptx::g_device_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(ptx::g_device_error, &z, sizeof(z));
  return v;
}

}  // namespace sdpa
