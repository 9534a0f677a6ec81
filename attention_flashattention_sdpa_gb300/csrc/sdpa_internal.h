// sdpa_internal.h — parameter blocks passed from the C-ABI layer to the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <set>
#include <utility>

namespace sdpa {

constexpr int kBlockM = 128;  // query rows per Q tile (one TMEM lane per row)
constexpr int kBlockN = 128;  // key/value rows per KV block

enum DType : int { kF16 = 0, kBF16 = 1, kE4M3 = 2 };

// Forward pass.  Tensor maps are 4-D (d, s, h, b) views over the caller's strides,
// 128-byte swizzled, box = (128 bytes of d, 128 rows, 1, 1).
struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  CUtensorMap tm_bias;        // bias tiles of 128 rows x 64 keys (bias with d <= 128), else unused
  float* lse;                 // [b][h_q][s_q] fp32 or nullptr
  const float* descale_q;     // E4M3 only
  const float* descale_k;
  const float* descale_v;
  int b, h_q, h_kv, s_q, s_kv;
  int group;                  // h_q / h_kv
  int causal;
  int num_m_blocks;           // ceil(s_q / (128 * q tiles per CTA))
  int one_tile;               // small problem: one Q tile per CTA even where two fit
  int ctas;                   // 0: one CTA per work unit; else this many persistent CTAs, each
                              // walking several units (plain 16-bit inputs, d <= 128)
  const int32_t* seq_lens_q;  // per-batch valid rows, or nullptr
  const int32_t* seq_lens_kv;
  int bottom_right;           // causal alignment: key j visible iff j <= i + len_kv - len_q
  float scale_log2;           // |attn_scale| * log2(e) (0 is replaced by a tiny positive value)
  int negate_scores;          // attn_scale < 0: the QK^T MMA negates its A operand
  int alibi;                  // add slope_hq * (j - i - off) to the scaled scores
  const float* alibi_slopes;  // [h_q] fp32, or nullptr for the geometric default
  const uint32_t* drop_rows;  // dropout keep bits [b*h_q][s_q][drop_kv_words], or nullptr
  int drop_kv_words;          // 32-bit words per row: ceil(s_kv / 128) * 4
  float drop_scale;           // 1 / (1 - p), or 1 without dropout
  const void* bias;           // additive bias [b][h_q][s_q][s_kv] (input dtype), or nullptr
  int64_t bias_sb, bias_sh, bias_ss;   // element strides (0 broadcasts b or h)
  long long wait_limit;       // bound on one mbarrier wait, SM cycles
};

// Number of Q tiles (of 128 rows) one forward CTA processes.
int fwd_q_tiles(int d, int in_dtype);

// Whether a plain 16-bit forward pass with d <= 128 should run one Q tile per CTA: when
// two-tile CTAs would not fill one wave of the GPU, twice as many CTAs of half the work
// finish sooner (measured: 64 CTAs +33%, 128 CTAs +5%; at 192 and 256 two tiles win).
bool fwd_prefer_one_tile(int b, int h_q, int s_q, int d, int in_dtype, bool plain, int num_sms);

// Persistent CTAs for a forward pass of `units` work units: the SM count when the units fill
// between one and four waves of the GPU (a launch with one CTA per unit would leave the last
// wave ragged and pay every CTA's set-up) and are short (s_kv <= 4096), else 0 (one CTA per
// unit).
int fwd_persistent_ctas(long long units, int s_kv, int d, int in_dtype, bool plain, int num_sms);

cudaError_t launch_fwd(const FwdParams& p, int d, int in_dtype, int out_dtype, cudaStream_t st);
uint32_t fwd_take_device_error();

// Backward pass.
struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;   // loads (128-byte swizzled)
  CUtensorMap tm_dk, tm_dv;              // stores
  CUtensorMap tm_dqacc;                  // fp32 [b*h_q*s_q_pad][d], reduce-add target
  const void* o;       // forward output, for Delta
  const void* dout;    // incoming gradient, for Delta
  const float* lse;    // [b][h_q][s_q]
  void* dq;            // output
  float* dq_acc;       // workspace [b][h_q][s_q_pad][d] fp32
  float* delta;        // workspace [b][h_q][s_q_pad] fp32 (-Delta_i)
  float* lse2;         // workspace [b][h_q][s_q_pad] fp32 (-LSE_i * log2 e)
  int64_t o_sb, o_sh, o_ss;     // element strides of O
  int64_t do_sb, do_sh, do_ss;  // element strides of dO
  int64_t dq_sb, dq_sh, dq_ss;  // element strides of dQ
  int b, h_q, h_kv, s_q, s_kv, d;
  int group;
  int causal;
  int s_q_pad;                  // s_q rounded up to 128
  float scale;                  // attn_scale
  float scale_log2;             // attn_scale * log2(e)
  const int32_t* seq_lens_q;    // per-batch valid rows, or nullptr
  const int32_t* seq_lens_kv;
  int bottom_right;             // causal alignment: key j visible iff j <= i + len_kv - len_q
  // Split groups: when a KV head's query heads are shared between `kv_split` CTAs, each CTA
  // adds its dK/dV partial into fp32 accumulators and a last pass writes dK, dV.
  int kv_split;                 // CTAs per (batch, KV head, KV block); 1 = no split
  int heads_per_split;          // query heads one such CTA visits
  int s_kv_pad;                 // s_kv rounded up to 128
  float* dk_acc;                // workspace, b * h_kv * s_kv_pad * d fp32 in 128-row key-block
                                // tiles (split only; layout at kv_acc_offset)
  float* dv_acc;
  void* dk;                     // outputs (split only: written by the convert pass)
  void* dv;
  int64_t dk_sb, dk_sh, dk_ss;
  int64_t dv_sb, dv_sh, dv_ss;
  int alibi;                    // add slope_hq * (j - i - off) to the scaled scores
  const float* alibi_slopes;    // [h_q] fp32, or nullptr for the geometric default
  const uint32_t* drop_cols;    // dropout keep bits, transposed: [b*h_q][s_kv][drop_q_words]
  int drop_q_words;             // 32-bit words per key row: ceil(s_q / 128) * 4
  float drop_scale;             // 1 / (1 - p), or 1 without dropout
  // FP8 inputs (widened exactly to the output dtype before the kernels run): per-tensor
  // descales of Q, K, V and dO, folded into the kernels' scale factors; nullptr otherwise.
  const float* descale_q;
  const float* descale_k;
  const float* descale_v;
  const float* descale_do;
  // Additive bias, transposed into the workspace: [bias_nb][bias_nh][s_kv][s_q_pad] in the
  // input dtype (bias_nb = 1 or b, bias_nh = 1 or h_q), or nullptr.
  const void* bias_t;
  int bias_nb, bias_nh;
  // Bias gradient: dS reduce-added into a zeroed fp32 workspace laid out like bias_t,
  // [bias_nb][bias_nh][s_kv][s_q_pad], or nullptr.
  float* dbias_acc;
  long long wait_limit;         // bound on one mbarrier wait, SM cycles
};

// dbias[nb][nh][s_q][s_kv] (16-bit, caller strides) from the transposed fp32 accumulator.
cudaError_t launch_dbias_convert(const float* acc, int nb, int nh, int s_q, int s_kv, int s_q_pad, void* dst,
                                 int64_t sb, int64_t sh, int64_t ss, int dtype, cudaStream_t st);

// Transposes a strided [nb][nh][s_q][s_kv] bias view into dense [nb][nh][s_kv][s_q_pad].
cudaError_t launch_bias_transpose(const void* src, int64_t sb, int64_t sh, int64_t ss, int nb, int nh,
                                  int s_q, int s_kv, int s_q_pad, int skip_above, int diag_off, void* dst,
                                  cudaStream_t st);

// Widens a strided FP8 (E4M3 or E5M2) [b][h][s][d] view into a dense F16 or BF16 copy.  Every
// FP8 value is exact in either 16-bit format; descales are applied later, by the kernels.
cudaError_t launch_fp8_widen(const void* src, int64_t sb, int64_t sh, int64_t ss, int b, int h, int s,
                             int d, int src_e5m2, void* dst, int dst_dtype, cudaStream_t st);

// Dropout keep mask (see sdpa_dropout.cu for the definition).
struct DropoutParams {
  uint32_t* rows;               // [b*h_q][s_q][kv_words] or nullptr
  uint32_t* cols;               // [b*h_q][s_kv][q_words] or nullptr
  uint64_t seed, offset;
  uint32_t threshold;           // keep iff the 16-bit draw >= threshold (<= 65536)
  int s_q, s_kv;
  int kv_words, q_words;        // ceil(s_kv / 128) * 4, ceil(s_q / 128) * 4
  int skip_above;               // skip 128x128 tiles whose keys all lie beyond row + diag_off
  int diag_off;                 // causal offset (0 top-left, s_kv - s_q bottom-right)
};

cudaError_t launch_dropout_mask(const DropoutParams& p, int bh, cudaStream_t st);

// How many CTAs share one (batch, KV head, KV block) in the backward pass.  A fixed policy
// of the shape alone (no device query), so workspace sizing and launch always agree.
int bwd_kv_split(int b, int h_q, int h_kv, int s_kv);

size_t bwd_workspace_bytes(int b, int h_q, int h_kv, int s_q, int s_kv, int d);
cudaError_t launch_bwd(const BwdParams& p, int dtype, cudaStream_t st);
uint32_t bwd_take_device_error();

// Raises a kernel's dynamic shared-memory limit once per (kernel, device): the setting lasts
// for the process, and the call costs microseconds that small problems would otherwise pay
// on every launch.
inline cudaError_t set_smem_once(const void* kern, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kern, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({kern, dev});
  return e;
}

// Default bound on one mbarrier wait, in SM cycles (about a second).
constexpr long long ptx_default_wait_limit() { return 1ll << 31; }

// Kernel feature bits (compile-time variants of the forward and backward kernels).
constexpr int kFeatAlibi = 1;
constexpr int kFeatDropout = 2;
constexpr int kFeatBias = 4;
constexpr int kFeatDBias = 8;   // only with kFeatBias
constexpr int kFeatOneTile = 16;  // forward: one Q tile per work unit at d <= 128
constexpr int kFeatPersist = 32;  // forward: persistent CTAs, each walking several work units

}  // namespace sdpa

namespace sdpa {

// Valid rows and causal offset of batch `bi`: key j is visible to query i < len_q iff
// j < len_kv and (no mask, or j <= i + off).
struct Lens {
  int len_q, len_kv, off;
};

template <typename P>
__device__ __forceinline__ Lens batch_lens(const P& p, int bi) {
  Lens L;
  L.len_q = p.seq_lens_q ? min(max(__ldg(p.seq_lens_q + bi), 0), p.s_q) : p.s_q;
  L.len_kv = p.seq_lens_kv ? min(max(__ldg(p.seq_lens_kv + bi), 0), p.s_kv) : p.s_kv;
  L.off = p.bottom_right ? L.len_kv - L.len_q : 0;
  return L;
}

// ALiBi slope of query head hq, in the log2 domain the kernels exponentiate in: the
// caller's slope (a negative one counts as 0), or the geometric sequence 2^(-8 (hq + 1) / h_q).
template <typename P>
__device__ __forceinline__ float alibi_slope_log2(const P& p, int hq) {
  const float m = p.alibi_slopes ? fmaxf(__ldg(p.alibi_slopes + hq), 0.f)
                                 : exp2f(-8.f * static_cast<float>(hq + 1) / static_cast<float>(p.h_q));
  return m * 1.4426950408889634f;
}

}  // namespace sdpa
