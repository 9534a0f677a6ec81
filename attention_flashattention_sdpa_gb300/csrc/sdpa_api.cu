// sdpa_api.cu — the C ABI declared in include/sdpa.h: argument validation, TMA tensor-map
// construction over the caller's strides, workspace sizing and kernel dispatch.
//
// Shape of the interface follows the pages' SDPA node: Q, K, V, attn_scale by value, a
// causal flag, an inference/training switch (here: lse == NULL or not), explicit dims and
// strides, a workspace the caller queries and allocates, asynchronous execution, and
// error codes with a last-error string [cuDNN 9 blog, SDPA walkthrough and error
// reporting; cuDNN-in-Python post, graph build / workspace / execute].  Unsupported
// requests return an error rather than falling back [attention codelab §6: the cuDNN path
// raises instead of silently using another implementation].
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/sdpa.h"
#include "sdpa_internal.h"

namespace {

thread_local std::string g_last_error;

sdpa_status_t fail(sdpa_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

sdpa_status_t ok() {
  g_last_error.clear();
  return SDPA_OK;
}

int log_level() {
  static int lvl = [] {
    const char* s = getenv("SDPA_LOG_LEVEL");
    return s ? atoi(s) : 0;
  }();
  return lvl;
}

bool debug_sync() {
  static bool v = [] {
    const char* s = getenv("SDPA_DEBUG_SYNC");
    return s && atoi(s) != 0;
  }();
  return v;
}

// Bound on every mbarrier wait inside the kernels, in SM cycles: about a second by default;
// SDPA_WAIT_LIMIT_CYCLES overrides it (read at every call), e.g. to make waits run out on
// purpose and check that a kernel gives up cleanly and reports SDPA_ERR_TIMEOUT.
long long wait_limit_cycles() {
  const char* s = getenv("SDPA_WAIT_LIMIT_CYCLES");
  const long long x = s ? atoll(s) : 0;
  return x > 0 ? x : sdpa::ptx_default_wait_limit();
}

int elem_bytes(int dt) { return (dt == SDPA_DTYPE_E4M3 || dt == SDPA_DTYPE_E5M2) ? 1 : 2; }

// Dense 16-bit copies of FP8 Q, K, V and dO that an E4M3 backward pass widens into the
// workspace after its own scratch (0 for 16-bit inputs).
size_t widen_bytes(const sdpa_problem_t* p, size_t* off_k, size_t* off_v, size_t* off_do) {
  auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t nq = a(static_cast<size_t>(p->b) * p->h_q * p->s_q * p->d * 2);
  const size_t nkv = a(static_cast<size_t>(p->b) * p->h_kv * p->s_kv * p->d * 2);
  if (off_k) *off_k = nq;
  if (off_v) *off_v = nq + nkv;
  if (off_do) *off_do = nq + 2 * nkv;
  return p->in_dtype == SDPA_DTYPE_E4M3 ? 2 * nq + 2 * nkv : 0;
}

// Transposed bias copy of a backward pass: [1 or b][1 or h_q] x 128 x 128 tiles over keys
// (s_kv rounded up to 128) and queries (s_q rounded up to 128).
size_t bias_t_bytes(const sdpa_problem_t* p) {
  if (p->bias == nullptr) return 0;
  const size_t nb = p->bias_strides.b == 0 ? 1 : p->b, nh = p->bias_strides.h == 0 ? 1 : p->h_q;
  const size_t pad = (p->s_q + 127) / 128 * 128, kpad = (p->s_kv + 127) / 128 * 128;
  return (nb * nh * kpad * pad * 2 + 255) & ~size_t(255);
}

// fp32 bias-gradient accumulator, laid out like the transposed bias copy.
size_t dbias_acc_bytes(const sdpa_problem_t* p) {
  if (p->bias == nullptr || p->dbias == nullptr) return 0;
  return 2 * bias_t_bytes(p);
}

size_t bwd_total_workspace(const sdpa_problem_t* p) {
  const size_t base = (sdpa::bwd_workspace_bytes(p->b, p->h_q, p->h_kv, p->s_q, p->s_kv, p->d) + 255) & ~size_t(255);
  return base + widen_bytes(p, nullptr, nullptr, nullptr) + bias_t_bytes(p) + dbias_acc_bytes(p);
}

bool valid_dtype(int dt) {
  return dt == SDPA_DTYPE_F16 || dt == SDPA_DTYPE_BF16 || dt == SDPA_DTYPE_E4M3 || dt == SDPA_DTYPE_E5M2;
}

// ---------------------------------------------------------------------------
// tensor maps
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

CUtensorMapDataType map_dtype(int dt) {
  switch (dt) {
    case SDPA_DTYPE_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case SDPA_DTYPE_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
  }
}

// Checks that a logical [b][h][s][d] view can be handed to the TMA unit.
sdpa_status_t check_view(const char* name, const void* ptr, const sdpa_strides_t& st, int b, int h,
                         int s, int d, int es) {
  if (ptr == nullptr) return fail(SDPA_ERR_INVALID_ARG, "%s: null pointer", name);
  if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
    return fail(SDPA_ERR_LAYOUT, "%s: base address must be 16-byte aligned", name);
  if (st.d != 1) return fail(SDPA_ERR_LAYOUT, "%s: innermost (d) stride must be 1, got %lld", name,
                             (long long)st.d);
  const int64_t strides[3] = {st.s, st.h, st.b};
  const int64_t sizes[3] = {s, h, b};
  const char* nm[3] = {"s", "h", "b"};
  for (int i = 0; i < 3; ++i) {
    if (sizes[i] == 1) continue;  // stride of a unit dimension is never used
    if (strides[i] <= 0)
      return fail(SDPA_ERR_LAYOUT, "%s: stride_%s must be positive, got %lld", name, nm[i],
                  (long long)strides[i]);
    if ((strides[i] * es) % 16 != 0)
      return fail(SDPA_ERR_LAYOUT, "%s: stride_%s * element size must be a multiple of 16 bytes",
                  name, nm[i]);
    if (strides[i] * es >= (int64_t(1) << 40))
      return fail(SDPA_ERR_LAYOUT, "%s: stride_%s too large for the TMA unit", name, nm[i]);
  }
  (void)d;
  return SDPA_OK;
}

sdpa_status_t make_map(CUtensorMap* map, const char* name, const void* ptr, const sdpa_strides_t& st,
                       int b, int h, int s, int d, int dt, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr)
    return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the CUDA driver");
  const int es = elem_bytes(dt);
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)s, (cuuint64_t)h, (cuuint64_t)b};
  // A unit dimension's stride is irrelevant; give it a legal value.
  const int64_t fallback = (int64_t)d * es * s * h;
  int64_t sb[3] = {st.s * es, st.h * es, st.b * es};
  int64_t sizes[3] = {s, h, b};
  for (int i = 0; i < 3; ++i)
    if (sizes[i] == 1) sb[i] = ((fallback + 15) / 16) * 16;
  cuuint64_t strides[3] = {(cuuint64_t)sb[0], (cuuint64_t)sb[1], (cuuint64_t)sb[2]};
  cuuint32_t box[4] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, map_dtype(dt), 4, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(SDPA_ERR_LAYOUT, "%s: cuTensorMapEncodeTiled rejected the view (CUresult %d)",
                name, (int)r);
  return SDPA_OK;
}

sdpa_status_t check_problem(const sdpa_problem_t* p, bool backward) {
  if (p == nullptr) return fail(SDPA_ERR_INVALID_ARG, "problem descriptor is NULL");
  if (p->b < 1 || p->h_q < 1 || p->h_kv < 1 || p->s_q < 1 || p->s_kv < 1 || p->d < 1)
    return fail(SDPA_ERR_INVALID_ARG,
                "sizes must be >= 1 (b=%d h_q=%d h_kv=%d s_q=%d s_kv=%d d=%d)", p->b, p->h_q,
                p->h_kv, p->s_q, p->s_kv, p->d);
  if (p->h_q % p->h_kv != 0)
    return fail(SDPA_ERR_INVALID_ARG, "h_q (%d) must be a multiple of h_kv (%d)", p->h_q, p->h_kv);
  if (p->d != 64 && p->d != 128 && p->d != 256)
    return fail(SDPA_ERR_UNSUPPORTED, "head dim %d not supported (64, 128 or 256)", p->d);
  if (!valid_dtype(p->in_dtype)) return fail(SDPA_ERR_INVALID_ARG, "unknown in_dtype %d", p->in_dtype);
  if (!valid_dtype(p->out_dtype))
    return fail(SDPA_ERR_INVALID_ARG, "unknown out_dtype %d", p->out_dtype);
  if (p->causal < 0 || p->causal > 2)
    return fail(SDPA_ERR_INVALID_ARG, "causal must be 0 (none), 1 (top-left) or 2 (bottom-right), got %d",
                p->causal);
  if ((p->seq_lens_q && reinterpret_cast<uintptr_t>(p->seq_lens_q) % 4) ||
      (p->seq_lens_kv && reinterpret_cast<uintptr_t>(p->seq_lens_kv) % 4))
    return fail(SDPA_ERR_LAYOUT, "seq_lens_q / seq_lens_kv must be 4-byte aligned");
  if (!std::isfinite(p->attn_scale))
    return fail(SDPA_ERR_INVALID_ARG, "attn_scale must be finite");
  if (p->alibi != 0 && p->alibi != 1)
    return fail(SDPA_ERR_INVALID_ARG, "alibi must be 0 or 1, got %d", p->alibi);
  if (p->alibi && p->alibi_slopes && reinterpret_cast<uintptr_t>(p->alibi_slopes) % 4)
    return fail(SDPA_ERR_LAYOUT, "alibi_slopes must be 4-byte aligned");
  // ALiBi penalises a query's distance to the earlier keys it sees (the ALiBi paper, §3);
  // without a causal mask the linear term would favour the farthest later keys instead.
  if (p->alibi && p->causal == 0)
    return fail(SDPA_ERR_UNSUPPORTED, "ALiBi needs a causal mask (causal = 1 or 2)");
  if (p->alibi && p->in_dtype == SDPA_DTYPE_E4M3)
    return fail(SDPA_ERR_UNSUPPORTED, "ALiBi takes F16 or BF16 inputs, not E4M3");
  if (!(p->dropout_p >= 0.f && p->dropout_p < 1.f))
    return fail(SDPA_ERR_INVALID_ARG, "dropout_p must be in [0, 1), got %g", p->dropout_p);
  if (p->dropout_p > 0.f && p->in_dtype == SDPA_DTYPE_E4M3)
    return fail(SDPA_ERR_UNSUPPORTED, "dropout takes F16 or BF16 inputs, not E4M3");
  if (p->bias != nullptr) {
    const sdpa_strides_t& bs = p->bias_strides;
    if (p->in_dtype == SDPA_DTYPE_E4M3)
      return fail(SDPA_ERR_UNSUPPORTED, "a bias tensor takes F16 or BF16 inputs, not E4M3");
    if (p->alibi) return fail(SDPA_ERR_UNSUPPORTED, "bias and alibi together: fold ALiBi into the bias");
    if (reinterpret_cast<uintptr_t>(p->bias) % 16)
      return fail(SDPA_ERR_LAYOUT, "bias must be 16-byte aligned");
    if (bs.d != 1 && p->s_kv > 1) return fail(SDPA_ERR_LAYOUT, "bias: the key stride (d field) must be 1");
    if (bs.b < 0 || bs.h < 0 || bs.s < 0 || bs.b % 8 || bs.h % 8 || bs.s % 8)
      return fail(SDPA_ERR_LAYOUT, "bias: strides must be non-negative multiples of 8 elements");
    if (p->s_q > 1 && bs.s < p->s_kv) return fail(SDPA_ERR_LAYOUT, "bias: row stride below s_kv");
  }
  if (backward && p->dbias != nullptr) {
    const sdpa_strides_t& ds = p->dbias_strides;
    if (p->bias == nullptr) return fail(SDPA_ERR_INVALID_ARG, "dbias needs a bias tensor");
    if (reinterpret_cast<uintptr_t>(p->dbias) % 16) return fail(SDPA_ERR_LAYOUT, "dbias must be 16-byte aligned");
    if ((ds.b == 0) != (p->bias_strides.b == 0) || (ds.h == 0) != (p->bias_strides.h == 0))
      return fail(SDPA_ERR_LAYOUT, "dbias must broadcast over the same dimensions as bias");
    if (ds.d != 1 && p->s_kv > 1) return fail(SDPA_ERR_LAYOUT, "dbias: the key stride (d field) must be 1");
    if (ds.b < 0 || ds.h < 0 || ds.s < 0 || ds.b % 8 || ds.h % 8 || ds.s % 8)
      return fail(SDPA_ERR_LAYOUT, "dbias: strides must be non-negative multiples of 8 elements");
    if (p->s_q > 1 && ds.s < p->s_kv) return fail(SDPA_ERR_LAYOUT, "dbias: row stride below s_kv");
  }
  if (p->in_dtype == SDPA_DTYPE_E5M2 || p->out_dtype == SDPA_DTYPE_E5M2)
    return fail(SDPA_ERR_UNSUPPORTED, "E5M2 is accepted only as dout_dtype of an FP8 backward pass");
  if (p->in_dtype == SDPA_DTYPE_E4M3) {
    if (p->out_dtype == SDPA_DTYPE_E4M3)
      return fail(SDPA_ERR_UNSUPPORTED, "E4M3 inputs give a BF16 or F16 output");
    if (!backward && p->d == 64) return fail(SDPA_ERR_UNSUPPORTED, "E4M3 forward supports d = 128 or 256");
    if (!p->descale_q || !p->descale_k || !p->descale_v)
      return fail(SDPA_ERR_INVALID_ARG, "E4M3 inputs need descale_q, descale_k and descale_v");
    if (backward) {
      if (p->dout_dtype != SDPA_DTYPE_E5M2 && p->dout_dtype != SDPA_DTYPE_E4M3)
        return fail(SDPA_ERR_UNSUPPORTED, "an E4M3 backward pass takes dO as E5M2 or E4M3 (dout_dtype %d)",
                    p->dout_dtype);
      if (!p->descale_do) return fail(SDPA_ERR_INVALID_ARG, "an FP8 dO needs descale_do");
    }
  } else if (p->out_dtype != p->in_dtype) {
    return fail(SDPA_ERR_UNSUPPORTED, "F16/BF16 inputs give an output of the same dtype");
  }
  // Row/column counts index int32 coordinates of the TMA unit.
  if ((int64_t)p->b * p->h_q * p->s_q >= (int64_t(1) << 31))
    return fail(SDPA_ERR_UNSUPPORTED, "b*h_q*s_q too large");
  return SDPA_OK;
}

float scale_log2_of(float attn_scale) {
  float a = std::fabs(attn_scale);
  if (a == 0.f) a = 1e-30f;  // exact zero scale: every score maps to exp2(0) = 1
  return a * 1.4426950408889634f;
}

sdpa_status_t finish_launch(cudaError_t e, cudaStream_t stream, const char* what) {
  if (e != cudaSuccess)
    return fail(SDPA_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
  if (debug_sync()) {
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    uint32_t flags = sdpa::fwd_take_device_error() | sdpa::bwd_take_device_error();
    if (flags) return fail(SDPA_ERR_TIMEOUT, "%s: a bounded device wait gave up (flags=%u)", what, flags);
  }
  return ok();
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Streaming multiprocessors of the current device (cached per device).
int num_sms() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    cache[dev] = (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) ? n : 152;
  }
  return cache[dev];
}

int words_of(int s) { return (s + 127) / 128 * 4; }   // keep-mask words per row or key

// Dropout mask pointer of a forward or backward call (checked only when dropout is on).
sdpa_status_t check_drop_mask(const sdpa_problem_t* p, const uint32_t* mask, const char* name) {
  if (p->dropout_p == 0.f) return SDPA_OK;
  if (mask == nullptr)
    return fail(SDPA_ERR_INVALID_ARG, "dropout_p > 0 needs %s (from sdpa_dropout_mask)", name);
  if (reinterpret_cast<uintptr_t>(mask) % 16)
    return fail(SDPA_ERR_LAYOUT, "%s must be 16-byte aligned", name);
  return SDPA_OK;
}

float drop_scale_of(const sdpa_problem_t* p) {
  return static_cast<float>(1.0 / (1.0 - static_cast<double>(p->dropout_p)));
}

}  // namespace

extern "C" {

sdpa_status_t sdpa_workspace_size(const sdpa_problem_t* p, int is_backward, size_t* bytes) {
  if (bytes == nullptr) return fail(SDPA_ERR_INVALID_ARG, "bytes is NULL");
  sdpa_status_t st = check_problem(p, is_backward != 0);
  if (st != SDPA_OK) return st;
  *bytes = is_backward ? bwd_total_workspace(p) : 0;
  return ok();
}

sdpa_status_t sdpa_fwd(const sdpa_problem_t* p, const void* q, const void* k, const void* v, void* o,
                       float* lse, void* workspace, size_t workspace_bytes, void* stream_) {
  (void)workspace;
  (void)workspace_bytes;
  sdpa_status_t st = check_problem(p, false);
  if (st != SDPA_OK) return st;
  const int es = elem_bytes(p->in_dtype);
  if ((st = check_view("q", q, p->q, p->b, p->h_q, p->s_q, p->d, es)) != SDPA_OK) return st;
  if ((st = check_view("k", k, p->k, p->b, p->h_kv, p->s_kv, p->d, es)) != SDPA_OK) return st;
  if ((st = check_view("v", v, p->v, p->b, p->h_kv, p->s_kv, p->d, es)) != SDPA_OK) return st;
  if ((st = check_view("o", o, p->o, p->b, p->h_q, p->s_q, p->d, 2)) != SDPA_OK) return st;
  if (lse != nullptr && reinterpret_cast<uintptr_t>(lse) % 4 != 0)
    return fail(SDPA_ERR_LAYOUT, "lse must be 4-byte aligned");
  if ((st = check_drop_mask(p, p->dropout_mask, "dropout_mask")) != SDPA_OK) return st;

  sdpa::FwdParams prm;
  memset(&prm, 0, sizeof(prm));
  if ((st = make_map(&prm.tm_q, "q", q, p->q, p->b, p->h_q, p->s_q, p->d, p->in_dtype, 128)) != SDPA_OK) return st;
  if ((st = make_map(&prm.tm_k, "k", k, p->k, p->b, p->h_kv, p->s_kv, p->d, p->in_dtype, 128)) != SDPA_OK) return st;
  if ((st = make_map(&prm.tm_v, "v", v, p->v, p->b, p->h_kv, p->s_kv, p->d, p->in_dtype, 128)) != SDPA_OK) return st;
  if ((st = make_map(&prm.tm_o, "o", o, p->o, p->b, p->h_q, p->s_q, p->d, p->out_dtype, 128)) != SDPA_OK) return st;
  if (p->bias != nullptr && p->d <= 128) {
    // Bias tiles for the forward kernel: [nb][nh][s_q][s_kv] (broadcast dimensions have size
    // 1), boxes of 128 rows x 64 keys (128 bytes), 128-byte swizzle.
    auto fn = encode_fn();
    if (fn == nullptr) return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const sdpa_strides_t& bs = p->bias_strides;
    const int64_t nb = bs.b == 0 ? 1 : p->b, nh = bs.h == 0 ? 1 : p->h_q;
    const int64_t row = p->s_q > 1 ? bs.s * 2 : ((int64_t)p->s_kv * 2 + 15) / 16 * 16;
    const int64_t head = nh > 1 ? bs.h * 2 : ((int64_t)p->s_q * row + 15) / 16 * 16;
    const int64_t batch = nb > 1 ? bs.b * 2 : ((int64_t)nh * head + 15) / 16 * 16;
    cuuint64_t dims[4] = {(cuuint64_t)p->s_kv, (cuuint64_t)p->s_q, (cuuint64_t)nh, (cuuint64_t)nb};
    cuuint64_t strides[3] = {(cuuint64_t)row, (cuuint64_t)head, (cuuint64_t)batch};
    cuuint32_t box[4] = {64, 128, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(&prm.tm_bias, map_dtype(p->in_dtype), 4, const_cast<void*>(p->bias), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(SDPA_ERR_LAYOUT, "bias: cuTensorMapEncodeTiled rejected the view (CUresult %d)", (int)r);
  }
  prm.lse = lse;
  prm.descale_q = p->descale_q;
  prm.descale_k = p->descale_k;
  prm.descale_v = p->descale_v;
  prm.b = p->b;
  prm.h_q = p->h_q;
  prm.h_kv = p->h_kv;
  prm.s_q = p->s_q;
  prm.s_kv = p->s_kv;
  prm.group = p->h_q / p->h_kv;
  prm.causal = p->causal != 0;
  prm.bottom_right = p->causal == 2;
  prm.seq_lens_q = p->seq_lens_q;
  prm.seq_lens_kv = p->seq_lens_kv;
  prm.alibi = p->alibi;
  prm.alibi_slopes = p->alibi ? p->alibi_slopes : nullptr;
  prm.drop_scale = drop_scale_of(p);
  prm.drop_rows = p->dropout_p > 0.f ? p->dropout_mask : nullptr;
  prm.drop_kv_words = words_of(p->s_kv);
  prm.bias = p->bias;
  prm.bias_sb = p->bias_strides.b;
  prm.bias_sh = p->bias_strides.h;
  prm.bias_ss = p->bias_strides.s;
  prm.wait_limit = wait_limit_cycles();
  const bool plain = !prm.alibi && !prm.drop_rows && !prm.bias;
  prm.one_tile = sdpa::fwd_prefer_one_tile(p->b, p->h_q, p->s_q, p->d, p->in_dtype, plain, num_sms()) ? 1 : 0;
  // With d <= 128 the bias instances run one Q tile per CTA (their bias tiles take the shared
  // memory of a second one).
  if (p->bias != nullptr && p->d <= 128) prm.one_tile = 1;
  // SDPA_FWD_Q_TILES=1 or 2 overrides the choice where both schedules exist (plain 16-bit,
  // d <= 128): a switch for testing and tuning.
  if (const char* qt = std::getenv("SDPA_FWD_Q_TILES")) {
    if (plain && p->in_dtype != SDPA_DTYPE_E4M3 && p->d <= 128 && (qt[0] == '1' || qt[0] == '2'))
      prm.one_tile = qt[0] == '1' ? 1 : 0;
  }
  const int rows_per_cta = 128 * (prm.one_tile ? 1 : sdpa::fwd_q_tiles(p->d, p->in_dtype));
  prm.num_m_blocks = (p->s_q + rows_per_cta - 1) / rows_per_cta;
  const long long units = static_cast<long long>(p->b) * p->h_q * prm.num_m_blocks;
  prm.ctas = sdpa::fwd_persistent_ctas(units, p->s_kv, p->d, p->in_dtype, plain, num_sms());
  // SDPA_FWD_PERSIST=N overrides the choice where both schedules exist (plain 16-bit,
  // d <= 128): 0 = one CTA per work unit, N >= 1 = min(N, units) CTAs walking the units (a
  // switch for testing and tuning).
  if (const char* ps = std::getenv("SDPA_FWD_PERSIST")) {
    const long long n = atoll(ps);
    if (plain && p->in_dtype != SDPA_DTYPE_E4M3 && p->d <= 128 && n >= 0)
      prm.ctas = static_cast<int>(n < units ? n : units);
  }
  prm.scale_log2 = scale_log2_of(p->attn_scale);
  prm.negate_scores = p->attn_scale < 0.f ? 1 : 0;
  if ((int64_t)p->b * p->h_q * prm.num_m_blocks > 0x7fffffff)
    return fail(SDPA_ERR_UNSUPPORTED, "grid too large");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (log_level() >= 1)
    fprintf(stderr, "[sdpa] fwd b=%d h_q=%d h_kv=%d s_q=%d s_kv=%d d=%d dt=%d causal=%d units=%lld "
            "(%d query tile(s) each) ctas=%lld%s\n",
            p->b, p->h_q, p->h_kv, p->s_q, p->s_kv, p->d, p->in_dtype, p->causal, units,
            prm.one_tile ? 1 : sdpa::fwd_q_tiles(p->d, p->in_dtype), prm.ctas ? (long long)prm.ctas : units,
            prm.ctas ? " persistent" : "");
  cudaError_t e = sdpa::launch_fwd(prm, p->d, p->in_dtype, p->out_dtype, stream);
  return finish_launch(e, stream, "sdpa_fwd");
}

sdpa_status_t sdpa_bwd(const sdpa_problem_t* p, const void* q, const void* k, const void* v,
                       const void* o, const void* dout, const float* lse, void* dq, void* dk,
                       void* dv, void* workspace, size_t workspace_bytes, void* stream_) {
  sdpa_status_t st = check_problem(p, true);
  if (st != SDPA_OK) return st;
  const bool fp8 = p->in_dtype == SDPA_DTYPE_E4M3;
  const int cdt = fp8 ? p->out_dtype : p->in_dtype;   // dtype the kernels compute in
  const int es = 2, es_in = fp8 ? 1 : 2;
  if ((st = check_view("q", q, p->q, p->b, p->h_q, p->s_q, p->d, es_in)) != SDPA_OK) return st;
  if ((st = check_view("k", k, p->k, p->b, p->h_kv, p->s_kv, p->d, es_in)) != SDPA_OK) return st;
  if ((st = check_view("v", v, p->v, p->b, p->h_kv, p->s_kv, p->d, es_in)) != SDPA_OK) return st;
  if ((st = check_view("o", o, p->o, p->b, p->h_q, p->s_q, p->d, es)) != SDPA_OK) return st;
  if ((st = check_view("dout", dout, p->dout, p->b, p->h_q, p->s_q, p->d, es_in)) != SDPA_OK) return st;
  if ((st = check_view("dq", dq, p->dq, p->b, p->h_q, p->s_q, p->d, es)) != SDPA_OK) return st;
  if ((st = check_view("dk", dk, p->dk, p->b, p->h_kv, p->s_kv, p->d, es)) != SDPA_OK) return st;
  if ((st = check_view("dv", dv, p->dv, p->b, p->h_kv, p->s_kv, p->d, es)) != SDPA_OK) return st;
  if (lse == nullptr) return fail(SDPA_ERR_INVALID_ARG, "lse: null pointer (the backward pass needs the forward statistics)");
  if (reinterpret_cast<uintptr_t>(lse) % 4 != 0) return fail(SDPA_ERR_LAYOUT, "lse must be 4-byte aligned");
  if ((st = check_drop_mask(p, p->dropout_mask_t, "dropout_mask_t")) != SDPA_OK) return st;
  const size_t need = bwd_total_workspace(p);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(SDPA_ERR_WORKSPACE, "workspace of %zu bytes required, %zu given%s", need,
                workspace_bytes, workspace ? "" : " (NULL)");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(SDPA_ERR_WORKSPACE, "workspace must be 256-byte aligned");

  sdpa::BwdParams prm;
  memset(&prm, 0, sizeof(prm));
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // FP8: widen Q, K, V and dO exactly into dense 16-bit copies after the scratch; the kernels
  // read those (the descales are folded into their scale factors).
  sdpa_strides_t sq = p->q, sk = p->k, sv = p->v, sdo = p->dout;
  if (fp8) {
    size_t off_k, off_v, off_do;
    widen_bytes(p, &off_k, &off_v, &off_do);
    uint8_t* wbase = static_cast<uint8_t*>(workspace) +
                     ((sdpa::bwd_workspace_bytes(p->b, p->h_q, p->h_kv, p->s_q, p->s_kv, p->d) + 255) & ~size_t(255));
    const sdpa_strides_t dq_st = {(int64_t)p->h_q * p->s_q * p->d, (int64_t)p->s_q * p->d, p->d, 1};
    const sdpa_strides_t dkv_st = {(int64_t)p->h_kv * p->s_kv * p->d, (int64_t)p->s_kv * p->d, p->d, 1};
    struct W { const void* src; const sdpa_strides_t* st; int h, s, e5m2; uint8_t* dst; };
    const W ws4[4] = {{q, &p->q, p->h_q, p->s_q, 0, wbase}, {k, &p->k, p->h_kv, p->s_kv, 0, wbase + off_k},
                      {v, &p->v, p->h_kv, p->s_kv, 0, wbase + off_v},
                      {dout, &p->dout, p->h_q, p->s_q, p->dout_dtype == SDPA_DTYPE_E5M2, wbase + off_do}};
    for (const W& w : ws4) {
      cudaError_t e = sdpa::launch_fp8_widen(w.src, w.st->b, w.st->h, w.st->s, p->b, w.h, w.s, p->d, w.e5m2,
                                             w.dst, cdt, stream);
      if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "FP8 widening launch failed: %s", cudaGetErrorString(e));
    }
    q = ws4[0].dst; k = ws4[1].dst; v = ws4[2].dst; dout = ws4[3].dst;
    sq = dq_st; sk = dkv_st; sv = dkv_st; sdo = dq_st;
    prm.descale_q = p->descale_q;
    prm.descale_k = p->descale_k;
    prm.descale_v = p->descale_v;
    prm.descale_do = p->descale_do;
  }
  if (p->bias != nullptr) {
    // The compute threads own key rows: give them a transposed, dense copy of the bias.
    const size_t base = (sdpa::bwd_workspace_bytes(p->b, p->h_q, p->h_kv, p->s_q, p->s_kv, p->d) + 255) & ~size_t(255);
    uint8_t* bt = static_cast<uint8_t*>(workspace) + base + widen_bytes(p, nullptr, nullptr, nullptr);
    prm.bias_nb = p->bias_strides.b == 0 ? 1 : p->b;
    prm.bias_nh = p->bias_strides.h == 0 ? 1 : p->h_q;
    // Causal without per-batch lengths: tiles that no query can see are left unwritten.
    const int skip = p->causal != 0 && !p->seq_lens_q && !p->seq_lens_kv;
    const int off = p->causal == 2 ? p->s_kv - p->s_q : 0;
    cudaError_t e = sdpa::launch_bias_transpose(p->bias, p->bias_strides.b, p->bias_strides.h, p->bias_strides.s,
                                                prm.bias_nb, prm.bias_nh, p->s_q, p->s_kv,
                                                (p->s_q + 127) / 128 * 128, skip, off, bt, stream);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "bias transpose launch failed: %s", cudaGetErrorString(e));
    prm.bias_t = bt;
    if (p->dbias != nullptr) {
      float* acc = reinterpret_cast<float*>(bt + bias_t_bytes(p));
      cudaError_t e2 = cudaMemsetAsync(acc, 0, dbias_acc_bytes(p), stream);
      if (e2 != cudaSuccess) return fail(SDPA_ERR_CUDA, "dbias accumulator clear failed: %s", cudaGetErrorString(e2));
      prm.dbias_acc = acc;
    }
  }
  // d = 256 walks 64-row query blocks (its kernel keeps only half of d of dK/dV in TMEM).
  const int q_rows = p->d == 256 ? 64 : 128;
  if ((st = make_map(&prm.tm_q, "q", q, sq, p->b, p->h_q, p->s_q, p->d, cdt, q_rows)) != SDPA_OK) return st;
  if ((st = make_map(&prm.tm_k, "k", k, sk, p->b, p->h_kv, p->s_kv, p->d, cdt, 128)) != SDPA_OK) return st;
  if ((st = make_map(&prm.tm_v, "v", v, sv, p->b, p->h_kv, p->s_kv, p->d, cdt, 128)) != SDPA_OK) return st;
  if ((st = make_map(&prm.tm_do, "dout", dout, sdo, p->b, p->h_q, p->s_q, p->d, cdt, q_rows)) != SDPA_OK) return st;
  if ((st = make_map(&prm.tm_dk, "dk", dk, p->dk, p->b, p->h_kv, p->s_kv, p->d, p->out_dtype, 128)) != SDPA_OK) return st;
  if ((st = make_map(&prm.tm_dv, "dv", dv, p->dv, p->b, p->h_kv, p->s_kv, p->d, p->out_dtype, 128)) != SDPA_OK) return st;
  const int s_q_pad = (p->s_q + 127) / 128 * 128;
  const size_t acc_bytes = align256((size_t)p->b * p->h_q * s_q_pad * p->d * 4);
  {
    // fp32 dQ accumulator [b*h_q*s_q_pad][d]: target of the kernel's TMA reduce-add, in
    // 32-column (128-byte) chunks of 128 rows.
    auto fn = encode_fn();
    if (fn == nullptr) return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    // d = 256 keeps the accumulator transposed, [b*h_q*d][s_q_pad] (its kernel produces dQᵀ).
    const bool tr = p->d == 256;
    cuuint64_t dims[2] = {tr ? (cuuint64_t)s_q_pad : (cuuint64_t)p->d,
                          tr ? (cuuint64_t)p->b * p->h_q * p->d : (cuuint64_t)p->b * p->h_q * s_q_pad};
    cuuint64_t strides[1] = {tr ? (cuuint64_t)s_q_pad * 4 : (cuuint64_t)p->d * 4};
    cuuint32_t box[2] = {32, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(&prm.tm_dqacc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, workspace, dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(SDPA_ERR_LAYOUT, "dQ accumulator: cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  }
  const size_t vec_bytes = align256((size_t)p->b * p->h_q * s_q_pad * 4);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  prm.o = o;
  prm.dout = dout;
  prm.lse = lse;
  prm.dq = dq;
  prm.dq_acc = reinterpret_cast<float*>(ws);
  prm.delta = reinterpret_cast<float*>(ws + acc_bytes);
  prm.lse2 = reinterpret_cast<float*>(ws + acc_bytes + vec_bytes);
  prm.o_sb = p->o.b; prm.o_sh = p->o.h; prm.o_ss = p->o.s;
  prm.do_sb = sdo.b; prm.do_sh = sdo.h; prm.do_ss = sdo.s;
  prm.dq_sb = p->dq.b; prm.dq_sh = p->dq.h; prm.dq_ss = p->dq.s;
  prm.b = p->b;
  prm.h_q = p->h_q;
  prm.h_kv = p->h_kv;
  prm.s_q = p->s_q;
  prm.s_kv = p->s_kv;
  prm.d = p->d;
  prm.group = p->h_q / p->h_kv;
  prm.causal = p->causal != 0;
  prm.bottom_right = p->causal == 2;
  prm.seq_lens_q = p->seq_lens_q;
  prm.seq_lens_kv = p->seq_lens_kv;
  prm.alibi = p->alibi;
  prm.alibi_slopes = p->alibi ? p->alibi_slopes : nullptr;
  prm.drop_scale = drop_scale_of(p);
  prm.drop_cols = p->dropout_p > 0.f ? p->dropout_mask_t : nullptr;
  prm.drop_q_words = words_of(p->s_q);
  prm.s_q_pad = s_q_pad;
  prm.wait_limit = wait_limit_cycles();
  prm.scale = p->attn_scale;
  prm.scale_log2 = p->attn_scale * 1.4426950408889634f;
  prm.kv_split = sdpa::bwd_kv_split(p->b, p->h_q, p->h_kv, p->s_kv);
  prm.heads_per_split = (prm.group + prm.kv_split - 1) / prm.kv_split;
  prm.s_kv_pad = (p->s_kv + 127) / 128 * 128;
  prm.dk = dk;
  prm.dv = dv;
  prm.dk_sb = p->dk.b; prm.dk_sh = p->dk.h; prm.dk_ss = p->dk.s;
  prm.dv_sb = p->dv.b; prm.dv_sh = p->dv.h; prm.dv_ss = p->dv.s;
  if (prm.kv_split > 1) {
    const size_t kv_bytes = align256((size_t)p->b * p->h_kv * prm.s_kv_pad * p->d * 4);
    prm.dk_acc = reinterpret_cast<float*>(ws + acc_bytes + 2 * vec_bytes);
    prm.dv_acc = reinterpret_cast<float*>(ws + acc_bytes + 2 * vec_bytes + kv_bytes);
  }
  // The per-row passes put (batch, head) on grid.y.
  if ((int64_t)p->b * p->h_q > 65535 ||
      (int64_t)p->b * p->h_kv * prm.kv_split * ((p->s_kv + 127) / 128) > 0x7fffffff)
    return fail(SDPA_ERR_UNSUPPORTED, "grid too large (b*h_q must be <= 65535 for the backward pass)");
  if (log_level() >= 1)
    fprintf(stderr, "[sdpa] bwd b=%d h_q=%d h_kv=%d s_q=%d s_kv=%d d=%d dt=%d causal=%d ws=%zu\n",
            p->b, p->h_q, p->h_kv, p->s_q, p->s_kv, p->d, p->in_dtype, p->causal, need);
  cudaError_t e = sdpa::launch_bwd(prm, cdt, stream);
  if (e == cudaSuccess && prm.dbias_acc != nullptr)
    e = sdpa::launch_dbias_convert(prm.dbias_acc, prm.bias_nb, prm.bias_nh, p->s_q, p->s_kv, s_q_pad, p->dbias,
                                   p->dbias_strides.b, p->dbias_strides.h, p->dbias_strides.s, cdt, stream);
  return finish_launch(e, stream, "sdpa_bwd");
}

}  // extern "C"

// Scratch for sdpa_bwd_noalloc: a fixed device array, so callers that cannot allocate still
// get a backward pass.  In host code its name is only a stand-in; the device address comes
// from cudaGetSymbolAddress, once per device, with that device current.
static __device__ __align__(256) uint8_t g_noalloc_scratch[SDPA_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

extern "C" {

sdpa_status_t sdpa_bwd_noalloc(const sdpa_problem_t* p, const void* q, const void* k,
                               const void* v, const void* o, const void* dout, const float* lse,
                               void* dq, void* dk, void* dv, void* stream) {
  sdpa_status_t st = check_problem(p, true);
  if (st != SDPA_OK) return st;
  // The whole workspace sdpa_bwd needs: the base scratch plus, where the problem asks for
  // them, the widened FP8 copies, the transposed bias and the bias-gradient accumulator.
  const size_t need = bwd_total_workspace(p);
  if (need > SDPA_NOALLOC_SCRATCH_BYTES)
    return fail(SDPA_ERR_UNSUPPORTED,
                "sdpa_bwd_noalloc: this problem needs %zu bytes of scratch but the built-in "
                "scratch holds %zu; call sdpa_bwd with a workspace instead",
                need, (size_t)SDPA_NOALLOC_SCRATCH_BYTES);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "sdpa_bwd_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(SDPA_ERR_UNSUPPORTED, "sdpa_bwd_noalloc: device %d out of range", dev);
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || ptr == nullptr)
        return fail(SDPA_ERR_CUDA, "sdpa_bwd_noalloc: cudaGetSymbolAddress of the scratch failed: %s",
                    cudaGetErrorString(e));
      g_noalloc_ptr[dev] = ptr;
    }
    scratch = g_noalloc_ptr[dev];
  }
  return sdpa_bwd(p, q, k, v, o, dout, lse, dq, dk, dv, scratch, SDPA_NOALLOC_SCRATCH_BYTES, stream);
}

sdpa_status_t sdpa_dropout_mask_size(const sdpa_problem_t* p, size_t* bytes, size_t* bytes_t) {
  if (p == nullptr || bytes == nullptr || bytes_t == nullptr)
    return fail(SDPA_ERR_INVALID_ARG, "problem, bytes and bytes_t must not be NULL");
  if (p->b < 1 || p->h_q < 1 || p->s_q < 1 || p->s_kv < 1)
    return fail(SDPA_ERR_INVALID_ARG, "sizes must be >= 1 (b=%d h_q=%d s_q=%d s_kv=%d)", p->b, p->h_q,
                p->s_q, p->s_kv);
  const size_t bh = static_cast<size_t>(p->b) * p->h_q;
  *bytes = bh * p->s_q * words_of(p->s_kv) * 4;
  *bytes_t = bh * p->s_kv * words_of(p->s_q) * 4;
  return ok();
}

sdpa_status_t sdpa_dropout_mask(const sdpa_problem_t* p, uint64_t seed, uint64_t offset, uint32_t* mask,
                                uint32_t* mask_t, void* stream_) {
  size_t n, n_t;
  sdpa_status_t st = sdpa_dropout_mask_size(p, &n, &n_t);
  if (st != SDPA_OK) return st;
  if (!(p->dropout_p >= 0.f && p->dropout_p < 1.f))
    return fail(SDPA_ERR_INVALID_ARG, "dropout_p must be in [0, 1), got %g", p->dropout_p);
  if ((mask && reinterpret_cast<uintptr_t>(mask) % 16) || (mask_t && reinterpret_cast<uintptr_t>(mask_t) % 16))
    return fail(SDPA_ERR_LAYOUT, "mask and mask_t must be 16-byte aligned");
  if (static_cast<int64_t>(p->b) * p->h_q > 65535)
    return fail(SDPA_ERR_UNSUPPORTED, "b*h_q = %lld exceeds 65535", static_cast<long long>(p->b) * p->h_q);
  if (mask == nullptr && mask_t == nullptr) return ok();
  sdpa::DropoutParams prm;
  prm.rows = mask;
  prm.cols = mask_t;
  prm.seed = seed;
  prm.offset = offset;
  const double t = std::floor(static_cast<double>(p->dropout_p) * 65536.0 + 0.5);
  prm.threshold = static_cast<uint32_t>(t > 65536.0 ? 65536.0 : t);
  prm.s_q = p->s_q;
  prm.s_kv = p->s_kv;
  prm.kv_words = words_of(p->s_kv);
  prm.q_words = words_of(p->s_q);
  // Causal without per-batch lengths: tiles wholly above the diagonal are never read.
  prm.skip_above = (p->causal == 1 || p->causal == 2) && !p->seq_lens_q && !p->seq_lens_kv;
  prm.diag_off = p->causal == 2 ? p->s_kv - p->s_q : 0;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaError_t e = sdpa::launch_dropout_mask(prm, p->b * p->h_q, stream);
  return finish_launch(e, stream, "sdpa_dropout_mask");
}

const char* sdpa_last_error_string(void) { return g_last_error.c_str(); }

sdpa_status_t sdpa_device_error(uint32_t* flags) {
  if (flags == nullptr) return fail(SDPA_ERR_INVALID_ARG, "flags is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "synchronize failed: %s", cudaGetErrorString(e));
  *flags = sdpa::fwd_take_device_error() | sdpa::bwd_take_device_error();
  return ok();
}

int sdpa_version(void) { return 100; }

size_t sdpa_problem_struct_size(void) { return sizeof(sdpa_problem_t); }

}  // extern "C"
