// C ABI of libtokengate.so (declared in include/tokengate.h): argument
// validation, TMA descriptor encoding, the device status word and kernel
// launches.  Every compute entry point validates on the host and launches
// nothing when an argument is invalid.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "tg_internal.h"
#include "../../include/tokengate.h"

namespace tg {

// The status word lives in this module's static device memory (one copy per
// device that loads the library); kernels receive its device address.
__device__ unsigned int g_device_status;

namespace {

thread_local std::string g_last_error;
long long g_watchdog_cycles = 1LL << 31;

tg_status fail(tg_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

tg_status ok() {
  g_last_error.clear();
  return TG_OK;
}

tg_status cuda_fail(cudaError_t e, const char* where) {
  return fail(TG_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready = false;
  unsigned int* status = nullptr;
  int num_sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

tg_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(TG_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    d.status = static_cast<unsigned int*>(p);
    d.ready = true;
  }
  *out = &d;
  return TG_OK;
}

// ---- TMA descriptors -------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor of `rank` dims (innermost first), 128-byte swizzle.
tg_status make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                   const uint32_t* box, const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(TG_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5];
  cuuint32_t es[5];
  for (int i = 0; i < rank; ++i) { gd[i] = dims[i]; bx[i] = box[i]; es[i] = 1; }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs,
                  bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TG_ERR_INVALID_ARG, "tensor map for %s rejected (CUresult %d)", what, (int)r);
  return TG_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace tg

using namespace tg;

extern "C" {

const char* tg_version(void) { return "tokengate-b300 0.1 (sm_103a)"; }

const char* tg_last_error_string(void) { return g_last_error.c_str(); }

void tg_set_watchdog_cycles(long long cycles) { g_watchdog_cycles = cycles > 0 ? cycles : (1LL << 31); }

tg_status tg_check_device_status(cudaStream_t stream) {
  DeviceInfo* di = nullptr;
  tg_status s = device_info(&di);
  if (s != TG_OK) return s;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "read status");
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "clear status");
  if (v == kStatusTimeout) return fail(TG_ERR_TIMEOUT, "a device-side wait exceeded its cycle limit");
  if (v == kStatusIndex) return fail(TG_ERR_DEVICE_INDEX, "a device-side index or size check failed");
  if (v != 0) return fail(TG_ERR_CUDA, "unknown device status %u", v);
  return ok();
}

// the gate on the document prefix (prunable null) or on a per-row mask
static tg_status gate_score_any(const void* x_bf16, int64_t n_rows, int32_t d, const int32_t* cu_seqlens,
                                const int32_t* n_doc, int32_t batch, bool masked, const uint8_t* prunable,
                                const void* w1_bf16,
                                const float* b1, const void* w2_bf16, float b2, int32_t h, float* s_out,
                                void* topk_ws, size_t topk_ws_bytes, cudaStream_t stream) {
  if (n_rows < 0 || n_rows > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "n_rows out of range");
  if (!masked && batch < 1) return fail(TG_ERR_INVALID_ARG, "batch must be >= 1");
  if (d < 64 || d % 64 != 0 || d > (1 << 20)) return fail(TG_ERR_INVALID_ARG, "d must be a positive multiple of 64");
  if (h < 16 || h > 256 || h % 16 != 0) return fail(TG_ERR_INVALID_ARG, "h must be a multiple of 16 in [16, 256]");
  if ((!masked && (!cu_seqlens || !n_doc)) || !w1_bf16 || !w2_bf16)
    return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (masked && topk_ws && (!cu_seqlens || batch < 1))
    return fail(TG_ERR_INVALID_ARG, "a top-K workspace needs cu_seqlens and batch >= 1");
  if (n_rows == 0) return ok();
  if (masked && !prunable) return fail(TG_ERR_INVALID_ARG, "null prunable mask");
  if (!x_bf16 || !s_out) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(x_bf16) || !aligned16(w1_bf16)) return fail(TG_ERR_INVALID_ARG, "x and w1 must be 16-byte aligned");
  if (!std::isfinite(b2)) return fail(TG_ERR_INVALID_ARG, "b2 must be finite");
  if (topk_ws) {
    if (batch > kTopkMaxHistBatch) return fail(TG_ERR_INVALID_ARG, "a top-K workspace needs batch <= %d", kTopkMaxHistBatch);
    if (topk_ws_bytes < tg_topk_workspace_size(batch))
      return fail(TG_ERR_WORKSPACE, "top-K workspace of %zu bytes needed, %zu given", tg_topk_workspace_size(batch),
                  topk_ws_bytes);
    if (!aligned16(topk_ws)) return fail(TG_ERR_INVALID_ARG, "top-K workspace must be 16-byte aligned");
  }
  DeviceInfo* di = nullptr;
  tg_status s = device_info(&di);
  if (s != TG_OK) return s;
  CUtensorMap mx, mw;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(n_rows)};
    const uint64_t str[1] = {static_cast<uint64_t>(d) * 2};
    const uint32_t box[2] = {64, 128};
    if ((s = make_map(&mx, x_bf16, 2, dims, str, box, "x")) != TG_OK) return s;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(h)};
    const uint64_t str[1] = {static_cast<uint64_t>(d) * 2};
    // each CTA of a pair stages one half of W1's rows
    const uint32_t box[2] = {64, static_cast<uint32_t>(h / 2)};
    if ((s = make_map(&mw, w1_bf16, 2, dims, str, box, "w1")) != TG_OK) return s;
  }
  GateArgs a{};
  a.hist = static_cast<uint32_t*>(topk_ws);
  a.prunable = prunable;
  a.b1 = b1;
  a.w2 = static_cast<const __nv_bfloat16*>(w2_bf16);
  a.b2 = b2;
  a.cu_seqlens = cu_seqlens;
  a.n_doc = n_doc;
  a.batch = batch;
  a.n_rows = n_rows;
  a.d = d;
  a.h = h;
  a.s_out = s_out;
  a.status = di->status;
  a.watchdog = g_watchdog_cycles;
  a.num_sms = di->num_sms;
  cudaError_t e = launch_gate(mx, mw, a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "gate kernel launch");
  return ok();
}

size_t tg_topk_workspace_size(int32_t batch) {
  if (batch <= 0 || batch > kTopkMaxHistBatch) return 0;
  return static_cast<size_t>(batch) * kHistWords * sizeof(uint32_t);
}

tg_status tg_gate_score(const void* x_bf16, int64_t n_rows, int32_t d, const int32_t* cu_seqlens,
                        const int32_t* n_doc, int32_t batch, const void* w1_bf16, const float* b1,
                        const void* w2_bf16, float b2, int32_t h, float* s_out, void* topk_ws,
                        size_t topk_ws_bytes, cudaStream_t stream) {
  return gate_score_any(x_bf16, n_rows, d, cu_seqlens, n_doc, batch, false, nullptr, w1_bf16, b1, w2_bf16, b2, h,
                        s_out, topk_ws, topk_ws_bytes, stream);
}

tg_status tg_gate_score_masked(const void* x_bf16, int64_t n_rows, int32_t d, const uint8_t* prunable,
                               const void* w1_bf16, const float* b1, const void* w2_bf16, float b2, int32_t h,
                               float* s_out, const int32_t* cu_seqlens, int32_t batch, void* topk_ws,
                               size_t topk_ws_bytes, cudaStream_t stream) {
  if (!topk_ws) { cu_seqlens = nullptr; batch = 0; }
  return gate_score_any(x_bf16, n_rows, d, cu_seqlens, nullptr, batch, true, prunable, w1_bf16, b1, w2_bf16, b2, h,
                        s_out, topk_ws, topk_ws_bytes, stream);
}

tg_status tg_topk_select(const float* s, int64_t n_rows, const int32_t* cu_seqlens, const int32_t* n_doc,
                         const int32_t* k, int32_t batch, int32_t max_n_doc, int32_t* kept_idx,
                         int32_t* cu_kept, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (batch < 0 || batch > (1 << 24)) return fail(TG_ERR_INVALID_ARG, "batch out of range");
  if (n_rows < 0 || n_rows > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "n_rows out of range");
  if (max_n_doc < 0) return fail(TG_ERR_INVALID_ARG, "max_n_doc must be >= 0");
  if (batch == 0) return ok();
  if (workspace) {
    if (batch > kTopkMaxHistBatch) return fail(TG_ERR_INVALID_ARG, "a top-K workspace needs batch <= %d", kTopkMaxHistBatch);
    if (ws_bytes < tg_topk_workspace_size(batch))
      return fail(TG_ERR_WORKSPACE, "top-K workspace of %zu bytes needed, %zu given", tg_topk_workspace_size(batch),
                  ws_bytes);
    if (!aligned16(workspace)) return fail(TG_ERR_INVALID_ARG, "top-K workspace must be 16-byte aligned");
  }
  if (!cu_seqlens || !n_doc || !k || !cu_kept) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (n_rows > 0 && (!s || !kept_idx)) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  DeviceInfo* di = nullptr;
  tg_status st = device_info(&di);
  if (st != TG_OK) return st;
  TopkArgs a{};
  a.hist = static_cast<uint32_t*>(workspace);
  a.s = s;
  a.cu_seqlens = cu_seqlens;
  a.n_doc = n_doc;
  a.k = k;
  a.batch = batch;
  a.max_n_doc = max_n_doc;
  a.kept_capacity = INT64_MAX;
  a.kept_idx = kept_idx;
  a.cu_kept = cu_kept;
  a.status = di->status;
  cudaError_t e = launch_topk(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "top-K kernel launch");
  return ok();
}

tg_status tg_topk_select_masked(const float* s, int64_t n_rows, const int32_t* cu_seqlens, const uint8_t* prunable,
                                const int32_t* k, int32_t batch, int32_t max_len, int64_t kept_capacity,
                                int32_t* kept_idx, int32_t* cu_kept, int32_t* n_prunable, void* workspace,
                                size_t ws_bytes, cudaStream_t stream) {
  if (batch < 0 || batch > (1 << 24)) return fail(TG_ERR_INVALID_ARG, "batch out of range");
  if (batch > 0 && workspace) {
    if (batch > kTopkMaxHistBatch) return fail(TG_ERR_INVALID_ARG, "a top-K workspace needs batch <= %d", kTopkMaxHistBatch);
    if (ws_bytes < tg_topk_workspace_size(batch))
      return fail(TG_ERR_WORKSPACE, "top-K workspace of %zu bytes needed, %zu given", tg_topk_workspace_size(batch),
                  ws_bytes);
    if (!aligned16(workspace)) return fail(TG_ERR_INVALID_ARG, "top-K workspace must be 16-byte aligned");
  }
  if (n_rows < 0 || n_rows > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "n_rows out of range");
  if (max_len < 0) return fail(TG_ERR_INVALID_ARG, "max_len must be >= 0");
  if (kept_capacity < 0) return fail(TG_ERR_INVALID_ARG, "kept_capacity must be >= 0");
  if (batch == 0) return ok();
  if (!cu_seqlens || !k || !cu_kept || !n_prunable) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (n_rows > 0 && (!s || !prunable || (kept_capacity > 0 && !kept_idx)))
    return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  DeviceInfo* di = nullptr;
  tg_status st = device_info(&di);
  if (st != TG_OK) return st;
  cudaError_t e = launch_topk_count(prunable, cu_seqlens, batch, n_prunable, di->status, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prunable count kernel launch");
  TopkArgs a{};
  a.hist = static_cast<uint32_t*>(workspace);
  a.s = s;
  a.cu_seqlens = cu_seqlens;
  a.n_doc = n_prunable;
  a.prunable = prunable;
  a.k = k;
  a.batch = batch;
  a.max_n_doc = max_len;
  a.kept_capacity = kept_capacity;
  a.kept_idx = kept_idx;
  a.cu_kept = cu_kept;
  a.status = di->status;
  e = launch_topk(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "top-K kernel launch");
  return ok();
}

tg_status tg_gather_kept(const void* x_bf16, int64_t n_rows, int32_t d, const float* s,
                         const int32_t* cu_seqlens, const int32_t* kept_idx, const int32_t* cu_kept,
                         int32_t batch, int64_t n_kept, void* x_kept_bf16, int32_t* pos_kept, float* s_kept,
                         cudaStream_t stream) {
  if (batch < 1) return fail(TG_ERR_INVALID_ARG, "batch must be >= 1");
  if (n_kept < 0 || n_kept > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "n_kept out of range");
  if (n_rows < 0 || n_rows > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "n_rows out of range");
  if (d < 8 || d % 8 != 0) return fail(TG_ERR_INVALID_ARG, "d must be a positive multiple of 8");
  if (!cu_seqlens || !cu_kept) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (n_kept == 0) return ok();
  if (!kept_idx) return fail(TG_ERR_INVALID_ARG, "null kept_idx");
  if (x_kept_bf16 && (!x_bf16 || !aligned16(x_bf16) || !aligned16(x_kept_bf16)))
    return fail(TG_ERR_INVALID_ARG, "x and x_kept must be non-null and 16-byte aligned");
  if (s_kept && !s) return fail(TG_ERR_INVALID_ARG, "s_kept requested without s");
  DeviceInfo* di = nullptr;
  tg_status st = device_info(&di);
  if (st != TG_OK) return st;
  GatherArgs a{};
  a.x = x_bf16;
  a.n_rows = n_rows;
  a.d = d;
  a.s = s;
  a.cu_seqlens = cu_seqlens;
  a.kept_idx = kept_idx;
  a.cu_kept = cu_kept;
  a.batch = batch;
  a.n_kept = n_kept;
  a.x_kept = x_kept_bf16;
  a.pos_kept = pos_kept;
  a.s_kept = s_kept;
  a.status = di->status;
  a.watchdog = g_watchdog_cycles;
  a.num_sms = di->num_sms;
  cudaError_t e = launch_gather(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch");
  return ok();
}

size_t tg_attention_workspace_size(int64_t n_kept, int32_t hq, int32_t hkv, int32_t head_dim,
                                   int32_t has_k_cache) {
  if (n_kept <= 0 || hq <= 0 || hkv <= 0 || head_dim <= 0) return 0;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  size_t b = up(static_cast<size_t>(n_kept) * hq * head_dim * 2);
  if (!has_k_cache) b += up(static_cast<size_t>(n_kept) * hkv * head_dim * 2);
  return b;
}

// shared argument checks of the attention calls
// RoPE rates theta^(-2i/D) / (2 pi) in turns per position, i < D/2, each as
// an fp32 pair hi + lo (formed in fp64).
static void rope_turns(float rope_theta, int32_t head_dim, RopeFreqs* f) {
  for (int i = 0; i < head_dim / 2; ++i) {
    const double t = std::pow(static_cast<double>(rope_theta), -2.0 * i / head_dim) / (2.0 * 3.141592653589793);
    f->turns_hi[i] = static_cast<float>(t);
    f->turns_lo[i] = static_cast<float>(t - static_cast<double>(f->turns_hi[i]));
  }
}

static tg_status check_attention_shape(int32_t batch, int64_t n_kept, int32_t hq, int32_t hkv, int32_t head_dim,
                                       const int32_t* cu_kept) {
  if (batch < 1) return fail(TG_ERR_INVALID_ARG, "batch must be >= 1");
  if (n_kept < 0 || n_kept > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "n_kept out of range");
  if (hq < 1 || hkv < 1 || hq % hkv != 0) return fail(TG_ERR_INVALID_ARG, "hq must be a positive multiple of hkv");
  if (head_dim != 64 && head_dim != 128) return fail(TG_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (!cu_kept) return fail(TG_ERR_INVALID_ARG, "null cu_kept");
  return TG_OK;
}

tg_status tg_rope_qk(const void* q, const void* k, const int32_t* pos_kept, float rope_theta, const int32_t* cu_kept,
                     int32_t batch, int64_t n_kept, int32_t hq, int32_t hkv, int32_t head_dim, void* q_out,
                     void* k_out, cudaStream_t stream) {
  tg_status st = check_attention_shape(batch, n_kept, hq, hkv, head_dim, cu_kept);
  if (st != TG_OK) return st;
  if (!(rope_theta > 0.0f) || !std::isfinite(rope_theta)) return fail(TG_ERR_INVALID_ARG, "rope_theta must be positive");
  if (n_kept == 0) return ok();
  if (!q || !k || !pos_kept || !q_out || !k_out) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_out) || !aligned16(k_out))
    return fail(TG_ERR_INVALID_ARG, "q, k, q_out and k_out must be 16-byte aligned");
  if (q_out == q || k_out == k) return fail(TG_ERR_INVALID_ARG, "q_out and k_out must not alias q and k");
  DeviceInfo* di = nullptr;
  st = device_info(&di);
  if (st != TG_OK) return st;
  RopeFreqs f{};
  rope_turns(rope_theta, head_dim, &f);
  RopeArgs ra{};
  ra.q = q; ra.k = k; ra.pos = pos_kept; ra.cu_kept = cu_kept; ra.batch = batch; ra.n_kept = n_kept;
  ra.hq = hq; ra.hkv = hkv; ra.head_dim = head_dim; ra.q_out = q_out; ra.k_out = k_out;
  ra.status = di->status; ra.num_sms = di->num_sms;
  const cudaError_t e = launch_rope(ra, f, stream);
  if (e != cudaSuccess) return cuda_fail(e, "RoPE kernel launch");
  return ok();
}

tg_status tg_gated_attention_rotated(const void* q_rot, const void* k_rot, const void* v, const int32_t* pos_kept,
                                     const float* s_kept, const float* gain, float tau, const int32_t* cu_kept,
                                     int32_t batch, int64_t n_kept, int32_t max_kept, int32_t hq, int32_t hkv,
                                     int32_t head_dim, void* o, float* lse, cudaStream_t stream) {
  tg_status st = check_attention_shape(batch, n_kept, hq, hkv, head_dim, cu_kept);
  if (st != TG_OK) return st;
  if (max_kept < 0) return fail(TG_ERR_INVALID_ARG, "max_kept must be >= 0");
  if (!(tau > 0.0f) || !std::isfinite(tau)) return fail(TG_ERR_INVALID_ARG, "tau must be positive and finite");
  if (n_kept == 0 || max_kept == 0) return ok();
  if (!q_rot || !k_rot || !v || !pos_kept || !s_kept || !gain || !o) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q_rot) || !aligned16(k_rot) || !aligned16(v) || !aligned16(o))
    return fail(TG_ERR_INVALID_ARG, "q_rot, k_rot, v and o must be 16-byte aligned");
  DeviceInfo* di = nullptr;
  st = device_info(&di);
  if (st != TG_OK) return st;
  CUtensorMap mq, mk, mv;
  const uint32_t box[3] = {64, 1, 128};
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(head_dim), static_cast<uint64_t>(hq), static_cast<uint64_t>(n_kept)};
    const uint64_t str[2] = {static_cast<uint64_t>(head_dim) * 2, static_cast<uint64_t>(hq) * head_dim * 2};
    if ((st = make_map(&mq, q_rot, 3, dims, str, box, "q'")) != TG_OK) return st;
  }
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(head_dim), static_cast<uint64_t>(hkv), static_cast<uint64_t>(n_kept)};
    const uint64_t str[2] = {static_cast<uint64_t>(head_dim) * 2, static_cast<uint64_t>(hkv) * head_dim * 2};
    if ((st = make_map(&mk, k_rot, 3, dims, str, box, "k'")) != TG_OK) return st;
    if ((st = make_map(&mv, v, 3, dims, str, box, "v")) != TG_OK) return st;
  }
  AttnArgs a{};
  a.pos = pos_kept; a.s_kept = s_kept; a.gain = gain; a.cu_kept = cu_kept; a.batch = batch;
  a.n_kept = n_kept; a.max_kept = max_kept; a.hq = hq; a.hkv = hkv; a.head_dim = head_dim;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / (std::sqrt(static_cast<double>(head_dim)) * tau));
  a.bias_unit = static_cast<float>(std::sqrt(static_cast<double>(head_dim)) * tau);
  a.o = o; a.lse = lse; a.status = di->status; a.watchdog = g_watchdog_cycles;
  const cudaError_t e = launch_attention(mq, mk, mv, a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
  return ok();
}

tg_status tg_gated_attention_fwd(const void* q, const void* k, const void* v, const int32_t* pos_kept,
                                 const float* s_kept, const float* gain, float tau, float rope_theta,
                                 const int32_t* cu_kept, int32_t batch, int64_t n_kept, int32_t max_kept,
                                 int32_t hq, int32_t hkv, int32_t head_dim, void* o, float* lse,
                                 void* k_cache, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
  tg_status st = check_attention_shape(batch, n_kept, hq, hkv, head_dim, cu_kept);
  if (st != TG_OK) return st;
  if (max_kept < 0) return fail(TG_ERR_INVALID_ARG, "max_kept must be >= 0");
  if (!(tau > 0.0f) || !std::isfinite(tau)) return fail(TG_ERR_INVALID_ARG, "tau must be positive and finite");
  if (!(rope_theta > 0.0f) || !std::isfinite(rope_theta)) return fail(TG_ERR_INVALID_ARG, "rope_theta must be positive");
  if (n_kept == 0) return ok();
  if (!q || !k || !v || !pos_kept || !s_kept || !gain || !o) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (k_cache && !aligned16(k_cache)))
    return fail(TG_ERR_INVALID_ARG, "q, k, v, o and k_cache must be 16-byte aligned");
  const size_t need = tg_attention_workspace_size(n_kept, hq, hkv, head_dim, k_cache ? 1 : 0);
  if (!workspace || workspace_bytes < need)
    return fail(TG_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(TG_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (max_kept == 0) return ok();
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* q_rot = ws;
  void* k_rot = k_cache;
  if (!k_rot) k_rot = ws + ((static_cast<size_t>(n_kept) * hq * head_dim * 2 + 255) & ~static_cast<size_t>(255));
  st = tg_rope_qk(q, k, pos_kept, rope_theta, cu_kept, batch, n_kept, hq, hkv, head_dim, q_rot, k_rot, stream);
  if (st != TG_OK) return st;
  return tg_gated_attention_rotated(q_rot, k_rot, v, pos_kept, s_kept, gain, tau, cu_kept, batch, n_kept, max_kept,
                                    hq, hkv, head_dim, o, lse, stream);
}

size_t tg_attention_bwd_workspace_size(int64_t n_kept, int32_t hq) {
  if (n_kept <= 0 || hq <= 0) return 0;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t plane = static_cast<size_t>(n_kept) * hq * 4;
  return up(plane) + 2 * up(2 * plane) + up(static_cast<size_t>(hq) * kBwdChunks * 2 * 4);
}

tg_status tg_gated_attention_bwd(const void* q_rot, const void* k_rot, const void* v, const void* o,
                                 const float* lse, const void* d_o, const int32_t* pos_kept, const float* s_kept,
                                 const float* gain, float tau, const int32_t* cu_kept, int32_t batch,
                                 int64_t n_kept, int32_t max_kept, int32_t hq, int32_t hkv, int32_t head_dim,
                                 float* d_s, float* d_gain, float* d_tau, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
  tg_status st = check_attention_shape(batch, n_kept, hq, hkv, head_dim, cu_kept);
  if (st != TG_OK) return st;
  if (hq / hkv > kBwdMaxGroup) return fail(TG_ERR_UNSUPPORTED, "hq / hkv must be at most %d", kBwdMaxGroup);
  if (hq > kBwdMaxHeads) return fail(TG_ERR_UNSUPPORTED, "hq must be at most %d", kBwdMaxHeads);
  if (max_kept < 0) return fail(TG_ERR_INVALID_ARG, "max_kept must be >= 0");
  if (!(tau > 0.0f) || !std::isfinite(tau)) return fail(TG_ERR_INVALID_ARG, "tau must be positive and finite");
  if (!d_gain || !d_tau || (n_kept > 0 && !d_s)) return fail(TG_ERR_INVALID_ARG, "null output pointer");
  if (n_kept == 0 || max_kept == 0) {
    // no sequence holds a row: every gradient is zero
    cudaError_t e = cudaMemsetAsync(d_gain, 0, static_cast<size_t>(hq) * 4, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_tau, 0, 4, stream);
    if (e == cudaSuccess && n_kept > 0) e = cudaMemsetAsync(d_s, 0, static_cast<size_t>(n_kept) * 4, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    return ok();
  }
  if (!q_rot || !k_rot || !v || !o || !lse || !d_o || !pos_kept || !s_kept || !gain)
    return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q_rot) || !aligned16(k_rot) || !aligned16(v) || !aligned16(o) || !aligned16(d_o))
    return fail(TG_ERR_INVALID_ARG, "q_rot, k_rot, v, o and d_o must be 16-byte aligned");
  const size_t need = tg_attention_bwd_workspace_size(n_kept, hq);
  if (!workspace || workspace_bytes < need)
    return fail(TG_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(TG_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  DeviceInfo* di = nullptr;
  st = device_info(&di);
  if (st != TG_OK) return st;
  // 2D views [n_kept rows, heads * head_dim columns]; a box is 64 columns of
  // one head by 128 keys (K, V) or 64 query rows (q', dO)
  CUtensorMap mq, mk, mv, mdo;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(hq) * head_dim, static_cast<uint64_t>(n_kept)};
    const uint64_t str[1] = {static_cast<uint64_t>(hq) * head_dim * 2};
    const uint32_t box[2] = {64, 64};
    if ((st = make_map(&mq, q_rot, 2, dims, str, box, "q'")) != TG_OK) return st;
    if ((st = make_map(&mdo, d_o, 2, dims, str, box, "dO")) != TG_OK) return st;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(hkv) * head_dim, static_cast<uint64_t>(n_kept)};
    const uint64_t str[1] = {static_cast<uint64_t>(hkv) * head_dim * 2};
    const uint32_t box[2] = {64, 128};
    if ((st = make_map(&mk, k_rot, 2, dims, str, box, "k'")) != TG_OK) return st;
    if ((st = make_map(&mv, v, 2, dims, str, box, "v")) != TG_OK) return st;
  }
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t plane = static_cast<size_t>(n_kept) * hq * 4;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AttnBwdArgs a{};
  a.o = o; a.d_o = d_o; a.lse = lse; a.pos = pos_kept; a.s_kept = s_kept; a.gain = gain; a.cu_kept = cu_kept;
  a.batch = batch; a.n_kept = n_kept; a.max_kept = max_kept; a.hq = hq; a.hkv = hkv; a.head_dim = head_dim;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / (std::sqrt(static_cast<double>(head_dim)) * tau));
  a.dtau_scale = static_cast<float>(-1.0 / (std::sqrt(static_cast<double>(head_dim)) * static_cast<double>(tau) * tau));
  a.delta = reinterpret_cast<float*>(ws);
  a.r_part = reinterpret_cast<float*>(ws + up(plane));
  a.t_part = reinterpret_cast<float*>(ws + up(plane) + up(2 * plane));
  a.part = reinterpret_cast<float*>(ws + up(plane) + 2 * up(2 * plane));
  a.ds = d_s; a.dgain = d_gain; a.dtau = d_tau;
  a.status = di->status; a.watchdog = g_watchdog_cycles; a.num_sms = di->num_sms;
  const cudaError_t e = launch_attention_bwd(mq, mk, mv, mdo, a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attention backward launch");
  return ok();
}

size_t tg_gated_delta_scan_workspace_size(int64_t n_kept, int32_t batch, int32_t hv, int32_t dk, int32_t dv) {
  if (batch < 1 || hv < 1 || n_kept < 0 || n_kept > 0x7FFFFFFF) return 0;
  if ((dk != 64 && dk != 128) || dv < 16 || dv > 128 || dv % 16 != 0) return 0;
  return delta_chunked_ws_bytes(n_kept, batch, hv, dk, dv);
}

tg_status tg_gated_delta_scan(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              const int32_t* cu_kept, int32_t batch, int64_t n_kept, int32_t hk, int32_t hv,
                              int32_t dk, int32_t dv, float scale, const float* initial_state, void* o,
                              float* final_state, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (batch < 1) return fail(TG_ERR_INVALID_ARG, "batch must be >= 1");
  if (n_kept < 0 || n_kept > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "n_kept out of range");
  if (hk < 1 || hv < 1 || hv % hk != 0) return fail(TG_ERR_INVALID_ARG, "hv must be a positive multiple of hk");
  if (dk != 64 && dk != 128) return fail(TG_ERR_UNSUPPORTED, "dk must be 64 or 128");
  if (dv < 16 || dv > 1024 || dv % 16 != 0) return fail(TG_ERR_INVALID_ARG, "dv must be a multiple of 16 in [16, 1024]");
  if (!(scale > 0.0f) || !std::isfinite(scale)) return fail(TG_ERR_INVALID_ARG, "scale must be positive and finite");
  if (!cu_kept) return fail(TG_ERR_INVALID_ARG, "null cu_kept");
  if (n_kept > 0 && (!q || !k || !v || !g || !beta || !o)) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (n_kept > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)))
    return fail(TG_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if ((initial_state && !aligned16(initial_state)) || (final_state && !aligned16(final_state)))
    return fail(TG_ERR_INVALID_ARG, "initial_state and final_state must be 16-byte aligned");
  const size_t ws_need = tg_gated_delta_scan_workspace_size(n_kept, batch, hv, dk, dv);
  const bool chunked = workspace != nullptr && ws_need > 0;
  if (chunked && workspace_bytes < ws_need) return fail(TG_ERR_WORKSPACE, "delta scan workspace too small");
  if (chunked && reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(TG_ERR_INVALID_ARG, "delta scan workspace must be 256-byte aligned");
  DeviceInfo* di = nullptr;
  tg_status st = device_info(&di);
  if (st != TG_OK) return st;
  ScanArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu_kept = cu_kept; a.batch = batch; a.n_kept = n_kept;
  a.hk = hk; a.hv = hv; a.dk = dk; a.dv = dv; a.scale = scale; a.initial_state = initial_state; a.o = o;
  a.final_state = final_state; a.status = di->status;
  a.ws = chunked ? workspace : nullptr;
  a.watchdog = g_watchdog_cycles;
  a.num_sms = di->num_sms;
  const cudaError_t e = chunked ? launch_delta_scan_chunked(a, stream) : launch_delta_scan(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "gated delta scan launch");
  return ok();
}

tg_status tg_rms_norm(const void* x, const void* w, int64_t rows, int32_t d, float eps, void* y,
                      cudaStream_t stream) {
  if (rows < 0) return fail(TG_ERR_INVALID_ARG, "rows must be >= 0");
  if (d < 8 || d % 8 != 0 || d > (1 << 16)) return fail(TG_ERR_INVALID_ARG, "d must be a multiple of 8 in [8, 65536]");
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(TG_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (rows == 0) return ok();
  if (!x || !w || !y) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return fail(TG_ERR_INVALID_ARG, "x, w and y must be 16-byte aligned");
  DeviceInfo* di = nullptr;
  tg_status st = device_info(&di);
  if (st != TG_OK) return st;
  const cudaError_t e = launch_rms_norm(x, w, rows, d, eps, y, di->num_sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "RMSNorm launch");
  return ok();
}

tg_status tg_swiglu(const void* gate_up, int64_t rows, int32_t f, void* y, cudaStream_t stream) {
  if (rows < 0) return fail(TG_ERR_INVALID_ARG, "rows must be >= 0");
  if (f < 8 || f % 8 != 0) return fail(TG_ERR_INVALID_ARG, "f must be a positive multiple of 8");
  if (rows == 0) return ok();
  if (!gate_up || !y) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(gate_up) || !aligned16(y)) return fail(TG_ERR_INVALID_ARG, "gate_up and y must be 16-byte aligned");
  DeviceInfo* di = nullptr;
  tg_status st = device_info(&di);
  if (st != TG_OK) return st;
  const cudaError_t e = launch_swiglu(gate_up, rows, f, y, di->num_sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "SwiGLU launch");
  return ok();
}

size_t tg_decode_workspace_size(int32_t batch, int32_t hq, int32_t head_dim, int32_t max_cache_len) {
  if (batch <= 0 || hq <= 0 || head_dim <= 0 || max_cache_len < 0) return 0;
  const long long n_split = max_cache_len > 0 ? (static_cast<long long>(max_cache_len) + kDecodeSplit - 1) / kDecodeSplit : 1;
  return static_cast<size_t>(batch) * hq * n_split * (head_dim + 2) * 4;
}

tg_status tg_decode_attention(const void* q_rot, const void* k_new_rot, const void* v_new, const void* k_cache,
                              const void* v_cache, const int32_t* cache_cu, int32_t batch, int64_t cache_rows,
                              int32_t max_cache_len, const float* s_cache, const float* gain, float tau, int32_t hq,
                              int32_t hkv, int32_t head_dim, void* o, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
  if (batch < 0) return fail(TG_ERR_INVALID_ARG, "batch must be >= 0");
  if (cache_rows < 0 || cache_rows > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "cache_rows out of range");
  if (max_cache_len < 0) return fail(TG_ERR_INVALID_ARG, "max_cache_len must be >= 0");
  if (hq < 1 || hkv < 1 || hq % hkv != 0) return fail(TG_ERR_INVALID_ARG, "hq must be a positive multiple of hkv");
  if (hq / hkv > kDecodeMaxGroup) return fail(TG_ERR_UNSUPPORTED, "hq / hkv must be at most %d", kDecodeMaxGroup);
  if (head_dim != 64 && head_dim != 128) return fail(TG_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (!(tau > 0.0f) || !std::isfinite(tau)) return fail(TG_ERR_INVALID_ARG, "tau must be positive and finite");
  if (batch == 0) return ok();
  if (!q_rot || !k_new_rot || !v_new || !cache_cu || !o) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (cache_rows > 0 && (!k_cache || !v_cache)) return fail(TG_ERR_INVALID_ARG, "null cache");
  if ((s_cache == nullptr) != (gain == nullptr)) return fail(TG_ERR_INVALID_ARG, "s_cache and gain go together");
  const size_t need = tg_decode_workspace_size(batch, hq, head_dim, max_cache_len);
  if (!workspace || workspace_bytes < need)
    return fail(TG_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (!aligned16(workspace)) return fail(TG_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  DeviceInfo* di = nullptr;
  tg_status st = device_info(&di);
  if (st != TG_OK) return st;
  DecodeArgs a{};
  a.q = q_rot; a.k_new = k_new_rot; a.v_new = v_new; a.k_cache = k_cache; a.v_cache = v_cache; a.cache_cu = cache_cu;
  a.s_cache = s_cache; a.gain = gain; a.batch = batch; a.cache_rows = cache_rows; a.hq = hq; a.hkv = hkv;
  a.head_dim = head_dim; a.split_len = kDecodeSplit;
  a.n_split = max_cache_len > 0 ? (max_cache_len + kDecodeSplit - 1) / kDecodeSplit : 1;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / (std::sqrt(static_cast<double>(head_dim)) * tau));
  a.part = static_cast<float*>(workspace); a.o = o; a.status = di->status;
  const cudaError_t e = launch_decode_attention(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
  return ok();
}

// TMA maps of a linear call: A [m, kdim] in 128-row boxes, W [n, kdim] in
// boxes of half a tile's rows (each CTA of a pair stages one half).
static tg_status linear_maps(const void* a_ptr, const void* w, int64_t m, int32_t n, int32_t kdim, CUtensorMap* ma,
                             CUtensorMap* mw) {
  tg_status st;
  const int bn = linear_tile_n(n);
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(kdim), static_cast<uint64_t>(m)};
    const uint64_t str[1] = {static_cast<uint64_t>(kdim) * 2};
    const uint32_t box[2] = {64, 128};
    if ((st = make_map(ma, a_ptr, 2, dims, str, box, "a")) != TG_OK) return st;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(kdim), static_cast<uint64_t>(n)};
    const uint64_t str[1] = {static_cast<uint64_t>(kdim) * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(bn / 2)};
    if ((st = make_map(mw, w, 2, dims, str, box, "w")) != TG_OK) return st;
  }
  return TG_OK;
}

tg_status tg_linear_bf16(const void* a_ptr, const void* w, const void* residual, void* out, int64_t m, int32_t n,
                         int32_t kdim, cudaStream_t stream) {
  if (m < 0 || m > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "m out of range");
  if (n < 16 || n % 16 != 0) return fail(TG_ERR_INVALID_ARG, "n must be a positive multiple of 16");
  if (kdim < 64 || kdim % 64 != 0) return fail(TG_ERR_INVALID_ARG, "kdim must be a positive multiple of 64");
  if (m == 0) return ok();
  if (!a_ptr || !w || !out) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(a_ptr) || !aligned16(w) || !aligned16(out) || (residual && !aligned16(residual)))
    return fail(TG_ERR_INVALID_ARG, "a, w, residual and out must be 16-byte aligned");
  DeviceInfo* di = nullptr;
  tg_status st = device_info(&di);
  if (st != TG_OK) return st;
  CUtensorMap ma, mw;
  if ((st = linear_maps(a_ptr, w, m, n, kdim, &ma, &mw)) != TG_OK) return st;
  LinearArgs la{};
  la.residual = residual; la.out = out; la.m = m; la.n = n; la.kdim = kdim;
  la.status = di->status; la.watchdog = g_watchdog_cycles; la.num_sms = di->num_sms;
  cudaError_t e = launch_linear(ma, mw, la, stream);
  if (e != cudaSuccess) return cuda_fail(e, "linear kernel launch");
  return ok();
}

tg_status tg_qkv_rope_bf16(const void* x, const void* w_qkv, int64_t m, int32_t kdim, int32_t hq, int32_t hkv,
                           int32_t head_dim, const int32_t* pos, float rope_theta, void* q_out, void* k_out,
                           void* v_out, cudaStream_t stream) {
  if (m < 0 || m > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "m out of range");
  if (kdim < 64 || kdim % 64 != 0) return fail(TG_ERR_INVALID_ARG, "kdim must be a positive multiple of 64");
  if (hq < 1 || hkv < 1) return fail(TG_ERR_INVALID_ARG, "hq and hkv must be >= 1");
  if (head_dim != 64 && head_dim != 128) return fail(TG_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  const int64_t n = static_cast<int64_t>(hq + 2 * hkv) * head_dim;
  if (n > 0x7FFFFFFF) return fail(TG_ERR_INVALID_ARG, "too many heads");
  if (!(rope_theta > 0.0f) || !std::isfinite(rope_theta)) return fail(TG_ERR_INVALID_ARG, "rope_theta must be positive");
  if (m == 0) return ok();
  if (!x || !w_qkv || !pos || !q_out || !k_out || !v_out) return fail(TG_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(q_out) || !aligned16(k_out) || !aligned16(v_out))
    return fail(TG_ERR_INVALID_ARG, "x, w_qkv, q_out, k_out and v_out must be 16-byte aligned");
  DeviceInfo* di = nullptr;
  tg_status st = device_info(&di);
  if (st != TG_OK) return st;
  CUtensorMap ma, mw;
  if ((st = linear_maps(x, w_qkv, m, static_cast<int32_t>(n), kdim, &ma, &mw)) != TG_OK) return st;
  LinearArgs la{};
  la.m = m; la.n = static_cast<int32_t>(n); la.kdim = kdim;
  la.status = di->status; la.watchdog = g_watchdog_cycles; la.num_sms = di->num_sms;
  la.q_out = q_out; la.k_out = k_out; la.v_out = v_out; la.pos = pos;
  la.hq = hq; la.hkv = hkv; la.head_dim = head_dim;
  rope_turns(rope_theta, head_dim, &la.freqs);
  cudaError_t e = launch_linear(ma, mw, la, stream);
  if (e != cudaSuccess) return cuda_fail(e, "QKV projection launch");
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Token-gated attention without a caller-provided workspace.
//
// For callers that cannot allocate device memory at call time (an engine
// that plans all of its device memory at start-up and forbids allocation
// afterwards, a plugin running under a host runtime that owns the allocator,
// a plain C program that does not want to manage a scratch buffer).  The
// scratch space that tg_gated_attention_fwd takes as `workspace` (the
// rotated queries, and the rotated keys when no K cache is given) lives in
// a fixed array of this library's device memory instead.
// ---------------------------------------------------------------------------
namespace tg {
namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;   // 64 MiB
// Every device that loads the library holds this array until the process exits.
__device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device.  In host code
// the symbol itself is only a host-side stand-in, so the address is asked
// from the runtime once per device (with that device current) and cached.
tg_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(TG_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TG_OK;
}

}  // namespace
}  // namespace tg

extern "C" size_t tg_attention_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" tg_status tg_gated_attention_fwd_noalloc(const void* q, const void* k, const void* v,
                                                   const int32_t* pos_kept, const float* s_kept,
                                                   const float* gain, float tau, float rope_theta,
                                                   const int32_t* cu_kept, int32_t batch, int64_t n_kept,
                                                   int32_t max_kept, int32_t hq, int32_t hkv,
                                                   int32_t head_dim, void* o, float* lse, void* k_cache,
                                                   cudaStream_t stream) {
  // the same shape checks and messages as tg_gated_attention_fwd, before the scratch is sized
  const tg_status shape_ok = check_attention_shape(batch, n_kept, hq, hkv, head_dim, cu_kept);
  if (shape_ok != TG_OK) return shape_ok;
  const size_t need = tg_attention_workspace_size(n_kept, hq, hkv, head_dim, k_cache ? 1 : 0);
  if (need > kStaticScratchBytes)
    return fail(TG_ERR_WORKSPACE,
                "this call needs %zu bytes of scratch; the library's fixed scratch holds %zu bytes "
                "(use tg_gated_attention_fwd with a caller-provided workspace)",
                need, kStaticScratchBytes);
  void* scratch = nullptr;
  tg_status s = scratch_address(&scratch);
  if (s != TG_OK) return s;
  return tg_gated_attention_fwd(q, k, v, pos_kept, s_kept, gain, tau, rope_theta, cu_kept, batch, n_kept,
                                max_kept, hq, hkv, head_dim, o, lse, k_cache, scratch, kStaticScratchBytes,
                                stream);
}
