// Pruned Gated DeltaNet: the gated delta rule run over the KEPT tokens of
// each sequence (TokenGate prunes the Gated DeltaNet layers of the hybrid
// model as well as its attention layers: MarkTechPost article, section "Does
// it work on hybrid attention models?"; pruned tokens never update the
// state, as pruned tokens get no KV entries in the attention layers).  Per
// sequence and value head h, with S (d_v x d_k) from the initial state (zero
// when none), token by token in order:
//   k^ = k / sqrt(|k|^2 + eps),   q^ = scale q / sqrt(|q|^2 + eps)
//   S  = exp(g) (S - beta (S k^) k^T) + beta v k^T,    o = S q^
// Value head h reads q/k head h / (hv / hk).
//
// The rows of S evolve independently: row r needs only k^, q^, g, beta and
// v[r].  One warp owns one row, its d_k entries spread over the lanes (fp32),
// so the whole recurrence runs in registers with two warp reductions per
// token (S_r . k^ and S_r . q^); every (sequence, value head, row) is an
// independent warp.  With the row form
//   S_r = exp(g) S_r + beta (v_r - exp(g) S_r . k^) k^
// the state update is one FMA per entry.
#include "tg_common.cuh"

namespace tg {

constexpr int kScanWarpsPerBlock = 8;
constexpr float kScanL2Eps = 1e-6f;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// per lane: kE = d_k / 32 consecutive entries of the row
template <int kE>
__device__ __forceinline__ void load_bf16_vec(const __nv_bfloat16* p, float (&x)[kE]) {
  if constexpr (kE == 4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  } else {
    const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
    x[0] = a.x; x[1] = a.y;
  }
}

template <int kDk>
__global__ void __launch_bounds__(kScanWarpsPerBlock * 32)
delta_scan_kernel(ScanArgs a) {
  constexpr int kE = kDk / 32;
  const int lane = lane_id();
  const long long row_id = static_cast<long long>(blockIdx.x) * kScanWarpsPerBlock + warp_id();
  const long long rows = static_cast<long long>(a.batch) * a.hv * a.dv;
  if (row_id >= rows) return;
  const int r = static_cast<int>(row_id % a.dv);
  const int h = static_cast<int>((row_id / a.dv) % a.hv);
  const int b = static_cast<int>(row_id / (static_cast<long long>(a.dv) * a.hv));
  const int lo = __ldg(a.cu_kept + b);
  const int hi = __ldg(a.cu_kept + b + 1);
  if (lo < 0 || hi < lo || hi > a.n_kept) {
    if (lane == 0) record_error(a.status, kStatusIndex);
    return;
  }
  const int kh = h / (a.hv / a.hk);
  float s[kE];
  const long long state_off = ((static_cast<long long>(b) * a.hv + h) * a.dv + r) * kDk + lane * kE;
#pragma unroll
  for (int e = 0; e < kE; ++e) s[e] = a.initial_state ? __ldg(a.initial_state + state_off + e) : 0.0f;

  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v);
  __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.o);
  const long long qk_stride = static_cast<long long>(a.hk) * kDk;     // elements per token
  const long long v_stride = static_cast<long long>(a.hv) * a.dv;
  for (int t = lo; t < hi; ++t) {
    float kx[kE], qx[kE];
    load_bf16_vec<kE>(kp + t * qk_stride + static_cast<long long>(kh) * kDk + lane * kE, kx);
    load_bf16_vec<kE>(qp + t * qk_stride + static_cast<long long>(kh) * kDk + lane * kE, qx);
    const float alpha = __expf(__ldg(a.g + static_cast<long long>(t) * a.hv + h));
    const float beta = __ldg(a.beta + static_cast<long long>(t) * a.hv + h);
    const float vr = __bfloat162float(__ldg(vp + t * v_stride + static_cast<long long>(h) * a.dv + r));
    float kk = 0.0f, qq = 0.0f, sk = 0.0f;
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      kk = fmaf(kx[e], kx[e], kk);
      qq = fmaf(qx[e], qx[e], qq);
      sk = fmaf(s[e], kx[e], sk);
    }
    kk = warp_sum(kk);
    qq = warp_sum(qq);
    sk = warp_sum(sk);
    const float kinv = rsqrtf(kk + kScanL2Eps);
    const float qinv = a.scale * rsqrtf(qq + kScanL2Eps);
    // S_r k^ = (S_r . k) kinv; S_r = alpha S_r + beta (v_r - alpha S_r k^) k^
    const float c = beta * (vr - alpha * sk * kinv) * kinv;
    float sq = 0.0f;
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      s[e] = fmaf(c, kx[e], alpha * s[e]);
      sq = fmaf(s[e], qx[e], sq);
    }
    sq = warp_sum(sq);
    if (lane == 0) op[t * v_stride + static_cast<long long>(h) * a.dv + r] = __float2bfloat16_rn(sq * qinv);
  }
  if (a.final_state) {
#pragma unroll
    for (int e = 0; e < kE; ++e) a.final_state[state_off + e] = s[e];
  }
}

cudaError_t launch_delta_scan(const ScanArgs& a, cudaStream_t st) {
  const long long rows = static_cast<long long>(a.batch) * a.hv * a.dv;
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows + kScanWarpsPerBlock - 1) / kScanWarpsPerBlock;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  if (a.dk == 128)
    delta_scan_kernel<128><<<static_cast<unsigned>(blocks), kScanWarpsPerBlock * 32, 0, st>>>(a);
  else
    delta_scan_kernel<64><<<static_cast<unsigned>(blocks), kScanWarpsPerBlock * 32, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tg
