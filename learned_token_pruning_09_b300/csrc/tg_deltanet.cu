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
// The rows of S evolve independently: with the row form
//   c = beta (v_r - exp(g) S_r . k^),   S_r = exp(g) S_r + c k^
// row r needs only k^, q^, g, beta and v[r].  A CTA owns kRows rows of one
// (sequence, value head); each row is split over kTpr threads holding 32
// state entries each in registers, so a token costs three 32-term dot
// products or updates per thread and two shuffle reductions over the row's
// threads.  The token stream comes through shared memory: the raw q, k, v,
// g and beta of the next 32 tokens are copied with cp.async while the
// current 32 are processed, and each block's k^ and q^ are normalised once
// (one warp per vector) and its decays exponentiated once, so the per-token
// loop never waits on global memory.  Outputs of a block are collected in
// shared memory and written as whole 64-byte row groups.
#include "tg_common.cuh"

namespace tg {

constexpr float kScanL2Eps = 1e-6f;
constexpr int kScanTok = 32;        // tokens per staged block
constexpr int kScanRows = 16;       // state rows per CTA
constexpr int kScanCols = 32;       // state entries per thread

template <int kDk>
struct ScanSmem {
  alignas(16) __nv_bfloat16 kraw[2][kScanTok][kDk];
  alignas(16) __nv_bfloat16 qraw[2][kScanTok][kDk];
  alignas(16) __nv_bfloat16 vraw[2][kScanTok][kScanRows];
  alignas(16) float graw[2][kScanTok];
  alignas(16) float braw[2][kScanTok];
  alignas(16) float kh[kScanTok][kDk];      // normalised k of the current block
  alignas(16) float qh[kScanTok][kDk];      // normalised, scaled q
  float alpha[kScanTok];                    // exp(g)
  alignas(16) __nv_bfloat16 o[kScanTok][kScanRows];
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <int kDk>
__global__ void __launch_bounds__(kScanRows * (kDk / kScanCols))
delta_scan_kernel(ScanArgs a) {
  constexpr int kTpr = kDk / kScanCols;             // threads per state row
  constexpr int kThreads = kScanRows * kTpr;
  constexpr int kV4 = kScanCols / 4;                // float4s of state per thread
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ScanSmem<kDk>& sm = *reinterpret_cast<ScanSmem<kDk>*>(smem_raw);
  const int tid = threadIdx.x;
  const int lane = lane_id();
  const int rr = tid / kTpr;                        // row of this CTA's block
  const int sl = tid % kTpr;                        // slice: float4 columns sl, sl + kTpr, ...
  const int row0 = blockIdx.x * kScanRows;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int lo = __ldg(a.cu_kept + b);
  const int hi = __ldg(a.cu_kept + b + 1);
  if (lo < 0 || hi < lo || hi > a.n_kept) {
    if (tid == 0) record_error(a.status, kStatusIndex);
    return;
  }
  const int kh = h / (a.hv / a.hk);
  const long long state_row = (static_cast<long long>(b) * a.hv + h) * a.dv + row0 + rr;
  float4 s[kV4];
#pragma unroll
  for (int j = 0; j < kV4; ++j) {
    s[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (a.initial_state) s[j] = __ldg(reinterpret_cast<const float4*>(a.initial_state + state_row * kDk) + kTpr * j + sl);
  }

  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v);
  __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.o);
  const int n_tok = hi - lo;
  const int n_blocks = (n_tok + kScanTok - 1) / kScanTok;

  // raw copies of block bi into buffer bi & 1 (tokens past the sequence end are not copied)
  auto issue = [&](int bi) {
    const int buf = bi & 1;
    const int t0 = lo + bi * kScanTok;
    const int nt = min(kScanTok, hi - t0);
    constexpr int kRowChunks = kDk * 2 / 16;        // 16-byte pieces of a q or k row
    for (int c = tid; c < nt * kRowChunks; c += kThreads) {
      const int tt = c / kRowChunks, pc = c - tt * kRowChunks;
      const long long src = (static_cast<long long>(t0 + tt) * a.hk + kh) * kDk + pc * 8;
      cp_async16(&sm.kraw[buf][tt][pc * 8], kp + src);
      cp_async16(&sm.qraw[buf][tt][pc * 8], qp + src);
    }
    constexpr int kVChunks = kScanRows * 2 / 16;    // 16-byte pieces of the rows' v
    for (int c = tid; c < nt * kVChunks; c += kThreads) {
      const int tt = c / kVChunks, pc = c - tt * kVChunks;
      cp_async16(&sm.vraw[buf][tt][pc * 8],
                 vp + (static_cast<long long>(t0 + tt) * a.hv + h) * a.dv + row0 + pc * 8);
    }
    for (int tt = tid; tt < nt; tt += kThreads) {
      cp_async4(&sm.graw[buf][tt], a.g + static_cast<long long>(t0 + tt) * a.hv + h);
      cp_async4(&sm.braw[buf][tt], a.beta + static_cast<long long>(t0 + tt) * a.hv + h);
    }
  };

  if (n_blocks > 0) issue(0);
  cp_async_commit();
  for (int bi = 0; bi < n_blocks; ++bi) {
    const int buf = bi & 1;
    const int t0 = lo + bi * kScanTok;
    const int nt = min(kScanTok, hi - t0);
    if (bi + 1 < n_blocks) issue(bi + 1);           // its buffer was last read in block bi - 1
    cp_async_commit();
    cp_async_wait_one();                            // this thread's copies of block bi landed
    __syncthreads();                                // everyone's did
    // normalise: one warp per vector (kScanTok k rows, then kScanTok q rows)
    for (int vec = warp_id(); vec < 2 * nt; vec += kThreads / 32) {
      const bool isq = vec >= nt;
      const int tt = isq ? vec - nt : vec;
      const __nv_bfloat16* src = isq ? sm.qraw[buf][tt] : sm.kraw[buf][tt];
      float x[kDk / 32];
      float ss = 0.0f;
#pragma unroll
      for (int e = 0; e < kDk / 32; ++e) {
        x[e] = __bfloat162float(src[e * 32 + lane]);
        ss = fmaf(x[e], x[e], ss);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = (isq ? a.scale : 1.0f) * rsqrtf(ss + kScanL2Eps);
      float* dst = isq ? sm.qh[tt] : sm.kh[tt];
#pragma unroll
      for (int e = 0; e < kDk / 32; ++e) dst[e * 32 + lane] = x[e] * inv;
    }
    for (int tt = tid; tt < nt; tt += kThreads) sm.alpha[tt] = __expf(sm.graw[buf][tt]);
    __syncthreads();

    for (int tt = 0; tt < nt; ++tt) {
      const float4* k4 = reinterpret_cast<const float4*>(sm.kh[tt]);
      const float4* q4 = reinterpret_cast<const float4*>(sm.qh[tt]);
      float4 kx[kV4];
#pragma unroll
      for (int j = 0; j < kV4; ++j) kx[j] = k4[kTpr * j + sl];
      float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
#pragma unroll
      for (int j = 0; j < kV4; ++j) {
        p0 = fmaf(s[j].x, kx[j].x, p0);
        p1 = fmaf(s[j].y, kx[j].y, p1);
        p2 = fmaf(s[j].z, kx[j].z, p2);
        p3 = fmaf(s[j].w, kx[j].w, p3);
      }
      float sk = (p0 + p1) + (p2 + p3);
#pragma unroll
      for (int o = 1; o < kTpr; o <<= 1) sk += __shfl_xor_sync(0xffffffffu, sk, o);
      const float alpha = sm.alpha[tt];
      const float c = sm.braw[buf][tt] * (__bfloat162float(sm.vraw[buf][tt][rr]) - alpha * sk);
      float r0 = 0.0f, r1 = 0.0f, r2 = 0.0f, r3 = 0.0f;
#pragma unroll
      for (int j = 0; j < kV4; ++j) {
        const float4 qx = q4[kTpr * j + sl];
        s[j].x = fmaf(c, kx[j].x, alpha * s[j].x);
        s[j].y = fmaf(c, kx[j].y, alpha * s[j].y);
        s[j].z = fmaf(c, kx[j].z, alpha * s[j].z);
        s[j].w = fmaf(c, kx[j].w, alpha * s[j].w);
        r0 = fmaf(s[j].x, qx.x, r0);
        r1 = fmaf(s[j].y, qx.y, r1);
        r2 = fmaf(s[j].z, qx.z, r2);
        r3 = fmaf(s[j].w, qx.w, r3);
      }
      float sq = (r0 + r1) + (r2 + r3);
#pragma unroll
      for (int o = 1; o < kTpr; o <<= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      if (sl == 0) sm.o[tt][rr] = __float2bfloat16_rn(sq);
    }
    __syncthreads();
    // the block's outputs: each token's kScanRows values are 32 contiguous bytes
    constexpr int kOChunks = kScanRows * 2 / 16;
    for (int c = tid; c < nt * kOChunks; c += kThreads) {
      const int tt = c / kOChunks, pc = c - tt * kOChunks;
      *reinterpret_cast<uint4*>(op + (static_cast<long long>(t0 + tt) * a.hv + h) * a.dv + row0 + pc * 8) =
          *reinterpret_cast<const uint4*>(&sm.o[tt][pc * 8]);
    }
  }
  if (a.final_state) {
#pragma unroll
    for (int j = 0; j < kV4; ++j) reinterpret_cast<float4*>(a.final_state + state_row * kDk)[kTpr * j + sl] = s[j];
  }
}

cudaError_t launch_delta_scan(const ScanArgs& a, cudaStream_t st) {
  if (a.batch == 0 || a.hv == 0 || a.dv == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(a.dv / kScanRows), static_cast<unsigned>(a.hv),
                  static_cast<unsigned>(a.batch));
  if (a.dk == 128) {
    const size_t smem = sizeof(ScanSmem<128>);
    cudaError_t e = cudaFuncSetAttribute(delta_scan_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    delta_scan_kernel<128><<<grid, kScanRows * (128 / kScanCols), smem, st>>>(a);
  } else {
    const size_t smem = sizeof(ScanSmem<64>);
    cudaError_t e = cudaFuncSetAttribute(delta_scan_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    delta_scan_kernel<64><<<grid, kScanRows * (64 / kScanCols), smem, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace tg
