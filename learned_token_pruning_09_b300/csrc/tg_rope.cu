// RoPE prologue of token-gated attention: rotates q and k by rotate-half
// RoPE at the ORIGINAL positions of the kept tokens (base theta, 1e6 for
// Qwen3) and writes them as bf16: q' into the workspace, k' into the
// kept-only KV cache.  Also checks that positions strictly increase inside
// each sequence, which the attention kernel's causal tile skipping relies on.
//
// Angles: a = pos * theta^(-2i/D) can reach 1.3e5 rad at 128k context, where
// an fp32 angle would be off by ~1e-2 rad.  The product and its reduction to
// [-pi, pi] are done in fp64 (inverse frequencies precomputed on the host in
// fp64), then sin/cos in fp32 of the reduced angle.
#include "tg_common.cuh"

namespace tg {

constexpr int kRopeThreads = 128;

__global__ void __launch_bounds__(kRopeThreads)
rope_kernel(RopeArgs a, RopeFreqs f) {
  __shared__ float cs[kMaxHeadDimHalf];
  __shared__ float sn[kMaxHeadDimHalf];
  const int D = a.head_dim;
  const int half = D >> 1;
  const int vph = half >> 3;                    // 8-element vectors per half-head
  const int nqv = a.hq * vph;
  const int ntot = nqv + a.hkv * vph;
  const double kTwoPi = 6.283185307179586;
  const double kInvTwoPi = 0.15915494309189535;
  for (long long t = blockIdx.x; t < a.n_kept; t += gridDim.x) {
    const int p = __ldg(a.pos + t);
    if (threadIdx.x < half) {
      const double ang = static_cast<double>(p) * f.inv_freq[threadIdx.x];
      const double r = fma(-rint(ang * kInvTwoPi), kTwoPi, ang);
      float sv, cv;
      sincosf(static_cast<float>(r), &sv, &cv);
      cs[threadIdx.x] = cv;
      sn[threadIdx.x] = sv;
    }
    if (threadIdx.x == 0) {
      // positions: non-negative and strictly increasing within a sequence
      int lo = 0, hi = a.batch;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<long long>(__ldg(a.cu_kept + mid)) <= t) lo = mid; else hi = mid - 1;
      }
      const bool first = static_cast<long long>(__ldg(a.cu_kept + lo)) == t;
      if (p < 0 || (!first && __ldg(a.pos + t - 1) >= p)) record_error(a.status, kStatusIndex);
    }
    __syncthreads();
    for (int w = threadIdx.x; w < ntot; w += kRopeThreads) {
      const bool isq = w < nqv;
      const int ww = isq ? w : w - nqv;
      const int head = ww / vph;
      const int v = ww - head * vph;
      const int nh = isq ? a.hq : a.hkv;
      const size_t row = (static_cast<size_t>(t) * nh + head) * D;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(isq ? a.q : a.k) + row);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(isq ? a.q_out : a.k_out) + row);
      const uint4 lo4 = __ldg(src + v);
      const uint4 hi4 = __ldg(src + vph + v);
      const __nv_bfloat162* l2 = reinterpret_cast<const __nv_bfloat162*>(&lo4);
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&hi4);
      uint4 olo, ohi;
      uint32_t* ol = reinterpret_cast<uint32_t*>(&olo);
      uint32_t* oh = reinterpret_cast<uint32_t*>(&ohi);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 xl = __bfloat1622float2(l2[e]);
        const float2 xh = __bfloat1622float2(h2[e]);
        const int i0 = v * 8 + 2 * e;
        const float c0 = cs[i0], s0 = sn[i0], c1 = cs[i0 + 1], s1 = sn[i0 + 1];
        ol[e] = pack_bf16x2(xl.x * c0 - xh.x * s0, xl.y * c1 - xh.y * s1);
        oh[e] = pack_bf16x2(xh.x * c0 + xl.x * s0, xh.y * c1 + xl.y * s1);
      }
      dst[v] = olo;
      dst[vph + v] = ohi;
    }
    __syncthreads();
  }
}

cudaError_t launch_rope(const RopeArgs& a, const RopeFreqs& f, cudaStream_t st) {
  if (a.n_kept == 0) return cudaSuccess;
  long long blocks = a.n_kept;
  const long long cap = static_cast<long long>(a.num_sms) * 16;
  if (blocks > cap) blocks = cap;
  rope_kernel<<<static_cast<unsigned>(blocks), kRopeThreads, 0, st>>>(a, f);
  return cudaGetLastError();
}

}  // namespace tg
