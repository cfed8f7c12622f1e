// RoPE prologue of token-gated attention: rotates q and k by rotate-half
// RoPE at the ORIGINAL positions of the kept tokens (base theta, 1e6 for
// Qwen3) and writes them as bf16.  Also checks that positions strictly
// increase inside each sequence, which the attention kernel's causal tile
// skipping relies on.
//
// Angles: a = pos * theta^(-2i/D) reaches 1.3e5 rad at 128k context, where a
// plain fp32 product would be off by ~1e-2 rad.  The angle is formed in turns,
// pos * t with t = theta^(-2i/D) / (2 pi) held as an unevaluated sum of two
// fp32 numbers (t_hi + t_lo, split on the host in fp64), and reduced exactly
// by rope_sincos (tg_common.cuh).  No fp64 arithmetic on the device.
//
// One warp per token (grid-stride), no block-wide synchronisation: every lane
// of the warp handles the same 8-element column v of several heads (the
// token's vector pairs are dealt round-robin and 32 is a multiple of the
// column count), so each lane needs the 8 frequencies of column v.  The
// lanes of a column compute one share of them each and exchange them by
// shuffles; every load of a lane is issued before the angle math.
#include "tg_common.cuh"

namespace tg {

constexpr int kRopeThreads = 256;
constexpr int kRopeChunk = 4;     // vector pairs per lane per pass

template <int kD>
__global__ void __launch_bounds__(kRopeThreads)
rope_kernel(RopeArgs a, RopeFreqs f) {
  constexpr int kHalf = kD / 2;
  constexpr int kVph = kHalf / 8;              // 8-element columns per half-head
  constexpr int kShare = 8 * kVph / 32;        // frequencies each lane computes
  __shared__ float th_s[kHalf], tl_s[kHalf];
  for (int i = threadIdx.x; i < kHalf; i += kRopeThreads) { th_s[i] = f.turns_hi[i]; tl_s[i] = f.turns_lo[i]; }
  __syncthreads();
  const int lane = lane_id();
  const int v = lane % kVph;                   // this lane's column, the same in all its pairs
  const int grp = lane / kVph;
  const int nqv = a.hq * kVph;
  const int per_tok = nqv + a.hkv * kVph;
  const long long wg = static_cast<long long>(blockIdx.x) * (kRopeThreads / 32) + warp_id();
  const long long nwarps = static_cast<long long>(gridDim.x) * (kRopeThreads / 32);
  for (long long t = wg; t < a.n_kept; t += nwarps) {
    const int p = __ldg(a.pos + t);
    for (int c0 = 0; c0 < per_tok; c0 += 32 * kRopeChunk) {
      uint4 lo4[kRopeChunk], hi4[kRopeChunk];
#pragma unroll
      for (int u = 0; u < kRopeChunk; ++u) {
        const int r = c0 + u * 32 + lane;
        if (r < per_tok) {
          const bool isq = r < nqv;
          const int head = (isq ? r : r - nqv) / kVph;
          const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(isq ? a.q : a.k) +
                                                            (t * (isq ? a.hq : a.hkv) + head) * kD);
          lo4[u] = __ldg(src + v);
          hi4[u] = __ldg(src + kVph + v);
        }
      }
      // cos and sin of the column's 8 frequencies: this lane's share, then
      // the rest from the lanes of the same column
      float cc[kShare], ss[kShare];
#pragma unroll
      for (int q = 0; q < kShare; ++q) {
        const int i = v * 8 + grp * kShare + q;
        rope_sincos(p, th_s[i], tl_s[i], &ss[q], &cc[q]);
      }
      float cs[8], sn[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int src_lane = v + kVph * (e / kShare);
        cs[e] = __shfl_sync(0xffffffffu, cc[e % kShare], src_lane);
        sn[e] = __shfl_sync(0xffffffffu, ss[e % kShare], src_lane);
      }
#pragma unroll
      for (int u = 0; u < kRopeChunk; ++u) {
        const int r = c0 + u * 32 + lane;
        if (r < per_tok) {
          const bool isq = r < nqv;
          const int head = (isq ? r : r - nqv) / kVph;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(isq ? a.q_out : a.k_out) +
                                                (t * (isq ? a.hq : a.hkv) + head) * kD);
          const __nv_bfloat162* l2 = reinterpret_cast<const __nv_bfloat162*>(&lo4[u]);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&hi4[u]);
          uint4 olo, ohi;
          uint32_t* ol = reinterpret_cast<uint32_t*>(&olo);
          uint32_t* oh = reinterpret_cast<uint32_t*>(&ohi);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 xl = __bfloat1622float2(l2[e]);
            const float2 xh = __bfloat1622float2(h2[e]);
            const float c0f = cs[2 * e], s0 = sn[2 * e], c1 = cs[2 * e + 1], s1 = sn[2 * e + 1];
            ol[e] = pack_bf16x2(xl.x * c0f - xh.x * s0, xl.y * c1 - xh.y * s1);
            oh[e] = pack_bf16x2(xh.x * c0f + xl.x * s0, xh.y * c1 + xl.y * s1);
          }
          dst[v] = olo;
          dst[kVph + v] = ohi;
        }
      }
    }
    if (lane == 0) {
      // positions: non-negative and strictly increasing within a sequence
      int lo = 0, hi = a.batch;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<long long>(__ldg(a.cu_kept + mid)) <= t) lo = mid; else hi = mid - 1;
      }
      const bool first = static_cast<long long>(__ldg(a.cu_kept + lo)) == t;
      if (p < 0 || (!first && __ldg(a.pos + t - 1) >= p)) record_error(a.status, kStatusIndex);
    }
  }
}

cudaError_t launch_rope(const RopeArgs& a, const RopeFreqs& f, cudaStream_t st) {
  if (a.n_kept == 0) return cudaSuccess;
  long long blocks = (a.n_kept + kRopeThreads / 32 - 1) / (kRopeThreads / 32);
  const long long cap = static_cast<long long>(a.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (a.head_dim == 128) rope_kernel<128><<<static_cast<unsigned>(blocks), kRopeThreads, 0, st>>>(a, f);
  else rope_kernel<64><<<static_cast<unsigned>(blocks), kRopeThreads, 0, st>>>(a, f);
  return cudaGetLastError();
}

}  // namespace tg
