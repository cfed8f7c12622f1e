// The pieces of the Qwen3-style layer around the pruned path, for the whole
// pruned prefill and its first decode step (TokenGate's three phases,
// MarkTechPost article, "How does TokenGate's learned token pruning work?";
// the model is Qwen3, "How does TokenGate perform on the benchmarks?"):
//
//  * rms_norm_kernel: y = x / sqrt(mean(x^2) + eps) * w per row, bf16 in and
//    out, fp32 arithmetic; one warp per row.  Rows of [T, d] give the
//    layer's pre-norms; rows of [T * heads, D] give the per-head QK-norm.
//  * swiglu_kernel: y = SiLU(a) * b from a fused gate/up projection
//    [T, 2f] (a = the first f columns, b = the last f), bf16 in and out.
//  * decode attention: one new query row per sequence against that
//    sequence's cache plus the new token's own key, with the score bias
//    gain_h s_j and the temperature (s of the new token 0; no bias in the
//    layers without one).  Split along the cache (flash-decoding): each CTA
//    takes a slice of one sequence's cache for one KV head and every query
//    head of its group, keeps a running max / sum / weighted sum per head,
//    and writes them to a workspace; a second kernel merges the slices.
//    HBM-bound: each cache row is read once per KV head.
#include <cfloat>

#include "tg_common.cuh"

namespace tg {

constexpr int kNormWarps = 8;

__global__ void __launch_bounds__(kNormWarps * 32)
rms_norm_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w, long long rows, int d,
                float eps, __nv_bfloat16* __restrict__ y) {
  const int lane = lane_id();
  const long long n_warps = static_cast<long long>(gridDim.x) * kNormWarps;
  const int n_vec = d / 8;                         // 16-byte vectors per row
  for (long long r = static_cast<long long>(blockIdx.x) * kNormWarps + warp_id(); r < rows; r += n_warps) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + r * d);
    float ss = 0.0f;
    for (int v = lane; v < n_vec; v += 32) {
      const uint4 u = __ldg(xr + v);
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(p[e]);
        ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss / static_cast<float>(d) + eps);
    uint4* yr = reinterpret_cast<uint4*>(y + r * d);
    const uint4* wr = reinterpret_cast<const uint4*>(w);
    for (int v = lane; v < n_vec; v += 32) {
      const uint4 u = __ldg(xr + v);
      const uint4 wu = __ldg(wr + v);
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
      const __nv_bfloat162* pw = reinterpret_cast<const __nv_bfloat162*>(&wu);
      uint4 out;
      uint32_t* po = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(p[e]);
        const float2 g = __bfloat1622float2(pw[e]);
        po[e] = pack_bf16x2(f.x * inv * g.x, f.y * inv * g.y);
      }
      yr[v] = out;
    }
  }
}

__global__ void __launch_bounds__(256)
swiglu_kernel(const __nv_bfloat16* __restrict__ gu, long long rows, int f, __nv_bfloat16* __restrict__ y) {
  const int n_vec = f / 8;
  const long long total = rows * n_vec;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / n_vec;
    const int v = static_cast<int>(i - r * n_vec);
    const uint4* row = reinterpret_cast<const uint4*>(gu + r * 2 * f);
    const uint4 a = __ldg(row + v);
    const uint4 b = __ldg(row + n_vec + v);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
    uint4 out;
    uint32_t* po = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 za = __bfloat1622float2(pa[e]);
      const float2 zb = __bfloat1622float2(pb[e]);
      const float s0 = za.x / (1.0f + __expf(-za.x));
      const float s1 = za.y / (1.0f + __expf(-za.y));
      po[e] = pack_bf16x2(s0 * zb.x, s1 * zb.y);
    }
    reinterpret_cast<uint4*>(y + r * f)[v] = out;
  }
}

cudaError_t launch_rms_norm(const void* x, const void* w, long long rows, int d, float eps, void* y, int num_sms,
                            cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  long long blocks = (rows + kNormWarps - 1) / kNormWarps;
  const long long cap = static_cast<long long>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  rms_norm_kernel<<<static_cast<unsigned>(blocks), kNormWarps * 32, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w), rows, d, eps,
      static_cast<__nv_bfloat16*>(y));
  return cudaGetLastError();
}

cudaError_t launch_swiglu(const void* gu, long long rows, int f, void* y, int num_sms, cudaStream_t st) {
  const long long total = rows * (f / 8);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  swiglu_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(gu), rows, f,
                                                                static_cast<__nv_bfloat16*>(y));
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// decode attention
// ---------------------------------------------------------------------------
constexpr int kDecodeWarps = 4;

// per (sequence, query head, slice): [m (log2 units), l, o[0..D)]
__host__ __device__ inline long long decode_part_index(int b, int h, int sp, int hq, int n_split, int d) {
  return ((static_cast<long long>(b) * hq + h) * n_split + sp) * (d + 2);
}

template <int kD>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_partial_kernel(DecodeArgs a) {
  constexpr int kE = kD / 32;
  __shared__ float sm_m[kDecodeWarps][kDecodeMaxGroup];
  __shared__ float sm_l[kDecodeWarps][kDecodeMaxGroup];
  __shared__ float sm_o[kDecodeWarps][kDecodeMaxGroup][kD];
  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = warp_id(), lane = lane_id();
  const int group = a.hq / a.hkv;
  const int lo = __ldg(a.cache_cu + b), hi = __ldg(a.cache_cu + b + 1);
  // a sequence longer than the slices cover (max_cache_len too small) is flagged, not cut short
  if (lo < 0 || hi < lo || hi > a.cache_rows ||
      static_cast<long long>(hi - lo) > static_cast<long long>(a.n_split) * a.split_len) {
    if (threadIdx.x == 0) record_error(a.status, kStatusIndex);
    return;
  }
  const int k0 = lo + sp * a.split_len;
  const int k1 = min(hi, k0 + a.split_len);
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(a.k_new);
  const __nv_bfloat16* vn = static_cast<const __nv_bfloat16*>(a.v_new);
  float qf[kDecodeMaxGroup][kE], acc[kDecodeMaxGroup][kE], m[kDecodeMaxGroup], l[kDecodeMaxGroup],
      gl[kDecodeMaxGroup];
#pragma unroll
  for (int hh = 0; hh < kDecodeMaxGroup; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.0f;
    gl[hh] = 0.0f;
#pragma unroll
    for (int e = 0; e < kE; ++e) { qf[hh][e] = 0.0f; acc[hh][e] = 0.0f; }
    if (hh < group) {
      const int h = g * group + hh;
      const __nv_bfloat16* qr = q + (static_cast<long long>(b) * a.hq + h) * kD + lane * kE;
#pragma unroll
      for (int e = 0; e < kE; ++e) qf[hh][e] = __bfloat162float(qr[e]);
      gl[hh] = a.gain ? __ldg(a.gain + h) * 1.4426950408889634f : 0.0f;
    }
  }
  // one key: logits of every head of the group, then the running softmax
  auto visit = [&](const __nv_bfloat16* kr, const __nv_bfloat16* vr, float sj) {
    float kf[kE], vf[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) { kf[e] = __bfloat162float(kr[e]); vf[e] = __bfloat162float(vr[e]); }
#pragma unroll
    for (int hh = 0; hh < kDecodeMaxGroup; ++hh) {
      if (hh < group) {
        float dot = 0.0f;
#pragma unroll
        for (int e = 0; e < kE; ++e) dot = fmaf(qf[hh][e], kf[e], dot);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        // an infinite score adds -inf (its key is invisible); a zero gain adds nothing
        const float bias = (gl[hh] == 0.0f) ? 0.0f : gl[hh] * sj;
        const float x = dot * a.scale_log2 + bias;
        const float m_new = fmaxf(m[hh], x);
        const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
        const float corr = exp2f(m[hh] - m_use);
        const float p = exp2f(x - m_use);
        l[hh] = l[hh] * corr + p;
#pragma unroll
        for (int e = 0; e < kE; ++e) acc[hh][e] = fmaf(p, vf[e], acc[hh][e] * corr);
        m[hh] = m_new;
      }
    }
  };
  const long long kstride = static_cast<long long>(a.hkv) * kD;
  for (int j = k0 + warp; j < k1; j += kDecodeWarps) {
    const float sj = a.s_cache ? __ldg(a.s_cache + j) : 0.0f;
    visit(kc + j * kstride + static_cast<long long>(g) * kD + lane * kE,
          vc + j * kstride + static_cast<long long>(g) * kD + lane * kE, sj);
  }
  if (sp == 0 && warp == kDecodeWarps - 1) {     // the new token's own key, score 0
    visit(kn + (static_cast<long long>(b) * a.hkv + g) * kD + lane * kE,
          vn + (static_cast<long long>(b) * a.hkv + g) * kD + lane * kE, 0.0f);
  }
  // merge the warps of this CTA, then write the slice's partial state
#pragma unroll
  for (int hh = 0; hh < kDecodeMaxGroup; ++hh) {
    if (hh < group) {
      if (lane == 0) { sm_m[warp][hh] = m[hh]; sm_l[warp][hh] = l[hh]; }
#pragma unroll
      for (int e = 0; e < kE; ++e) sm_o[warp][hh][lane * kE + e] = acc[hh][e];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < group * kD; i += kDecodeWarps * 32) {
    const int hh = i / kD, dd = i - hh * kD;
    float mm = -INFINITY;
    for (int w = 0; w < kDecodeWarps; ++w) mm = fmaxf(mm, sm_m[w][hh]);
    const float mu = (mm == -INFINITY) ? 0.0f : mm;
    float ll = 0.0f, oo = 0.0f;
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float c = exp2f(sm_m[w][hh] - mu);
      ll = fmaf(sm_l[w][hh], c, ll);
      oo = fmaf(sm_o[w][hh][dd], c, oo);
    }
    float* part = a.part + decode_part_index(b, g * group + hh, sp, a.hq, a.n_split, kD);
    if (dd == 0) { part[0] = mm; part[1] = ll; }
    part[2 + dd] = oo;
  }
}

template <int kD>
__global__ void __launch_bounds__(kD)
decode_merge_kernel(DecodeArgs a) {
  const int bh = blockIdx.x;
  const int b = bh / a.hq, h = bh - b * a.hq;
  const int dd = threadIdx.x;
  float mm = -INFINITY;
  for (int sp = 0; sp < a.n_split; ++sp) mm = fmaxf(mm, a.part[decode_part_index(b, h, sp, a.hq, a.n_split, kD)]);
  const float mu = (mm == -INFINITY) ? 0.0f : mm;
  float ll = 0.0f, oo = 0.0f;
  for (int sp = 0; sp < a.n_split; ++sp) {
    const float* part = a.part + decode_part_index(b, h, sp, a.hq, a.n_split, kD);
    const float c = exp2f(part[0] - mu);
    ll = fmaf(part[1], c, ll);
    oo = fmaf(part[2 + dd], c, oo);
  }
  static_cast<__nv_bfloat16*>(a.o)[(static_cast<long long>(b) * a.hq + h) * kD + dd] = __float2bfloat16_rn(oo / ll);
}

cudaError_t launch_decode_attention(const DecodeArgs& a, cudaStream_t st) {
  if (a.batch == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(a.n_split), static_cast<unsigned>(a.hkv), static_cast<unsigned>(a.batch));
  if (a.head_dim == 128) {
    decode_partial_kernel<128><<<grid, kDecodeWarps * 32, 0, st>>>(a);
  } else {
    decode_partial_kernel<64><<<grid, kDecodeWarps * 32, 0, st>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned blocks = static_cast<unsigned>(a.batch * a.hq);
  if (a.head_dim == 128) decode_merge_kernel<128><<<blocks, 128, 0, st>>>(a);
  else decode_merge_kernel<64><<<blocks, 64, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tg
