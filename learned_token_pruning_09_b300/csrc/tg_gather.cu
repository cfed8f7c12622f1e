// Gather of the kept rows (TokenGate's pruned forward: the layers above the
// gate run on the kept tokens only).  One warp moves one residual row at a
// time with 16-byte vector loads (eight in flight per lane before the stores),
// and writes the row's original position and gate score.  Launched early
// behind the top-K (programmatic dependent launch), it waits for the kept ids
// before reading anything.
#include "tg_common.cuh"

namespace tg {

constexpr int kGatherThreads = 256;

__device__ __forceinline__ int find_seq(const int32_t* cu, int batch, long long i) {
  // largest b with cu[b] <= i  (cu ascending, cu[0] = 0)
  int lo = 0, hi = batch;   // answer in [0, batch)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<long long>(__ldg(cu + mid)) <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kGatherThreads)
gather_kernel(GatherArgs a) {
  pdl_wait();     // launched early behind the top-K: its kept ids must be complete
  const int lane = threadIdx.x & 31;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * kGatherThreads + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * kGatherThreads) >> 5;
  const int nvec = a.d >> 3;   // 16-byte vectors per row
  const uint4* __restrict__ x = static_cast<const uint4*>(a.x);
  uint4* __restrict__ y = static_cast<uint4*>(a.x_kept);
  for (long long i = warp0; i < a.n_kept; i += nwarps) {
    // the row's loads go out first, checked only against x's extent; the
    // sequence bounds are checked while they are in flight
    const long long r = __ldg(a.kept_idx + i);
    // x and s are read only for the outputs asked for (a call for positions
    // alone passes neither)
    const bool in_x = (!y && !a.s_kept) || (r >= 0 && r < a.n_rows);
    const uint4* src = x + r * nvec;
    uint4 buf[8];
    if (y && in_x) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = u * 32 + lane;
        if (v < nvec) buf[u] = __ldcs(src + v);
      }
    }
    const float sr = (a.s_kept && in_x) ? __ldg(a.s + r) : 0.0f;
    const int b = find_seq(a.cu_kept, a.batch, i);
    const int lo = __ldg(a.cu_seqlens + b);
    const int hi = __ldg(a.cu_seqlens + b + 1);
    if (!in_x || i >= __ldg(a.cu_kept + a.batch) || r < lo || r >= hi) {
      if (lane == 0) record_error(a.status, kStatusIndex);
      continue;
    }
    if (lane == 0) {
      if (a.pos_kept) a.pos_kept[i] = static_cast<int32_t>(r - lo);
      if (a.s_kept) a.s_kept[i] = sr;
    }
    if (!y) continue;
    uint4* dst = y + i * nvec;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int v = u * 32 + lane;
      if (v < nvec) dst[v] = buf[u];
    }
    for (int v0 = 32 * 8; v0 < nvec; v0 += 32 * 8) {   // rows wider than 4 KB
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < nvec) buf[u] = __ldcs(src + v);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < nvec) dst[v] = buf[u];
      }
    }
  }
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t st) {
  if (a.n_kept == 0) return cudaSuccess;
  const long long warps_needed = a.n_kept;
  long long blocks = (warps_needed * 32 + kGatherThreads - 1) / kGatherThreads;
  const long long cap = static_cast<long long>(a.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  // programmatic dependent launch behind the previous kernel (the top-K)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kGatherThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_kernel, a);
}

}  // namespace tg
