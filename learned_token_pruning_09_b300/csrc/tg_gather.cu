// Gather of the kept rows (TokenGate's pruned forward: the layers above the
// gate run on the kept tokens only).  One warp moves one residual row at a
// time with 16-byte vector loads (eight in flight per lane before the stores),
// and writes the row's original position and gate score.
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
  const int lane = threadIdx.x & 31;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * kGatherThreads + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * kGatherThreads) >> 5;
  const int nvec = a.d >> 3;   // 16-byte vectors per row
  const uint4* __restrict__ x = static_cast<const uint4*>(a.x);
  uint4* __restrict__ y = static_cast<uint4*>(a.x_kept);
  for (long long i = warp0; i < a.n_kept; i += nwarps) {
    const int b = find_seq(a.cu_kept, a.batch, i);
    const long long r = __ldg(a.kept_idx + i);
    const int lo = __ldg(a.cu_seqlens + b);
    const int hi = __ldg(a.cu_seqlens + b + 1);
    if (i >= __ldg(a.cu_kept + a.batch) || r < lo || r >= hi) {
      if (lane == 0) record_error(a.status, kStatusIndex);
      continue;
    }
    if (lane == 0) {
      if (a.pos_kept) a.pos_kept[i] = static_cast<int32_t>(r - lo);
      if (a.s_kept) a.s_kept[i] = __ldg(a.s + r);
    }
    if (!y) continue;
    const uint4* src = x + r * nvec;
    uint4* dst = y + i * nvec;
    for (int v0 = 0; v0 < nvec; v0 += 32 * 8) {
      uint4 buf[8];
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
  gather_kernel<<<static_cast<unsigned>(blocks), kGatherThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tg
