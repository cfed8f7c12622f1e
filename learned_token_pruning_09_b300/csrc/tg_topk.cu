// Top-K selection of document tokens per sequence, question tokens always
// kept (TokenGate gate module: "a top-K selector keeps the tokens with the
// highest score"; "only the document part of the prompt is prunable").
//
// One thread-block cluster of kCluster CTAs per sequence.  Each CTA owns a
// contiguous slice of the sequence's document rows, converts its scores to
// 32-bit order keys once (kept in shared memory when they fit) and the
// cluster runs an MSB-first radix select (4 passes x 8 bits): every CTA
// builds a 256-bin histogram of its slice and stores it into its own slot of
// every CTA's shared memory (distributed shared memory stores, which the
// storing CTA does not wait for); after one cluster barrier each CTA sums the
// slots locally and every CTA derives the same next digit.  The result is
// the exact K-th key and the number of keys equal to it that are taken
// (lowest row index first).  A final ordered compaction (warp ballots +
// prefix sums; slice counts exchanged the same way) writes the kept rows in
// ascending order, then the question rows.  No CTA reads another's shared
// memory, and none writes into another's after the last cluster barrier, so
// the CTAs may leave as soon as they are done.
//
// General prunable spans (a per-row mask instead of a document prefix): the
// slices cover the whole sequence; a row outside the mask gets the key
// 0xFFFFFFFF, which no score maps to (NaN maps to 0, +inf to 0xFF800000), so
// it stays out of every histogram, ranks above the K-th key and is kept by
// the same ordered compaction, in its place in row order.  The number of
// prunable rows of each sequence comes from a counting kernel run first.
#include <cooperative_groups.h>

#include "tg_common.cuh"

namespace cg = cooperative_groups;

namespace tg {

constexpr int kTopkClusterMax = 16;   // non-portable cluster size, when the device allows it
constexpr int kTopkClusterPortable = 8;
constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkMaxSmemKeys = (180 * 1024) / 4;
constexpr int kTopkBalChunks = 32;      // 32-key chunks per warp whose ballots the compaction keeps
constexpr uint32_t kFixedKey = 0xFFFFFFFFu;   // a row outside the prunable mask
constexpr uint32_t kNoneKey = 0xFFFFFFFEu;    // "K-th key" when no prunable row is kept

struct TopkShared {
  uint32_t slot[2][kTopkClusterMax][256];   // per pass parity: each CTA's histogram, stored by that CTA
  uint32_t local[256];                      // this CTA's histogram of the current pass
  uint32_t warp_tot[8];
  uint32_t warp_gt[kTopkWarps];
  uint32_t warp_eq[kTopkWarps];
  uint32_t slice_gt[kTopkClusterMax];       // each CTA's kept-above and equal counts, stored by that CTA
  uint32_t slice_eq[kTopkClusterMax];
  uint32_t bal_gt[kTopkWarps][kTopkBalChunks];   // per warp and 32-key chunk: keys above / equal to the K-th
  uint32_t bal_eq[kTopkWarps][kTopkBalChunks];

  uint32_t digit;
  int32_t remaining;
  int32_t found;
  uint32_t total;
  long long base;           // first output slot of this sequence
};

// The radix digit of the K-th key from 256 bin counts (bin t held by thread
// t < 256, every thread of the CTA calls): d with suffix(d + 1) < remaining
// <= suffix(d).  On success *digit is d and *rem the rank of the K-th key
// inside bin d; *total is the sum of all bins.  Returns false when no bin
// qualifies (the counts are inconsistent with `remaining`).
__device__ __forceinline__ bool pick_digit(TopkShared& sh, uint32_t tot, int remaining, uint32_t* digit, int* rem,
                                           uint32_t* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t suf = tot;
  if (warp < 8) {
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += v;
    }
    if (lane == 0) sh.warp_tot[warp] = suf;
  }
  if (tid == 0) sh.found = 0;
  __syncthreads();
  if (warp < 8) {
    for (int w2 = warp + 1; w2 < 8; ++w2) suf += sh.warp_tot[w2];
    // digit d is the one with suffix(d+1) < remaining <= suffix(d)
    const uint32_t above = suf - tot;
    if (static_cast<uint32_t>(remaining) <= suf && above < static_cast<uint32_t>(remaining)) {
      sh.digit = static_cast<uint32_t>(tid);
      sh.remaining = remaining - static_cast<int>(above);
      sh.found = 1;
    }
    if (tid == 0) sh.total = suf;
  }
  __syncthreads();
  *digit = sh.digit;
  *rem = sh.remaining;
  *total = sh.total;
  const bool found = sh.found != 0;
  __syncthreads();          // sh is reused by the next call
  return found;
}

// This CTA's share of zeroing sequence b's score histograms (the cluster
// covers them all), so the workspace is zero for the next gate call.
__device__ __forceinline__ void zero_hist(uint32_t* hist, int b, int rank, int n_ranks) {
  constexpr int kVecs = kHistWords / 4;
  uint4* h = reinterpret_cast<uint4*>(hist + static_cast<long long>(b) * kHistWords);
  const int per = (kVecs + n_ranks - 1) / n_ranks;
  const int v1 = min(kVecs, (rank + 1) * per);
  for (int v = rank * per + static_cast<int>(threadIdx.x); v < v1; v += kTopkThreads) h[v] = make_uint4(0u, 0u, 0u, 0u);
}

template <bool kSmemKeys, bool kMasked>
__global__ void __launch_bounds__(kTopkThreads, 1)
topk_kernel(TopkArgs a) {
  extern __shared__ __align__(16) uint32_t keys_smem[];
  __shared__ TopkShared sh;
  // launched early behind the gate (programmatic dependent launch): wait for
  // it to finish before any global memory is read or written, and let the
  // gather behind this kernel start launching
  pdl_wait();
  pdl_trigger();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int kTopkCluster = static_cast<int>(cluster.num_blocks());   // 8 or 16
  const int b = blockIdx.x / kTopkCluster;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  const int lo = a.cu_seqlens[b];
  const int hi = a.cu_seqlens[b + 1];
  const int nd = a.n_doc[b];
  const int kb = a.k[b];
  // every CTA of the cluster sees the same values, so all leave together
  if (hi < lo || nd < 0 || nd > hi - lo || (kMasked ? hi - lo : nd) > a.max_n_doc || kb < 0) {
    if (rank == 0 && tid == 0) record_error(a.status, kStatusIndex);
    return;
  }
  const int ke = min(kb, nd);
  const int nq = hi - lo - nd;

  // output offset of this sequence: sum of the kept lengths of earlier ones
  if (tid == 0) sh.base = 0;
  __syncthreads();
  {
    long long part = 0;
    for (int bb = tid; bb < b; bb += kTopkThreads) {
      const int l2 = a.cu_seqlens[bb], h2 = a.cu_seqlens[bb + 1], n2 = a.n_doc[bb], k2 = a.k[bb];
      part += static_cast<long long>(min(max(k2, 0), n2)) + (h2 - l2 - n2);
    }
    for (int o = 16; o > 0; o >>= 1) part += __shfl_down_sync(0xffffffffu, part, o);
    if (lane == 0 && part) atomicAdd(reinterpret_cast<unsigned long long*>(&sh.base),
                                     static_cast<unsigned long long>(part));
  }
  __syncthreads();
  const long long base = sh.base;
  if (base + ke + nq > a.kept_capacity) {   // the same verdict in every CTA of the cluster
    if (rank == 0 && tid == 0) record_error(a.status, kStatusIndex);
    return;
  }
  if (rank == 0 && tid == 0) {
    a.cu_kept[b + 1] = static_cast<int32_t>(base + ke + nq);
    if (b == 0) a.cu_kept[0] = 0;
  }
  // question rows, spread over the cluster (with a mask they are placed by
  // the compaction)
  if (!kMasked)
    for (int t = rank * kTopkThreads + tid; t < nq; t += kTopkCluster * kTopkThreads)
      a.kept_idx[base + ke + t] = lo + nd + t;

  // this CTA's slice of the document (of the whole sequence with a mask)
  const int span = kMasked ? hi - lo : nd;
  const int chunk = (span + kTopkCluster - 1) / kTopkCluster;
  const int s0 = min(span, rank * chunk);
  const int n_loc = min(span, s0 + chunk) - s0;
  const float* src = a.s + lo + s0;
  const uint8_t* msk = kMasked ? a.prunable + lo + s0 : nullptr;
  int32_t* out = a.kept_idx + base;

  if (ke == nd) {             // every prunable row kept, so every row (also nd == 0)
    for (int i = tid; i < n_loc; i += kTopkThreads) out[s0 + i] = lo + s0 + i;
    if (a.hist) zero_hist(a.hist, b, rank, kTopkCluster);
    return;
  }
  if (!kMasked && ke == 0) {  // question only
    if (a.hist) zero_hist(a.hist, b, rank, kTopkCluster);
    return;
  }
  const bool none = kMasked && ke == 0;   // only the rows outside the mask
  // the gate's histograms of this sequence's scores (the first two digits);
  // read before the keys so that the two loads overlap
  const uint32_t* hc = a.hist ? a.hist + static_cast<long long>(b) * kHistWords : nullptr;
  const uint32_t cnt0 = (hc && tid < 256) ? __ldcg(hc + tid) : 0u;
  // every CTA of the cluster must be running before any stores into its
  // shared memory: arrive here, wait before the first remote store
  cluster_arrive_relaxed();

  if (kSmemKeys) {
    // sixteen loads in flight per thread before any is used (the scores were
    // just written and sit in L2; one at a time would serialise its latency):
    // a 131k-row sequence's slice is one round
    for (int i0 = tid; i0 < n_loc; i0 += 16 * kTopkThreads) {
      float v[16];
      uint8_t m[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + u * kTopkThreads;
        v[u] = i < n_loc ? __ldg(src + i) : 0.0f;
        m[u] = (kMasked && i < n_loc) ? __ldg(msk + i) : 1;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + u * kTopkThreads;
        if (i < n_loc) keys_smem[i] = m[u] ? order_key(v[u]) : kFixedKey;
      }
    }
  }
  auto key_at = [&](int i) -> uint32_t {
    if (kSmemKeys) return keys_smem[i];
    if (kMasked && __ldg(msk + i) == 0) return kFixedKey;
    return order_key(__ldg(src + i));
  };

  // ---- radix select, 4 passes of 8 bits --------------------------------
  uint32_t prefix = 0, mask = 0;
  int remaining = ke;
  int pass_begin = 0;
  if (hc) {
    // the first two digits from the gate's counts: every CTA reads the same
    // bins and derives the same digits, with no exchange.  Counts that do not
    // add up (a gate call whose histograms no top-K consumed) fall back to
    // the four passes.
    uint32_t d0 = 0, d1 = 0, tot0 = 0, tot1 = 0;
    int r0 = 0, r1 = 0;
    bool ok = pick_digit(sh, cnt0, ke, &d0, &r0, &tot0) && tot0 == static_cast<uint32_t>(nd);
    if (ok) {
      const uint32_t cnt1 = tid < 256 ? __ldcg(hc + kHistCoarse + fine_slot((d0 << 8) | tid)) : 0u;
      ok = pick_digit(sh, cnt1, r0, &d1, &r1, &tot1) && tot1 == __ldcg(hc + d0);
    }
    if (ok) {
      prefix = (d0 << 24) | (d1 << 16);
      mask = 0xFFFF0000u;
      remaining = r1;
      pass_begin = 2;
    }
  }
  for (int pass = pass_begin; pass < (none ? 0 : 4); ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) sh.local[tid] = 0;
    __syncthreads();
    for (int i = tid; i < n_loc; i += kTopkThreads) {
      const uint32_t key = key_at(i);
      if ((!kMasked || key != kFixedKey) && (key & mask) == prefix) atomicAdd(&sh.local[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    // this CTA's histogram into its slot of every CTA (two threads per bin,
    // each covering half of the ranks)
    if (pass == pass_begin) cluster_wait();
    {
      const uint32_t bin = static_cast<uint32_t>(tid) & 255u;
      const uint32_t v = sh.local[bin];
      const uint32_t dst = smem_u32(&sh.slot[pass & 1][rank][bin]);
      for (int r = tid >> 8; r < kTopkCluster; r += 2) st_cluster_u32(mapa_shared(dst, static_cast<uint32_t>(r)), v);
    }
    cluster.sync();
    // bin tid summed over the cluster, then this pass's digit
    uint32_t tot = 0;
    if (tid < 256) {
      for (int r = 0; r < kTopkCluster; ++r) tot += sh.slot[pass & 1][r][tid];
    }
    uint32_t digit = 0, total = 0;
    int rem = 0;
    if (!pick_digit(sh, tot, remaining, &digit, &rem, &total)) {   // cannot happen for valid input
      if (tid == 0) record_error(a.status, kStatusIndex);
      return;                 // every CTA sees the same sums, so all leave here
    }
    prefix |= digit << shift;
    mask |= 255u << shift;
    remaining = rem;
  }
  const uint32_t kth = none ? kNoneKey : prefix;   // exact K-th largest key
  const int take_eq = none ? 0 : remaining;         // keys equal to kth that are kept

  // ---- ordered compaction ---------------------------------------------
  // each warp a segment of the slice, in 32-key chunks; the counting pass
  // keeps each chunk's ballots when they fit, so that the writing pass needs
  // neither the keys nor the comparisons again
  const int seg = ((n_loc + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
  const int w0 = min(n_loc, warp * seg);
  const int w1 = min(n_loc, w0 + seg);
  const bool keep_bal = seg / 32 <= kTopkBalChunks;      // the same in every warp
  const int n_chunks = (w1 - w0 + 31) / 32;
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t gt = 0, eq = 0;
  if (keep_bal) {
    for (int c = 0; c < n_chunks; ++c) {
      const int i = w0 + c * 32 + lane;
      const uint32_t key = i < w1 ? key_at(i) : 0u;
      const uint32_t gb = __ballot_sync(0xffffffffu, i < w1 && key > kth);
      const uint32_t eb = __ballot_sync(0xffffffffu, i < w1 && key == kth);
      if (lane == 0) { sh.bal_gt[warp][c] = gb; sh.bal_eq[warp][c] = eb; }
      gt += __popc(gb);
      eq += __popc(eb);
    }
  } else {
    for (int i = w0 + lane; i < w1; i += 32) {
      const uint32_t key = key_at(i);
      gt += key > kth;
      eq += key == kth;
    }
    for (int o = 16; o > 0; o >>= 1) {
      gt += __shfl_down_sync(0xffffffffu, gt, o);
      eq += __shfl_down_sync(0xffffffffu, eq, o);
    }
  }
  if (lane == 0) { sh.warp_gt[warp] = gt; sh.warp_eq[warp] = eq; }
  __syncthreads();
  if (none) cluster_wait();   // no radix pass ran, so the first remote store is here
  if (tid < kTopkCluster) {
    // this CTA's counts into its slots of CTA `tid`
    uint32_t g = 0, e = 0;
    for (int w2 = 0; w2 < kTopkWarps; ++w2) { g += sh.warp_gt[w2]; e += sh.warp_eq[w2]; }
    st_cluster_u32(mapa_shared(smem_u32(&sh.slice_gt[rank]), static_cast<uint32_t>(tid)), g);
    st_cluster_u32(mapa_shared(smem_u32(&sh.slice_eq[rank]), static_cast<uint32_t>(tid)), e);
  }
  cluster.sync();   // the last cluster barrier: no CTA touches another's memory after it
  // every CTA read the histograms before its first push, so they can be cleared
  if (a.hist) zero_hist(a.hist, b, rank, kTopkCluster);
  // offsets of this CTA's slice (CTAs of lower rank come first)
  uint32_t gt_before = 0, eq_before = 0;
  for (int r = 0; r < rank; ++r) {
    gt_before += sh.slice_gt[r];
    eq_before += sh.slice_eq[r];
  }
  const int eq_take_cta = max(0, min(static_cast<int>(sh.slice_eq[rank]), take_eq - static_cast<int>(eq_before)));
  const long long cta_out = static_cast<long long>(gt_before) + min(static_cast<int>(eq_before), take_eq);
  uint32_t gt_w = 0, eq_w = 0;
  for (int w2 = 0; w2 < warp; ++w2) { gt_w += sh.warp_gt[w2]; eq_w += sh.warp_eq[w2]; }
  long long pos = cta_out + gt_w + min(static_cast<int>(eq_w), eq_take_cta);
  int eq_seen = static_cast<int>(eq_w);
  if (keep_bal) {
    for (int c = 0; c < n_chunks; ++c) {
      uint32_t kb = sh.bal_gt[warp][c];
      const uint32_t eb = sh.bal_eq[warp][c];
      if (eb) {           // keys equal to the K-th: the first eq_take_cta of them in row order
        const bool take = ((eb >> lane) & 1u) && eq_seen + __popc(eb & lt_mask) < eq_take_cta;
        kb |= __ballot_sync(0xffffffffu, take);
        eq_seen += __popc(eb);
      }
      if ((kb >> lane) & 1u) out[pos + __popc(kb & lt_mask)] = lo + s0 + w0 + c * 32 + lane;
      pos += __popc(kb);
    }
    return;
  }
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = (i < w1) ? key_at(i) : 0u;
    const bool is_eq = (i < w1) && key == kth;
    const uint32_t eq_bal = __ballot_sync(0xffffffffu, is_eq);
    const int my_eq_rank = eq_seen + __popc(eq_bal & lt_mask);
    const bool keep = (i < w1) && (key > kth || (is_eq && my_eq_rank < eq_take_cta));
    const uint32_t keep_bal = __ballot_sync(0xffffffffu, keep);
    if (keep) out[pos + __popc(keep_bal & lt_mask)] = lo + s0 + i;
    pos += __popc(keep_bal);
    eq_seen += __popc(eq_bal);
  }
}

// Launch with `csize` CTAs per cluster; returns the launch error.
template <bool kSmemKeys, bool kMasked>
static cudaError_t launch_topk_cluster(const TopkArgs& a, int csize, cudaStream_t st) {
  auto kernel = topk_kernel<kSmemKeys, kMasked>;
  const int chunk = (a.max_n_doc + csize - 1) / csize;
  const size_t smem = kSmemKeys ? static_cast<size_t>(max(chunk, 4)) * sizeof(uint32_t) : 0;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (csize > kTopkClusterPortable) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.batch) * csize);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // a cluster size the device cannot co-schedule is refused here, not at run time
  int n_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&n_clusters, kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (n_clusters < 1) return cudaErrorInvalidConfiguration;
  // programmatic dependent launch behind the previous kernel (the gate): the
  // kernel waits for it before touching memory
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <bool kMasked>
static cudaError_t launch_topk_masked(const TopkArgs& a, cudaStream_t st) {
  // 16-CTA clusters halve the per-CTA slice when the device allows them
  for (int csize : {kTopkClusterMax, kTopkClusterPortable}) {
    const int chunk = (a.max_n_doc + csize - 1) / csize;
    const cudaError_t e = chunk <= kTopkMaxSmemKeys ? launch_topk_cluster<true, kMasked>(a, csize, st)
                                                    : launch_topk_cluster<false, kMasked>(a, csize, st);
    if (e == cudaSuccess) return cudaSuccess;
    if (csize == kTopkClusterPortable) return e;
    (void)cudaGetLastError();   // clear the refusal of the larger cluster, try the portable size
  }
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st) {
  if (a.batch == 0) return cudaSuccess;
  return a.prunable ? launch_topk_masked<true>(a, st) : launch_topk_masked<false>(a, st);
}

// ---------------------------------------------------------------------------
// prunable rows per sequence (one block per sequence)
// ---------------------------------------------------------------------------
constexpr int kCountThreads = 1024;

__global__ void __launch_bounds__(kCountThreads)
topk_count_kernel(const uint8_t* __restrict__ prunable, const int32_t* __restrict__ cu_seqlens,
                  int32_t* __restrict__ n_prun, unsigned int* status) {
  __shared__ int part[kCountThreads / 32];
  const int b = blockIdx.x;
  const int lo = __ldg(cu_seqlens + b);
  const int hi = __ldg(cu_seqlens + b + 1);
  if (hi < lo) {
    if (threadIdx.x == 0) { record_error(status, kStatusIndex); n_prun[b] = 0; }
    return;
  }
  // the 16-byte aligned middle of the span as uint4 words, four in flight
  // per thread; the unaligned head and tail byte by byte
  const int head = static_cast<int>((16u - (reinterpret_cast<uintptr_t>(prunable + lo) & 15u)) & 15u);
  const int a0 = min(hi, lo + head);                     // first 16-byte aligned row
  const int a1 = a0 + (((hi - a0) >> 4) << 4);           // end of the whole words
  int c = 0;
  for (int i = lo + static_cast<int>(threadIdx.x); i < a0; i += kCountThreads) c += __ldg(prunable + i) != 0;
  for (int i = a1 + static_cast<int>(threadIdx.x); i < hi; i += kCountThreads) c += __ldg(prunable + i) != 0;
  const uint4* w = reinterpret_cast<const uint4*>(prunable + a0);
  const int nw = (a1 - a0) >> 4;
  auto nonzero_bytes = [](uint32_t x) {
    // per byte: 1 when nonzero (x | x >> 1 | ... folds each byte's bits into its low bit)
    x |= x >> 4;
    x |= x >> 2;
    x |= x >> 1;
    return __popc(x & 0x01010101u);
  };
  for (int j0 = static_cast<int>(threadIdx.x); j0 < nw; j0 += 4 * kCountThreads) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u * kCountThreads;
      v[u] = j < nw ? __ldg(w + j) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      c += nonzero_bytes(v[u].x) + nonzero_bytes(v[u].y) + nonzero_bytes(v[u].z) + nonzero_bytes(v[u].w);
  }
  for (int o = 16; o > 0; o >>= 1) c += __shfl_down_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x < 32) {
    int t = part[threadIdx.x];
    for (int o = 16; o > 0; o >>= 1) t += __shfl_down_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) n_prun[b] = t;
  }
}

cudaError_t launch_topk_count(const uint8_t* prunable, const int32_t* cu_seqlens, int32_t batch,
                              int32_t* n_prun, unsigned int* status, cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  topk_count_kernel<<<static_cast<unsigned>(batch), kCountThreads, 0, st>>>(prunable, cu_seqlens, n_prun, status);
  return cudaGetLastError();
}

}  // namespace tg
